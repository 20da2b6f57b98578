// Interpreter specialisation: MH=2, MF=6, head_dim=128, q heads per kv head=4
// (0 = chosen at run time).
#include "mk_kernel.cuh"

namespace mk {
KernelVariant variant_h2_f6_d128_r4() { return make_variant<2, 6, 128, 4>(); }
}  // namespace mk
