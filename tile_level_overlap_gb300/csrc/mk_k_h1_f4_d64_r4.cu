// Interpreter specialisation: MH=1, MF=4, head_dim=64, q heads per kv head=4
// (0 = chosen at run time).
#include "mk_kernel.cuh"

namespace mk {
KernelVariant variant_h1_f4_d64_r4() { return make_variant<1, 4, 64, 4>(); }
}  // namespace mk
