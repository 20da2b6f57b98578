// Interpreter specialisation: MH=0, MF=0, head_dim=0, q heads per kv head=0
// (0 = chosen at run time).
#include "mk_kernel.cuh"

namespace mk {
KernelVariant variant_generic() { return make_variant<0, 0, 0, 0>(); }
}  // namespace mk
