// General backward kernel instances without the norm (g = R^T d only).
#include "instances.cuh"

namespace qkvp {
const void* bwd_kernel_nonorm(const BwdVariant& v) { return inst::BwdPick<false, false>::pick(v); }
}  // namespace qkvp
