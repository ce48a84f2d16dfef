// General forward kernel instances: head_dim 128, with the q/k RMSNorm.
#include "instances.cuh"

namespace qkvp {
const void* fwd_kernel_d128_norm(const FwdVariant& v) { return inst::FwdPick<128, true, false>::pick(v); }
}  // namespace qkvp
