// General forward kernel instances: head_dim 64, with the q/k RMSNorm.
#include "instances.cuh"

namespace qkvp {
const void* fwd_kernel_d64_norm(const FwdVariant& v) { return inst::FwdPick<64, true, false>::pick(v); }
}  // namespace qkvp
