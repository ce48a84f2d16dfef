// General forward kernel instances: head_dim 64, without the norm (split -> RoPE).
#include "instances.cuh"

namespace qkvp {
const void* fwd_kernel_d64_nonorm(const FwdVariant& v) { return inst::FwdPick<64, false, false>::pick(v); }
}  // namespace qkvp
