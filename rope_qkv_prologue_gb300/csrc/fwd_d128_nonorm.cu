// General forward kernel instances: head_dim 128, without the norm (split -> RoPE).
#include "instances.cuh"

namespace qkvp {
const void* fwd_kernel_d128_nonorm(const FwdVariant& v) { return inst::FwdPick<128, false, false>::pick(v); }
}  // namespace qkvp
