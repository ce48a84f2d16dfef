// Pipelined forward kernel instances: head_dim 128, without the norm (split -> RoPE).
#include "instances.cuh"

namespace qkvp {
const void* fwd_stream_kernel_d128_nonorm(const FwdVariant& v) { return inst::FwdPick<128, false, true>::pick(v); }
}  // namespace qkvp
