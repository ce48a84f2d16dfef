// Pipelined forward kernel instances: head_dim 64, without the norm (split -> RoPE).
#include "instances.cuh"

namespace qkvp {
const void* fwd_stream_kernel_d64_nonorm(const FwdVariant& v) { return inst::FwdPick<64, false, true>::pick(v); }
}  // namespace qkvp
