// Pipelined forward kernel instances: head_dim 128, with the q/k RMSNorm.
#include "instances.cuh"

namespace qkvp {
const void* fwd_stream_kernel_d128_norm(const FwdVariant& v) { return inst::FwdPick<128, true, true>::pick(v); }
}  // namespace qkvp
