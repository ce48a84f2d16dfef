// Pipelined forward kernel instances: head_dim 64, with the q/k RMSNorm.
#include "instances.cuh"

namespace qkvp {
const void* fwd_stream_kernel_d64_norm(const FwdVariant& v) { return inst::FwdPick<64, true, true>::pick(v); }
}  // namespace qkvp
