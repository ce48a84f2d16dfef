// Forward kernel instances for head_dim 128 (contiguous and pool destinations).
#include "gqa_kernels.cuh"

namespace qkvp {

namespace {
template <bool S, bool R, bool SV, bool P>
const void* fwd_ptr() {
  return reinterpret_cast<const void*>(&qkvp_fwd_kernel<128, S, R, SV, P>);
}
template <bool S, bool R>
const void* fwd_pick(const FwdVariant& v) {
  if (v.pool) return fwd_ptr<S, R, false, true>();
  return v.save_pre ? fwd_ptr<S, R, true, false>() : fwd_ptr<S, R, false, false>();
}
}  // namespace

const void* fwd_kernel_d128(const FwdVariant& v) {
  if (v.sectioned) return v.rope ? fwd_pick<true, true>(v) : fwd_pick<true, false>(v);
  return v.rope ? fwd_pick<false, true>(v) : fwd_pick<false, false>(v);
}

}  // namespace qkvp
