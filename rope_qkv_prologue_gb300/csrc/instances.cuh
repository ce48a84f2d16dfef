// Kernel instance pickers: the template arguments of each kernel family for
// a run-time variant. Every instance file includes this header and
// instantiates one slice (head_dim x norm on/off), so the slices compile in
// parallel.
#pragma once

#include "gqa_stream.cuh"

namespace qkvp {
namespace inst {

// Forward, pipelined (STREAM) or general, for one head_dim and norm setting.
template <int HD, bool NORM, bool STREAM>
struct FwdPick {
  template <bool S, bool R, bool SV, bool P, bool B>
  static const void* get() {
    if constexpr (STREAM) {
      constexpr StreamShape sh = fwd_stream_shape(SV);
      return reinterpret_cast<const void*>(
          &qkvp_fwd_stream_kernel<HD, S, R, SV, P, NORM, B, sh.warps, sh.ctas_per_sm>);
    } else {
      return reinterpret_cast<const void*>(&qkvp_fwd_kernel<HD, S, R, SV, P, NORM, B>);
    }
  }
  template <bool S, bool R, bool B>
  static const void* dest(const FwdVariant& v) {
    if (v.pool) return get<S, R, false, true, B>();
    return v.save_pre ? get<S, R, true, false, B>() : get<S, R, false, false, B>();
  }
  template <bool S, bool R>
  static const void* bias(const FwdVariant& v) {
    return v.bias ? dest<S, R, true>(v) : dest<S, R, false>(v);
  }
  static const void* pick(const FwdVariant& v) {
    if (v.sectioned) return v.rope ? bias<true, true>(v) : bias<true, false>(v);
    return v.rope ? bias<false, true>(v) : bias<false, false>(v);
  }
};

// Backward, pipelined or general, for one norm setting (both head_dims).
template <bool NORM, bool STREAM>
struct BwdPick {
  template <int HD, bool S, bool R, bool B>
  static const void* get() {
    if constexpr (STREAM) {
      constexpr StreamShape sh = bwd_stream_shape();
      return reinterpret_cast<const void*>(&qkvp_bwd_stream_kernel<HD, S, R, NORM, B, sh.warps, sh.ctas_per_sm, 0>);
    } else {
      return reinterpret_cast<const void*>(&qkvp_bwd_kernel<HD, S, R, NORM, B>);
    }
  }
  template <int HD, bool S, bool R>
  static const void* bias(const BwdVariant& v) {
    return v.bias ? get<HD, S, R, true>() : get<HD, S, R, false>();
  }
  template <int HD>
  static const void* layout(const BwdVariant& v) {
    if (v.sectioned) return v.rope ? bias<HD, true, true>(v) : bias<HD, true, false>(v);
    return v.rope ? bias<HD, false, true>(v) : bias<HD, false, false>(v);
  }
  static const void* pick(const BwdVariant& v) {
    if constexpr (STREAM && NORM) {
      // two chunk pairs per thread (head_dim 64 rows of up to 640 chunk pairs):
      // the weight-gradient sums are kept per step
      constexpr StreamShape sh = bwd_stream_shape();
      if (v.steps == 2 && v.head_dim == 64 && !v.bias) {
        if (v.sectioned)
          return v.rope ? reinterpret_cast<const void*>(&qkvp_bwd_stream_kernel<64, true, true, true, false, sh.warps, sh.ctas_per_sm, 2>)
                        : reinterpret_cast<const void*>(&qkvp_bwd_stream_kernel<64, true, false, true, false, sh.warps, sh.ctas_per_sm, 2>);
        return v.rope ? reinterpret_cast<const void*>(&qkvp_bwd_stream_kernel<64, false, true, true, false, sh.warps, sh.ctas_per_sm, 2>)
                      : reinterpret_cast<const void*>(&qkvp_bwd_stream_kernel<64, false, false, true, false, sh.warps, sh.ctas_per_sm, 2>);
      }
    }
    return v.head_dim == 64 ? layout<64>(v) : layout<128>(v);
  }
};

}  // namespace inst
}  // namespace qkvp
