"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""

import numpy as np
import pytest

import oracle.bf16 as B
import oracle.prologue as P
import oracle_checks as C
import workloads


def test_bf16_rounding_is_exact_nearest_even(rng):
    C.check_to_bf16_rne(B, rng)


def test_bf16_widening_all_patterns():
    C.check_bf16_widen(B)


def test_bf16_rounding_matches_torch_on_float32_inputs(rng):
    # float32 -> bf16 is a single rounding in torch, so it must agree on values
    # that are exactly float32.
    import torch

    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(B.to_bf16_rne(x.astype(np.float64)), want)


@pytest.mark.parametrize("name", ["head_blocks_8q_over_2kv.txt", "head_blocks_muse_spark_16kv.txt"])
def test_head_block_order_matches_pages(name):
    C.check_head_block_fixture(P, name)


@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
@pytest.mark.parametrize("shape", [(8, 2, 64), (128, 16, 64), (32, 8, 128), (4, 4, 8)])
def test_split_is_pure_permutation(kind, shape):
    C.check_split_is_permutation(P, P.PackedLayout(kind, *shape))


def test_fused_total_and_block_count():
    # the row holds exactly (n_q + 2 n_kv) * head_dim values: 12 blocks for 8 q over 2 kv
    L = P.PackedLayout("interleaved", 8, 2, 64)
    assert L.n_blocks == 12 and L.row_width == 768
    assert P.PackedLayout("sectioned", 128, 16, 64).row_width == 160 * 64
    with pytest.raises(ValueError):
        P.PackedLayout("interleaved", 8, 3, 64)


def test_merge_inverts_split(rng):
    for kind in ("interleaved", "sectioned"):
        L = P.PackedLayout(kind, 8, 2, 64)
        x = rng.standard_normal((4, L.row_width))
        assert np.array_equal(P.merge_heads(L, *P.split_heads(L, x)), x)


def test_tiny_layouts_give_identical_outputs():
    C.check_layout_equivalence(P, B, workloads.tiny())


def test_layouts_identical_muse_spark_shape():
    C.check_layout_equivalence(P, B, workloads.decode_pool(8))


def test_rms_norm_closed_forms(rng):
    C.check_rms_norm(P, rng)


def test_rope_closed_forms(rng):
    C.check_rope(P, rng)


@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
def test_nope_equals_rope_at_position_zero(kind, rng):
    C.check_nope_is_rope_at_zero(P, P.PackedLayout(kind, 8, 2, 64), rng)


def test_fwd_copies_are_bitwise(rng):
    L = P.PackedLayout("interleaved", 8, 2, 64)
    bits = B.to_bf16_rne(rng.standard_normal((6, L.row_width)))
    out = P.prologue_fwd(L, bits, np.arange(6), np.ones(64), np.ones(64), 1e-6, 1e4)
    x = bits.reshape(6, 12, 64)
    assert np.array_equal(out["v_bits"], x[:, [5, 11]])
    assert np.array_equal(out["k_pre_bits"], x[:, [4, 10]])
    assert np.array_equal(out["q_pre_bits"], x[:, [0, 1, 2, 3, 6, 7, 8, 9]])


@pytest.mark.parametrize("nope", [False, True])
@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
def test_backward_finite_differences_small(kind, nope, rng):
    C.check_finite_differences(P, P.PackedLayout(kind, 2, 1, 8), rng, T=3, nope=nope)


@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
def test_backward_finite_differences_head_dim_64(kind, rng):
    C.check_finite_differences(P, P.PackedLayout(kind, 4, 2, 64), rng, T=2, n_probe=120, base=5e5)


@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
def test_backward_invariants(kind, rng):
    C.check_backward_invariants(P, P.PackedLayout(kind, 8, 2, 64), rng)


def test_backward_layouts_agree(rng):
    T, D = 4, 64
    Li, Ls = P.PackedLayout("interleaved", 8, 2, D), P.PackedLayout("sectioned", 8, 2, D)
    xq, xk = rng.standard_normal((T, 8, D)), rng.standard_normal((T, 2, D))
    dq, dk, dv = rng.standard_normal((T, 8, D)), rng.standard_normal((T, 2, D)), rng.standard_normal((T, 2, D))
    w = rng.uniform(0.5, 1.5, D)
    a = P.prologue_bwd_f64(Li, dq, dk, dv, xq, xk, np.arange(T), w, w, 1e-6, 5e5)
    b = P.prologue_bwd_f64(Ls, dq, dk, dv, xq, xk, np.arange(T), w, w, 1e-6, 5e5)
    for u, v in zip(P.split_heads(Li, a["dpacked"]), P.split_heads(Ls, b["dpacked"])):
        assert np.array_equal(u, v)
    assert np.array_equal(a["dw_q"], b["dw_q"]) and np.array_equal(a["dw_k"], b["dw_k"])


def test_pool_write_placement(rng):
    C.check_pool_placement(P, B, rng)


def test_mla_rows(rng):
    C.check_mla_rows(P, rng)


def test_workload_repack_matches_layout_definition():
    # the input generator's sectioned repack is the page's sectioned order
    wl = workloads.tiny()
    L = P.PackedLayout("interleaved", 8, 2, 64)
    Ls = P.PackedLayout("sectioned", 8, 2, 64)
    xi = workloads.bits_u16(wl.packed_rows())
    xs = workloads.bits_u16(wl.sectioned_rows())
    for u, v in zip(P.split_heads(L, xi), P.split_heads(Ls, xs)):
        assert np.array_equal(u, v)


def test_variant_forward_options(rng):
    C.check_variant_forward(P, rng)


def test_rope_frequency_table_and_factor(rng):
    C.check_rope_extras(P, rng)


def test_variant_backward_finite_differences(rng):
    C.check_variant_backward(P, rng)


# ---------------------------------------------- per-head Newton-Schulz ----

import oracle.newton_schulz as N  # noqa: E402


def test_ns_known_svd_closed_forms(rng):
    C.check_ns_svd_closed_form(N, rng)


def test_ns_orthogonal_equivariance(rng):
    C.check_ns_equivariance(N, rng)


def test_ns_blocks_independent_and_scaled(rng):
    C.check_ns_per_head(N, rng)


def test_ns_sectioned_equals_interleaved(rng):
    C.check_ns_layout_equivalence(N, P, rng)


def test_ns_page_split_cases_and_scales():
    C.check_ns_page_facts(N)


def test_ns_constants_are_muons_published_defaults():
    assert N.NS_COEFFS == (3.4445, -4.7750, 2.0315) and N.NS_STEPS == 5 and N.NS_EPS == 1e-7


def test_ns_bits_entry_checks_the_fused_total(rng):
    L = P.PackedLayout("interleaved", 8, 2, 16)
    m = B.to_bf16_rne(rng.standard_normal((12 * 16, 32)))
    out = N.qkv_newton_schulz(L, m)
    assert out.shape == (192, 32)
    assert np.array_equal(out, N.per_head_newton_schulz(B.bf16_bits_to_f64(m), 16))
    with pytest.raises(ValueError):
        N.qkv_newton_schulz(L, m[:-16])


def test_ns_dispatch_per_head_or_whole(rng):
    C.check_ns_dispatch(N, rng)


def test_projection_exact_sums_one_rounding_and_hand_over(rng):
    # x . W^T against exact rational sums (square and non-square W), one
    # rounding past a bf16 tie, and W = identity / permutation into the prologue
    C.check_projection(P, rng)
