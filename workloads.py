"""Seeded synthetic inputs for the packed-QKV prologue.

This module only draws and lays out random inputs; it holds none of the
prologue's arithmetic (no norm, no rotation, no rounding of results). Both the
CUDA path's tests / benchmark and the fp64 oracle consume what it returns, so
the two sides always see the same bits.

Every draw uses ``torch.Generator('cpu').manual_seed(seed)`` and float32
samples rounded to bf16. Norm weights are drawn U(0.5, 1.5), rounded to
bf16-representable values and kept as float32 (so the float32 weights the
kernels take and a bf16 reading of them are the same numbers).

The five workloads mirror the shapes the pages measure: the Muse Spark packed
projection [T, 16 kv heads, 10, 64] of "[muse_spark][perf] Split the packed
qkv inside the q/k region" (Problem 1), and the 576-wide MLA kv latent rows
(512 normed + 64 roped) written into a 64-token-page pool in "MLA DSpark: run
each drafter layer's kv path beside its q path". No dataset is involved.
"""

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

EPS = 1e-6


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, g):
    """N(0, 1) float32 draws rounded to bf16."""
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def norm_weight(n, g):
    """U(0.5, 1.5) draws rounded to bf16-representable values, kept as float32."""
    u = torch.rand(n, generator=g, dtype=torch.float32) + 0.5
    return u.to(torch.bfloat16).to(torch.float32)


def random_slots(T, num_pages, page_size, g):
    """Distinct (page, offset) pairs for T tokens: a seeded random permutation
    of all pool slots, first T taken; no two tokens share a slot."""
    if T > num_pages * page_size:
        raise ValueError("more tokens than pool slots")
    slot = torch.randperm(num_pages * page_size, generator=g)[:T]
    return (slot // page_size).to(torch.int32), (slot % page_size).to(torch.int32)


def sectioned_from_interleaved(packed, n_q, n_kv, head_dim):
    """Re-lay interleaved rows [T, n_kv, G+2, D] as sectioned rows
    [T, (n_q + 2 n_kv) * D] holding the same heads: q heads 0..n_q-1 (head
    g*G + j is slot j of group g), then k heads (slot G), then v heads
    (slot G+1)."""
    G = n_q // n_kv
    x = packed.reshape(packed.shape[0], n_kv, G + 2, head_dim)
    q = x[:, :, :G, :].reshape(x.shape[0], n_q, head_dim)
    k = x[:, :, G, :]
    v = x[:, :, G + 1, :]
    return torch.cat([q, k, v], dim=1).reshape(x.shape[0], -1).contiguous()


@dataclass
class GQAWorkload:
    """Inputs of one GQA prologue call (all CPU tensors)."""

    name: str
    n_q: int
    n_kv: int
    head_dim: int
    packed: torch.Tensor          # bf16 [T, n_kv, G+2, D] (interleaved)
    pos: torch.Tensor             # int32 [T]
    w_q: torch.Tensor             # float32 [D]
    w_k: torch.Tensor             # float32 [D]
    rope_base: float
    nope: bool = False
    eps: float = EPS
    # training
    dq: Optional[torch.Tensor] = None   # bf16 [T, n_q, D]
    dk: Optional[torch.Tensor] = None   # bf16 [T, n_kv, D]
    dv: Optional[torch.Tensor] = None   # bf16 [T, n_kv, D]
    # paged pool destination
    page: Optional[torch.Tensor] = None    # int32 [T]
    offset: Optional[torch.Tensor] = None  # int32 [T]
    num_pages: int = 0
    page_size: int = 0
    # the GQAttention variant options (Llama 3, Qwen3, GPT-OSS)
    norm: bool = True
    bias: Optional[torch.Tensor] = None   # float32 [row_width], interleaved packed order
    inv_freq: Optional[np.ndarray] = None  # float64 [head_dim / 2], or None: base**(-2i/D)
    rope_scale: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def T(self):
        return self.packed.shape[0]

    @property
    def row_width(self):
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    def packed_rows(self):
        """Interleaved packed input as [T, row_width]."""
        return self.packed.reshape(self.T, self.row_width)

    def sectioned_rows(self):
        return sectioned_from_interleaved(self.packed, self.n_q, self.n_kv, self.head_dim)

    def bias_for(self, kind):
        """The bias in the packed order of `kind` (None without a bias)."""
        if self.bias is None:
            return None
        if kind == "interleaved":
            return self.bias
        G = self.n_q // self.n_kv
        b = self.bias.reshape(1, self.n_kv, G + 2, self.head_dim)
        return sectioned_from_interleaved(b, self.n_q, self.n_kv, self.head_dim).reshape(-1).contiguous()

    def variant(self, kind="interleaved"):
        """Keyword options of the GQAttention variant (for oracle and library calls)."""
        return dict(norm=self.norm, bias=self.bias_for(kind), inv_freq=self.inv_freq, rope_scale=self.rope_scale)


@dataclass
class MLAWorkload:
    name: str
    rows: torch.Tensor            # bf16 [T, norm_dim + rope_dim]
    pos: torch.Tensor             # int32 [T]
    w: torch.Tensor               # float32 [norm_dim]
    page: torch.Tensor
    offset: torch.Tensor
    num_pages: int
    page_size: int
    rope_base: float = 10000.0
    norm_dim: int = 512
    rope_dim: int = 64
    eps: float = EPS

    @property
    def T(self):
        return self.rows.shape[0]


def gqa_inputs(T, n_q, n_kv, head_dim, seed, rope_base, nope=False, pos_high=None,
               name="gqa", with_grads=False):
    """Packed [T, n_kv, G+2, D] N(0,1) bf16, norm weights, positions.

    Positions are 0..T-1 when pos_high is None, else uniform in [0, pos_high).
    With with_grads, upstream gradients dq, dk, dv are N(0,1) bf16.
    """
    g = _gen(seed)
    G = n_q // n_kv
    packed = normal_bf16((T, n_kv, G + 2, head_dim), g)
    w_q = norm_weight(head_dim, g)
    w_k = norm_weight(head_dim, g)
    if pos_high is None:
        pos = torch.arange(T, dtype=torch.int32)
    else:
        pos = torch.randint(0, pos_high, (T,), generator=g, dtype=torch.int32)
    wl = GQAWorkload(name, n_q, n_kv, head_dim, packed, pos, w_q, w_k, float(rope_base), nope)
    if with_grads:
        wl.dq = normal_bf16((T, n_q, head_dim), g)
        wl.dk = normal_bf16((T, n_kv, head_dim), g)
        wl.dv = normal_bf16((T, n_kv, head_dim), g)
    return wl


# --- the GQAttention variant (Llama 3, Qwen3, GPT-OSS) -------------------------
#
# Frequency tables and the bias are inputs of the library call (the library
# never computes them); these build them the way those models do.

def llama3_inv_freq(head_dim, base=500000.0, factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0,
                    original_max_position=8192):
    """Llama 3.1-style frequency table: a frequency whose wavelength is shorter
    than original_max_position / high_freq_factor keeps its value, one longer
    than original_max_position / low_freq_factor is divided by factor, and the
    ones between blend the two linearly in original_max_position / wavelength."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    f = base ** (-2.0 * i / head_dim)
    wavelen = 2.0 * np.pi / f
    smooth = (original_max_position / wavelen - low_freq_factor) / (high_freq_factor - low_freq_factor)
    mid = (1.0 - smooth) * f / factor + smooth * f
    out = np.where(wavelen > original_max_position / low_freq_factor, f / factor, mid)
    return np.where(wavelen < original_max_position / high_freq_factor, f, out)


def yarn_inv_freq(head_dim, base, factor, original_max_position, beta_fast=32.0, beta_slow=1.0):
    """YaRN-style frequency table: frequencies that turn more than beta_fast
    times over the original context keep their value, those turning fewer than
    beta_slow times are divided by factor, with a linear ramp over the
    dimensions between."""
    def dim_of(turns):
        return head_dim * math.log(original_max_position / (turns * 2.0 * math.pi)) / (2.0 * math.log(base))

    lo = max(math.floor(dim_of(beta_fast)), 0)
    hi = min(math.ceil(dim_of(beta_slow)), head_dim - 1)
    i = np.arange(head_dim // 2, dtype=np.float64)
    keep = base ** (-2.0 * i / head_dim)
    ramp = np.clip((i - lo) / max(hi - lo, 1e-3), 0.0, 1.0)  # 0: keep, 1: divide by factor
    return keep * (1.0 - ramp) + keep / factor * ramp


def yarn_attention_factor(factor):
    """YaRN's factor on cos and sin: 0.1 ln(factor) + 1."""
    return 0.1 * math.log(factor) + 1.0


def qkv_bias(row_width, g):
    """A fused linear's qkv bias: float32 N(0, 0.5^2) [row_width]."""
    return (torch.randn(row_width, generator=g, dtype=torch.float32) * 0.5).contiguous()


def llama3(T, seed=6, pos_high=None, with_grads=True):
    """Llama 3 8B attention: 32 q heads over 8 kv heads, head_dim 128, no q/k
    norm, RoPE base 5e5 with the Llama 3.1 frequency scaling."""
    wl = gqa_inputs(T, 32, 8, 128, seed, 500000.0, pos_high=pos_high, name=f"llama3_T{T}", with_grads=with_grads)
    wl.norm = False
    wl.inv_freq = llama3_inv_freq(128)
    return wl


def qwen3(T, seed=7, pos_high=None, with_grads=True):
    """Qwen3 8B attention: 32 q heads over 8 kv heads, head_dim 128, per-head
    q/k RMSNorm, RoPE base 1e6."""
    return gqa_inputs(T, 32, 8, 128, seed, 1000000.0, pos_high=pos_high, name=f"qwen3_T{T}",
                      with_grads=with_grads)


def gpt_oss(T, seed=8, pos_high=None, with_grads=True):
    """GPT-OSS 20b attention: 64 q heads over 8 kv heads, head_dim 64, no q/k
    norm, a qkv bias, RoPE base 150000 with a YaRN-style table (factor 32,
    original context 4096) and its cos/sin factor."""
    wl = gqa_inputs(T, 64, 8, 64, seed, 150000.0, pos_high=pos_high, name=f"gpt_oss_T{T}", with_grads=with_grads)
    wl.norm = False
    wl.bias = qkv_bias(wl.row_width, _gen(seed * 1000 + 11))
    wl.inv_freq = yarn_inv_freq(64, 150000.0, 32.0, 4096)
    wl.rope_scale = yarn_attention_factor(32.0)
    return wl


# --- the projection to the left of the path -------------------------------------

def gemm_inputs(T, hidden, n_q, n_kv, head_dim, seed, exact=True):
    """x [T, hidden] and the fused weight W [(n_q + 2 n_kv) * head_dim, hidden],
    bf16. exact: x = k / 8 (|k| <= 16) and W = k / 64 (|k| <= 32), so every
    product and every partial sum of up to 4096 terms is exact in float32 and a
    GEMM gives the exact product whatever its summation order; else x N(0,1)
    and W N(0, 1/hidden) (the scale of a trained projection)."""
    g = _gen(seed)
    rows = (n_q + 2 * n_kv) * head_dim
    if exact:
        x = torch.clamp(torch.round(torch.randn(T, hidden, generator=g) * 4), -16, 16) / 8
        w = torch.clamp(torch.round(torch.randn(rows, hidden, generator=g) * 8), -32, 32) / 64
    else:
        x = torch.randn(T, hidden, generator=g)
        w = torch.randn(rows, hidden, generator=g) / math.sqrt(hidden)
    return x.to(torch.bfloat16), w.to(torch.bfloat16)


def fused_qkv_update(n_q, n_kv, head_dim, cols, seed, scale=1.0):
    """A fused QKV weight's update (a gradient or a momentum)
    [(n_q + 2 n_kv) * head_dim, cols] bf16, N(0, scale^2), rows in the
    interleaved-per-KV-group order. The whole tensor is one draw, so every
    head block looks like any other."""
    g = _gen(seed)
    rows = (n_q + 2 * n_kv) * head_dim
    return (torch.randn(rows, cols, generator=g) * scale).to(torch.bfloat16)


def sectioned_weight_from_interleaved(w, n_q, n_kv, head_dim):
    """The same fused weight with its dim-0 head blocks in sectioned order
    (q heads, then k heads, then v heads): a row permutation of w."""
    return sectioned_from_interleaved(w.t().contiguous(), n_q, n_kv, head_dim).t().contiguous()


# Fused QKV weights the per-head Newton-Schulz path runs on:
#  - the page's model ("[muon] Per-head Newton-Schulz for fused QKV
#    projections", End-to-end training): a LLaMA-shaped model, 6 layers,
#    hidden 512, 8 query heads over 2 KV heads of 64, so a [768, 512] fused
#    weight per layer;
#  - the Muse Spark packing of the prologue ([T, 16 kv heads, 10, 64]): a
#    [10240, hidden] fused weight; hidden 5120 stands in for the model's
#    (the pages give none).
NS_PAGE_MODEL = dict(n_q=8, n_kv=2, head_dim=64, cols=512, layers=6)
NS_MUSE_SPARK = dict(n_q=128, n_kv=16, head_dim=64, cols=5120, layers=1)


# --- the five workloads ------------------------------------------------------

def tiny(seed=1):
    """T=16, [16, 2 kv, 4 q + 1 k + 1 v, 64], base 10000, positions 0..15."""
    return gqa_inputs(16, 8, 2, 64, seed, 10000.0, name="tiny_fwd_T16")


def decode_pool(T, seed=2, num_pages=4096, page_size=64):
    """Decode with a paged pool: [T,16,10,64], positions U[0,131072), base 5e5,
    4096 pages x 64 tokens x 16 heads x 64, distinct random slots."""
    wl = gqa_inputs(T, 128, 16, 64, seed, 500000.0, pos_high=131072, name=f"decode_pool_T{T}")
    g = _gen(seed * 1000 + 7)
    wl.page, wl.offset = random_slots(T, num_pages, page_size, g)
    wl.num_pages, wl.page_size = num_pages, page_size
    return wl


def prefill(T, seed=3, nope=False):
    """Prefill: [T,16,10,64], positions 0..T-1, base 5e5 (or NoPE)."""
    return gqa_inputs(T, 128, 16, 64, seed, 500000.0, nope=nope,
                      name=f"prefill_T{T}" + ("_nope" if nope else ""))


def train(T, seed=4):
    """Training fwd+bwd: [T,16,10,64], positions 0..T-1, base 5e5, N(0,1) grads."""
    return gqa_inputs(T, 128, 16, 64, seed, 500000.0, name=f"train_T{T}", with_grads=True)


def mla(T, seed=5, num_pages=8192, page_size=64):
    """MLA latent rows [T, 576] N(0,1), positions U[0,393216), base 1e4,
    pool of 8192 pages x 64 tokens x 576, distinct random slots."""
    g = _gen(seed)
    rows = normal_bf16((T, 576), g)
    w = norm_weight(512, g)
    pos = torch.randint(0, 393216, (T,), generator=g, dtype=torch.int32)
    page, offset = random_slots(T, num_pages, page_size, _gen(seed * 1000 + 7))
    return MLAWorkload(f"mla_T{T}", rows, pos, w, page, offset, num_pages, page_size)


def random_pool_bits(shape, seed, device="cpu"):
    """A pool pre-filled with random bits (int16 view of bf16 storage)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    bits = torch.randint(-32768, 32768, tuple(shape), generator=g, dtype=torch.int16, device=device)
    return bits.view(torch.bfloat16)


def bits_u16(t):
    """The raw bits of a bf16 tensor as a NumPy uint16 array (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
