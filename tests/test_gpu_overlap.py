"""The MLA drafter-layer schedule ("MLA DSpark: run each drafter layer's kv path
beside its q path", Description): the kv path (kv_a projection -> latent
norm/RoPE -> direct pool write) forked to a side stream with
functional.mla_kv_path_beside, the q path on the current stream, joined before
a reader of the pool. Captured in a CUDA graph and replayed, then checked

  * against the fp64 oracle: the rows written into the pool are
    oracle.mla_pool_write of the kv rows the graph produced (prologue
    tolerance), and every other pool byte is the pool's initial bits;
  * for ordering: a gather of the written slots queued on the current stream
    after the join reads exactly the rows the side stream wrote;
  * against the same work on one stream: identical bits everywhere.
"""

import numpy as np
import pytest
import torch

import oracle.prologue as P
import workloads
from parity import assert_bf16_close
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu


def _layer(T, dev, hidden=1024, q_rank=384):
    g = torch.Generator(device="cpu")
    g.manual_seed(4321 + T)
    bf = dict(dtype=torch.bfloat16, device=dev)
    h = torch.randn(T, hidden, generator=g).to(**bf)
    wkva = (torch.randn(hidden, 576, generator=g) / hidden ** 0.5).to(**bf)
    wqa = (torch.randn(hidden, q_rank, generator=g) / hidden ** 0.5).to(**bf)
    wqb = (torch.randn(q_rank, 16 * 192, generator=g) / q_rank ** 0.5).to(**bf)
    return h, wkva, wqa, wqb


@pytest.mark.parametrize("T", [16, 64])
def test_kv_path_beside_q_path_in_a_graph_matches_oracle(lib, cuda, T):
    F = lib.functional
    wl = workloads.mla(T, num_pages=512)
    h, wkva, wqa, wqb = _layer(T, cuda)
    pos, w, page, off = wl.pos.to(cuda), wl.w.to(cuda), wl.page.to(cuda), wl.offset.to(cuda)
    slots = (page.long() * wl.page_size + off.long())
    init = workloads.random_pool_bits((wl.num_pages, wl.page_size, 576), 99, cuda)
    pools = {m: init.clone() for m in ("two", "one")}
    side = torch.cuda.Stream(cuda)

    def q_path():
        qa = torch.nn.functional.rms_norm(h @ wqa, (wqa.shape[1],), None, 1e-6)
        return qa @ wqb

    def step(mode):
        pool = pools[mode]
        if mode == "two":
            rows, done = F.mla_kv_path_beside(side, pos, w, page, off, pool, kv_proj=lambda: h @ wkva,
                                              eps=wl.eps, rope_base=wl.rope_base)
            q = q_path()
            F.join(done)
        else:
            rows = h @ wkva
            F.latent_pool_write(rows, pos, w, page, off, pool, wl.eps, wl.rope_base)
            q = q_path()
        read = pool.view(-1, 576)[slots]  # a reader of the pool, after the join
        return rows, q, read

    graphs, outs = {}, {}
    cap = torch.cuda.Stream(cuda)
    cap.wait_stream(torch.cuda.current_stream(cuda))
    with torch.cuda.stream(cap):
        for mode in ("two", "one"):
            step(mode)  # warm-up outside the graph (cuBLAS handles, workspaces)
            torch.cuda.synchronize()
            pools[mode].copy_(init)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=cap):
                outs[mode] = step(mode)
            graphs[mode] = gr
    torch.cuda.synchronize()
    for mode in ("two", "one"):
        pools[mode].copy_(init)
        graphs[mode].replay()
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=False) == 0

    rows, q, read = outs["two"]
    exact, want_pool = P.mla_pool_write(u16(rows), wl.pos.numpy(), wl.w.numpy(), wl.eps, wl.rope_base,
                                        wl.page.numpy(), wl.offset.numpy(), u16(init))
    got_pool = u16(pools["two"]).reshape(-1, 576)
    s = slots.cpu().numpy()
    assert_bf16_close(got_pool[s], exact, "pool rows written on the side stream")
    untouched = np.ones(got_pool.shape[0], dtype=bool)
    untouched[s] = False
    assert np.array_equal(got_pool[untouched], u16(init).reshape(-1, 576)[untouched]), "untouched pool bytes"
    assert np.array_equal(u16(read), got_pool[s]), "the reader after the join sees the written rows"
    # the one-stream schedule gives the same bits
    for a, b in zip(outs["two"], outs["one"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(pools["two"].view(torch.int16), pools["one"].view(torch.int16))


def test_kv_path_beside_needs_one_source(lib, cuda):
    F = lib.functional
    with pytest.raises(ValueError):
        F.mla_kv_path_beside(torch.cuda.Stream(cuda), None, None, None, None, None)


def test_on_side_stream_orders_work(lib, cuda):
    # the side stream sees what the current stream queued before the fork, and the
    # join makes its result visible after
    F = lib.functional
    side = torch.cuda.Stream(cuda)
    x = torch.zeros(1 << 20, device=cuda)
    x.fill_(3.0)  # queued on the current stream
    y, done = F.on_side_stream(side, lambda t: t * 2.0, x)
    F.join(done)
    assert torch.all(y == 6.0)
