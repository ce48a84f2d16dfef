"""The MLA drafter-layer scheduling: the kv path (projection -> latent norm/RoPE
-> direct pool write) on a side stream beside the q path, under CUDA graph
capture, gives exactly the results of running both on one stream."""

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [16, 64])
def test_side_stream_kv_path_equals_one_stream(lib, cuda, T):
    import bench

    r = bench.mla_two_stream_overlap(cuda, T, layers=2, reps=3)
    assert r["same_results"], r
    assert r["serial_us_per_step"] > 0 and r["two_stream_us_per_step"] > 0


def test_on_side_stream_orders_work(lib, cuda):
    # the side stream sees what the current stream queued before the fork, and the
    # join makes its result visible after
    F = lib.functional
    side = torch.cuda.Stream(cuda)
    x = torch.zeros(1 << 20, device=cuda)
    x.fill_(3.0)  # queued on the current stream
    y, done = F.on_side_stream(side, lambda t: t * 2.0, x)
    torch.cuda.current_stream().wait_event(done)
    assert torch.all(y == 6.0)
