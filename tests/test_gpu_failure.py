"""Failure detection on the GPU without a fault: a bounded wait gives up, records
SITU_ERR_TIMEOUT in the device status, and the context stays usable."""
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(cuda_dev):
    situ.selftest_bounded_wait(limit_us=2000)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 5  # SITU_ERR_TIMEOUT
    assert situ.device_status(clear=True) == 0
    g = wl.normal((4, 16), 1.0, seed=0).to(cuda_dev)
    out = situ.situ_glu_act(g)
    torch.cuda.synchronize()
    assert out.shape == (4, 8)


# Every case has a long contraction (M = 4096): its waits for an accumulator last many
# microseconds.
def _ffn_dense(dev):
    x, wgu, wd = wl.ffn_inputs(4096, 1536, 4096, seed=1)
    x, wgu, wd = x.to(dev), wgu.to(dev), wd.to(dev)
    return lambda: situ.situ_ffn_forward(x, wgu, wd)


def _grouped(dev, sizes):
    E, M, I = len(sizes), 4096, 512
    ids = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(2))][:, None]
    x = wl.normal((ids.shape[0], M), 1.0, seed=3).to(dev)
    wgu, wd = (w.to(dev) for w in wl.expert_weights(E, M, I, seed=4))
    off, tix = situ.situ_moe_build_index(ids.to(dev), E)
    return lambda: situ.situ_moe_grouped_forward(x, off, tix, wgu, wd, 1)


def _grouped_backward(dev):
    """The grouped training step's backward: K-grouped weight-gradient GEMMs."""
    E, M, I, T = 4, 4096, 384, 96
    g = torch.Generator().manual_seed(5)
    ids = torch.stack([torch.randperm(E, generator=g)[:2] for _ in range(T)]).to(torch.int32)
    x = wl.normal((T, M), 1.0, seed=6).to(dev)
    dy = wl.normal((T, 2, M), 1.0, seed=7).to(dev)
    wgu, wd = (w.to(dev) for w in wl.expert_weights(E, M, I, seed=8))
    off, tix = situ.situ_moe_build_index(ids.to(dev), E)
    _, gu, h = situ.situ_moe_grouped_forward_train(x, off, tix, wgu, wd, 2)
    torch.cuda.synchronize()
    return lambda: situ.situ_moe_grouped_backward(x, off, tix, wgu, wd, gu, h, dy)


def _dense_backward(dev):
    """The dense training step's backward: the two-CTA dh GEMM whose loader warp stages
    the saved (g, u) and stores d(g, u) with TMA."""
    x, wgu, wd = wl.ffn_inputs(4096, 512, 512, seed=10)
    x, wgu, wd = x.to(dev), wgu.to(dev), wd.to(dev)
    dy = wl.normal((512, 4096), 1.0, seed=11).to(dev)
    _, gu, h = situ.situ_ffn_forward_train(x, wgu, wd)
    torch.cuda.synchronize()
    return lambda: situ.situ_ffn_backward(x, wgu, wd, gu, h, dy)


def _grouped_backward_two_cta(dev):
    """A grouped backward whose experts average >= 128 routes: two-CTA dh (staged) and dx
    GEMMs, half-pair tails."""
    sizes, M, I = (300, 290, 140), 4096, 384
    E = len(sizes)
    ids = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(12))][:, None]
    T = ids.shape[0]
    x = wl.normal((T, M), 1.0, seed=13).to(dev)
    dy = wl.normal((T, 1, M), 1.0, seed=14).to(dev)
    wgu, wd = (w.to(dev) for w in wl.expert_weights(E, M, I, seed=15))
    off, tix = situ.situ_moe_build_index(ids.to(dev), E)
    _, gu, h = situ.situ_moe_grouped_forward_train(x, off, tix, wgu, wd, 1)
    torch.cuda.synchronize()
    return lambda: situ.situ_moe_grouped_backward(x, off, tix, wgu, wd, gu, h, dy)


def _mx_dense(dev):
    x, wgu, wd = wl.ffn_inputs(4096, 1536, 2048, seed=9)
    wq = situ.mx_quantize_weights(wgu.to(dev), situ.MX_GATE_UP, situ.MX_E2M1)
    dq = situ.mx_quantize_weights(wd.to(dev), situ.MX_DOWN, situ.MX_E2M1)
    x = x.to(dev)
    return lambda: situ.situ_ffn_forward_mxfp8(x, wq, dq)


@pytest.mark.parametrize("case", ["dense_one_launch", "grouped_two_cta", "grouped_one_cta",
                                  "grouped_backward", "dense_backward",
                                  "grouped_backward_two_cta", "mx_dense"])
def test_gemm_waits_time_out_and_recover(cuda_dev, case):
    """With a 1 us bound every pipelined GEMM's waits run out (a tile's MMAs alone take
    several microseconds): the call records SITU_ERR_TIMEOUT, drains, frees its tensor
    memory and returns.  Restoring the default bound, the next call's results equal
    those of a call made before, bit for bit (the context, tensor memory and
    barriers are all usable again)."""
    run = {"dense_one_launch": lambda: _ffn_dense(cuda_dev),
           "grouped_two_cta": lambda: _grouped(cuda_dev, (300, 290, 140)),
           "grouped_one_cta": lambda: _grouped(cuda_dev, (20, 7, 33, 1, 12)),
           "grouped_backward": lambda: _grouped_backward(cuda_dev),
           "dense_backward": lambda: _dense_backward(cuda_dev),
           "grouped_backward_two_cta": lambda: _grouped_backward_two_cta(cuda_dev),
           "mx_dense": lambda: _mx_dense(cuda_dev)}[case]()
    flat = lambda out: [t.contiguous().view(torch.uint8).clone()
                        for t in (out if isinstance(out, tuple) else (out,))]
    before = flat(run())
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    old = situ.set_wait_limit_ns(1000)
    try:
        run()
        torch.cuda.synchronize()
        assert situ.device_status(clear=True) == 5  # SITU_ERR_TIMEOUT
    finally:
        situ.set_wait_limit_ns(old)
    for _ in range(2):
        after = flat(run())
        torch.cuda.synchronize()
        assert situ.device_status(clear=True) == 0
        assert all(torch.equal(a, b) for a, b in zip(before, after))
