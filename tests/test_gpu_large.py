"""Buffers past 4 GiB: the dense FFN over 700 000 tokens (h alone is 4.3 GB, more than
2^31 elements) and the standalone activation over a 4.9 GB input, so that any 32-bit
element or byte offset in the kernels' or the ABI's indexing would show.  Seeded
sampled rows (first and last included) against the FP64 oracle, in the launch
configuration the benchmark uses."""
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_ffn_close, assert_within_ulp, oracle_input, to_f64

pytestmark = pytest.mark.gpu


def _rows(n, count, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.cat([torch.tensor([0, n - 1, n // 2]), torch.randint(0, n, (count - 3,), generator=g)])


def test_dense_ffn_past_4gib(oracle, cuda_dev):
    R, M, I = 700_000, 2048, 3072
    assert R * I > 2 ** 31
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=21, device=cuda_dev)
    y = situ.situ_ffn_forward(x, wgu, wd)
    torch.cuda.synchronize()
    assert situ.ffn_last_path() == situ.FFN_PATH_FUSED
    rd = _rows(R, 24, 22).to(cuda_dev)
    ref = oracle.ffn_forward(oracle_input(x[rd]), oracle_input(wgu), oracle_input(wd))
    assert_ffn_close(to_f64(y[rd]), ref, "dense FFN past 4 GiB")
    del x, y
    torch.cuda.empty_cache()


def test_act_past_4gib(oracle, cuda_dev):
    rows, I = 400_000, 3072
    assert rows * 2 * I > 2 ** 31
    w = wl.WORKLOADS["act"]
    gate_up = wl.gate_up_input(w, seed=23, device=cuda_dev, rows=rows)
    assert gate_up.shape == (rows, 2 * I)
    out = situ.situ_glu_act(gate_up)
    torch.cuda.synchronize()
    rd = _rows(rows, 64, 24).to(cuda_dev)
    ref = oracle.situ_glu_act(oracle_input(gate_up[rd].cpu()))
    assert_within_ulp(to_f64(out[rd]), ref, "activation past 4 GiB")
    del gate_up, out
    torch.cuda.empty_cache()
