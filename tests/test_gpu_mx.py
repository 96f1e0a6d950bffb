"""MXFP8 experts on the GPU against the FP64 oracle.

Quantization (codes and scales): bit-exact -- every decision is taken on the bf16
input by both sides.  GEMMs: the oracle multiplies the decoded MX values in FP64.
The GPU accumulates in FP32 and rounds the output to bf16, so
    |err| <= 2^-8 |ref| + K 2^-24 sum_k |terms_k|
(bf16 rounding; worst-case FP32 accumulation over K terms), well inside the stated
FFN tolerance 2e-2 (1 + |ref|), which every FFN output must also meet.  The MX FFN
rounds h to bf16 and quantizes it on the GPU, where h carries the FP32 arithmetic
of the activation: a code can differ from the oracle's by one step where h sits at
a rounding boundary, so the end-to-end check allows exactly the differences of the
codes that differ, sum_j |dec(h_gpu)_j - dec(h_ref)_j| |W_down[m, j]|.
"""
import math

import numpy as np
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_ffn_close, oracle_input, to_f64

pytestmark = pytest.mark.gpu
INF = float("inf")


# ----- scale-tile layouts (as include/situ.h documents them), read on the host -----
def untile_act_scales(sf: np.ndarray, R: int, K: int) -> np.ndarray:
    ks, nt = K // 128, (R + 127) // 128
    a = sf[: nt * ks * 512].reshape(nt, ks, 32, 4, 4)      # [tile, stage, l, g, k]
    return a.transpose(0, 3, 2, 1, 4).reshape(nt * 128, ks * 4)[:R]


def untile_weight_scales(sf: np.ndarray, E: int, rows: int, K: int, split: int) -> np.ndarray:
    ks = K // 128
    nt = math.ceil(split / 96) if split else math.ceil(rows / 192)
    a = sf.reshape(E, nt, ks, 2, 32, 4, 4)                  # [e, t, s, half, l, g, k]
    by_n = a.transpose(0, 1, 3, 5, 4, 2, 6).reshape(E, nt, 256, ks * 4)  # n = 128h + 32g + l
    out = np.zeros((E, rows, ks * 4), dtype=np.uint8)
    for t in range(nt):
        for n in range(192):
            if split:
                j = n % 96
                if 96 * t + j >= split:
                    continue
                r = 96 * t + j if n < 96 else split + 96 * t + j
            else:
                r = 192 * t + n
                if r >= rows:
                    continue
            out[:, r, :] = by_n[:, t, n, :]
    return out


def _gpu_mx_act(x_dev):
    codes, sf = situ.mx_quantize_act(x_dev)
    torch.cuda.synchronize()
    R, K = codes.shape
    return codes.cpu().numpy(), untile_act_scales(sf.cpu().numpy(), R, K)


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _special_rows(K=256):
    """Blocks with zeros, negative zeros, bf16 subnormals, clamping and outliers."""
    rows = np.zeros((6, K))
    rows[0, :32] = -0.0
    rows[1, :32] = np.linspace(-1, 1, 32) * 1e-39          # subnormal bf16
    rows[2, :32] = 1.9 * 2.0 ** 5                           # clamps to 448 after scaling
    rows[3, :32] = np.r_[5000.0, np.full(31, 0.01)]         # outlier flattens its block
    rows[4, :] = np.tile(np.r_[2.0 ** -10, -(2.0 ** -10) * 1.5, np.full(30, 1.0)], K // 32)
    rows[5, :32] = 3.0e38
    return torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("R,K", [(300, 256), (1, 128), (128, 2048), (129, 384)])
def test_quantize_act_bit_exact(oracle, cuda_dev, R, K):
    x = wl.normal((R, K), 3.0, seed=R + K)
    wl.add_outliers(x, 0.01, 50.0, 5000.0, seed=R)
    if R >= 6:
        x[:6] = _special_rows(K)
    codes, scales = _gpu_mx_act(x.to(cuda_dev))
    rc, rs = oracle.mx_quantize(_bf16_bits(x))
    assert np.array_equal(codes, rc)
    assert np.array_equal(scales, rs)


@pytest.mark.parametrize("order", ["shuffled", "sorted"])
def test_quantize_every_bf16_value(oracle, cuda_dev, order):
    """Every finite bf16 value, in seeded-shuffled blocks (mixed magnitudes: many
    values scaled far down against a large block maximum) and in magnitude-sorted
    blocks (neighbouring values, every scale from 2^-127 up)."""
    bits = np.arange(65536, dtype=np.uint32)
    finite = bits[(bits & 0x7F80) != 0x7F80].astype(np.uint16)
    if order == "shuffled":
        finite = np.random.default_rng(7).permutation(finite)
    else:
        finite = finite[np.argsort(finite & 0x7FFF, kind="stable")]
    K = 256
    n = -(-finite.size // K) * K
    v = np.zeros(n, dtype=np.uint16)
    v[: finite.size] = finite
    x = torch.from_numpy(v.view(np.int16).reshape(-1, K).copy()).view(torch.bfloat16)
    codes, scales = _gpu_mx_act(x.to(cuda_dev))
    rc, rs = oracle.mx_quantize(v.reshape(-1, K))
    assert np.array_equal(scales, rs)
    bad = np.flatnonzero(codes.ravel() != rc.ravel())
    assert bad.size == 0, f"{bad.size} codes differ, first at {bad[:4]}"


FMTS = [situ.MX_E4M3, situ.MX_E2M1]
FMT_IDS = ["mxfp8_w", "mxfp4_w"]


def _oracle_wq(oracle, t, fmt):
    """The oracle's quantization of weight rows in format fmt."""
    bits = _bf16_bits(t.reshape(-1, t.shape[-1]))
    return oracle.mxfp4_quantize(bits) if fmt == situ.MX_E2M1 else oracle.mx_quantize(bits)


def _wdeq(oracle, q, fmt):
    return oracle.mxfp4_dequantize(*q) if fmt == situ.MX_E2M1 else oracle.mx_dequantize(*q)


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("kind", [situ.MX_GATE_UP, situ.MX_DOWN], ids=["gate_up", "down"])
def test_quantize_weights_bit_exact(oracle, cuda_dev, kind, fmt):
    E, M, I = 2, 256, 384
    wgu, wd = wl.expert_weights(E, M, I, seed=11)
    W = wgu if kind == situ.MX_GATE_UP else wd
    codes, sf, _ = situ.mx_quantize_weights(W.to(cuda_dev), kind, fmt)
    torch.cuda.synchronize()
    rows, K = W.shape[1], W.shape[2]
    split = I if kind == situ.MX_GATE_UP else 0
    got_s = untile_weight_scales(sf.cpu().numpy(), E, rows, K, split)
    rc, rs = _oracle_wq(oracle, W, fmt)
    assert np.array_equal(codes.cpu().numpy().reshape(rc.shape), rc)
    assert np.array_equal(got_s.reshape(E * rows, K // 32), rs)


def test_quantize_fp4_every_bf16_value(oracle, cuda_dev):
    """Every finite bf16 value through the MXFP4 weight quantizer (seeded-shuffled
    into 32-blocks of mixed magnitudes), codes and scales bit-exact."""
    bits = np.arange(65536, dtype=np.uint32)
    finite = np.random.default_rng(8).permutation(bits[(bits & 0x7F80) != 0x7F80].astype(np.uint16))
    M, I = 256, 256
    v = np.zeros(M * I, dtype=np.uint16)
    v[: finite.size] = finite
    W = torch.from_numpy(v.view(np.int16).reshape(1, M, I).copy()).view(torch.bfloat16)
    codes, sf, _ = situ.mx_quantize_weights(W.to(cuda_dev), situ.MX_DOWN, situ.MX_E2M1)
    torch.cuda.synchronize()
    rc, rs = oracle.mxfp4_quantize(v.reshape(M, I))
    got_s = untile_weight_scales(sf.cpu().numpy(), 1, M, I, 0).reshape(M, I // 32)
    assert np.array_equal(got_s, rs)
    bad = np.flatnonzero(codes.cpu().numpy().reshape(M, I // 2) != rc)
    assert bad.size == 0, f"{bad.size} code bytes differ, first at {bad[:4]}"


def _mx_inputs(R, M, I, seed):
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=seed)
    return x, wgu, wd


def _oracle_q(oracle, t):
    return oracle.mx_quantize(_bf16_bits(t.reshape(-1, t.shape[-1])))


def _gemm_close(got, ref, abs_terms, K, what):
    g = to_f64(got) if isinstance(got, torch.Tensor) else got
    err = np.abs(g - ref)
    tol = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -24 * abs_terms + 1e-30
    assert np.isfinite(g).all(), what
    assert (err <= tol).all(), f"{what}: worst err/tol {float((err / tol).max()):.3g}"
    assert_ffn_close(g, ref, what)


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("R,M,I", [(300, 256, 384), (1, 128, 128), (513, 512, 1152)])
def test_gate_up_mxfp8(oracle, cuda_dev, R, M, I, fmt):
    """h of the block-scaled gate_up GEMM against the oracle's FFN on the decoded MX
    operands (activation at the FP64 gu; FFN tolerance)."""
    x, wgu, wd = _mx_inputs(R, M, I, seed=R + I)
    xq = situ.mx_quantize_act(x.to(cuda_dev))
    wq = situ.mx_quantize_weights(wgu.to(cuda_dev), situ.MX_GATE_UP, fmt)
    h = situ.situ_ffn_gate_up_mxfp8(xq, wq)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    xd = oracle.mx_dequantize(*_oracle_q(oracle, x))
    wgud = _wdeq(oracle, _oracle_wq(oracle, wgu, fmt), fmt)
    _, h_ref = oracle.ffn_forward(xd, wgud, to_f64(wd), want_h=True)
    assert_ffn_close(to_f64(h), h_ref, f"MX h {R}x{M}x{I}")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("R,M,I", [(300, 256, 384), (129, 128, 256), (513, 512, 1152)])
def test_ffn_forward_mxfp8(oracle, cuda_dev, R, M, I, fmt):
    x, wgu, wd = _mx_inputs(R, M, I, seed=3 * R + I)
    xd_, wgud_, wdd_ = x.to(cuda_dev), wgu.to(cuda_dev), wd.to(cuda_dev)
    wguq = situ.mx_quantize_weights(wgud_, situ.MX_GATE_UP, fmt)
    wdq = situ.mx_quantize_weights(wdd_, situ.MX_DOWN, fmt)
    ws = torch.empty(situ.ffn_mxfp8_workspace_bytes(R, M, I), dtype=torch.uint8, device=cuda_dev)
    y = situ.situ_ffn_forward_mxfp8(xd_, wguq, wdq, workspace=ws)
    h_bf16 = situ.situ_ffn_gate_up_mxfp8(situ.mx_quantize_act(xd_), wguq)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    # Workspace regions (256-byte aligned, in order): x codes, x scales, h codes, h scales.
    up = lambda n: -(-n // 256) * 256
    o_hc = up(R * M) + up(situ.mx_act_scales_bytes(R, M))
    o_hs = o_hc + up(R * I)
    wsn = ws.cpu().numpy()
    hc = wsn[o_hc:o_hc + R * I].reshape(R, I)
    hs = untile_act_scales(wsn[o_hs:o_hs + situ.mx_act_scales_bytes(R, I)], R, I)
    # 1. The fused quantization of h is the oracle's quantization of the GPU's bf16 h.
    rc, rs = oracle.mx_quantize(_bf16_bits(h_bf16))
    assert np.array_equal(hs, rs)
    assert np.array_equal(hc, rc)
    # 2. The down GEMM against the FP64 product of the decoded operands.
    wdd = _wdeq(oracle, _oracle_wq(oracle, wd, fmt), fmt)
    hdec = oracle.mx_dequantize(hc, hs)
    _gemm_close(y, hdec @ wdd.T, np.abs(hdec) @ np.abs(wdd).T, I, f"MX down {R}x{M}x{I}")
    # 3. End to end against the oracle's MX FFN, allowing the codes that differ.
    y_ref, _, (hc_r, hs_r) = oracle.mx_ffn_forward(
        _oracle_q(oracle, x), _oracle_wq(oracle, wgu, fmt), _oracle_wq(oracle, wd, fmt),
        weights_fp4=fmt == situ.MX_E2M1)
    diff = np.abs(hdec - oracle.mx_dequantize(hc_r, hs_r))
    assert (hc != hc_r).mean() < 0.02, "more than 2% of the h codes differ"
    err = np.abs(to_f64(y) - y_ref)
    tol = 2e-2 * (1 + np.abs(y_ref)) + diff @ np.abs(wdd).T
    assert (err <= tol).all(), f"MX FFN end to end: worst err/tol {float((err / tol).max()):.3g}"


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("R,M,I,caps", [(300, 256, 384, (4.0, 25.0)), (129, 128, 256, (INF, INF)),
                                        (513, 512, 1152, (4.0, INF)),
                                        (4096, 2048, 3072, (4.0, 25.0))])
def test_ffn_mxfp8_single_launch_matches_two_launches(cuda_dev, R, M, I, caps, fmt):
    """The one-launch MX FFN (down tiles wait on per-row-tile h-ready counts) gives the
    bits of the gate_up launch followed by the down launch; repeated calls reset the
    counts."""
    x, wgu, wd = _mx_inputs(R, M, I, seed=R + I)
    xd_ = x.to(cuda_dev)
    wguq = situ.mx_quantize_weights(wgu.to(cuda_dev), situ.MX_GATE_UP, fmt)
    wdq = situ.mx_quantize_weights(wd.to(cuda_dev), situ.MX_DOWN, fmt)
    ws = torch.empty(situ.ffn_mxfp8_workspace_bytes(R, M, I), dtype=torch.uint8, device=cuda_dev)
    assert situ.ffn_set_single_launch(False) is True
    try:
        y2 = situ.situ_ffn_forward_mxfp8(xd_, wguq, wdq, *caps, workspace=ws)
        assert situ.ffn_last_path() == situ.FFN_PATH_TWO_LAUNCHES
    finally:
        situ.ffn_set_single_launch(True)
    for _ in range(3):
        y = situ.situ_ffn_forward_mxfp8(xd_, wguq, wdq, *caps, workspace=ws)
        assert situ.ffn_last_path() == situ.FFN_PATH_FUSED
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert situ.device_status() == 0


def test_ffn_mxfp8_variants(oracle, cuda_dev):
    """Both caps removed (SwiGLU) and the up cap removed, through the MX path."""
    R, M, I = 200, 256, 384
    x, wgu, wd = _mx_inputs(R, M, I, seed=77)
    xq = situ.mx_quantize_act(x.to(cuda_dev))
    wq = situ.mx_quantize_weights(wgu.to(cuda_dev), situ.MX_GATE_UP)
    inf = float("inf")
    xd = oracle.mx_dequantize(*_oracle_q(oracle, x))
    wgud = oracle.mx_dequantize(*_oracle_q(oracle, wgu))
    for caps, oc in (((inf, inf), (0.0, 0.0)), ((4.0, inf), (4.0, 0.0))):
        h = situ.situ_ffn_gate_up_mxfp8(xq, wq, *caps)
        torch.cuda.synchronize()
        _, h_ref = oracle.ffn_forward(xd, wgud, to_f64(wd), *oc, want_h=True)
        assert_ffn_close(to_f64(h), h_ref, f"MX h caps {caps}")


def _grouped_case(T, k, E, M, I, seed, dev, fmt=situ.MX_E4M3):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E - 1, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    x = wl.normal((T, M), 1.0, seed=seed)
    wgu, wd = wl.expert_weights(E, M, I, seed=seed + 1)
    off, tix = situ.situ_moe_build_index(ids.to(dev), E)
    wguq = situ.mx_quantize_weights(wgu.to(dev), situ.MX_GATE_UP, fmt)
    wdq = situ.mx_quantize_weights(wd.to(dev), situ.MX_DOWN, fmt)
    return ids, x, wgu, wd, off, tix, wguq, wdq


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("T,k,E,M,I", [
    (50, 3, 6, 256, 384),
    (300, 2, 3, 128, 256),
    # 1600 routes over 3 experts (at least 512 rows per expert on average): two-CTA
    # MMAs; experts 0 and 1 hold 800 rows (7 m-tiles, so each has a pair whose second
    # m-tile is past its rows), expert 2 none; K of 2 and of 3 128-wide k-blocks.
    (800, 2, 3, 256, 256),
    (800, 2, 3, 384, 256),
])
def test_grouped_mxfp8_equals_dense_per_expert(cuda_dev, T, k, E, M, I, fmt):
    """Each (token, slot) row of the grouped MX forward equals the dense MX FFN of its
    expert on the token, bit for bit: rows are quantized and multiplied
    independently of the other rows of their tile."""
    ids, x, wgu, wd, off, tix, wguq, wdq = _grouped_case(T, k, E, M, I, T + E, cuda_dev, fmt)
    y = situ.situ_moe_grouped_forward_mxfp8(x.to(cuda_dev), off, tix, wguq, wdq, k)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    y = y.cpu()
    for e in range(E):
        t_idx, s_idx = (ids == e).nonzero(as_tuple=True)
        if len(t_idx) == 0:
            continue
        we = situ.MxWeights(wguq[0][e].contiguous(), wguq[1].view(E, -1)[e].contiguous(), fmt)
        wde = situ.MxWeights(wdq[0][e].contiguous(), wdq[1].view(E, -1)[e].contiguous(), fmt)
        ye = situ.situ_ffn_forward_mxfp8(x.to(cuda_dev), we, wde).cpu()
        assert torch.equal(y[t_idx, s_idx].view(torch.int16), ye[t_idx].view(torch.int16)), e


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_grouped_mxfp8_against_oracle(oracle, cuda_dev, fmt):
    T, k, E, M, I = 40, 4, 9, 256, 384
    ids, x, wgu, wd, off, tix, wguq, wdq = _grouped_case(T, k, E, M, I, 5, cuda_dev, fmt)
    y = situ.situ_moe_grouped_forward_mxfp8(x.to(cuda_dev), off, tix, wguq, wdq, k)
    torch.cuda.synchronize()
    y = to_f64(y)
    xq = _oracle_q(oracle, x)
    for e in range(E):
        t_idx, s_idx = (ids == e).nonzero(as_tuple=True)
        if len(t_idx) == 0:
            continue
        t_np = t_idx.numpy()
        xe = (xq[0][t_np], xq[1][t_np])
        y_ref, _, _ = oracle.mx_ffn_forward(xe, _oracle_wq(oracle, wgu[e], fmt),
                                            _oracle_wq(oracle, wd[e], fmt),
                                            weights_fp4=fmt == situ.MX_E2M1)
        assert_ffn_close(y[t_idx, s_idx], y_ref, f"grouped MX expert {e}")


def test_ffn_mxfp8_full_size_sampled(oracle, cuda_dev):
    """The 16384-token dense workload (M=2048, I=3072) through the MX path at full
    size; 24 sampled rows (first, last, random) against the oracle's MX FFN."""
    w = wl.WORKLOADS["dense"]
    x, wgu, wd = wl.ffn_inputs(w.M, w.I, w.rows, seed=0, device=cuda_dev)
    wguq = situ.mx_quantize_weights(wgu, situ.MX_GATE_UP)
    wdq = situ.mx_quantize_weights(wd, situ.MX_DOWN)
    y = situ.situ_ffn_forward_mxfp8(x, wguq, wdq)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    g = torch.Generator().manual_seed(3)
    rows = [0, w.rows - 1] + torch.randint(1, w.rows - 1, (22,), generator=g).tolist()
    xs = x[torch.tensor(rows, device=cuda_dev)].cpu()
    y_ref, _, _ = oracle.mx_ffn_forward(_oracle_q(oracle, xs), _oracle_q(oracle, wgu.cpu()),
                                        _oracle_q(oracle, wd.cpu()))
    assert_ffn_close(to_f64(y[torch.tensor(rows, device=cuda_dev)]), y_ref, "MX FFN full size")


def test_mxfp8_bad_shapes(cuda_dev):
    x = torch.zeros(4, 136, dtype=torch.bfloat16, device=cuda_dev)
    with pytest.raises(situ.SituError, match="UNSUPPORTED"):
        situ.mx_quantize_act(x)


@pytest.mark.parametrize("name", ["k3_decode", "k3_prefill", "grouped"])
@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_moe_mx_full_size_sampled(oracle, cuda_dev, fmt, name):
    """The routed-expert workloads the benchmark times through the grouped MX path at
    full size -- the Kimi-K3-shaped layer (896 routed + 2 shared experts, M=2048,
    I=3072) at 512 and 32768 tokens, and the 64-expert Zipf workload; 16 sampled routes
    (first and last rows of expert groups, random rows) against the oracle's MX FFN of
    their expert on their token."""
    w = wl.WORKLOADS[name]
    E = w.num_experts
    ids = wl.routes(w, seed=0)
    x = wl.normal((w.T, w.M), 1.0, seed=0, device=cuda_dev)
    wgu, wd = wl.expert_weights(E, w.M, w.I, seed=0, device=cuda_dev)
    wguq = situ.mx_quantize_weights(wgu, situ.MX_GATE_UP, fmt)
    wdq = situ.mx_quantize_weights(wd, situ.MX_DOWN, fmt)
    off, tix = situ.situ_moe_build_index(ids.to(cuda_dev), E)
    y = situ.situ_moe_grouped_forward_mxfp8(x, off, tix, wguq, wdq, w.k_eff)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    off_c, tix_c = off.cpu().numpy(), tix.cpu().numpy()
    nonempty = np.flatnonzero(np.diff(off_c) > 0)
    g = torch.Generator().manual_seed(12)
    pick = [int(off_c[nonempty[0]]), int(off_c[nonempty[-1] + 1] - 1)]
    pick += torch.randint(0, w.T * w.k_eff, (14,), generator=g).tolist()
    for r in pick:
        flat = int(tix_c[r])
        t, s = divmod(flat, w.k_eff)
        e = int(ids[t, s])
        y_ref, _, _ = oracle.mx_ffn_forward(_oracle_q(oracle, x[t:t + 1].cpu()),
                                            _oracle_wq(oracle, wgu[e].cpu(), fmt),
                                            _oracle_wq(oracle, wd[e].cpu(), fmt),
                                            weights_fp4=fmt == situ.MX_E2M1)
        assert_ffn_close(to_f64(y[t, s:s + 1]), y_ref, f"K3 MX route {r} (t={t}, s={s}, e={e})")
    del wgu, wd, wguq, wdq
    torch.cuda.empty_cache()
