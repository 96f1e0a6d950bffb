"""Seeded synthetic inputs shaped like the SiTU-GLU pages' workloads.

Shared by the tests, the benchmark and the smoke check; both the CUDA path and
the CPU oracle are fed from here.  This module draws random numbers and arranges
them into tensors; it contains none of SiTU-GLU's arithmetic.

Recipes (all seed 0 unless a test says otherwise):
  * normal(shape, std): torch's seeded normal generator on the requested device,
    drawn in float32 and rounded to the storage dtype (bf16 rounding is
    round-to-nearest-even).  Weights use std = 1/sqrt(fan_in).
  * add_outliers: each entry independently, with probability p, replaced by
    sign * U(lo, hi) with a fair random sign.
  * zipf_routes: expert popularity p(rank) proportional to rank^-s over E ranks,
    ranks mapped to expert ids by a seeded permutation; n_empty seeded experts get
    probability zero; each token draws k distinct experts by sequential weighted
    sampling without replacement (Gumbel top-k).
  * uniform_routes: k distinct experts per token, uniformly, then every shared
    expert id appended as extra slots.
Routes are always drawn on the CPU so they are identical whichever device the
tensors live on.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

M_MODEL = 2048       # synthetic expert width
I_FFN = 3072         # expert d_ff (moe_intermediate_size)
BETA, LINEAR_BETA = 4.0, 25.0


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "act" | "ffn" | "moe"
    rows: int = 0        # act / ffn rows
    M: int = M_MODEL
    I: int = I_FFN
    dtype: torch.dtype = torch.bfloat16
    std: float = 1.0     # input std
    outlier_p: float = 0.0
    outlier_lo: float = 50.0
    outlier_hi: float = 5000.0
    # MoE
    T: int = 0
    E: int = 0
    k: int = 0
    shared: tuple = field(default_factory=tuple)
    routing: str = ""    # "zipf" | "uniform"
    zipf_s: float = 1.1
    n_empty: int = 0

    @property
    def k_eff(self) -> int:
        return self.k + len(self.shared)

    @property
    def num_experts(self) -> int:
        return self.E + len(self.shared)


WORKLOADS = {
    # Tiny fp32 dense FFN: x [2, 8, 128], W_gate_up [512, 128], W_down [128, 256].
    "tiny_fp32": Workload("tiny dense SiTU-GLU FFN, fp32, x[2,8,128], I=256", "ffn",
                          rows=16, M=128, I=256, dtype=torch.float32),
    # Standalone activation, memory bound: gate_up bf16 [65536, 6144] ~ N(0, 3) + 1% outliers.
    "act": Workload("standalone SiTU-GLU activation, bf16 [65536, 2x3072], N(0,3) + 1% "
                    "outliers U(50,5000)", "act", rows=65536, I=3072, std=3.0, outlier_p=0.01),
    # Dense FFN, compute bound: 16384 tokens, M=2048, I=3072.
    "dense": Workload("dense SiTU-GLU FFN, bf16, 16384 tokens, M=2048, I=3072", "ffn",
                      rows=16384),
    # Grouped routed experts: E=64, top-8 Zipf(1.1) with 4 empty experts.
    "grouped": Workload("grouped SiTU-GLU experts, bf16, E=64, 16384 tokens top-8 Zipf(1.1)",
                        "moe", T=16384, E=64, k=8, routing="zipf", n_empty=4),
    # The grouped shapes at a quarter of the tokens (16 experts, one of them empty): the
    # same per-expert GEMM shapes with about 2 GB on the device, for profiling.
    "grouped_slice": Workload("16 routed experts, 4096 tokens top-8 Zipf(1.1) with 1 empty "
                              "expert (the grouped shapes, for profiling)", "moe", T=4096, E=16,
                              k=8, routing="zipf", n_empty=1),
    # Kimi-K3-shaped layer: 896 routed + 2 shared experts.
    "k3_decode": Workload("Kimi-K3-shaped MoE layer, 896 routed + 2 shared experts, 512 tokens",
                          "moe", T=512, E=896, k=8, shared=(896, 897), routing="uniform"),
    "k3_prefill": Workload("Kimi-K3-shaped MoE layer, 896 routed + 2 shared experts, "
                           "32768 tokens", "moe", T=32768, E=896, k=8, shared=(896, 897),
                           routing="uniform"),
    # A 64-expert slice with the prefill's rows per expert (about 293): the same
    # per-expert GEMM shapes with 2.4 GB of weights, for profiling.
    "k3_prefill_slice": Workload("64 routed experts, 2344 tokens top-8 uniform (about 293 rows "
                                 "per expert, the K3 prefill shape)", "moe", T=2344, E=64, k=8,
                                 routing="uniform"),
    # A 64-expert slice with the decode's rows per expert (about 6): the same
    # weight-streaming GEMM shapes with 2.4 GB of weights, for profiling.
    "k3_decode_slice": Workload("64 routed experts, 48 tokens top-8 uniform (about 6 rows per "
                                "expert, the K3 decode shape)", "moe", T=48, E=64, k=8,
                                routing="uniform"),
}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, device="cpu", dtype=torch.bfloat16,
           chunk: int = 1 << 27) -> torch.Tensor:
    """Seeded N(0, std^2) tensor; drawn in float32 chunks, rounded to dtype."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    g = generator(seed, device)
    n = flat.numel()
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        tmp = torch.randn(m, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[i:i + m].copy_(tmp)
    return out


def add_outliers(t: torch.Tensor, p: float, lo: float, hi: float, seed: int,
                 chunk: int = 1 << 26) -> torch.Tensor:
    """In place: each entry with probability p becomes sign * U(lo, hi)."""
    flat = t.view(-1)
    g = generator(seed, t.device)
    n = flat.numel()
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        u = torch.rand(3, m, generator=g, device=t.device, dtype=torch.float32)
        mask = u[0] < p
        val = (lo + (hi - lo) * u[1]) * torch.where(u[2] < 0.5, -1.0, 1.0)
        seg = flat[i:i + m]
        seg[mask] = val[mask].to(t.dtype)
    return t


def gate_up_input(w: Workload, seed: int = 0, device="cpu", rows: int | None = None):
    """gate_up [rows, 2I] for an activation workload."""
    r = w.rows if rows is None else rows
    t = normal((r, 2 * w.I), w.std, seed, device, w.dtype)
    if w.outlier_p:
        add_outliers(t, w.outlier_p, w.outlier_lo, w.outlier_hi, seed + 1)
    return t


def ffn_inputs(M: int, I: int, rows: int, seed: int = 0, device="cpu",
               dtype=torch.bfloat16):
    """x [rows, M] ~ N(0,1); W_gate_up [2I, M] ~ N(0, 1/M); W_down [M, I] ~ N(0, 1/I)."""
    x = normal((rows, M), 1.0, seed, device, dtype)
    w_gu = normal((2 * I, M), 1.0 / math.sqrt(M), seed + 1, device, dtype)
    w_d = normal((M, I), 1.0 / math.sqrt(I), seed + 2, device, dtype)
    return x, w_gu, w_d


def expert_weights(E: int, M: int, I: int, seed: int = 0, device="cpu",
                   dtype=torch.bfloat16):
    """Stacked expert weights W_gate_up [E, 2I, M], W_down [E, M, I]."""
    w_gu = normal((E, 2 * I, M), 1.0 / math.sqrt(M), seed + 1, device, dtype)
    w_d = normal((E, M, I), 1.0 / math.sqrt(I), seed + 2, device, dtype)
    return w_gu, w_d


def zipf_routes(T: int, E: int, k: int, s: float = 1.1, n_empty: int = 0,
                seed: int = 0) -> torch.Tensor:
    """expert_ids [T, k] int32: k distinct experts per token, Zipf(s) popularity."""
    g = generator(seed)
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    p_rank = ranks.pow(-s)
    perm = torch.randperm(E, generator=g)          # rank i -> expert perm[i]
    p = torch.empty(E, dtype=torch.float64)
    p[perm] = p_rank
    if n_empty:
        empty = torch.randperm(E, generator=g)[:n_empty]
        p[empty] = 0.0
    logp = torch.log(p / p.sum())
    gumbel = -torch.log(-torch.log(torch.rand(T, E, generator=g, dtype=torch.float64)))
    keys = logp.unsqueeze(0) + gumbel
    return keys.topk(k, dim=1).indices.to(torch.int32).contiguous()


def uniform_routes(T: int, E: int, k: int, shared=(), seed: int = 0) -> torch.Tensor:
    """expert_ids [T, k + len(shared)] int32: k distinct uniform experts, then shared ids."""
    g = generator(seed)
    ids = torch.rand(T, E, generator=g).topk(k, dim=1).indices.to(torch.int32)
    if shared:
        sh = torch.tensor(shared, dtype=torch.int32).expand(T, len(shared))
        ids = torch.cat([ids, sh], dim=1)
    return ids.contiguous()


def combine_weights(T: int, k: int, n_shared: int = 0, seed: int = 0) -> torch.Tensor:
    """Router combine weights [T, k + n_shared] float32: for the k routed slots a
    softmax of seeded N(0, 1) logits (positive, summing to 1 per token), then
    weight 1 for every shared-expert slot."""
    g = generator(seed)
    w = torch.softmax(torch.randn(T, k, generator=g, dtype=torch.float32), dim=1)
    if n_shared:
        w = torch.cat([w, torch.ones(T, n_shared, dtype=torch.float32)], dim=1)
    return w.contiguous()


def routes(w: Workload, seed: int = 0, T: int | None = None) -> torch.Tensor:
    T = w.T if T is None else T
    if w.routing == "zipf":
        return zipf_routes(T, w.E, w.k, w.zipf_s, w.n_empty, seed)
    return uniform_routes(T, w.E, w.k, w.shared, seed)


# Activation rows of the tiny configuration: the worked example, the bound at
# |g|, |u| = 1e4 in every sign pair, one saturated branch at a time, and gate
# values deep in the negative tail whose outputs are subnormal.
SPECIAL_PAIRS = [
    (2.0, 2.0),
    (1e4, 1e4), (1e4, -1e4), (-1e4, 1e4), (-1e4, -1e4),
    (1e4, 2.0), (2.0, 1e4),
    (-90.0, 2.0), (-100.0, 2.0), (-90.0, 25.0), (-100.0, -7.0),
]


def special_gate_up(dtype=torch.float32, pad_to: int | None = None) -> torch.Tensor:
    """One row [2n]: the gate values of SPECIAL_PAIRS, then their up values."""
    g = [p[0] for p in SPECIAL_PAIRS]
    u = [p[1] for p in SPECIAL_PAIRS]
    if pad_to:
        g += [0.0] * (pad_to - len(g))
        u += [0.0] * (pad_to - len(u))
    return torch.tensor([g + u], dtype=dtype)
