"""Seeded synthetic inputs for the DSA hot path.

This module only draws random tensors: it holds none of the path's arithmetic
and is shared by the tests, the oracle checks and ``bench.py``.  Everything is
drawn on the CPU with a ``torch.Generator`` seeded per workload, in a fixed
order, then rounded to the workload's storage dtype (bf16, or kept fp32), so
the CUDA path and the oracle see bit-identical values.

Shapes follow the released DeepSeek-V3.2 configuration (config_671B_v3.2.json
excerpt on the "DeepSeek-V3.2-Exp - Block input" page: 128 heads, kv_lora_rank
512, qk_rope_head_dim 64, qk_nope_head_dim 128, v_head_dim 128,
index_n_heads 64, index_head_dim 128, index_topk 2048).

Distributions: ``N(0, s)`` means standard deviation s.  The latent c^KV is an
"RMS-normalised Gaussian": x ~ N(0, 1) scaled by 1/sqrt(mean(x^2) + 1e-6) per
row in fp32 (unit gain, the kv_norm RMSNorm of the "Attention input" page),
then rounded.  The latent cache is stored packed, one row per key:
``kv_cache[s] = [c^KV[s] (d_c values) | k_pe[s] (d_r values)]``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Shape:
    """Head shapes of one workload."""
    H_I: int = 64          # indexer heads
    D_I: int = 128         # indexer head dim
    k: int = 2048          # top-k
    H: int = 128           # MLA heads
    d_n: int = 128         # qk_nope_head_dim
    d_r: int = 64          # qk_rope_head_dim
    d_c: int = 512         # kv_lora_rank (latent width)
    d_v: int = 128         # v_head_dim
    softmax_scale: float = 1.0 / math.sqrt(192.0)
    dtype: str = "bf16"    # storage dtype of every tensor: "bf16" or "f32"
    idx_fp8: bool = False  # quantise the indexer q^I / k^I to e4m3 + ue8m0 block scales
    w_std: float = 1.0 / 8.0
    W_std: float = 1.0 / math.sqrt(512.0)


TINY = Shape(H_I=4, D_I=32, k=64, H=4, d_n=32, d_r=16, d_c=64, d_v=32,
             softmax_scale=1.0 / math.sqrt(48.0), dtype="f32", w_std=1.0, W_std=1.0 / math.sqrt(64.0))
FULL = Shape()
FULL_FP8 = Shape(idx_fp8=True)


@dataclass
class Workload:
    """A batch of sequences: query rows of sequence b are rows cu_q[b]..cu_q[b+1]-1,
    its keys are cache rows cu_k[b]..cu_k[b+1]-1, query t sits at start_pos[b] + t."""
    name: str
    shape: Shape
    seed: int
    T: list
    S: list
    start_pos: list
    tensors: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return len(self.T)

    @property
    def cu_q(self) -> list:
        out = [0]
        for t in self.T:
            out.append(out[-1] + t)
        return out

    @property
    def cu_k(self) -> list:
        out = [0]
        for s in self.S:
            out.append(out[-1] + s)
        return out

    @property
    def total_q(self) -> int:
        return sum(self.T)

    @property
    def total_k(self) -> int:
        return sum(self.S)

    def row_positions(self, b: int) -> list:
        return [self.start_pos[b] + t for t in range(self.T[b])]

    def causal_pairs(self) -> int:
        """Number of (query, key) pairs with key <= query position."""
        return sum(sum(p + 1 for p in self.row_positions(b)) for b in range(self.B))

    def selected_pairs(self) -> int:
        k = self.shape.k
        return sum(sum(min(k, p + 1) for p in self.row_positions(b)) for b in range(self.B))


def _store(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x.to(torch.float32)
    raise ValueError(dtype)


def _normal(g: torch.Generator, shape, std: float) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std


def generate(name: str, shape: Shape, seed: int, T: list, S: list, start_pos: list) -> Workload:
    """Draw every tensor of a workload, in this order: q^I, k^I, w, q_nope, q_pe,
    the raw latent, k_pe, W_UK, W_UV."""
    assert len(T) == len(S) == len(start_pos)
    for t, s, p in zip(T, S, start_pos):
        assert t >= 0 and p >= 0 and p + t <= s, (t, s, p)
    sh = shape
    g = torch.Generator().manual_seed(seed + 7919)  # tensors; sizes use the bare seed
    nq, nk = sum(T), sum(S)
    t = {}
    t["qI"] = _store(_normal(g, (nq, sh.H_I, sh.D_I), 1.0), sh.dtype)
    t["kI"] = _store(_normal(g, (nk, sh.D_I), 1.0), sh.dtype)
    t["w"] = _store(_normal(g, (nq, sh.H_I), sh.w_std), sh.dtype).float()  # weights are passed as fp32
    t["q_nope"] = _store(_normal(g, (nq, sh.H, sh.d_n), 1.0), sh.dtype)
    t["q_pe"] = _store(_normal(g, (nq, sh.H, sh.d_r), 1.0), sh.dtype)
    raw = _normal(g, (nk, sh.d_c), 1.0)
    latent = raw * torch.rsqrt(raw.pow(2).mean(-1, keepdim=True) + 1e-6)
    kpe = _normal(g, (nk, sh.d_r), 1.0)
    t["kv_cache"] = _store(torch.cat([latent, kpe], dim=1), sh.dtype)
    t["W_UK"] = _store(_normal(g, (sh.H, sh.d_n, sh.d_c), sh.W_std), sh.dtype)
    t["W_UV"] = _store(_normal(g, (sh.H, sh.d_c, sh.d_v), sh.W_std), sh.dtype)
    return Workload(name=name, shape=sh, seed=seed, T=list(T), S=list(S), start_pos=list(start_pos), tensors=t)


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------
WORKLOADS = {
    0: "tiny fp32 prefill, T=S=256, 4 heads, top-64",
    1: "prefill T=S=4096 causal, 671B head shapes, bf16, top-2048",
    2: "long-context prefill T=S=32768 causal, bf16, top-2048",
    3: "batched decode, 64 sequences x 1 query, caches of 8192-65536 keys",
    4: "chunked prefill, 8 sequences x 8192 new queries on caches of 8192-57344, FP8 indexer",
}


def decode_lengths(seed: int = 1, B: int = 64, lo: int = 8192, hi: int = 65536) -> list:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


def chunk_prefixes(seed: int = 2, B: int = 8, lo: int = 8192, hi: int = 57344) -> list:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


def workload(cfg: int, seed: int | None = None) -> Workload:
    """Generate workload ``cfg`` (0..4) at its full size.  ``seed`` replaces the workload's own tensor
    seed (the sequence lengths stay those of the configuration)."""
    def sd(default):
        return default if seed is None else seed
    if cfg == 0:
        return generate("tiny", TINY, sd(0), [256], [256], [0])
    if cfg == 1:
        return generate("prefill-4k", FULL, sd(0), [4096], [4096], [0])
    if cfg == 2:
        return generate("prefill-32k", FULL, sd(0), [32768], [32768], [0])
    if cfg == 3:
        S = decode_lengths()
        return generate("decode-64", FULL, sd(1), [1] * len(S), S, [s - 1 for s in S])
    if cfg == 4:
        P = chunk_prefixes()
        return generate("chunked-8x8192-fp8", FULL_FP8, sd(2), [8192] * len(P), [p + 8192 for p in P], P)
    raise ValueError(cfg)


def sample_rows(wl: Workload, n: int = 256, seed: int | None = None) -> list:
    """A fixed sample of global query rows: the first and last rows, the rows
    around t = k-1 of each sequence, then random rows (seed 100 + workload seed
    unless given)."""
    nq = wl.total_q
    if nq <= n:
        return list(range(nq))
    rows = {0, nq - 1}
    cu = wl.cu_q
    for b in range(wl.B):
        for dt in (-2, -1, 0, 1):
            t = wl.shape.k - 1 - wl.start_pos[b] + dt
            if 0 <= t < wl.T[b]:
                rows.add(cu[b] + t)
        rows.add(cu[b])
        rows.add(cu[b + 1] - 1)
    g = torch.Generator().manual_seed(100 + wl.seed if seed is None else seed)
    while len(rows) < n:
        rows.add(int(torch.randint(0, nq, (1,), generator=g)))
    return sorted(rows)[:n] if len(rows) > n else sorted(rows)


def random_selection(wl: Workload, seed: int, density: float = 0.5) -> torch.Tensor:
    """A seeded selection input for stand-alone attention tests: for each row,
    up to k distinct causal keys drawn at random (-1 padded, random order)."""
    g = torch.Generator().manual_seed(seed)
    k = wl.shape.k
    rows = []
    for b in range(wl.B):
        for p in wl.row_positions(b):
            n_causal = p + 1
            n = min(k, max(1, int(round(n_causal * density))))
            perm = torch.randperm(n_causal, generator=g)[:n].to(torch.int32)
            row = torch.full((k,), -1, dtype=torch.int32)
            slots = torch.randperm(k, generator=g)[:n]
            row[slots] = perm
            rows.append(row)
    return torch.stack(rows) if rows else torch.empty((0, k), dtype=torch.int32)
