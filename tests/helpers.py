"""Shared helpers of the parity tests: moving a workload to the device,
running the oracle on a subset of rows, and the acceptance rules.

Acceptance rules (the tolerances the path is held to):
  * indexer scores: |gpu - ref| <= 1e-3 * |ref| + 1e-5 * A, where A is the
    absolute-term sum 1/sqrt(H_I D_I) sum_h |w| ReLU(q.k).  The first term is
    the stated "1e-3 relative"; the second is a floor of the size of the fp32
    accumulation error (the kernels add the exact input products and the 64
    weighted heads in fp32, whose rounding is a few 1e-7 of A), so that a
    score that cancels to ~0 is not held to an impossible relative bound.
    Masked keys must be exactly -inf;
  * top-k: the GPU set equals the oracle set except for keys whose oracle
    score lies within tau = 1e-3 * |S_n| + 1e-5 * A_n of the oracle's n-th
    score S_n; the GPU row holds exactly n = min(k, p+1) distinct causal keys
    followed by -1 padding;
  * attention output: max |gpu - ref| <= 2e-2 (unit-scale bf16 data);
    fp32 workloads are held to 1e-4.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_latent_attention_indexer_gb300 as dsa

SCORE_RTOL = 1e-3
SCORE_ATOL_A = 1e-5  # times the absolute-term sum A of the same score
OUT_ATOL_BF16 = 2e-2
OUT_ATOL_F32 = 1e-4
# The stated tolerances bound the outputs only; the lse (natural log) bound is derived from the
# rounding the bf16 path performs: q~ rounded to bf16 (relative 2^-9 per element) perturbs a
# unit-scale logit by a few 1e-3, and the fp16 exchange of the log2-scaled partial scores between
# the two CTAs of a cluster (relative 2^-11 of scores below about 8) adds about 3e-3 more.
LSE_ATOL_BF16 = 1e-2
LSE_ATOL_F32 = 1e-4


def seqs_of(wl) -> dsa.Seqs:
    return dsa.Seqs(wl.cu_q, wl.cu_k, wl.start_pos)


def to_device(wl, dev="cuda"):
    t = {k: v.to(dev) for k, v in wl.tensors.items()}
    d_c = wl.shape.d_c
    t["ckv"] = t["kv_cache"][:, :d_c]
    t["kpe"] = t["kv_cache"][:, d_c:]
    return t


def gpu_forward(wl, t, **kw):
    sh = wl.shape
    return dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], t["ckv"], t["kpe"], t["W_UK"],
                           t["W_UV"], seqs_of(wl), sh.k, sh.softmax_scale, idx_fp8=sh.idx_fp8, **kw)


def f32np(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().numpy()


def rows_by_sequence(wl, rows):
    """Group global row ids by sequence: {b: [(row, t), ...]}."""
    cu = wl.cu_q
    out = {}
    for r in rows:
        b = int(np.searchsorted(cu, r, side="right") - 1)
        while cu[b + 1] <= r:  # skip empty sequences
            b += 1
        out.setdefault(b, []).append((r, r - cu[b]))
    return out


def oracle_rows(wl, rows, with_attention=True):
    """The oracle's view of the given global rows: per row the score row,
    absolute-term row, selection, output and lse (absorbed form for the
    attention: pinned equal to the unabsorbed form)."""
    sh = wl.shape
    T = wl.tensors
    res = {}
    for b, items in rows_by_sequence(wl, rows).items():
        k0, k1 = wl.cu_k[b], wl.cu_k[b + 1]
        q0 = wl.cu_q[b]
        glob = [r for r, _ in items]
        loc = [t for _, t in items]
        pos = np.array([wl.start_pos[b] + t for t in loc], np.int64)
        qI = f32np(T["qI"][glob])
        kI = f32np(T["kI"][k0:k1])
        if sh.idx_fp8:
            qc, qe = oracle.quant_e4m3_ue8m0(qI.reshape(-1, 128))
            qI = oracle.dequant_e4m3(qc, qe).reshape(qI.shape)
            kc, ke = oracle.quant_e4m3_ue8m0(kI)
            kI = oracle.dequant_e4m3(kc, ke).reshape(kI.shape)
        w = f32np(T["w"][glob])
        scores, absterm = oracle.indexer_scores(qI, w, kI, pos, with_absterm=True)
        idx = oracle.topk(scores, pos, sh.k)
        entry = dict(scores=scores, absterm=absterm, idx=idx, pos=pos, b=b)
        if with_attention:
            cache = f32np(T["kv_cache"][k0:k1])
            out, lse = oracle.sparse_mla_absorbed(f32np(T["q_nope"][glob]), f32np(T["q_pe"][glob]),
                                                  cache[:, :sh.d_c], cache[:, sh.d_c:], f32np(T["W_UK"]),
                                                  f32np(T["W_UV"]), idx, pos, sh.softmax_scale)
            entry["out"], entry["lse"] = out, lse
        for i, r in enumerate(glob):
            row = dict(scores=scores[i], absterm=absterm[i], idx=idx[i], pos=int(pos[i]), b=b)
            if with_attention:
                row["out"], row["lse"] = entry["out"][i], entry["lse"][i]
            res[r] = row
    return res


def score_band(ref, absterm):
    """The allowed |gpu - ref| of each score."""
    return SCORE_RTOL * np.abs(ref) + SCORE_ATOL_A * absterm


def check_score_row(gpu_row, ref_row, abs_row, p, S):
    """gpu_row: the first S columns of the GPU score row.  Returns the row's
    error statistics: the largest error over its band ("ratio", <= 1), over A
    ("err_over_A") and relative to |ref| where |ref| >= 1e-2 A ("rel")."""
    gpu_row = np.asarray(gpu_row, np.float64)
    causal = slice(0, p + 1)
    fut = gpu_row[p + 1:S]
    assert np.all(np.isneginf(fut)), "future keys must be -inf"
    g, r, a = gpu_row[causal], ref_row[causal], abs_row[causal]
    assert np.all(np.isfinite(g)), "causal scores must be finite"
    band = score_band(r, a)
    err = np.abs(g - r)
    bad = err > band
    assert not bad.any(), (f"{bad.sum()} scores out of tolerance; worst err {err[bad].max():.3e} "
                           f"(band {band[bad][err[bad].argmax()]:.3e})")
    pos = a > 0
    big = np.abs(r) >= 1e-2 * a
    big &= pos
    return {"ratio": float((err[pos] / band[pos]).max()) if pos.any() else 0.0,
            "err_over_A": float((err[pos] / a[pos]).max()) if pos.any() else 0.0,
            "rel": float((err[big] / np.abs(r[big])).max()) if big.any() else 0.0}


def merge_stats(acc, st):
    for key, v in st.items():
        acc[key] = max(acc.get(key, 0.0), v)
    return acc


def check_selection_row(gpu_idx, ref_scores, ref_abs, p, k):
    gpu_idx = np.asarray(gpu_idx)
    n = min(k, p + 1)
    live = gpu_idx[:n]
    assert np.all(gpu_idx[n:] == -1), "padding must be -1"
    assert np.all((live >= 0) & (live <= p)), "selected keys must be causal"
    assert len(np.unique(live)) == n, "duplicate keys in the selection"
    causal = ref_scores[:p + 1]
    order = np.lexsort((np.arange(p + 1), -causal))
    ref_set = set(order[:n].tolist())
    gpu_set = set(live.tolist())
    if ref_set == gpu_set:
        return 0
    s_n = causal[order[n - 1]]
    tau = SCORE_RTOL * abs(s_n) + SCORE_ATOL_A * ref_abs[order[n - 1]]
    diff = ref_set ^ gpu_set
    far = [s for s in diff if abs(causal[s] - s_n) > tau]
    assert not far, f"selection differs outside the tie band: keys {far[:8]}"
    return len(diff)


def cpu_topk_same_buffer(score_row, p, k):
    """The top-k of an fp32 buffer on the CPU: value descending, then key
    ascending; -0.0 and +0.0 are equal."""
    causal = np.asarray(score_row[:p + 1], np.float32).astype(np.float64) + 0.0
    order = np.lexsort((np.arange(p + 1), -causal))
    n = min(k, p + 1)
    return order[:n]
