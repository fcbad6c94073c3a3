"""The five workloads at their full sizes, in the launch configuration the
bench times (one dsa_forward over the whole batch), checked on sampled rows
that the oracle computes one by one: the selection (tie band), the output
(max-abs), and the indexer scores of a few rows (through dsa_indexer_scores
on that row alone, same kernels)."""
import gc

import numpy as np
import pytest
import torch

import dsa_inputs as di
import sparse_latent_attention_indexer_gb300 as dsa
from tests import helpers as H

pytestmark = pytest.mark.gpu

SAMPLE = {0: 256, 1: 40, 2: 16, 3: 16, 4: 16}
SCORE_ROWS = 6


def _row_scores(wl, t, r, b):
    k0, k1 = wl.cu_k[b], wl.cu_k[b + 1]
    p = wl.start_pos[b] + (r - wl.cu_q[b])
    seqs = dsa.Seqs([0, 1], [0, k1 - k0], [p])
    q, k, w = t["qI"][r:r + 1], t["kI"][k0:k1], t["w"][r:r + 1]
    if wl.shape.idx_fp8:
        qc, qs = dsa.dsa_quant_e4m3_ue8m0(q)
        kc, ks = dsa.dsa_quant_e4m3_ue8m0(k)
        return dsa.dsa_indexer_scores(qc, kc, w, seqs, q_scale=qs, k_scale=ks)[0].cpu().numpy(), p
    return dsa.dsa_indexer_scores(q, k, w, seqs)[0].cpu().numpy(), p


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_workload(cfg):
    wl = di.workload(cfg)
    t = H.to_device(wl)
    out, lse, idx = H.gpu_forward(wl, t)
    st, site = dsa.dsa_check_device_error()
    assert st == 0, (st, site)
    rows = di.sample_rows(wl, SAMPLE[cfg])
    ref = H.oracle_rows(wl, rows)
    out_np = out[rows].float().cpu().numpy()
    idx_np = idx[rows].cpu().numpy()
    lse_np = lse[rows].cpu().numpy()
    atol = H.OUT_ATOL_F32 if wl.shape.dtype == "f32" else H.OUT_ATOL_BF16
    swaps = 0
    for i, r in enumerate(rows):
        o = ref[r]
        swaps += H.check_selection_row(idx_np[i], o["scores"], o["absterm"], o["pos"], wl.shape.k)
        err = float(np.abs(out_np[i] - o["out"]).max())
        assert err <= atol, f"cfg {cfg} row {r}: max abs err {err:.3e}"
        assert np.all(np.isfinite(lse_np[i]))
    for r in rows[:: max(1, len(rows) // SCORE_ROWS)][:SCORE_ROWS]:
        o = ref[r]
        S = wl.S[o["b"]]
        sc, p = _row_scores(wl, t, r, o["b"])
        H.check_score_row(sc[:S], o["scores"], o["absterm"], p, S)
    print(f"cfg {cfg}: {len(rows)} rows ok, {swaps} near-tie swaps, kernels {sorted(dsa.last_kernels())}")
    del t, out, lse, idx
    gc.collect()
    torch.cuda.empty_cache()
