"""The fused indexer + top-k (one persistent kernel: each SM scores a group of
4 query rows into its own slot and selects their top-k from it) against the
unfused path on the same inputs: dsa_indexer_scores over the whole batch, then
dsa_topk_select on that buffer.  Both compute the same fp32 scores and apply
the same selection rule, so the index rows must be identical -- same keys, same
order, ties at the k-th score resolved to the lower key index -- including
rows that see at most k keys (dense), rows whose candidates overflow the
candidate list (all scores equal), and a ragged batch of sequences with
different prefixes.  The oracle then checks a sample of the fused rows."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import sparse_latent_attention_indexer_gb300 as dsa
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _unfused_idx(wl, t):
    sh = wl.shape
    seqs = H.seqs_of(wl)
    q, k, qs, ks = t["qI"], t["kI"], None, None
    if sh.idx_fp8:
        q, qs = dsa.dsa_quant_e4m3_ue8m0(t["qI"])
        k, ks = dsa.dsa_quant_e4m3_ue8m0(t["kI"])
    scores = dsa.dsa_indexer_scores(q, k, t["w"], seqs, q_scale=qs, k_scale=ks)
    return dsa.dsa_topk_select(scores, seqs, sh.k)


@pytest.mark.parametrize("fp8", [False, True])
def test_fused_selection_equals_unfused(fp8):
    shape = di.Shape(k=256, idx_fp8=fp8)
    T, S, P = [700, 513, 900, 130], [3000, 513, 5000, 10000], [2300, 0, 4100, 9870]
    wl = di.generate(f"fused-{fp8}", shape, 31, T, S, P)
    # rows of the last sequence get zero weights: every score 0, so ties decide the whole row and
    # its candidates (all 10000 keys) overflow the candidate list
    r0 = wl.cu_q[3]
    wl.tensors["w"][r0:r0 + 40] = 0.0
    t = H.to_device(wl)
    dsa.dsa_set_fused_topk(True)
    try:
        out, lse, idx = H.gpu_forward(wl, t)
        kern = dsa.last_kernels()
    finally:
        dsa.dsa_set_fused_topk(-1)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert "indexer_topk" in kern and "topk" not in kern, kern
    ref = _unfused_idx(wl, t)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert torch.equal(idx, ref)
    # a zero-weight row selects keys 0 .. k-1
    assert torch.equal(idx[r0], torch.arange(shape.k, dtype=torch.int32, device=idx.device))
    # dense rows (the second sequence's first k rows see at most k keys)
    r1 = wl.cu_q[1]
    for t_ in (0, 100, 255):
        row = idx[r1 + t_].cpu().numpy()
        assert np.array_equal(row[:t_ + 1], np.arange(t_ + 1)) and (row[t_ + 1:] == -1).all()
    rows = di.sample_rows(wl, 24)
    refo = H.oracle_rows(wl, rows)
    idx_np, out_np = idx.cpu().numpy(), out.float().cpu().numpy()
    for r in rows:
        o = refo[r]
        H.check_selection_row(idx_np[r], o["scores"], o["absterm"], o["pos"], shape.k)
        assert np.abs(out_np[r] - o["out"]).max() <= H.OUT_ATOL_BF16
