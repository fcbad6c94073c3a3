"""Every option of dsa_forward at once on one ragged batch: the FP8 indexer (e4m3 + ue8m0), the fused
indexer + top-k kernel, the FP8 latent cache and the output projection wo, with a dense-only sequence,
a decode row and chunked-prefill rows in the same launch.  Each option must change nothing but what it
is for:
  * the selection equals the unfused path's (indexer scores, then the top-k kernel) exactly;
  * the attention output over the e4m3 latent cache equals, bit for bit, the forward over a bf16 cache
    that holds the dequantised values (the dequantisation in the gather is exact);
  * y is wo applied to that output (within the GEMM's bf16 rounding);
  * sampled rows match the oracle's whole path on the dequantised cache."""
import math

import numpy as np
import pytest
import torch

import dsa_inputs as di
import sparse_latent_attention_indexer_gb300 as dsa
from tests import helpers as H
from tests.test_gpu_fp8_latent import _fp8_cache
from tests.test_gpu_fused_topk import _unfused_idx
from tests.test_gpu_projections import _check_linear

pytestmark = pytest.mark.gpu


def test_fp8_indexer_fused_topk_fp8_latent_and_wo_together():
    shape = di.Shape(k=256, idx_fp8=True)
    # enough query groups (at least two per SM) for the fused kernel to take the batch
    T, S, P = [700, 1, 90, 900], [3000, 5000, 90, 6200], [2300, 4999, 0, 5300]
    wl = di.generate("all-options", shape, 81, T, S, P)
    sh = wl.shape
    t = H.to_device(wl)
    codes, scales, deq = _fp8_cache(t)
    g = torch.Generator().manual_seed(82)
    d_model = 1024
    wo = (torch.randn(d_model, sh.H * sh.d_v, generator=g) / math.sqrt(sh.H * sh.d_v)).to(torch.bfloat16).cuda()
    seqs = H.seqs_of(wl)
    dsa.dsa_set_fused_topk(True)
    try:
        out8, lse8, idx8, y8 = dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], codes, t["kpe"],
                                               t["W_UK"], t["W_UV"], seqs, sh.k, sh.softmax_scale, idx_fp8=True,
                                               kv_scale=scales, wo=wo)
        kern = dsa.last_kernels()
    finally:
        dsa.dsa_set_fused_topk(-1)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert {"indexer_topk", "quant", "mla_tc", "gemm_tc"} <= kern, kern
    # the selection: the unfused path on the same inputs
    assert torch.equal(idx8, _unfused_idx(wl, t))
    # the attention: the bf16 path on the dequantised cache, bit for bit (same selection)
    out_b, lse_b, idx_b = dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], deq, t["kpe"],
                                          t["W_UK"], t["W_UV"], seqs, sh.k, sh.softmax_scale, idx_fp8=True)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert torch.equal(idx_b, idx8) and torch.equal(out_b, out8) and torch.equal(lse_b, lse8)
    # y = out wo^T on sampled rows
    rows = list(range(0, wl.total_q, 29)) + [wl.total_q - 1]
    _check_linear(y8[rows], out8.reshape(wl.total_q, -1), wo, rows)
    # the oracle's whole path on sampled rows (its cache is the dequantised one)
    wl.tensors["kv_cache"][:, :sh.d_c] = deq.cpu()
    sample = di.sample_rows(wl, 24)
    ref = H.oracle_rows(wl, sample)
    idx_np, out_np = idx8.cpu().numpy(), out8.float().cpu().numpy()
    for r in sample:
        o = ref[r]
        H.check_selection_row(idx_np[r], o["scores"], o["absterm"], o["pos"], sh.k)
        assert np.abs(out_np[r] - o["out"]).max() <= H.OUT_ATOL_BF16
