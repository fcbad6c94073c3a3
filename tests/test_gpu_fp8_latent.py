"""The sparse attention over an FP8 latent cache (e4m3 codes + one ue8m0 scale
per 128 latent values, k_pe in bf16), on the GPU:

  * against the oracle's attention over the dequantised cache (code * scale,
    exact in bf16), under the attention tolerance;
  * bit-identical to the bf16 kernel run on a bf16 cache that holds the same
    dequantised values (the dequantisation in the gather is exact, so nothing
    after it may differ);
  * through dsa_forward (kv_fp8), with the selection made by the indexer.
"""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import oracle
import sparse_latent_attention_indexer_gb300 as dsa
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _fp8_cache(t, d_c=512):
    """(codes [S, d_c] uint8, scales [S, d_c/128] fp32, the dequantised latent as bf16)."""
    lat = t["ckv"].contiguous()
    codes, scales = dsa.dsa_quant_e4m3_ue8m0(lat)
    deq = codes.view(torch.float8_e4m3fn).float() * scales.view(-1, d_c // 128).repeat_interleave(128, dim=1)
    return codes, scales.view(-1, d_c // 128), deq.to(torch.bfloat16)


@pytest.mark.parametrize("case", ["decode", "prefill"])
def test_fp8_latent_attention_matches_oracle_and_bf16_kernel(case):
    if case == "decode":
        g = torch.Generator().manual_seed(61)
        S = [int(x) for x in torch.randint(300, 6000, (20,), generator=g)]
        wl = di.generate("fp8kv-decode", di.FULL, 61, [1] * len(S), S, [s - 1 for s in S])
    else:
        wl = di.generate("fp8kv-prefill", di.FULL, 62, [300, 90], [300, 2200], [0, 2110])
    t = H.to_device(wl)
    sh = wl.shape
    sel = di.random_selection(wl, seed=7, density=0.7).cuda()
    codes, scales, deq = _fp8_cache(t)
    # the quantiser's codes are the oracle's
    oc, oe = oracle.quant_e4m3_ue8m0(t["ckv"].float().cpu().numpy())
    assert np.array_equal(codes.cpu().numpy().reshape(-1, 128), oc)
    out8, lse8 = dsa.dsa_sparse_mla_fwd_fp8kv(t["q_nope"], t["q_pe"], codes, scales, t["kpe"], t["W_UK"], t["W_UV"],
                                              sel, H.seqs_of(wl), sh.softmax_scale)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert "mla_tc" in dsa.last_kernels()
    # the bf16 kernel on the same values, bit for bit
    out_b, lse_b = dsa.dsa_sparse_mla_fwd(t["q_nope"], t["q_pe"], deq, t["kpe"], t["W_UK"], t["W_UV"], sel,
                                          H.seqs_of(wl), sh.softmax_scale)
    assert torch.equal(out8, out_b) and torch.equal(lse8, lse_b)
    # the oracle over the dequantised latent
    deq_np = oracle.dequant_e4m3(oc, oe).reshape(-1, sh.d_c)
    kpe_np = t["kpe"].float().cpu().numpy()
    sel_np = sel.cpu().numpy()
    rows = list(range(0, wl.total_q, max(1, wl.total_q // 24)))
    for b, items in H.rows_by_sequence(wl, rows).items():
        k0, k1 = wl.cu_k[b], wl.cu_k[b + 1]
        glob = [r for r, _ in items]
        pos = [wl.start_pos[b] + tt for _, tt in items]
        ref, lse_ref = oracle.sparse_mla_absorbed(
            t["q_nope"][glob].float().cpu().numpy(), t["q_pe"][glob].float().cpu().numpy(), deq_np[k0:k1],
            kpe_np[k0:k1], t["W_UK"].float().cpu().numpy(), t["W_UV"].float().cpu().numpy(), sel_np[glob], pos,
            sh.softmax_scale)
        err = np.abs(out8[glob].float().cpu().numpy() - ref).max()
        assert err <= H.OUT_ATOL_BF16, f"max abs err {err:.3e}"
        assert np.abs(lse8[glob].cpu().numpy() - lse_ref).max() <= H.LSE_ATOL_BF16


def test_forward_with_fp8_latent_cache():
    wl = di.generate("fp8kv-forward", di.Shape(k=64), 63, [96, 40, 700], [96, 300, 900], [0, 260, 200])
    t = H.to_device(wl)
    codes, scales, deq = _fp8_cache(t)
    out8, lse8, idx8 = dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], codes, t["kpe"], t["W_UK"],
                                       t["W_UV"], H.seqs_of(wl), wl.shape.k, wl.shape.softmax_scale, kv_scale=scales)
    assert dsa.dsa_check_device_error() == (0, 0)
    out_b, lse_b, idx_b = dsa.dsa_forward(t["qI"], t["kI"], t["w"], t["q_nope"], t["q_pe"], deq, t["kpe"],
                                          t["W_UK"], t["W_UV"], H.seqs_of(wl), wl.shape.k, wl.shape.softmax_scale)
    assert torch.equal(idx8, idx_b)
    assert torch.equal(out8, out_b) and torch.equal(lse8, lse_b)
