"""Failure detection on the GPU without a GPU fault: a kernel's bounded wait on
a barrier phase that nothing completes gives up after its limit, records its
site in the device error word and returns.  The host reads DSA_ERR_TIMEOUT and
the site, the word is cleared, and the next calls run normally."""
import pytest
import torch

import sparse_latent_attention_indexer_gb300 as dsa
from sparse_latent_attention_indexer_gb300 import _abi

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_its_site():
    assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    # about a millisecond of SM clock: the wait ends by itself
    dsa.dsa_selftest_bounded_wait(2_000_000, flag)
    assert "selftest" in dsa.last_kernels()
    st, site = dsa.dsa_check_device_error()
    assert st == _abi.DSA_ERR_TIMEOUT and site == 90
    assert int(flag.item()) == 1  # the wait gave up, and a wait on a completed phase succeeded
    # the word was cleared and the context is usable
    assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
    scores = torch.randn((3, 64), device="cuda")
    idx = dsa.dsa_topk_select(scores, dsa.Seqs([0, 3], [0, 64], [61]), 8)
    torch.cuda.synchronize()
    assert idx.shape == (3, 8) and bool((idx >= 0).all())
    assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)


def test_production_kernels_give_up_and_recover():
    """The failure path of the production tensor-core kernels (indexer, top-k
    input, absorption, sparse attention): with a wait limit of 64 SM cycles the
    first wait that is not already satisfied gives up, the CTA records its site,
    drains what it has in flight, frees its tensor memory and exits.  The host
    reads DSA_ERR_TIMEOUT and a production site; with the limit restored the
    same call matches the oracle."""
    import numpy as np

    import dsa_inputs as di
    from tests import helpers as H

    wl = di.generate("abort-path", di.Shape(k=64), 5, [96, 40], [96, 300], [0, 260])
    t = H.to_device(wl)
    assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
    try:
        dsa.dsa_set_wait_limit(64)
        H.gpu_forward(wl, t)
        launched = dsa.last_kernels()
        st, site = dsa.dsa_check_device_error()
    finally:
        dsa.dsa_set_wait_limit(0)
    assert {"indexer_tc", "absorb_tc", "mla_tc"} <= launched, launched
    assert st == _abi.DSA_ERR_TIMEOUT, st
    assert 1 <= site <= 40, site  # a production kernel's site (the self-test uses 90 and 91)
    assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
    out, lse, idx = H.gpu_forward(wl, t)
    assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
    ref = H.oracle_rows(wl, list(range(wl.total_q)))
    out_np, idx_np = out.float().cpu().numpy(), idx.cpu().numpy()
    for r, o in ref.items():
        H.check_selection_row(idx_np[r], o["scores"], o["absterm"], o["pos"], wl.shape.k)
        assert float(np.abs(out_np[r] - o["out"]).max()) <= H.OUT_ATOL_BF16
    with pytest.raises(dsa.DSAError):
        dsa.dsa_set_wait_limit(-1)


def test_fused_indexer_topk_and_gemm_give_up_and_recover():
    """The same failure path through the kernels of the chunked-prefill configuration: the fused FP8
    indexer + top-k (its producer, MMA, epilogue and six selecting warps), the attention and the
    output-projection GEMM, with a 64-cycle wait limit: a production site is reported and every kernel
    returns; with the limit restored the selection equals the unfused path's exactly."""
    import math

    import dsa_inputs as di
    from tests import helpers as H
    from tests.test_gpu_fused_topk import _unfused_idx

    shape = di.Shape(k=256, idx_fp8=True)
    wl = di.generate("abort-fused", shape, 6, [700, 513, 900], [3000, 513, 5000], [2300, 0, 4100])
    t = H.to_device(wl)
    g = torch.Generator().manual_seed(7)
    wo = (torch.randn(512, shape.H * shape.d_v, generator=g) / math.sqrt(shape.H * shape.d_v)).to(torch.bfloat16)
    wo = wo.cuda()
    assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
    dsa.dsa_set_fused_topk(True)
    try:
        try:
            dsa.dsa_set_wait_limit(64)
            H.gpu_forward(wl, t, wo=wo)
            launched = dsa.last_kernels()
            st, site = dsa.dsa_check_device_error()
        finally:
            dsa.dsa_set_wait_limit(0)
        assert {"indexer_topk", "mla_tc", "gemm_tc"} <= launched, launched
        assert st == _abi.DSA_ERR_TIMEOUT, st
        assert 1 <= site <= 60, site
        assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
        out, lse, idx, y = H.gpu_forward(wl, t, wo=wo)
        assert dsa.dsa_check_device_error() == (_abi.DSA_OK, 0)
    finally:
        dsa.dsa_set_fused_topk(-1)
    assert torch.equal(idx, _unfused_idx(wl, t))
