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
