"""dsa_sparse_mla_fwd_noalloc: the attention entry point for callers that
cannot give the library a workspace (e.g. a runtime that owns all device
memory through its own pool and hands a plugin only input and output
tensors).  It must give the same result as dsa_sparse_mla_fwd, call after
call, while using the library's reserved scratch; and it must refuse a call
that needs more scratch than it reserves, without launching anything.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test; it also passes on its own in a
fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import dsa_inputs as di
import sparse_latent_attention_indexer_gb300 as dsa
from sparse_latent_attention_indexer_gb300 import _abi
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _decode_batch(seed, n=24):
    """A decode step: n sequences with one query each, at the 671B head
    shapes, and a seeded selection of up to 2048 keys per query."""
    g = torch.Generator().manual_seed(seed)
    S = [int(x) for x in torch.randint(200, 5000, (n,), generator=g)]
    wl = di.generate(f"noalloc-{seed}", di.FULL, seed, [1] * len(S), S, [s - 1 for s in S])
    sel = di.random_selection(wl, seed=seed + 1, density=0.6)
    return wl, H.to_device(wl), sel.cuda()


def _noalloc(wl, t, sel, out, lse):
    sh = wl.shape
    lib = _abi.load()
    seqs = H.seqs_of(wl)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dsa_sparse_mla_fwd_noalloc(
        ctypes.c_void_p(t["q_nope"].data_ptr()), ctypes.c_void_p(t["q_pe"].data_ptr()), _abi.DSA_BF16,
        ctypes.c_void_p(t["ckv"].data_ptr()), t["ckv"].stride(0), ctypes.c_void_p(t["kpe"].data_ptr()),
        t["kpe"].stride(0), ctypes.c_void_p(t["W_UK"].data_ptr()), ctypes.c_void_p(t["W_UV"].data_ptr()),
        sh.H, sh.d_n, sh.d_r, sh.d_c, sh.d_v, ctypes.c_void_p(sel.data_ptr()), sel.shape[1], seqs.ref(),
        ctypes.c_float(sh.softmax_scale), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)


def test_noalloc_zero_rows_is_set_up_only():
    """A call with no query rows does the per-device set-up and launches nothing."""
    wl, t, sel = _decode_batch(40, n=2)
    empty = di.Workload("empty", wl.shape, 0, [0], [16], [0], {})
    st = _noalloc(empty, t, sel, torch.empty(0, device="cuda"), torch.empty(0, device="cuda"))
    assert st == _abi.DSA_OK, _abi.load().dsa_status_string(st)
    assert _abi.load().dsa_last_launch_count() == 0


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    # two calls in a row; the second is the largest batch the scratch holds (128 rows)
    batches = [_decode_batch(41), _decode_batch(42, n=128)]
    for wl, t, sel in batches:  # two calls in a row, different inputs
        sh = wl.shape
        ref_out, ref_lse = dsa.dsa_sparse_mla_fwd(t["q_nope"], t["q_pe"], t["ckv"], t["kpe"], t["W_UK"], t["W_UV"],
                                                  sel, H.seqs_of(wl), sh.softmax_scale)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _noalloc(wl, t, sel, out, lse)
        assert st == _abi.DSA_OK, _abi.load().dsa_status_string(st)
        torch.cuda.synchronize()
        err = (out.float() - ref_out.float()).abs().max().item()
        assert err <= H.OUT_ATOL_BF16, f"max abs difference {err:.3e}"
        assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=0, atol=H.LSE_ATOL_BF16)


def test_noalloc_rejects_calls_beyond_its_scratch():
    wl, t, sel = _decode_batch(43)
    sh = wl.shape
    rows = 4096  # needs far more than DSA_NOALLOC_SCRATCH_BYTES at these head shapes
    need = dsa.dsa_sparse_mla_workspace_size(_abi.DSA_BF16, sh.H, sh.d_n, sh.d_r, sh.d_c, sh.d_v, sh.k,
                                             dsa.Seqs([0, rows], [0, rows], [0]))
    assert need > _abi.DSA_NOALLOC_SCRATCH_BYTES
    big = di.Workload("big", sh, 0, [rows], [rows], [0], {})
    # Real buffers of the full size, so that even a wrongly accepted call would stay in bounds.
    tb = {
        "q_nope": torch.zeros((rows, sh.H, sh.d_n), dtype=torch.bfloat16, device="cuda"),
        "q_pe": torch.zeros((rows, sh.H, sh.d_r), dtype=torch.bfloat16, device="cuda"),
        "W_UK": t["W_UK"], "W_UV": t["W_UV"],
    }
    cache = torch.zeros((rows, sh.d_c + sh.d_r), dtype=torch.bfloat16, device="cuda")
    tb["ckv"], tb["kpe"] = cache[:, :sh.d_c], cache[:, sh.d_c:]
    sel_b = torch.full((rows, sh.k), -1, dtype=torch.int32, device="cuda")
    out = torch.zeros((rows, sh.H, sh.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((rows, sh.H), dtype=torch.float32, device="cuda")
    st = _noalloc(big, tb, sel_b, out, lse)
    assert st == _abi.DSA_ERR_WORKSPACE
    assert _abi.load().dsa_last_launch_count() == 0
