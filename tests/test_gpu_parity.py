"""GPU parity of every stage against the oracle, at sizes the oracle finishes
in seconds that still span several tiles and ragged tails, plus edge cases.
All calls go through the C ABI (libdsa.so) via the thin binding."""
import math

import numpy as np
import pytest
import torch

import dsa_inputs as di
import oracle
import sparse_latent_attention_indexer_gb300 as dsa
from tests import helpers as H

pytestmark = pytest.mark.gpu

FULL_K64 = di.Shape(k=64)
CASES = {
    # full head shapes, three sequences: ragged tile tails, start_pos > 0, rows above and below k
    "bf16-ragged": lambda: di.generate("bf16-ragged", di.FULL, 11, [300, 1, 77], [300, 2100, 2200], [0, 2099, 2123]),
    # small k so most rows select a strict subset
    "bf16-k64": lambda: di.generate("bf16-k64", FULL_K64, 12, [333], [333], [0]),
    # FP8 indexer on the ragged batch
    "fp8-ragged": lambda: di.generate("fp8-ragged", di.Shape(idx_fp8=True), 13, [129, 65], [129, 2300], [0, 2235]),
    # the tiny fp32 workload in full
    "f32-tiny": lambda: di.workload(0),
}
_cache = {}


def case(name):
    if name not in _cache:
        wl = CASES[name]()
        _cache[name] = (wl, H.to_device(wl))
    return _cache[name]


def _oracle(name):
    key = ("oracle", name)
    if key not in _cache:
        wl, _ = case(name)
        _cache[key] = H.oracle_rows(wl, list(range(wl.total_q)))
    return _cache[key]


def out_atol(wl):
    return H.OUT_ATOL_F32 if wl.shape.dtype == "f32" else H.OUT_ATOL_BF16


# ---------------------------------------------------------------------------
# quantiser: bit-exact codes and scales
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quant_bit_exact(dtype):
    g = torch.Generator().manual_seed(21)
    x = torch.randn(300, 128, generator=g) * torch.exp2(torch.randint(-30, 30, (300, 1), generator=g).float())
    x[0] = 0.0
    x[1] = 0.0
    x[1, 3] = 448.0
    x[2] = 0.0
    x[2, 100] = -448.5
    x[3] = 0.0
    x[3, 0] = 1e-38
    x[4] = -0.0
    x = x.to(dtype)
    codes, scales = dsa.dsa_quant_e4m3_ue8m0(x.cuda())
    rc, re = oracle.quant_e4m3_ue8m0(x.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), np.ldexp(1.0, re).astype(np.float32))


# ---------------------------------------------------------------------------
# indexer scores
# ---------------------------------------------------------------------------
def _gpu_scores(wl, t):
    seqs = H.seqs_of(wl)
    if wl.shape.idx_fp8:
        qc, qs = dsa.dsa_quant_e4m3_ue8m0(t["qI"])
        kc, ks = dsa.dsa_quant_e4m3_ue8m0(t["kI"])
        return dsa.dsa_indexer_scores(qc, kc, t["w"], seqs, q_scale=qs, k_scale=ks)
    return dsa.dsa_indexer_scores(t["qI"], t["kI"], t["w"], seqs)


@pytest.mark.parametrize("name", list(CASES))
def test_indexer_scores(name):
    wl, t = case(name)
    ref = _oracle(name)
    scores = _gpu_scores(wl, t).cpu().numpy()
    for r, o in ref.items():
        S = wl.S[o["b"]]
        H.check_score_row(scores[r, :S], o["scores"], o["absterm"], o["pos"], S)


# ---------------------------------------------------------------------------
# top-k: exact on the GPU's own buffer; tie band against the oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", list(CASES))
def test_topk(name):
    wl, t = case(name)
    ref = _oracle(name)
    seqs = H.seqs_of(wl)
    scores = _gpu_scores(wl, t)
    idx = dsa.dsa_topk_select(scores, seqs, wl.shape.k).cpu().numpy()
    sc = scores.cpu().numpy()
    for r, o in ref.items():
        p, k = o["pos"], wl.shape.k
        n = min(k, p + 1)
        want = H.cpu_topk_same_buffer(sc[r], p, k)
        assert sorted(idx[r, :n].tolist()) == sorted(want.tolist()), f"row {r}"
        assert np.all(idx[r, n:] == -1)
        H.check_selection_row(idx[r], o["scores"], o["absterm"], p, k)


# A launch with fewer than 2 x 152 rows of at least 8192 causal keys takes the cluster top-k kernel
# (decode: eight CTAs per row), or the wide one-CTA-per-row kernel when a row's slices would not fit
# the CTAs' shared memory; every other launch takes the filter kernel (a candidate list, or the global
# row when the list would overflow).  The cases below run on every side of those switches.
@pytest.mark.parametrize("T", [700, 100])
@pytest.mark.parametrize("fill", [1.0, 0.0, -3.5])
def test_topk_all_equal_scores(fill, T):
    """Every score equal: the lowest key indices win."""
    S = 700
    k = 100
    seqs = dsa.Seqs.from_lengths([T], [S], [S - T])
    scores = torch.full((T, S), fill, dtype=torch.float32, device="cuda")
    if fill == 0.0:
        scores[:, ::2] = -0.0  # -0 and +0 are the same score
    idx = dsa.dsa_topk_select(scores, seqs, k).cpu().numpy()
    for r in range(T):
        n = min(k, S - T + r + 1)
        assert sorted(idx[r, :n].tolist()) == list(range(n))
        assert np.all(idx[r, n:] == -1)


@pytest.mark.parametrize("rows", [24, 320])
def test_topk_threshold_ties_and_large_rows(rows):
    """Scores on a coarse grid (many exact ties at the threshold), rows up to
    65536 keys (cluster kernel for 24 rows, beyond the many-rows kernel's key
    cache for 320 rows); exact equality with the CPU top-k of the same buffer."""
    g = torch.Generator().manual_seed(5)
    S = 65536
    seqs = dsa.Seqs([0, rows], [0, S], [S - rows])
    scores = torch.randint(-40, 40, (rows, S), generator=g).float() / 8
    idx = dsa.dsa_topk_select(scores.cuda(), seqs, 2048).cpu().numpy()
    sc = scores.numpy()
    for r in range(rows):
        p = S - rows + r
        want = H.cpu_topk_same_buffer(sc[r], p, 2048)
        assert sorted(idx[r].tolist()) == sorted(want.tolist())


def test_topk_candidate_overflow_falls_back_to_the_global_row():
    """Many rows (the many-rows kernel) whose threshold bin holds more keys
    than its shared-memory candidate list: almost every score ties at 1.0 and
    a few keys score 2.0, so the select runs on the global row; exact equality
    with the CPU top-k of the same buffer (lowest indices win the ties)."""
    g = torch.Generator().manual_seed(7)
    rows, S, k = 320, 12000, 2048
    seqs = dsa.Seqs([0, rows], [0, S], [S - rows])
    scores = torch.ones((rows, S))
    hot = torch.randint(0, S, (rows, 300), generator=g)
    scores.scatter_(1, hot, 2.0)
    idx = dsa.dsa_topk_select(scores.cuda(), seqs, k).cpu().numpy()
    sc = scores.numpy()
    for r in range(rows):
        want = H.cpu_topk_same_buffer(sc[r], S - rows + r, k)
        assert sorted(idx[r].tolist()) == sorted(want.tolist())


@pytest.mark.parametrize("rows", [24, 320])
def test_topk_odd_row_stride(rows):
    """A score buffer whose rows are not 16-byte aligned (odd row stride): the
    kernels take their scalar loads; exact equality with the CPU top-k."""
    g = torch.Generator().manual_seed(8)
    S, k = 9001, 512
    seqs = dsa.Seqs([0, rows], [0, S], [S - rows])
    full = torch.randn((rows, S + 1), generator=g)
    scores = full.cuda()[:, 1:]
    assert scores.stride(0) % 4 != 0 or scores.data_ptr() % 16 != 0
    idx = dsa.dsa_topk_select(scores, seqs, k).cpu().numpy()
    sc = full[:, 1:].numpy()
    for r in range(rows):
        want = H.cpu_topk_same_buffer(sc[r], S - rows + r, k)
        assert sorted(idx[r].tolist()) == sorted(want.tolist())


def test_topk_rows_longer_than_the_cluster_cache():
    """Two rows of 400,000 causal keys (beyond eight CTAs' shared memory: the
    wide kernel, which re-reads global memory); exact equality with the CPU
    top-k of the same buffer, ties included."""
    g = torch.Generator().manual_seed(6)
    rows, S, k = 2, 400_000, 2048
    seqs = dsa.Seqs([0, rows], [0, S], [S - rows])
    scores = torch.randint(-400, 400, (rows, S), generator=g).float() / 16
    idx = dsa.dsa_topk_select(scores.cuda(), seqs, k).cpu().numpy()
    sc = scores.numpy()
    for r in range(rows):
        want = H.cpu_topk_same_buffer(sc[r], S - rows + r, k)
        assert sorted(idx[r].tolist()) == sorted(want.tolist())


# ---------------------------------------------------------------------------
# sparse attention on a seeded selection (same idx on both sides)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", list(CASES))
def test_sparse_mla_given_selection(name):
    wl, t = case(name)
    sh = wl.shape
    sel = di.random_selection(wl, seed=31, density=0.7)
    out, lse = dsa.dsa_sparse_mla_fwd(t["q_nope"], t["q_pe"], t["ckv"], t["kpe"], t["W_UK"], t["W_UV"],
                                      sel.cuda(), H.seqs_of(wl), sh.softmax_scale)
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    T = wl.tensors
    for b in range(wl.B):
        q0, q1, k0, k1 = wl.cu_q[b], wl.cu_q[b + 1], wl.cu_k[b], wl.cu_k[b + 1]
        if q0 == q1:
            continue
        pos = np.arange(wl.start_pos[b], wl.start_pos[b] + wl.T[b])
        cache = H.f32np(T["kv_cache"][k0:k1])
        ro, rl = oracle.sparse_mla_absorbed(H.f32np(T["q_nope"][q0:q1]), H.f32np(T["q_pe"][q0:q1]),
                                            cache[:, :sh.d_c], cache[:, sh.d_c:], H.f32np(T["W_UK"]),
                                            H.f32np(T["W_UV"]), sel[q0:q1].numpy(), pos, sh.softmax_scale)
        err = np.abs(out[q0:q1] - ro).max()
        assert err <= out_atol(wl), f"seq {b}: max abs err {err:.3e}"
        assert np.allclose(lse[q0:q1], rl, rtol=0, atol=H.LSE_ATOL_BF16 if sh.dtype == "bf16" else H.LSE_ATOL_F32)


def test_sparse_mla_masked_rows_and_out_of_window_indices():
    """A row whose selection holds only -1, future or out-of-range keys has
    no live key: out = 0, lse = -inf.  Such entries inside a row are ignored."""
    wl, t = case("bf16-k64")
    sh = wl.shape
    k = sh.k
    sel = torch.full((wl.total_q, k), -1, dtype=torch.int32)
    sel[5, :3] = torch.tensor([6, 7, 100000])     # row 5 (p = 5): all masked
    sel[9, :4] = torch.tensor([2, 10, -7, 4])     # row 9: keys 2 and 4 live
    out, lse = dsa.dsa_sparse_mla_fwd(t["q_nope"], t["q_pe"], t["ckv"], t["kpe"], t["W_UK"], t["W_UV"], sel.cuda(),
                                      H.seqs_of(wl), sh.softmax_scale)
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(out[5] == 0) and np.all(np.isneginf(lse[5]))
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    T = wl.tensors
    cache = H.f32np(T["kv_cache"])
    ro, rl = oracle.sparse_mla_absorbed(H.f32np(T["q_nope"][9:10]), H.f32np(T["q_pe"][9:10]), cache[:, :sh.d_c],
                                        cache[:, sh.d_c:], H.f32np(T["W_UK"]), H.f32np(T["W_UV"]),
                                        np.array([[2, 4]], np.int32), np.array([9]), sh.softmax_scale)
    assert np.abs(out[9] - ro[0]).max() <= H.OUT_ATOL_BF16


# ---------------------------------------------------------------------------
# the whole path
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", list(CASES))
def test_forward_end_to_end(name):
    wl, t = case(name)
    ref = _oracle(name)
    out, lse, idx = H.gpu_forward(wl, t)
    out, idx = out.float().cpu().numpy(), idx.cpu().numpy()
    for r, o in ref.items():
        H.check_selection_row(idx[r], o["scores"], o["absterm"], o["pos"], wl.shape.k)
    err = max(np.abs(out[r] - o["out"]).max() for r, o in ref.items())
    assert err <= out_atol(wl), f"max abs err {err:.3e}"


def test_forward_dense_when_k_covers_the_sequence():
    """k >= S: every causal key is selected (rows keep t + 1 keys) and the
    result is plain causal attention (nnterp deepseek_v32 note)."""
    wl = di.generate("dense", di.Shape(k=512), 14, [200], [200], [0])
    t = H.to_device(wl)
    out, _, idx = H.gpu_forward(wl, t)
    idx = idx.cpu().numpy()
    assert ((idx >= 0).sum(1) == np.arange(1, 201)).all()
    sh = wl.shape
    T = wl.tensors
    cache = H.f32np(T["kv_cache"])
    KC, V = oracle.kv_up(cache[:, :sh.d_c], H.f32np(T["W_UK"]), H.f32np(T["W_UV"]))
    rows = [0, 1, 57, 199]
    ref, _ = oracle.dense_masked_mla(H.f32np(T["q_nope"][rows]), H.f32np(T["q_pe"][rows]), KC, cache[:, sh.d_c:], V,
                                     np.array(rows), sh.softmax_scale)
    assert np.abs(out.float().cpu().numpy()[rows] - ref).max() <= H.OUT_ATOL_BF16


INDEXER_AND_TOPK = {"quant", "indexer_simt", "indexer_tc", "indexer_fp8", "topk", "indexer_topk"}


@pytest.mark.parametrize("shape", ["bf16", "fp8", "f32"])
def test_forward_dense_batch_launches_no_indexer_or_topk(shape):
    """Every row of the batch sees at most k keys (k >= S; the second sequence
    continues at position 100 with 37 rows): the selection is every causal key,
    known without scores, so no quantiser, indexer or top-k kernel runs.  The
    index output is the dense pattern the top-k writes for such rows, and the
    outputs match the oracle's whole path on sampled rows."""
    sh = {"bf16": di.Shape(k=512), "fp8": di.Shape(k=512, idx_fp8=True),
          "f32": di.workload(0).shape}[shape]
    if shape == "f32":
        wl = di.generate("dense-f32", sh, 16, [40, 9], [40, 70], [0, 55])   # k = 64 covers p + 1 <= 64
    else:
        wl = di.generate("dense-" + shape, sh, 15, [200, 37], [200, 300], [0, 100])
    t = H.to_device(wl)
    out, lse, idx = H.gpu_forward(wl, t)
    kernels = dsa.last_kernels()
    assert not kernels & INDEXER_AND_TOPK, kernels
    assert "dense_idx" in kernels, kernels
    idx = idx.cpu().numpy()
    for b in range(wl.B):
        for tt in range(wl.T[b]):
            r, p = wl.cu_q[b] + tt, wl.start_pos[b] + tt
            n = min(p + 1, wl.S[b])
            want = np.full(sh.k, -1, np.int32)
            want[:n] = np.arange(n)
            assert np.array_equal(idx[r], want), (b, tt)
    rows = [0, 1, wl.cu_q[1] - 1, wl.cu_q[1], wl.cu_q[2] - 1]
    ref = H.oracle_rows(wl, rows)
    out = out.float().cpu().numpy()
    err = max(np.abs(out[r] - o["out"]).max() for r, o in ref.items())
    assert err <= out_atol(wl), f"max abs err {err:.3e}"


@pytest.mark.parametrize("name", ["bf16-ragged", "f32-tiny"])
def test_sparse_mla_null_selection_is_the_dense_causal_one(name):
    """idx = NULL means entry e of a row is key e: bit-identical to passing the
    explicit selection 0 .. min(k, p+1, S)-1 followed by -1 padding."""
    wl, t = case(name)
    sh = wl.shape
    explicit = np.full((wl.cu_q[-1], sh.k), -1, np.int32)
    for b in range(wl.B):
        for tt in range(wl.T[b]):
            n = min(sh.k, wl.start_pos[b] + tt + 1, wl.S[b])
            explicit[wl.cu_q[b] + tt, :n] = np.arange(n)
    args = (t["q_nope"], t["q_pe"], t["ckv"], t["kpe"], t["W_UK"], t["W_UV"])
    o1, l1 = dsa.dsa_sparse_mla_fwd(*args, torch.from_numpy(explicit).cuda(), H.seqs_of(wl), sh.softmax_scale)
    o2, l2 = dsa.dsa_sparse_mla_fwd(*args, None, H.seqs_of(wl), sh.softmax_scale, k=sh.k)
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


def test_forward_yarn_scale_and_empty_sequence():
    """The released model's YaRN-scaled softmax scale 0.1352, and a batch
    holding an empty sequence (T = 0) between two others."""
    sh = di.Shape(k=128, softmax_scale=192 ** -0.5 * (0.1 * math.log(40) + 1) ** 2)
    wl = di.generate("yarn", sh, 15, [40, 0, 3], [300, 50, 200], [260, 10, 197])
    t = H.to_device(wl)
    ref = H.oracle_rows(wl, list(range(wl.total_q)))
    out, _, idx = H.gpu_forward(wl, t)
    out, idx = out.float().cpu().numpy(), idx.cpu().numpy()
    for r, o in ref.items():
        H.check_selection_row(idx[r], o["scores"], o["absterm"], o["pos"], sh.k)
        assert np.abs(out[r] - o["out"]).max() <= H.OUT_ATOL_BF16


def test_forward_deterministic():
    wl, t = case("bf16-ragged")
    a = H.gpu_forward(wl, t)
    b = H.gpu_forward(wl, t)
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])
    assert torch.equal(a[1], b[1])


@pytest.mark.parametrize("rows", [256, 24])
def test_sparse_mla_repeatable_over_runs(rows):
    """Long selections (about 32 key tiles per row) run eight times in a row:
    every run is bit-identical and sampled rows match the oracle.  The two
    CTAs of a row exchange partial scores through double-buffered shared
    memory every tile, so a buffer reused before its transfer finished shows
    up as run-to-run differences in a few rows.  24 rows take the split path
    (several clusters per row plus the merge kernel)."""
    wl = di.generate("repeat", di.FULL, 17, [rows], [4096], [4096 - rows])
    t = H.to_device(wl)
    sh = wl.shape
    sel = di.random_selection(wl, seed=5, density=0.7)
    seqs = H.seqs_of(wl)
    sel_d = sel.cuda()
    runs = [dsa.dsa_sparse_mla_fwd(t["q_nope"], t["q_pe"], t["ckv"], t["kpe"], t["W_UK"], t["W_UV"], sel_d, seqs,
                                   sh.softmax_scale) for _ in range(8)]
    for k, (o, l) in enumerate(runs[1:], 1):
        bad = (o != runs[0][0]).flatten(1).any(1).nonzero().flatten().tolist()
        assert not bad and torch.equal(l, runs[0][1]), f"run {k} differs from run 0 in rows {bad[:8]}"
    sample = sorted({0, rows // 3, rows // 2, rows - 1})
    T = wl.tensors
    pos = np.array([wl.start_pos[0] + r for r in sample], np.int64)
    cache = H.f32np(T["kv_cache"])
    ro, rl = oracle.sparse_mla_absorbed(H.f32np(T["q_nope"][sample]), H.f32np(T["q_pe"][sample]), cache[:, :sh.d_c],
                                        cache[:, sh.d_c:], H.f32np(T["W_UK"]), H.f32np(T["W_UV"]),
                                        sel[sample].numpy(), pos, sh.softmax_scale)
    out = runs[0][0].float().cpu().numpy()[sample]
    assert np.abs(out - ro).max() <= H.OUT_ATOL_BF16
    assert np.abs(runs[0][1].cpu().numpy()[sample] - rl).max() <= H.LSE_ATOL_BF16


@pytest.mark.parametrize("name", ["bf16-ragged", "bf16-k64", "fp8-ragged"])
def test_indexer_tensor_core_matches_generic(name, monkeypatch):
    """The tcgen05 indexer and the CUDA-core indexer on the same inputs agree
    to fp32 summation-order noise, and the tensor-core kernel is the one the
    default dispatch runs for the 64 x 128 indexer shape."""
    wl, t = case(name)
    tc_scores = _gpu_scores(wl, t)
    kernels = dsa.last_kernels()
    assert ("indexer_fp8" if wl.shape.idx_fp8 else "indexer_tc") in kernels, kernels
    monkeypatch.setenv("DSA_FORCE_GENERIC", "1")
    gen_scores = _gpu_scores(wl, t)
    assert "indexer_simt" in dsa.last_kernels()
    monkeypatch.delenv("DSA_FORCE_GENERIC")
    a, b = tc_scores.cpu().numpy(), gen_scores.cpu().numpy()
    for bq in range(wl.B):
        rows = slice(wl.cu_q[bq], wl.cu_q[bq + 1])
        S = wl.S[bq]
        x, y = a[rows, :S], b[rows, :S]
        assert np.array_equal(np.isneginf(x), np.isneginf(y))
        fin = np.isfinite(y)
        scale = np.abs(y[fin]).max() if fin.any() else 1.0
        assert np.abs(x[fin] - y[fin]).max() <= 1e-5 * scale


@pytest.mark.parametrize("name", ["bf16-ragged", "bf16-k64"])
def test_attention_stage_tensor_core_matches_generic(name, monkeypatch):
    """The tensor-core attention stage (tcgen05 absorption GEMMs, bf16 q~ and
    latent context) against the generic fp32 stage on the same selection:
    equal within the bf16 output tolerance."""
    wl, t = case(name)
    sh = wl.shape
    sel = di.random_selection(wl, seed=37, density=0.8).cuda()
    args = (t["q_nope"], t["q_pe"], t["ckv"], t["kpe"], t["W_UK"], t["W_UV"], sel, H.seqs_of(wl), sh.softmax_scale)
    fast, lf = dsa.dsa_sparse_mla_fwd(*args)
    assert {"absorb_tc", "mla_tc"} <= dsa.last_kernels(), dsa.last_kernels()
    monkeypatch.setenv("DSA_FORCE_GENERIC", "1")
    gen, lg = dsa.dsa_sparse_mla_fwd(*args)
    assert "absorb_simt" in dsa.last_kernels()
    monkeypatch.delenv("DSA_FORCE_GENERIC")
    assert (fast.float() - gen.float()).abs().max().item() <= H.OUT_ATOL_BF16
    assert (lf - lg).abs().max().item() <= H.LSE_ATOL_BF16


@pytest.mark.parametrize("B", [700, dsa._abi.DSA_MAX_SEQS])
def test_forward_decode_batch_beyond_512_sequences(B):
    """A decode step of 700 and of the maximum 1024 sequences (one query each, caches of 300..3000
    keys, top-256): more sequences than one launch carried before; sampled rows match the oracle's
    whole path."""
    g = torch.Generator().manual_seed(77)
    S = [int(x) for x in torch.randint(300, 3000, (B,), generator=g)]
    wl = di.generate(f"decode-{B}", di.Shape(k=256), 77, [1] * len(S), S, [s - 1 for s in S])
    t = H.to_device(wl)
    out, lse, idx = H.gpu_forward(wl, t)
    st, site = dsa.dsa_check_device_error()
    assert st == 0, (st, site)
    rows = di.sample_rows(wl, 24)
    ref = H.oracle_rows(wl, rows)
    out_np, idx_np = out.float().cpu().numpy(), idx.cpu().numpy()
    for r in rows:
        o = ref[r]
        H.check_selection_row(idx_np[r], o["scores"], o["absterm"], o["pos"], wl.shape.k)
        assert np.abs(out_np[r] - o["out"]).max() <= H.OUT_ATOL_BF16


def _documented_order(row, p, k):
    """The selection's documented order: the keys above the k-th score T in increasing key index, then
    the first keys equal to T in increasing key index."""
    sel = H.cpu_topk_same_buffer(row, p, k)
    causal = np.asarray(row[:p + 1], np.float32).astype(np.float64) + 0.0
    T = causal[sel[-1]]
    above = np.sort(sel[causal[sel] > T])
    equal = np.sort(sel[causal[sel] == T])
    return np.concatenate([above, equal])


@pytest.mark.parametrize("kind", ["random", "coarse", "equal", "rising"])
def test_topk_cluster_rows_exact_order(kind):
    """Few long rows (the cluster kernel: eight CTAs per row, 9K to 62K keys) with random scores, a
    coarse grid (ties at the k-th score), all-equal scores and rising scores (every top key in the last
    CTA's slice): the output is the documented order exactly -- keys above the k-th score in increasing
    index, then the first keys equal to it -- ties to the lower key index."""
    g = torch.Generator().manual_seed(11)
    rows, k = 24, 2048
    S = [9000 + 2300 * r for r in range(rows)]
    cu = np.concatenate([[0], np.cumsum(S)]).tolist()
    seqs = dsa.Seqs(list(range(rows + 1)), cu, [s - 1 for s in S])
    ld = max(S)
    if kind == "random":
        scores = torch.randn((rows, ld), generator=g)
    elif kind == "coarse":
        scores = torch.randint(-30, 30, (rows, ld), generator=g).float() / 4
    elif kind == "equal":
        scores = torch.full((rows, ld), 0.5)
    else:
        scores = torch.arange(ld, dtype=torch.float32).repeat(rows, 1) / ld
    idx = dsa.dsa_topk_select(scores.cuda(), seqs, k).cpu().numpy()
    assert "topk" in dsa.last_kernels()
    sc = scores.numpy()
    for r in range(rows):
        want = _documented_order(sc[r], S[r] - 1, k)
        assert np.array_equal(idx[r], want), f"row {r}"
