"""Pins for the oracle: checks against what the pages and the mathematics fix,
not against the oracle itself.

Each test names what it pins: hand-worked examples (tests/golden), values the
pages print, closed forms, invariants, and special cases that reduce to a
library routine (Python's sort, torch's scaled_dot_product_attention, torch's
float8_e4m3fn conversion, a plain matmul).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _num(x):
    return -math.inf if x == "-inf" else float(x)


# --------------------------------------------------------------------------
# Indexer: hand-worked example (golden)
# --------------------------------------------------------------------------
def test_indexer_worked_example():
    g = _gold("indexer_worked_example.json")
    scores, absterm = oracle.indexer_scores(g["qI"], g["w"], g["kI"], g["pos"], with_absterm=True)
    exp = np.array([[_num(v) for v in row] for row in g["scores"]])
    assert np.array_equal(np.isinf(scores), np.isinf(exp))
    fin = np.isfinite(exp)
    assert np.allclose(scores[fin], exp[fin], rtol=0, atol=1e-15)
    assert np.allclose(absterm, np.array(g["absterm"]), rtol=0, atol=1e-15)
    idx = oracle.topk(scores, g["pos"], g["k"])
    assert idx.tolist() == g["idx"]


def test_indexer_page_constant_and_reduced_case():
    """The pages' constant 1/(sqrt(64) sqrt(128)); and with one head, w = 1 the
    score reduces to ReLU(q.k)/sqrt(D_I)."""
    rng = np.random.default_rng(1)
    n, S, D = 5, 7, 128
    q = rng.standard_normal((n, 64, D)).astype(np.float32)
    k = rng.standard_normal((S, D)).astype(np.float32)
    w = np.zeros((n, 64), np.float32)
    w[:, 3] = 1.0  # only head 3 counts
    pos = np.full(n, S - 1)
    s = oracle.indexer_scores(q, w, k, pos)
    dots = q[:, 3, :].astype(np.float64) @ k.T.astype(np.float64)
    exp = np.maximum(dots, 0.0) / (math.sqrt(64) * math.sqrt(128))
    assert np.allclose(s, exp, rtol=1e-13, atol=1e-13)
    # one head in total: ReLU(q.k) / sqrt(D)
    s1 = oracle.indexer_scores(q[:, :1, :], np.ones((n, 1), np.float32), k, pos)
    dots0 = q[:, 0, :].astype(np.float64) @ k.T.astype(np.float64)
    assert np.allclose(s1, np.maximum(dots0, 0)
                       / math.sqrt(D), rtol=1e-13, atol=1e-13)


def test_indexer_invariants():
    """Homogeneity (ReLU is positively homogeneous), reversal under w -> -w,
    equivariance under a permutation of the keys, and -inf exactly on the
    future keys."""
    rng = np.random.default_rng(2)
    n, S, H, D = 6, 11, 4, 16
    q = rng.standard_normal((n, H, D)).astype(np.float32)
    k = rng.standard_normal((S, D)).astype(np.float32)
    w = rng.standard_normal((n, H)).astype(np.float32)
    pos = np.array([0, 3, 5, 7, 10, 10])
    s = oracle.indexer_scores(q, w, k, pos)
    future = np.arange(S)[None, :] > pos[:, None]
    assert np.all(np.isneginf(s[future])) and np.all(np.isfinite(s[~future]))
    s2 = oracle.indexer_scores(q, 4.0 * w, k, pos)          # power-of-two scale: exact in fp32
    assert np.allclose(s2[~future], 4.0 * s[~future], rtol=1e-14, atol=0)
    s3 = oracle.indexer_scores(2.0 * q, w, k, pos)
    assert np.allclose(s3[~future], 2.0 * s[~future], rtol=1e-14, atol=0)
    s4 = oracle.indexer_scores(q, -w, k, pos)
    assert np.allclose(s4[~future], -s[~future], rtol=1e-14, atol=0)
    # key permutation among the keys every row can see (all rows at the last position)
    posl = np.full(n, S - 1)
    sa = oracle.indexer_scores(q, w, k, posl)
    perm = rng.permutation(S)
    sb = oracle.indexer_scores(q, w, k[perm], posl)
    assert np.allclose(sb, sa[:, perm], rtol=1e-14, atol=1e-14)
    # a key whose dot product is negative for every head contributes exactly 0
    kneg = -np.abs(k[:1])
    qpos = np.abs(q)
    z = oracle.indexer_scores(qpos, w, kneg, np.zeros(n, np.int64))
    assert np.all(z == 0.0)


# --------------------------------------------------------------------------
# Top-k: reduces to a full sort (Python's sorted) on small inputs
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_topk_equals_full_sort(seed):
    rng = np.random.default_rng(seed)
    n, S, k = 9, 40, 8
    # coarse values force many exact ties
    scores = rng.integers(-5, 6, size=(n, S)).astype(np.float64)
    pos = np.array([0, 1, 6, 7, 8, 20, 38, 39, 39])
    scores[np.arange(S)[None, :] > pos[:, None]] = -np.inf
    idx = oracle.topk(scores, pos, k)
    for r in range(n):
        cand = sorted(range(pos[r] + 1), key=lambda s: (-scores[r, s], s))
        want = cand[:k] + [-1] * (k - min(k, len(cand)))
        assert idx[r].tolist() == want


def test_topk_row_counts_plain_causal():
    """While the sequence is no longer than k every causal key is selected:
    row t keeps t + 1 keys (the nnterp deepseek_v32 note prints
    rows == arange(1, n + 1))."""
    rng = np.random.default_rng(3)
    S = k = 32
    scores = rng.standard_normal((S, S))
    pos = np.arange(S)
    scores[np.arange(S)[None, :] > pos[:, None]] = -np.inf
    idx = oracle.topk(scores, pos, k)
    counts = (idx >= 0).sum(1)
    assert counts.tolist() == list(range(1, S + 1))
    for t in range(S):
        assert sorted(idx[t][idx[t] >= 0].tolist()) == list(range(t + 1))


# --------------------------------------------------------------------------
# Latent up-projection: a plain matmul (library routine)
# --------------------------------------------------------------------------
def test_kv_up_is_matmul():
    rng = np.random.default_rng(4)
    S, H, d_n, d_c, d_v = 5, 3, 4, 6, 2
    ckv = rng.standard_normal((S, d_c + 2)).astype(np.float32)  # wider rows: packed cache
    W_UK = rng.standard_normal((H, d_n, d_c)).astype(np.float32)
    W_UV = rng.standard_normal((H, d_c, d_v)).astype(np.float32)
    KC, V = oracle.kv_up(ckv, W_UK, W_UV)
    c = ckv[:, :d_c].astype(np.float64)
    for h in range(H):
        assert np.allclose(KC[:, h, :], c @ W_UK[h].astype(np.float64).T, rtol=1e-13, atol=1e-13)
        assert np.allclose(V[:, h, :], c @ W_UV[h].astype(np.float64), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Attention: hand-worked example, closed forms, SDPA, equivalences
# --------------------------------------------------------------------------
def test_attention_worked_example():
    g = _gold("attention_worked_example.json")
    cache = np.array(g["kv_cache"], np.float32)
    ckv, kpe = cache[:, :2], cache[:, 2:]
    KC, V = oracle.kv_up(ckv, g["W_UK"], g["W_UV"])
    out, lse = oracle.sparse_mla_unabsorbed(g["q_nope"], g["q_pe"], KC, kpe, V, g["idx"], g["pos"], g["scale"])
    e2 = math.exp(2.0)
    want_out = [(3 * e2 + 5) / (e2 + 1), 3.0, 5.0]
    want_lse = [math.log(e2 + 1), 2.0, 0.0]
    assert np.allclose(out[:, 0, 0], want_out, rtol=1e-14, atol=1e-14)
    assert np.allclose(lse[:, 0], want_lse, rtol=1e-14, atol=1e-14)
    out2, lse2 = oracle.sparse_mla_absorbed(g["q_nope"], g["q_pe"], ckv, kpe, g["W_UK"], g["W_UV"],
                                            g["idx"], g["pos"], g["scale"])
    assert np.allclose(out2[:, 0, 0], want_out, rtol=1e-14, atol=1e-14)
    assert np.allclose(lse2[:, 0], want_lse, rtol=1e-14, atol=1e-14)


def _small_case(rng, n=7, S=13, H=3, d_n=8, d_r=4, d_c=10, d_v=6):
    return dict(
        q_nope=rng.standard_normal((n, H, d_n)).astype(np.float32),
        q_pe=rng.standard_normal((n, H, d_r)).astype(np.float32),
        ckv=rng.standard_normal((S, d_c)).astype(np.float32),
        kpe=rng.standard_normal((S, d_r)).astype(np.float32),
        W_UK=(rng.standard_normal((H, d_n, d_c)) / 3).astype(np.float32),
        W_UV=(rng.standard_normal((H, d_c, d_v)) / 3).astype(np.float32),
    )


def test_attention_closed_forms():
    """q = 0: every live logit is 0, so out is the plain mean of V over the
    live selected keys and lse = log(n).  A single live key gives out = V."""
    rng = np.random.default_rng(5)
    c = _small_case(rng)
    n, H = c["q_nope"].shape[:2]
    S = c["ckv"].shape[0]
    KC, V = oracle.kv_up(c["ckv"], c["W_UK"], c["W_UV"])
    pos = np.array([12, 12, 3, 0, 5, 12, 8])
    idx = np.array([[0, 5, 7, -1], [12, 11, 10, 9], [3, 4, 1, 2], [0, 1, 2, 3],
                    [-1, -1, -1, -1], [40, 2, -5, 2], [8, 7, 6, 5]], np.int32)
    zq = np.zeros_like(c["q_nope"]), np.zeros_like(c["q_pe"])
    out, lse = oracle.sparse_mla_unabsorbed(zq[0], zq[1], KC, c["kpe"], V, idx, pos, 0.3)
    for r in range(n):
        live = [s for s in idx[r] if 0 <= s < S and s <= pos[r]]
        for h in range(H):
            if live:
                assert np.allclose(out[r, h], V[live, h, :].mean(0), rtol=1e-13, atol=1e-13)
                assert math.isclose(lse[r, h], math.log(len(live)), rel_tol=1e-13, abs_tol=1e-13)
            else:
                assert np.all(out[r, h] == 0) and lse[r, h] == -math.inf
    # a single live key
    one = np.array([[4, -1, -1, -1]] * n, np.int32)
    pos5 = np.full(n, 5)
    out1, _ = oracle.sparse_mla_unabsorbed(c["q_nope"], c["q_pe"], KC, c["kpe"], V, one, pos5, 0.3)
    for r in range(n):
        assert np.allclose(out1[r], V[4], rtol=1e-13, atol=1e-13)


def test_attention_matches_sdpa():
    """The unabsorbed sparse attention is softmax attention with the
    selection mask: torch's scaled_dot_product_attention (float64, CPU) on
    Q = [q_nope; q_pe], K = [K^C; k_pe], V and the boolean mask of the live
    selected keys gives the same output."""
    rng = np.random.default_rng(6)
    c = _small_case(rng, n=9, S=17)
    n, H, d_n = c["q_nope"].shape
    S = c["ckv"].shape[0]
    pos = rng.integers(0, S, size=n)
    k = 6
    idx = np.full((n, k), -1, np.int32)
    for r in range(n):
        cand = rng.permutation(pos[r] + 1)[:k]
        idx[r, :len(cand)] = cand
    scale = 0.37
    KC, V = oracle.kv_up(c["ckv"], c["W_UK"], c["W_UV"])
    out, lse = oracle.sparse_mla_unabsorbed(c["q_nope"], c["q_pe"], KC, c["kpe"], V, idx, pos, scale)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    ckv = t(c["ckv"])
    Kc = torch.einsum("hdc,sc->hsd", t(c["W_UK"]), ckv)                  # [H,S,d_n]
    Vv = torch.einsum("sc,hce->hse", ckv, t(c["W_UV"]))                  # [H,S,d_v]
    K = torch.cat([Kc, t(c["kpe"]).unsqueeze(0).expand(H, S, -1)], -1)   # [H,S,d_n+d_r]
    Q = torch.cat([t(c["q_nope"]), t(c["q_pe"])], -1).transpose(0, 1)   # [H,n,d_n+d_r]
    mask = torch.zeros(n, S, dtype=torch.bool)
    for r in range(n):
        for s in idx[r]:
            if 0 <= s <= pos[r]:
                mask[r, s] = True
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, attn_mask=mask, scale=scale)
    assert np.allclose(out, ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_absorbed_equals_unabsorbed():
    """Regrouping the products (q^C W_UK^T c = (q^C W_UK) . c and
    (sum P c) W_UV = sum P (c W_UV)) leaves the result unchanged."""
    rng = np.random.default_rng(7)
    c = _small_case(rng, n=8, S=21, H=4, d_n=16, d_r=8, d_c=24, d_v=12)
    n = c["q_nope"].shape[0]
    S = c["ckv"].shape[0]
    pos = rng.integers(0, S, size=n)
    idx = np.stack([np.concatenate([rng.permutation(S)[:9]]).astype(np.int32) for _ in range(n)])
    KC, V = oracle.kv_up(c["ckv"], c["W_UK"], c["W_UV"])
    a, la = oracle.sparse_mla_unabsorbed(c["q_nope"], c["q_pe"], KC, c["kpe"], V, idx, pos, 0.21)
    b, lb = oracle.sparse_mla_absorbed(c["q_nope"], c["q_pe"], c["ckv"], c["kpe"], c["W_UK"], c["W_UV"],
                                       idx, pos, 0.21)
    assert np.allclose(a, b, rtol=1e-10, atol=1e-10)
    assert np.allclose(la, lb, rtol=1e-10, atol=1e-10)


def test_sparse_equals_dense_masked_and_plain_causal():
    """(a) The sparse form over the top-k selection equals the dense softmax
    with M^sel written out over every key (the atlas equations).  (b) While
    S <= k the selection holds every causal key, so the result is plain
    causal attention (nnterp deepseek_v32 note)."""
    rng = np.random.default_rng(8)
    n = S = 12
    H_I, D_I = 3, 8
    c = _small_case(rng, n=n, S=S)
    qI = rng.standard_normal((n, H_I, D_I)).astype(np.float32)
    kI = rng.standard_normal((S, D_I)).astype(np.float32)
    w = rng.standard_normal((n, H_I)).astype(np.float32)
    pos = np.arange(n)
    KC, V = oracle.kv_up(c["ckv"], c["W_UK"], c["W_UV"])
    scores = oracle.indexer_scores(qI, w, kI, pos)
    for k in (4, S):
        idx = oracle.topk(scores, pos, k)
        sel = np.zeros((n, S), np.uint8)
        for r in range(n):
            for s in idx[r]:
                if s >= 0:
                    sel[r, s] = 1
        sp, lsp = oracle.sparse_mla_unabsorbed(c["q_nope"], c["q_pe"], KC, c["kpe"], V, idx, pos, 0.3)
        de, lde = oracle.dense_masked_mla(c["q_nope"], c["q_pe"], KC, c["kpe"], V, pos, 0.3, sel=sel)
        assert np.allclose(sp, de, rtol=1e-12, atol=1e-12) and np.allclose(lsp, lde, rtol=1e-12, atol=1e-12)
    causal, lc = oracle.dense_masked_mla(c["q_nope"], c["q_pe"], KC, c["kpe"], V, pos, 0.3, sel=None)
    assert np.allclose(sp, causal, rtol=1e-12, atol=1e-12) and np.allclose(lsp, lc, rtol=1e-12, atol=1e-12)


def test_probabilities_sum_to_one_shift_invariance():
    """Adding the same constant to every live logit of a row leaves the
    output unchanged and shifts lse by that constant: the k_pe term with a
    constant rope key is such a shift."""
    rng = np.random.default_rng(9)
    c = _small_case(rng, n=4, S=9, d_r=2)
    n = c["q_nope"].shape[0]
    pos = np.full(n, 8)
    idx = np.tile(np.arange(9, dtype=np.int32), (n, 1))
    KC, V = oracle.kv_up(c["ckv"], c["W_UK"], c["W_UV"])
    kz = np.zeros_like(c["kpe"])
    kc = np.ones_like(c["kpe"]) * 0.5
    o0, l0 = oracle.sparse_mla_unabsorbed(c["q_nope"], c["q_pe"], KC, kz, V, idx, pos, 0.4)
    o1, l1 = oracle.sparse_mla_unabsorbed(c["q_nope"], c["q_pe"], KC, kc, V, idx, pos, 0.4)
    shift = 0.4 * 0.5 * c["q_pe"].astype(np.float64).sum(-1)
    assert np.allclose(o0, o1, rtol=1e-12, atol=1e-12)
    assert np.allclose(l1 - l0, shift, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Values the pages print: scale constants, parameter count, config
# --------------------------------------------------------------------------
def test_page_constants():
    g = _gold("config_671B_v32_excerpt.json")
    qk_head_dim = g["qk_nope_head_dim"] + g["qk_rope_head_dim"]
    plain = qk_head_dim ** -0.5
    mscale = 0.1 * g["mscale_all_dim"] * math.log(g["rope_factor"]) + 1.0
    assert round(plain, 4) == g["softmax_scale_plain"]
    assert round(mscale * mscale, 2) == g["yarn_factor"]
    assert round(plain * mscale * mscale, 4) == g["softmax_scale_yarn"]
    # the sparse-attention parameter count from the module shapes the pages print
    d, H = g["dim"], g["n_heads"]
    qlr, kvr = g["q_lora_rank"], g["kv_lora_rank"]
    dn, dr, dv = g["qk_nope_head_dim"], g["qk_rope_head_dim"], g["v_head_dim"]
    HI, DI = g["index_n_heads"], g["index_head_dim"]
    W_UK = H * dn * kvr  # [H, d_n, d_c] -- half of wkv_b
    W_UV = H * kvr * dv  # [H, d_c, d_v] -- the other half
    params = (d * qlr + qlr + qlr * H * (dn + dr) + d * (kvr + dr) + kvr + W_UK + W_UV + H * dv * d
              + qlr * HI * DI + d * DI + 2 * DI + d * HI)
    assert params == g["sparse_attention_params_per_block"]


def test_workload_shapes_follow_config():
    import dsa_inputs
    g = _gold("config_671B_v32_excerpt.json")
    f = dsa_inputs.FULL
    assert (f.H, f.d_n, f.d_r, f.d_c, f.d_v) == (g["n_heads"], g["qk_nope_head_dim"], g["qk_rope_head_dim"],
                                                 g["kv_lora_rank"], g["v_head_dim"])
    assert (f.H_I, f.D_I, f.k) == (g["index_n_heads"], g["index_head_dim"], g["index_topk"])
    assert math.isclose(f.softmax_scale, (g["qk_nope_head_dim"] + g["qk_rope_head_dim"]) ** -0.5)


# --------------------------------------------------------------------------
# FP8 e4m3 + ue8m0 quantiser
# --------------------------------------------------------------------------
def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2  # 0x7F, 0xFF
    assert np.array_equal(mine[~nan], ref[~nan])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6


def test_e4m3_encode_matches_torch_rne():
    """In range (|v| <= 448) the encoder is round-to-nearest-even, which is
    what torch's float -> float8_e4m3fn conversion does; exact midpoints
    between neighbouring codes are included."""
    fin = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (fin[:-1] + fin[1:]) / 2
    rng = np.random.default_rng(10)
    vals = np.concatenate([fin, mids, rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 0.01,
                           -mids, np.ldexp(rng.uniform(-1, 1, 500), -9)])
    vals = vals.astype(np.float32)  # exactly representable: all are dyadic with short mantissas or float32 draws
    blocks = np.zeros((len(vals) + 127) // 128 * 128, np.float32)
    blocks[:len(vals)] = vals
    # force each block's scale to 1 by planting 448 in its last slot
    blocks = blocks.reshape(-1, 128)
    planted = np.concatenate([blocks[:, :127], np.full((blocks.shape[0], 1), 448.0, np.float32)], 1)
    codes, exps = oracle.quant_e4m3_ue8m0(planted)
    assert np.all(exps == 0)
    ref = torch.from_numpy(planted.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_ue8m0_scale_rules():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 128)).astype(np.float32) * np.ldexp(1.0, rng.integers(-20, 20, (64, 1)))
    x[0] = 0.0
    x[1] = 0.0
    x[1, 5] = 448.0          # amax exactly 448 -> scale 1
    x[2] = 0.0
    x[2, 7] = -448.5         # just above -> scale 2
    x[3] = 0.0
    x[3, 0] = 1e-38          # tiny: exponent clamps at -127
    codes, exps = oracle.quant_e4m3_ue8m0(x)
    amax = np.abs(x.astype(np.float64)).max(1)
    assert exps[0] == 0 and exps[1] == 0 and exps[2] == 1 and exps[3] == -127
    for b in range(4, 64):
        e = int(exps[b])
        assert amax[b] <= 448.0 * 2.0 ** e and amax[b] > 448.0 * 2.0 ** (e - 1)
    deq = oracle.dequant_e4m3(codes, exps).astype(np.float64)
    # round to nearest: the error is at most half the local code spacing (3 mantissa bits)
    for b in range(64):
        e = float(2.0 ** exps[b])
        for i in range(128):
            v = x[b, i] / e
            if abs(v) >= 2.0 ** -6:
                assert abs(deq[b, i] - x[b, i]) <= 2.0 ** (math.floor(math.log2(abs(v))) - 4) * e * (1 + 1e-12)
            else:
                assert abs(deq[b, i] - x[b, i]) <= 2.0 ** -10 * e * (1 + 1e-12)


# ---------------------------------------------------------------------------
# The projections on either side of the path (the step before: wkv_a, kv_norm,
# rotary k_pe, wk + k_norm, weights_proj; the step after: wo)
# ---------------------------------------------------------------------------
def test_linear_is_the_matmul_with_the_weight_stored_out_by_in():
    """nn.Linear without bias: y = x W^T, W stored [out, in] (the printout's
    Linear(in_features, out_features)); a plain float64 matmul."""
    g = np.random.default_rng(11)
    x = g.standard_normal((7, 33)).astype(np.float32)
    W = g.standard_normal((5, 33)).astype(np.float32)
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    assert np.allclose(oracle.linear(x, W), ref, rtol=1e-13, atol=1e-12)
    # an identity weight copies its inputs; a one-hot row picks one input
    assert np.array_equal(oracle.linear(x, np.eye(33, dtype=np.float32)), x.astype(np.float64))
    e = np.zeros((1, 33), np.float32)
    e[0, 4] = 1.0
    assert np.array_equal(oracle.linear(x, e)[:, 0], x[:, 4].astype(np.float64))


def test_rmsnorm_matches_the_library_and_its_closed_form():
    g = np.random.default_rng(12)
    x = g.standard_normal((6, 512)) * 3.0
    gain = g.uniform(0.5, 1.5, 512).astype(np.float32)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (512,), torch.tensor(gain, dtype=torch.float64), eps=1e-6)
    assert np.allclose(oracle.rmsnorm(x, gain), ref.numpy(), rtol=1e-12, atol=1e-12)
    # a constant row c: y = gain * c / sqrt(c^2 + eps)
    c = 0.25
    y = oracle.rmsnorm(np.full((1, 512), c), np.ones(512, np.float32))
    assert np.allclose(y, c / math.sqrt(c * c + 1e-6), rtol=1e-14)
    # unit gain: the mean square of the output is ms / (ms + eps)
    y = oracle.rmsnorm(x, np.ones(512, np.float32))
    ms = (x ** 2).mean(-1)
    assert np.allclose((y ** 2).mean(-1), ms / (ms + 1e-6), rtol=1e-12)


def test_layernorm_matches_the_library_and_its_closed_form():
    g = np.random.default_rng(13)
    x = g.standard_normal((6, 128)) * 2.0 + 0.7
    gain = g.uniform(0.5, 1.5, 128).astype(np.float32)
    bias = g.standard_normal(128).astype(np.float32)
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (128,), torch.tensor(gain, dtype=torch.float64),
                                         torch.tensor(bias, dtype=torch.float64), eps=1e-6)
    assert np.allclose(oracle.layernorm(x, gain, bias), ref.numpy(), rtol=1e-12, atol=1e-12)
    # x = a + b * (+1, -1, +1, ...): mean a, variance b^2, so y = +-b / sqrt(b^2 + eps) * gain + bias
    a, b = 3.0, 0.5
    sgn = np.tile([1.0, -1.0], 64)
    y = oracle.layernorm((a + b * sgn)[None, :], gain, bias)[0]
    want = sgn * b / math.sqrt(b * b + 1e-6) * gain.astype(np.float64) + bias.astype(np.float64)
    assert np.allclose(y, want, rtol=1e-13, atol=1e-13)


def test_rotary_is_served_de_interleaved():
    """The nnterp deepseek_v32 note: at position 0, where the rotary step is the
    identity, the served rotary part is the projection's even dimensions
    followed by its odd ones; at any angle, pair (2i, 2i+1) is turned as the
    complex number x[2i] + i x[2i+1] times e^{i theta_i} into dims i, 32 + i."""
    g = np.random.default_rng(14)
    x = g.standard_normal((5, 64))
    ones, zeros = np.ones((5, 32), np.float32), np.zeros((5, 32), np.float32)
    y0 = oracle.rope_deinterleave(x, ones, zeros)
    assert np.array_equal(y0, np.concatenate([x[:, 0::2], x[:, 1::2]], axis=1))
    theta = g.uniform(-math.pi, math.pi, (5, 32))
    c, s = np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)
    y = oracle.rope_deinterleave(x, c, s)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * (c.astype(np.float64) + 1j * s.astype(np.float64))
    assert np.allclose(y[:, :32], z.real, rtol=1e-14, atol=1e-14)
    assert np.allclose(y[:, 32:], z.imag, rtol=1e-14, atol=1e-14)
    # turning back by -theta restores the pairs
    back = oracle.rope_deinterleave(np.stack([y[:, :32], y[:, 32:]], axis=2).reshape(5, 64), c, -s)
    assert np.allclose(back, y0, rtol=1e-6, atol=1e-6)


def test_kv_prologue_split_and_scale_invariance():
    """The step before the path, composed in the pages' order: the first 512
    outputs of wkv_a are normalised (RMSNorm: invariant to a positive scale of
    x up to eps), the next 64 rotated (linear in x), wk's 128 outputs
    layer-normalised (invariant to scale and shift of the outputs), and the 64
    head weights are weights_proj(x) as they come."""
    g = np.random.default_rng(15)
    dim = 96
    x = g.standard_normal((4, dim)).astype(np.float32)
    W = (g.standard_normal((512 + 64 + 128 + 64, dim)) / math.sqrt(dim)).astype(np.float32)
    kvg = g.uniform(0.5, 1.5, 512).astype(np.float32)
    kg = g.uniform(0.5, 1.5, 128).astype(np.float32)
    kb = g.standard_normal(128).astype(np.float32)
    th = g.uniform(-3, 3, (4, 32))
    c, s = np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)
    r = oracle.kv_prologue(x, W, kvg, kg, kb, c, s)
    lin = x.astype(np.float64) @ W.astype(np.float64).T
    assert np.allclose(r["w"], lin[:, 704:768], rtol=1e-12, atol=1e-12)
    # the rotated key keeps each pair's length
    assert np.allclose(r["k_pe"][:, :32] ** 2 + r["k_pe"][:, 32:] ** 2, lin[:, 512:576:2] ** 2 + lin[:, 513:576:2] ** 2,
                       rtol=1e-6)  # cos^2 + sin^2 = 1 to float32 precision
    r2 = oracle.kv_prologue(x * 4.0, W, kvg, kg, kb, c, s)
    assert np.allclose(r2["latent"], r["latent"], rtol=1e-5)
    assert np.allclose(r2["kI"], r["kI"], rtol=1e-5, atol=1e-5)
    assert np.allclose(r2["k_pe"], 4.0 * r["k_pe"], rtol=1e-12, atol=1e-12)
    assert np.allclose(r2["w"], 4.0 * r["w"], rtol=1e-12, atol=1e-12)
    # the latent rows have mean square ~ gain^2 weighted; with unit gain it is ~1
    r3 = oracle.kv_prologue(x, W, np.ones(512, np.float32), kg, kb, c, s)
    assert np.allclose((r3["latent"] ** 2).mean(-1), 1.0, atol=1e-4)


def test_output_projection_of_the_heads_side_by_side():
    """wo reads the attention output with the heads side by side
    ([n, H * d_v], the printout's attention_premix): y = sum_h out_h wo_h^T."""
    g = np.random.default_rng(16)
    out = g.standard_normal((3, 4, 8)).astype(np.float32)
    wo = g.standard_normal((6, 32)).astype(np.float32)
    y = oracle.output_proj(out, wo)
    per_head = sum(out[:, h, :].astype(np.float64) @ wo[:, h * 8:(h + 1) * 8].astype(np.float64).T for h in range(4))
    assert np.allclose(y, per_head, rtol=1e-12, atol=1e-12)
