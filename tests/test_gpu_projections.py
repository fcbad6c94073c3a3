"""The projections on either side of the path, on the GPU, against the oracle:

  * the tensor-core GEMM behind them (dsa_output_proj) on ragged sizes: a
    row tail, a partial last column block, several K slabs;
  * the output projection wo at the released shapes (16384 -> 7168) on
    sampled rows, and inside dsa_forward (W_UV and wo chunk by chunk), where
    it must equal wo applied to the forward's own attention output;
  * the step before the path (dsa_kv_prologue): the normalised latent, the
    rotated k_pe and the layer-normalised indexer key appended to the caches,
    the per-head weights, with the bf16 and the FP8 indexer cache.

Tolerances: a bf16 result is held to 2^-8 of its value (one rounding to
bf16 is 2^-9) plus 1e-5 of its absolute product sum (the fp32 accumulation's
rounding, sum_i |x_i| |w_i|); fp32 results to the second term only."""
import math

import numpy as np
import pytest
import torch

import dsa_inputs as di
import oracle
import sparse_latent_attention_indexer_gb300 as dsa
from tests import helpers as H

pytestmark = pytest.mark.gpu

RTOL_BF16 = 2.0 ** -8
ACC = 1e-5


def _f64(t):
    return t.detach().double().cpu().numpy()


def _check_linear(y_gpu, x, W, rows=None, bf16=True):
    """y_gpu [len(rows), N] against oracle.linear(x[rows], W)."""
    xs = x if rows is None else x[rows]
    ref = oracle.linear(_f64(xs).astype(np.float32), _f64(W).astype(np.float32))
    absum = np.abs(_f64(xs)) @ np.abs(_f64(W)).T
    band = (RTOL_BF16 * np.abs(ref) if bf16 else 0.0) + ACC * absum
    err = np.abs(_f64(y_gpu) - ref)
    assert (err <= band).all(), f"worst error {err.max():.3e} over band {band[np.unravel_index(err.argmax(), err.shape)]:.3e}"
    return float((err / band).max())


@pytest.mark.parametrize("M,K,N", [(300, 512, 384), (128, 64, 64), (1, 1024, 256), (1000, 192, 640)])
def test_gemm_ragged_sizes(M, K, N):
    g = torch.Generator().manual_seed(M + K + N)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(N, K, generator=g) / math.sqrt(K)).to(torch.bfloat16).cuda()
    y = dsa.dsa_output_proj(x, W)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert "gemm_tc" in dsa.last_kernels()
    _check_linear(y, x, W)


def test_output_projection_at_the_released_shapes():
    """wo: 128 heads x 128 values = 16384 -> 7168, 4096 rows; 24 sampled rows."""
    g = torch.Generator().manual_seed(7)
    M, K, N = 4096, 16384, 7168
    out = torch.randn(M, 128, 128, generator=g).to(torch.bfloat16).cuda()
    wo = (torch.randn(N, K, generator=g) / math.sqrt(K)).to(torch.bfloat16).cuda()
    y = dsa.dsa_output_proj(out, wo)
    assert dsa.dsa_check_device_error() == (0, 0)
    rows = sorted({0, M - 1, *torch.randint(0, M, (22,), generator=g).tolist()})
    _check_linear(y[rows], out.reshape(M, K), wo, rows)


@pytest.mark.parametrize("want_out", [True, False])
def test_forward_applies_wo_to_its_attention_output(want_out):
    wl = di.generate("wo-fused", di.Shape(k=64), 9, [96, 40, 2100], [96, 300, 2400], [0, 260, 300])
    t = H.to_device(wl)
    sh = wl.shape
    g = torch.Generator().manual_seed(10)
    d_model = 7168
    wo = (torch.randn(d_model, sh.H * sh.d_v, generator=g) / math.sqrt(sh.H * sh.d_v)).to(torch.bfloat16).cuda()
    out0, lse0, idx0 = H.gpu_forward(wl, t)
    out, lse, idx, y = H.gpu_forward(wl, t, wo=wo, want_out=want_out)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert "gemm_tc" in dsa.last_kernels()
    assert torch.equal(idx, idx0) and torch.equal(lse, lse0)
    if want_out:
        assert torch.equal(out, out0)
    else:
        assert out is None
    # y is wo applied to the forward's attention output (3 chunks of 2048 rows: the last one ragged)
    rows = list(range(0, wl.total_q, 37)) + [wl.total_q - 1]
    _check_linear(y[rows], out0.reshape(wl.total_q, -1), wo, rows)


def _prologue_inputs(seed, T, S, P, dim=7168):
    g = torch.Generator().manual_seed(seed)
    n = sum(T)
    x = torch.randn(n, dim, generator=g).to(torch.bfloat16)
    W = (torch.randn(512 + 64 + 128 + 64, dim, generator=g) / math.sqrt(dim)).to(torch.bfloat16)
    kv_gain = 1.0 + 0.1 * torch.randn(512, generator=g)
    k_gain = 1.0 + 0.1 * torch.randn(128, generator=g)
    k_bias = 0.1 * torch.randn(128, generator=g)
    n_pos = max(p + t for p, t in zip(P, T))
    theta = 10000.0 ** (-torch.arange(32, dtype=torch.float64) / 32.0)
    ang = torch.arange(n_pos, dtype=torch.float64)[:, None] * theta[None, :]
    return dict(x=x, W=W, kv_gain=kv_gain, k_gain=k_gain, k_bias=k_bias, cos=torch.cos(ang).float(),
                sin=torch.sin(ang).float())


@pytest.mark.parametrize("fp8", [False, True])
def test_kv_prologue_appends_the_new_tokens(fp8):
    T, S, P = [200, 1, 57], [1300, 4000, 60], [1100, 3999, 3]
    inp = _prologue_inputs(21, T, S, P)
    cu_q, cu_k = [0], [0]
    for t_, s_ in zip(T, S):
        cu_q.append(cu_q[-1] + t_)
        cu_k.append(cu_k[-1] + s_)
    seqs = dsa.Seqs(cu_q, cu_k, P)
    dev = {k: v.cuda() for k, v in inp.items()}
    sentinel = -3.0
    kv_cache = torch.full((cu_k[-1], 576), sentinel, dtype=torch.bfloat16, device="cuda")
    kc_bf16 = torch.full((cu_k[-1], 128), sentinel, dtype=torch.bfloat16, device="cuda")
    w = dsa.dsa_kv_prologue(dev["x"], dev["W"], dev["kv_gain"], dev["k_gain"], dev["k_bias"], dev["cos"], dev["sin"],
                            seqs, kv_cache, kc_bf16)
    assert dsa.dsa_check_device_error() == (0, 0)
    assert {"gemm_tc", "prologue"} <= dsa.last_kernels()
    if fp8:
        kc = torch.full((cu_k[-1], 128), 0x5A, dtype=torch.uint8, device="cuda")
        ks = torch.full((cu_k[-1],), -1.0, device="cuda")
        dsa.dsa_kv_prologue(dev["x"], dev["W"], dev["kv_gain"], dev["k_gain"], dev["k_bias"], dev["cos"], dev["sin"],
                            seqs, kv_cache, kc, k_scale=ks)
        assert dsa.dsa_check_device_error() == (0, 0)
    slots = [cu_k[b] + P[b] + t for b in range(len(T)) for t in range(T[b])]
    pos = [P[b] + t for b in range(len(T)) for t in range(T[b])]
    untouched = sorted(set(range(cu_k[-1])) - set(slots))
    assert bool((kv_cache[untouched] == sentinel).all()) and bool((kc_bf16[untouched] == sentinel).all())
    x64 = inp["x"].float().numpy()
    r = oracle.kv_prologue(x64, inp["W"].float().numpy(), inp["kv_gain"].numpy(), inp["k_gain"].numpy(),
                           inp["k_bias"].numpy(), inp["cos"].numpy()[pos], inp["sin"].numpy()[pos])
    absum = np.abs(x64.astype(np.float64)) @ np.abs(inp["W"].double().numpy()).T  # [n, 768]
    got = _f64(kv_cache[slots])
    # the latent and k^I are normalised: their rounding is relative to the normalised values
    for name, g_, lo, hi in (("latent", got[:, :512], 0, 512), ("k_pe", got[:, 512:], 512, 576),
                             ("kI", _f64(kc_bf16[slots]), 576, 704)):
        ref = r[name]
        band = RTOL_BF16 * np.abs(ref) + 1e-4
        err = np.abs(g_ - ref)
        assert (err <= band).all(), f"{name}: worst {err.max():.3e}"
    wref = r["w"]
    assert (np.abs(_f64(w) - wref) <= ACC * absum[:, 704:768]).all()
    if fp8:
        codes, exps = oracle.quant_e4m3_ue8m0(kc_bf16[slots].float().cpu().numpy())
        assert np.array_equal(kc[slots].cpu().numpy(), codes)
        assert np.array_equal(ks[slots].cpu().numpy(), np.ldexp(1.0, exps).astype(np.float32))
        assert bool((kc[untouched] == 0x5A).all()) and bool((ks[untouched] == -1.0).all())
