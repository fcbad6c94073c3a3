"""Oracle for the DSA hot path (lightning indexer -> top-k -> sparse latent
attention): ctypes bindings to the plain fp64 C code in ``oracle.c``.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  It shares no code with the CUDA library and never calls it.

Every function takes numpy arrays whose values are the exact input values
(bf16 / fp32 / dequantised e4m3, held as float32) and returns float64 results.
One call covers rows of ONE sequence; ``pos`` gives each row's absolute
position p = start_pos + t, keys are numbered 0..S-1 within the sequence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc into ``liboracle.so`` (in-tree)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_indexer_scores.argtypes = [P, P, P, P, I64, I64, I, I, P, P]
    lib.oracle_topk.argtypes = [P, P, I64, I64, I, P]
    lib.oracle_kv_up.argtypes = [P, I64, I64, P, P, I, I, I, I, P, P]
    lib.oracle_sparse_mla_unabsorbed.argtypes = [P, P, P, P, I64, P, P, P, I64, I, I64, I, I, I, I, D, P, P]
    lib.oracle_sparse_mla_absorbed.argtypes = [P, P, P, I64, P, I64, P, P, P, P, I64, I, I64, I, I, I, I, I,
                                               D, P, P, P, P]
    lib.oracle_dense_masked_mla.argtypes = [P, P, P, P, I64, P, P, P, I64, I64, I, I, I, I, D, P, P]
    lib.oracle_quant_e4m3_ue8m0.argtypes = [P, I64, P, P]
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = D
    lib.oracle_num_threads.restype = I
    lib.oracle_linear.argtypes = [P, P, I64, I64, I64, P]
    lib.oracle_rmsnorm.argtypes = [P, I64, I64, P, D, P]
    lib.oracle_layernorm.argtypes = [P, I64, I64, P, P, D, P]
    lib.oracle_rope_deinterleave.argtypes = [P, I64, I64, P, P, P]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def swap_library(path):
    """Load another build of the oracle source (the mutation tests compile
    copies with a planted mistake); returns the previous handle for
    ``restore_library``."""
    global _lib
    prev = _load()
    _lib = _bind(ctypes.CDLL(path))
    return prev


def restore_library(prev):
    global _lib
    _lib = prev


def _f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32:
        a = a.astype(np.float32)
    return np.ascontiguousarray(a)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return _load().oracle_num_threads()


def indexer_scores(qI, w, kI, pos, with_absterm: bool = False):
    """S~^I for rows of one sequence. qI [n,H_I,D_I], w [n,H_I], kI [S,D_I], pos [n].
    Returns scores [n,S] (and the |w| absolute-term sums when asked)."""
    qI, w, kI, pos = _f32(qI), _f32(w), _f32(kI), _i64(pos)
    n, H_I, D_I = qI.shape
    S = kI.shape[0]
    assert w.shape == (n, H_I) and kI.shape[1] == D_I and pos.shape == (n,)
    scores = np.empty((n, S), np.float64)
    absterm = np.empty((n, S), np.float64) if with_absterm else None
    _load().oracle_indexer_scores(_p(qI), _p(w), _p(kI), _p(pos), n, S, H_I, D_I, _p(scores), _p(absterm))
    return (scores, absterm) if with_absterm else scores


def topk(scores, pos, k: int):
    """Top-k causal keys per row (ties: lower key first), -1 padded. Returns int32 [n,k]."""
    scores, pos = _f64(scores), _i64(pos)
    n, S = scores.shape
    idx = np.empty((n, k), np.int32)
    _load().oracle_topk(_p(scores), _p(pos), n, S, k, _p(idx))
    return idx


def kv_up(ckv, W_UK, W_UV):
    """K^C [S,H,d_n] and V [S,H,d_v] from the latent ckv [S,d_c] (rows may be wider)."""
    ckv = _f32(ckv)
    W_UK, W_UV = _f32(W_UK), _f32(W_UV)
    H, d_n, d_c = W_UK.shape
    d_v = W_UV.shape[2]
    assert W_UV.shape == (H, d_c, d_v) and ckv.shape[1] >= d_c
    S = ckv.shape[0]
    KC = np.empty((S, H, d_n), np.float64)
    V = np.empty((S, H, d_v), np.float64)
    _load().oracle_kv_up(_p(ckv), S, ckv.shape[1], _p(W_UK), _p(W_UV), H, d_n, d_c, d_v, _p(KC), _p(V))
    return KC, V


def sparse_mla_unabsorbed(q_nope, q_pe, KC, kpe, V, idx, pos, scale: float):
    q_nope, q_pe, kpe = _f32(q_nope), _f32(q_pe), _f32(kpe)
    KC, V, idx, pos = _f64(KC), _f64(V), _i32(idx), _i64(pos)
    n, H, d_n = q_nope.shape
    d_r = q_pe.shape[2]
    S, _, d_v = V.shape
    k = idx.shape[1]
    out = np.empty((n, H, d_v), np.float64)
    lse = np.empty((n, H), np.float64)
    _load().oracle_sparse_mla_unabsorbed(_p(q_nope), _p(q_pe), _p(KC), _p(kpe), kpe.shape[1], _p(V), _p(idx),
                                         _p(pos), n, k, S, H, d_n, d_r, d_v, float(scale), _p(out), _p(lse))
    return out, lse


def sparse_mla_absorbed(q_nope, q_pe, ckv, kpe, W_UK, W_UV, idx, pos, scale: float, want_intermediates=False):
    q_nope, q_pe, ckv, kpe = _f32(q_nope), _f32(q_pe), _f32(ckv), _f32(kpe)
    W_UK, W_UV, idx, pos = _f32(W_UK), _f32(W_UV), _i32(idx), _i64(pos)
    n, H, d_n = q_nope.shape
    d_r = q_pe.shape[2]
    d_c = W_UK.shape[2]
    d_v = W_UV.shape[2]
    S = ckv.shape[0]
    k = idx.shape[1]
    out = np.empty((n, H, d_v), np.float64)
    lse = np.empty((n, H), np.float64)
    qt = np.empty((n, H, d_c), np.float64) if want_intermediates else None
    ol = np.empty((n, H, d_c), np.float64) if want_intermediates else None
    _load().oracle_sparse_mla_absorbed(_p(q_nope), _p(q_pe), _p(ckv), ckv.shape[1], _p(kpe), kpe.shape[1],
                                       _p(W_UK), _p(W_UV), _p(idx), _p(pos), n, k, S, H, d_n, d_r, d_c, d_v,
                                       float(scale), _p(out), _p(lse), _p(qt), _p(ol))
    if want_intermediates:
        return out, lse, qt, ol
    return out, lse


def dense_masked_mla(q_nope, q_pe, KC, kpe, V, pos, scale: float, sel=None):
    q_nope, q_pe, kpe = _f32(q_nope), _f32(q_pe), _f32(kpe)
    KC, V, pos = _f64(KC), _f64(V), _i64(pos)
    n, H, d_n = q_nope.shape
    d_r = q_pe.shape[2]
    S, _, d_v = V.shape
    sel_arr = None if sel is None else np.ascontiguousarray(np.asarray(sel, dtype=np.uint8))
    out = np.empty((n, H, d_v), np.float64)
    lse = np.empty((n, H), np.float64)
    _load().oracle_dense_masked_mla(_p(q_nope), _p(q_pe), _p(KC), _p(kpe), kpe.shape[1], _p(V), _p(sel_arr),
                                    _p(pos), n, S, H, d_n, d_r, d_v, float(scale), _p(out), _p(lse))
    return out, lse


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code) & 0xFF)


def quant_e4m3_ue8m0(x):
    """Blocks of 128 values -> (codes uint8 [nb,128], exps int32 [nb]); scale = 2**exps."""
    x = _f32(x).reshape(-1)
    assert x.size % 128 == 0
    nb = x.size // 128
    codes = np.empty((nb, 128), np.uint8)
    exps = np.empty((nb,), np.int32)
    _load().oracle_quant_e4m3_ue8m0(_p(x), nb, _p(codes), _p(exps))
    return codes, exps


def dequant_e4m3(codes, exps):
    """Exact dequantised values code * 2**exp as float32 (exactly representable)."""
    table = np.array([e4m3_value(c) for c in range(256)], np.float64)
    vals = table[np.asarray(codes, np.int64)] * np.ldexp(1.0, np.asarray(exps, np.int64))[..., None]
    return vals.astype(np.float32)


def dsa_rows(qI, w, kI, q_nope, q_pe, ckv, kpe, W_UK, W_UV, pos, k: int, scale: float, KC=None, V=None):
    """The whole path for rows of one sequence, as the pages define it:
    indexer scores with the causal mask -> top-k -> unabsorbed sparse latent
    attention.  Returns dict(scores, absterm, idx, out, lse)."""
    scores, absterm = indexer_scores(qI, w, kI, pos, with_absterm=True)
    idx = topk(scores, pos, k)
    if KC is None or V is None:
        KC, V = kv_up(ckv, W_UK, W_UV)
    out, lse = sparse_mla_unabsorbed(q_nope, q_pe, KC, kpe, V, idx, pos, scale)
    return dict(scores=scores, absterm=absterm, idx=idx, out=out, lse=lse)


# ---------------------------------------------------------------------------
# The projections on either side of the path (oracle.c section 8)
# ---------------------------------------------------------------------------
def linear(x, W):
    """y = x W^T for x [n, D] and W [N, D] (nn.Linear without bias), in float64."""
    x, W = _f32(x), _f32(W)
    n, D = x.shape
    N = W.shape[0]
    assert W.shape[1] == D
    y = np.empty((n, N), np.float64)
    _load().oracle_linear(_p(x), _p(W), n, D, N, _p(y))
    return y


def rmsnorm(x, gain, eps: float = 1e-6):
    x, gain = _f64(x), _f32(gain)
    n, d = x.shape
    y = np.empty((n, d), np.float64)
    _load().oracle_rmsnorm(_p(x), n, d, _p(gain), float(eps), _p(y))
    return y


def layernorm(x, gain, bias, eps: float = 1e-6):
    x, gain, bias = _f64(x), _f32(gain), _f32(bias)
    n, d = x.shape
    y = np.empty((n, d), np.float64)
    _load().oracle_layernorm(_p(x), n, d, _p(gain), _p(bias), float(eps), _p(y))
    return y


def rope_deinterleave(x, cos_t, sin_t):
    """x [n, 2*half] float64; cos_t, sin_t [n, half] (each row's angles)."""
    x, cos_t, sin_t = _f64(x), _f32(cos_t), _f32(sin_t)
    n, d = x.shape
    half = d // 2
    assert cos_t.shape == (n, half) and sin_t.shape == (n, half)
    y = np.empty((n, d), np.float64)
    _load().oracle_rope_deinterleave(_p(x), n, half, _p(cos_t), _p(sin_t), _p(y))
    return y


def kv_prologue(x, W_proj, kv_gain, k_gain, k_bias, cos_t, sin_t, d_c: int = 512, d_r: int = 64,
                D_I: int = 128, H_I: int = 64, eps: float = 1e-6):
    """The step before the path for rows x [n, dim], in the pages' order.
    W_proj stacks the three projections that read x: rows 0 .. d_c+d_r-1 are
    wkv_a, the next D_I rows wk, the last H_I rows weights_proj.  Returns
    dict(latent [n, d_c], k_pe [n, d_r], kI [n, D_I], w [n, H_I]) in float64."""
    y = linear(x, W_proj)
    kv, k_pe = y[:, :d_c], y[:, d_c:d_c + d_r]
    kI = y[:, d_c + d_r:d_c + d_r + D_I]
    w = y[:, d_c + d_r + D_I:d_c + d_r + D_I + H_I]
    return dict(latent=rmsnorm(kv, kv_gain, eps), k_pe=rope_deinterleave(k_pe, cos_t, sin_t),
                kI=layernorm(kI, k_gain, k_bias, eps), w=np.array(w))


def output_proj(out, wo):
    """y = out wo^T for the attention output out [n, H, d_v] (heads side by
    side, [n, H * d_v]) and wo [dim, H * d_v]."""
    out = np.asarray(out)
    return linear(out.reshape(out.shape[0], -1), wo)
