"""DeepSeek sparse attention (DSA) hot path on GB300: lightning indexer ->
top-k -> absorbed sparse latent attention, in hand-written sm_103a CUDA
behind the C ABI of ``libdsa.so`` (include/dsa.h).

This module is the thin Python binding: it marshals torch tensors (device
memory, the current stream) into the C calls of the same names.  Every
arithmetic step runs in the CUDA kernels; there is no CPU fallback, and a
missing ``libdsa.so`` raises.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import DSA_BF16, DSA_E4M3, DSA_F32, KERNEL_BITS

__all__ = [
    "Seqs", "DSAError", "dsa_quant_e4m3_ue8m0", "dsa_indexer_scores", "dsa_topk_select",
    "dsa_sparse_mla_workspace_size", "dsa_sparse_mla_fwd", "dsa_forward_workspace_size", "dsa_forward",
    "dsa_check_device_error", "dsa_selftest_bounded_wait", "dsa_set_wait_limit", "dsa_set_fused_topk", "dsa_kv_prologue",
    "dsa_output_proj", "dsa_sparse_mla_fwd_fp8kv", "dsa_forward_host", "last_kernels", "last_launch_count", "build",
]


class DSAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = _abi.load()
        msg = lib.dsa_status_string(status).decode()
        if status == _abi.DSA_ERR_CUDA:
            msg += f" (cudaError {lib.dsa_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")
        self.status = status


def build(force: bool = False) -> str:
    from .build import build as _b
    return _b(force=force)


def _check(fn: str, status: int):
    if status != _abi.DSA_OK:
        raise DSAError(fn, status)


class Seqs:
    """A batch description (host arrays): cu_q [B+1], cu_k [B+1], start_pos [B]."""

    def __init__(self, cu_q, cu_k, start_pos):
        B = len(start_pos)
        assert len(cu_q) == B + 1 and len(cu_k) == B + 1
        self._q = (ctypes.c_int32 * (B + 1))(*[int(x) for x in cu_q])
        self._k = (ctypes.c_int32 * (B + 1))(*[int(x) for x in cu_k])
        self._p = (ctypes.c_int32 * max(B, 1))(*[int(x) for x in start_pos])
        self.struct = _abi.dsa_seqs(B, self._q, self._k, self._p)
        self.B = B
        self.total_q = int(cu_q[-1])
        self.total_k = int(cu_k[-1])
        self.max_S = max(int(cu_k[b + 1]) - int(cu_k[b]) for b in range(B)) if B else 0

    @classmethod
    def from_lengths(cls, T, S, start_pos):
        cu_q, cu_k = [0], [0]
        for t, s in zip(T, S):
            cu_q.append(cu_q[-1] + int(t))
            cu_k.append(cu_k[-1] + int(s))
        return cls(cu_q, cu_k, start_pos)

    def ref(self):
        return ctypes.byref(self.struct)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DSA_F32
    if t.dtype == torch.bfloat16:
        return DSA_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return DSA_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _row_stride(t: torch.Tensor) -> int:
    assert t.dim() == 2 and t.stride(1) == 1, "rows must be contiguous"
    return t.stride(0)


def last_kernels() -> set:
    bits = _abi.load().dsa_last_kernels()
    return {k for k, v in KERNEL_BITS.items() if bits & v}


def last_launch_count() -> int:
    return _abi.load().dsa_last_launch_count()


def dsa_check_device_error(stream=None):
    site = ctypes.c_int(0)
    st = _abi.load().dsa_check_device_error(_stream(stream), ctypes.byref(site))
    return st, site.value


def dsa_selftest_bounded_wait(limit_cycles: int, completed_ok=None, stream=None):
    """Launch the bounded-wait self-test (a wait that runs out after limit_cycles);
    read its outcome with dsa_check_device_error."""
    _check("dsa_selftest_bounded_wait",
           _abi.load().dsa_selftest_bounded_wait(int(limit_cycles), _ptr(completed_ok) if completed_ok is not None else None,
                                                 _stream(stream)))


def dsa_set_wait_limit(cycles: int):
    """Wait limit (SM cycles) of the tensor-core kernels' bounded waits; 0 restores the default."""
    _check("dsa_set_wait_limit", _abi.load().dsa_set_wait_limit(int(cycles)))


def dsa_set_fused_topk(mode):
    """Fused indexer + top-k for the dsa_forward calls that follow on large batches:
    True/1 wherever it applies, False/0 never, -1 the library's choice (default)."""
    m = -1 if mode == -1 else (1 if mode else 0)
    _check("dsa_set_fused_topk", _abi.load().dsa_set_fused_topk(m))


def dsa_quant_e4m3_ue8m0(x: torch.Tensor, codes=None, scales=None, stream=None):
    """x: [..., 128k] f32/bf16 -> (codes uint8 same shape, scales f32 [numel/128])."""
    x = x.contiguous()
    nb = x.numel() // 128
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = torch.empty(nb, dtype=torch.float32, device=x.device) if scales is None else scales
    _check("dsa_quant_e4m3_ue8m0", _abi.load().dsa_quant_e4m3_ue8m0(_ptr(x), _dt(x), nb, _ptr(codes), _ptr(scales),
                                                                    _stream(stream)))
    return codes, scales


def dsa_indexer_scores(q_idx, k_idx, w, seqs: Seqs, q_scale=None, k_scale=None, scores=None, ld=None, stream=None):
    H_I, D_I = q_idx.shape[-2], q_idx.shape[-1]
    if ld is None:
        ld = (max(seqs.max_S, 1) + 3) // 4 * 4
    if scores is None:
        scores = torch.empty((seqs.total_q, ld), dtype=torch.float32, device=q_idx.device)
    st = _abi.load().dsa_indexer_scores(_ptr(q_idx), _ptr(q_scale), _ptr(k_idx), _ptr(k_scale), _dt(q_idx), _ptr(w),
                                        H_I, D_I, seqs.ref(), _ptr(scores), scores.stride(0), _stream(stream))
    _check("dsa_indexer_scores", st)
    return scores


def dsa_topk_select(scores, seqs: Seqs, k: int, idx=None, stream=None):
    if idx is None:
        idx = torch.empty((seqs.total_q, k), dtype=torch.int32, device=scores.device)
    st = _abi.load().dsa_topk_select(_ptr(scores), scores.stride(0), seqs.ref(), k, _ptr(idx), _stream(stream))
    _check("dsa_topk_select", st)
    return idx


def dsa_sparse_mla_workspace_size(dtype: int, H: int, d_n: int, d_r: int, d_c: int, d_v: int, k: int,
                                  seqs: Seqs) -> int:
    return _abi.load().dsa_sparse_mla_workspace_size(dtype, H, d_n, d_r, d_c, d_v, k, seqs.ref())


def dsa_sparse_mla_fwd(q_nope, q_pe, kv_cache, k_pe, W_UK, W_UV, idx, seqs: Seqs, softmax_scale: float, out=None,
                       lse=None, workspace=None, want_lse=True, stream=None, k=None):
    """kv_cache and k_pe are 2-D views [sum S, d_c] / [sum S, d_r] with contiguous rows
    (k_pe may be a column slice of a packed cache).  idx=None selects the dense causal
    pattern (entry e of a row is key e) for k entries per row."""
    M, H, d_n = q_nope.shape
    d_r = q_pe.shape[2]
    d_c = W_UK.shape[2]
    d_v = W_UV.shape[2]
    if idx is not None:
        k = idx.shape[1]
    elif k is None:
        raise ValueError("dsa_sparse_mla_fwd: idx=None needs k")
    dt = _dt(q_nope)
    dev = q_nope.device
    if out is None:
        out = torch.empty((M, H, d_v), dtype=q_nope.dtype, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((M, H), dtype=torch.float32, device=dev)
    need = dsa_sparse_mla_workspace_size(dt, H, d_n, d_r, d_c, d_v, k, seqs)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = _abi.load().dsa_sparse_mla_fwd(_ptr(q_nope), _ptr(q_pe), dt, _ptr(kv_cache), _row_stride(kv_cache), _ptr(k_pe),
                                        _row_stride(k_pe), _ptr(W_UK), _ptr(W_UV), H, d_n, d_r, d_c, d_v, _ptr(idx), k,
                                        seqs.ref(), float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                        workspace.numel(), _stream(stream))
    _check("dsa_sparse_mla_fwd", st)
    return out, lse


def dsa_kv_prologue(x, W_proj, kv_gain, k_gain, k_bias, rope_cos, rope_sin, seqs: Seqs, kv_cache, k_cache, w=None,
                    k_scale=None, d_c=512, d_r=64, D_I=128, H_I=64, workspace=None, stream=None):
    """The step before the path for the new tokens x [sum T, dim]: writes their
    rows of kv_cache ([sum S, >= d_c + d_r] bf16) and k_cache ([sum S, D_I] bf16,
    or uint8 e4m3 codes with k_scale [sum S]) and returns w [sum T, H_I]."""
    dim = x.shape[1]
    dev = x.device
    if w is None:
        w = torch.empty((seqs.total_q, H_I), dtype=torch.float32, device=dev)
    k_dtype = DSA_E4M3 if k_cache.dtype in (torch.uint8, torch.float8_e4m3fn) else DSA_BF16
    lib = _abi.load()
    need = lib.dsa_kv_prologue_workspace_size(dim, d_c, d_r, D_I, H_I, seqs.ref())
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = lib.dsa_kv_prologue(_ptr(x), dim, _ptr(W_proj), _ptr(kv_gain), _ptr(k_gain), _ptr(k_bias), _ptr(rope_cos),
                             _ptr(rope_sin), rope_cos.shape[0], d_c, d_r, D_I, H_I, seqs.ref(), _ptr(kv_cache),
                             _row_stride(kv_cache), _ptr(k_cache), k_dtype, _ptr(k_scale), _ptr(w), _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check("dsa_kv_prologue", st)
    return w


def dsa_output_proj(out, wo, y=None, stream=None):
    """y = out wo^T with out [M, H, d_v] (or [M, H * d_v]) and wo [d_model, H * d_v], bf16."""
    M = out.shape[0]
    K = out[0].numel() if M else wo.shape[1]
    d_model = wo.shape[0]
    if y is None:
        y = torch.empty((M, d_model), dtype=out.dtype, device=out.device)
    _check("dsa_output_proj", _abi.load().dsa_output_proj(_ptr(out), _ptr(wo), M, K, d_model, _ptr(y), _stream(stream)))
    return y


def dsa_sparse_mla_fwd_fp8kv(q_nope, q_pe, kv_codes, kv_scale, k_pe, W_UK, W_UV, idx, seqs: Seqs,
                             softmax_scale: float, out=None, lse=None, workspace=None, stream=None):
    """The sparse attention over an FP8 latent cache: kv_codes [sum S, >= d_c] uint8
    e4m3 codes with kv_scale [sum S, d_c / 128] fp32 block scales; k_pe bf16."""
    M, H, d_n = q_nope.shape
    d_r, d_c, d_v = q_pe.shape[2], W_UK.shape[2], W_UV.shape[2]
    k = idx.shape[1]
    dev = q_nope.device
    if out is None:
        out = torch.empty((M, H, d_v), dtype=q_nope.dtype, device=dev)
    if lse is None:
        lse = torch.empty((M, H), dtype=torch.float32, device=dev)
    need = dsa_sparse_mla_workspace_size(DSA_BF16, H, d_n, d_r, d_c, d_v, k, seqs)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = _abi.load().dsa_sparse_mla_fwd_fp8kv(_ptr(q_nope), _ptr(q_pe), _ptr(kv_codes), _row_stride(kv_codes),
                                              _ptr(kv_scale), _ptr(k_pe), _row_stride(k_pe), _ptr(W_UK), _ptr(W_UV), H,
                                              d_n, d_r, d_c, d_v, _ptr(idx), k, seqs.ref(), float(softmax_scale),
                                              _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                              _stream(stream))
    _check("dsa_sparse_mla_fwd_fp8kv", st)
    return out, lse


def _problem(q_idx, k_idx, w, q_nope, q_pe, kv_cache, k_pe, W_UK, W_UV, top_k, softmax_scale, idx_fp8, out, lse,
             idx_out, wo=None, y=None, kv_scale=None):
    p = _abi.dsa_problem()
    p.H_I, p.D_I = q_idx.shape[-2], q_idx.shape[-1]
    p.top_k = top_k
    p.H, p.d_n = q_nope.shape[1], q_nope.shape[2]
    p.d_r = q_pe.shape[2]
    p.d_c = W_UK.shape[2]
    p.d_v = W_UV.shape[2]
    p.dtype = _dt(q_nope)
    p.idx_fp8 = 1 if idx_fp8 else 0
    p.softmax_scale = float(softmax_scale)
    p.q_idx, p.k_idx, p.w = q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr()
    p.q_nope, p.q_pe = q_nope.data_ptr(), q_pe.data_ptr()
    p.kv_cache, p.ld_kv = kv_cache.data_ptr(), _row_stride(kv_cache)
    p.k_pe, p.ld_pe = k_pe.data_ptr(), _row_stride(k_pe)
    p.W_UK, p.W_UV = W_UK.data_ptr(), W_UV.data_ptr()
    p.out = out.data_ptr() if out is not None else None
    p.lse = lse.data_ptr() if lse is not None else None
    p.idx_out = idx_out.data_ptr() if idx_out is not None else None
    if wo is not None:
        p.wo, p.d_model, p.y = wo.data_ptr(), wo.shape[0], y.data_ptr()
    if kv_scale is not None:
        p.kv_fp8, p.kv_scale = 1, kv_scale.data_ptr()
    return p


def dsa_forward_workspace_size(problem, seqs: Seqs) -> int:
    return _abi.load().dsa_forward_workspace_size(ctypes.byref(problem), seqs.ref())


def dsa_forward(q_idx, k_idx, w, q_nope, q_pe, kv_cache, k_pe, W_UK, W_UV, seqs: Seqs, top_k: int,
                softmax_scale: float, idx_fp8: bool = False, out=None, lse=None, idx_out=None, workspace=None,
                want_lse=True, want_idx=True, stream=None, wo=None, y=None, want_out=True, kv_scale=None):
    """The whole path.  Returns (out [sum T, H, d_v] or None, lse [sum T, H] or None,
    idx [sum T, top_k] or None), plus y [sum T, d_model] = out wo^T when wo is given
    (the step after the path; with want_out=False the attention output stays in
    the workspace).  With kv_scale, kv_cache holds the latent rows as e4m3 codes
    (uint8) with kv_scale [sum S, d_c / 128] block scales."""
    dev = q_nope.device
    M, H = q_nope.shape[0], q_nope.shape[1]
    if out is None and (want_out or wo is None):
        out = torch.empty((M, H, W_UV.shape[2]), dtype=q_nope.dtype, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((M, H), dtype=torch.float32, device=dev)
    if idx_out is None and want_idx:
        idx_out = torch.empty((M, top_k), dtype=torch.int32, device=dev)
    if wo is not None and y is None:
        y = torch.empty((M, wo.shape[0]), dtype=q_nope.dtype, device=dev)
    p = _problem(q_idx, k_idx, w, q_nope, q_pe, kv_cache, k_pe, W_UK, W_UV, top_k, softmax_scale, idx_fp8, out, lse,
                 idx_out, wo, y, kv_scale)
    need = dsa_forward_workspace_size(p, seqs)
    if need == 0 and M > 0:
        raise DSAError("dsa_forward_workspace_size", _abi.DSA_ERR_INVALID_ARG)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        if stream is not None:  # freed on return while the call's kernels may still run on `stream`
            workspace.record_stream(stream)
    st = _abi.load().dsa_forward(ctypes.byref(p), seqs.ref(), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("dsa_forward", st)
    if wo is not None:
        return out, lse, idx_out, y
    return out, lse, idx_out


def dsa_forward_host(host: dict, q_idx, k_idx, w, q_nope, q_pe, kv_cache, k_pe, W_UK, W_UV, seqs: Seqs, top_k: int,
                     softmax_scale: float, idx_fp8: bool = False, out=None, lse=None, idx_out=None, workspace=None,
                     stream=None, wo=None, y=None, kv_scale=None, compute_after=None, compute_done=None,
                     copy_after=None, copy_done=None):
    """One step from HOST tensors (the end-to-end call).  ``host`` maps names to CPU
    tensors (pinned for asynchronous copies): inputs ``q_idx``, ``w``, ``q_nope``,
    ``q_pe`` (the step's queries) and ``kv_new``, ``k_pe_new``, ``k_idx_new``,
    ``kv_scale_new`` (the cache rows the step appends: rows start_pos[b] .. S_b - 1
    of every sequence, concatenated), outputs ``out`` (y with wo), ``lse``, ``idx``;
    a missing name is not copied.  The device tensors are the buffers the copies fill
    and the forward reads and writes.  Everything is enqueued on ``stream``, except the
    copies of q_nope and q_pe, which run on the library's side stream while the indexer
    runs (the attention waits for them on ``stream``); returns without synchronising.  ``compute_after`` / ``compute_done`` (torch.cuda.Event):
    the forward waits for the first after the input copies and records the second
    before the output copies, to chain the forwards of calls on two streams;
    ``copy_after`` / ``copy_done``: the input copies wait for the first and the
    second is recorded once they (and the append kernel) are enqueued, to chain
    the input copies of calls on two streams."""
    lib = _abi.load()
    p = _problem(q_idx, k_idx, w, q_nope, q_pe, kv_cache, k_pe, W_UK, W_UV, top_k, softmax_scale, idx_fp8, out, lse,
                 idx_out, wo, y, kv_scale)
    io = _abi.dsa_host_io()
    for name in ("q_idx", "w", "q_nope", "q_pe", "kv_new", "k_pe_new", "k_idx_new", "kv_scale_new", "out", "lse",
                 "idx"):
        ten = host.get(name)
        if ten is not None:
            if ten.device.type != "cpu" or not ten.is_contiguous():
                raise ValueError(f"host tensor {name} must be a contiguous CPU tensor")
            setattr(io, name, ten.data_ptr())
    for name, ev in (("compute_after", compute_after), ("compute_done", compute_done), ("copy_after", copy_after),
                     ("copy_done", copy_done)):
        if ev is not None:
            if not ev.cuda_event:  # torch creates the CUDA event on its first record
                ev.record()
            setattr(io, name, ev.cuda_event)
    need = dsa_forward_workspace_size(p, seqs)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q_nope.device)
        if stream is not None:  # freed on return while the call's kernels may still run on `stream`
            workspace.record_stream(stream)
    st = lib.dsa_forward_host(ctypes.byref(p), seqs.ref(), ctypes.byref(io), _ptr(workspace), workspace.numel(),
                              _stream(stream))
    _check("dsa_forward_host", st)


def set_stage_events(events):
    """Record ``events`` (DSA_STAGE_EVENTS torch.cuda.Event objects, or None to
    switch off) at the stage boundaries of the next dsa_forward calls."""
    lib = _abi.load()
    if events is None:
        _check("dsa_set_stage_events", lib.dsa_set_stage_events(None, 0))
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check("dsa_set_stage_events", lib.dsa_set_stage_events(arr, len(events)))
