"""ctypes declarations of libdsa's C ABI (include/dsa.h)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_WORKSPACE = range(6)
DSA_F32, DSA_BF16, DSA_E4M3 = 0, 1, 2
DSA_MAX_SEQS = 1024
DSA_NOALLOC_SCRATCH_BYTES = 64 << 20

KERNEL_BITS = {
    "quant": 1 << 0, "indexer_simt": 1 << 1, "indexer_tc": 1 << 2, "indexer_fp8": 1 << 3, "topk": 1 << 4,
    "absorb_simt": 1 << 5, "absorb_tc": 1 << 6, "mla_simt": 1 << 7, "mla_tc": 1 << 8, "combine": 1 << 9,
    "selftest": 1 << 10, "dense_idx": 1 << 11, "gemm_tc": 1 << 12, "prologue": 1 << 13,
    "indexer_topk": 1 << 14, "append": 1 << 15,
}


class dsa_seqs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("cu_q", ctypes.POINTER(ctypes.c_int32)),
                ("cu_k", ctypes.POINTER(ctypes.c_int32)), ("start_pos", ctypes.POINTER(ctypes.c_int32))]


class dsa_problem(ctypes.Structure):
    _fields_ = [
        ("H_I", ctypes.c_int32), ("D_I", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("H", ctypes.c_int32), ("d_n", ctypes.c_int32), ("d_r", ctypes.c_int32), ("d_c", ctypes.c_int32),
        ("d_v", ctypes.c_int32), ("dtype", ctypes.c_int32), ("idx_fp8", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("q_idx", ctypes.c_void_p), ("k_idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
        ("q_nope", ctypes.c_void_p), ("q_pe", ctypes.c_void_p), ("kv_cache", ctypes.c_void_p),
        ("ld_kv", ctypes.c_int64), ("k_pe", ctypes.c_void_p), ("ld_pe", ctypes.c_int64),
        ("W_UK", ctypes.c_void_p), ("W_UV", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("idx_out", ctypes.c_void_p),
        ("wo", ctypes.c_void_p), ("d_model", ctypes.c_int32), ("y", ctypes.c_void_p),
        ("kv_fp8", ctypes.c_int32), ("kv_scale", ctypes.c_void_p),
    ]


class dsa_host_io(ctypes.Structure):
    _fields_ = [
        ("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p), ("q_nope", ctypes.c_void_p), ("q_pe", ctypes.c_void_p),
        ("kv_new", ctypes.c_void_p), ("k_pe_new", ctypes.c_void_p), ("k_idx_new", ctypes.c_void_p),
        ("kv_scale_new", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("idx", ctypes.c_void_p),
        ("compute_after", ctypes.c_void_p), ("compute_done", ctypes.c_void_p),
        ("copy_after", ctypes.c_void_p), ("copy_done", ctypes.c_void_p),
    ]


# (name, restype, argtypes) of every exported function
P, I, I64, F, SZ, U32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint32
SEQS = ctypes.POINTER(dsa_seqs)
PROB = ctypes.POINTER(dsa_problem)
SIGNATURES = [
    ("dsa_quant_e4m3_ue8m0", I, [P, I, I64, P, P, P]),
    ("dsa_indexer_scores", I, [P, P, P, P, I, P, I, I, SEQS, P, I64, P]),
    ("dsa_topk_select", I, [P, I64, SEQS, I, P, P]),
    ("dsa_sparse_mla_workspace_size", SZ, [I, I, I, I, I, I, I, SEQS]),
    ("dsa_sparse_mla_fwd", I, [P, P, I, P, I64, P, I64, P, P, I, I, I, I, I, P, I, SEQS, F, P, P, P, SZ, P]),
    ("dsa_sparse_mla_fwd_fp8kv", I, [P, P, P, I64, P, P, I64, P, P, I, I, I, I, I, P, I, SEQS, F, P, P, P, SZ, P]),
    ("dsa_sparse_mla_fwd_noalloc", I, [P, P, I, P, I64, P, I64, P, P, I, I, I, I, I, P, I, SEQS, F, P, P, P]),
    ("dsa_kv_prologue_workspace_size", SZ, [I, I, I, I, I, SEQS]),
    ("dsa_kv_prologue", I, [P, I, P, P, P, P, P, P, I, I, I, I, I, SEQS, P, I64, P, I, P, P, P, SZ, P]),
    ("dsa_output_proj", I, [P, P, I, I, I, P, P]),
    ("dsa_forward_workspace_size", SZ, [PROB, SEQS]),
    ("dsa_forward", I, [PROB, SEQS, P, SZ, P]),
    ("dsa_forward_host", I, [PROB, SEQS, ctypes.POINTER(dsa_host_io), P, SZ, P]),
    ("dsa_status_string", ctypes.c_char_p, [I]),
    ("dsa_last_cuda_error", I, []),
    ("dsa_check_device_error", I, [P, ctypes.POINTER(ctypes.c_int)]),
    ("dsa_selftest_bounded_wait", I, [I64, P, P]),
    ("dsa_set_wait_limit", I, [I64]),
    ("dsa_set_fused_topk", I, [I]),
    ("dsa_last_kernels", U32, []),
    ("dsa_last_launch_count", I, []),
    ("dsa_set_stage_events", I, [ctypes.POINTER(ctypes.c_void_p), I]),
]
DSA_STAGE_EVENTS = 6

_lib = None


def load(path: str = LIB_PATH):
    """Load libdsa.so.  There is no fallback: a missing library is an error."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdsa.so is not built ({path}); run __graft_entry__.build() "
                           "or python -m sparse_latent_attention_indexer_gb300.build")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib
