"""CPU-only checks of the C ABI: the library loads, exports every function
include/dsa.h declares, and validates arguments on the host (an invalid call
returns an error status before any CUDA call is made)."""
import ctypes
import os
import re

import pytest

import sparse_latent_attention_indexer_gb300 as dsa
from sparse_latent_attention_indexer_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(dsa_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function():
    lib = _abi.load()
    names = _declared_functions()
    assert len(names) >= 12, names
    for n in names:
        assert hasattr(lib, n), f"libdsa.so does not export {n}"
    assert sorted(n for n, _, _ in _abi.SIGNATURES) == names


def test_status_strings():
    lib = _abi.load()
    assert lib.dsa_status_string(0) == b"DSA_OK"
    assert lib.dsa_status_string(5) == b"DSA_ERR_WORKSPACE"


def _seqs(T, S, P):
    return dsa.Seqs.from_lengths(T, S, P)


def test_invalid_sequences_rejected_before_launch():
    lib = _abi.load()
    bad = _seqs([4], [3], [0])         # start_pos + T > S
    st = lib.dsa_topk_select(ctypes.c_void_p(16), 4, bad.ref(), 8, ctypes.c_void_p(16), None)
    assert st == _abi.DSA_ERR_INVALID_ARG
    good = _seqs([4], [8], [2])
    assert lib.dsa_topk_select(ctypes.c_void_p(16), 8, good.ref(), 0, ctypes.c_void_p(16), None) == 1  # k = 0
    assert lib.dsa_topk_select(ctypes.c_void_p(16), 4, good.ref(), 8, ctypes.c_void_p(16), None) == 1  # ld < S
    none = _abi.dsa_seqs(0, None, None, None)
    assert lib.dsa_topk_select(ctypes.c_void_p(16), 8, ctypes.byref(none), 8, ctypes.c_void_p(16), None) == 1


def test_indexer_shape_checks():
    lib = _abi.load()
    s = _seqs([2], [4], [0])
    P = ctypes.c_void_p(256)
    # E4M3 needs D_I = 128 and scales
    assert lib.dsa_indexer_scores(P, None, P, None, _abi.DSA_E4M3, P, 4, 64, s.ref(), P, 4, None) == 2
    assert lib.dsa_indexer_scores(P, None, P, None, _abi.DSA_E4M3, P, 4, 128, s.ref(), P, 4, None) == 1
    assert lib.dsa_indexer_scores(P, None, P, None, _abi.DSA_BF16, P, 256, 128, s.ref(), P, 4, None) == 2
    assert lib.dsa_indexer_scores(P, None, P, None, _abi.DSA_BF16, P, 4, 32, s.ref(), P, 3, None) == 1  # ld % 4


def _problem(**over):
    p = _abi.dsa_problem()
    p.H_I, p.D_I, p.top_k = 64, 128, 2048
    p.H, p.d_n, p.d_r, p.d_c, p.d_v = 128, 128, 64, 512, 128
    p.dtype, p.idx_fp8, p.softmax_scale = _abi.DSA_BF16, 0, 192 ** -0.5
    for n in ("q_idx", "k_idx", "w", "q_nope", "q_pe", "kv_cache", "k_pe", "W_UK", "W_UV", "out"):
        setattr(p, n, 4096)
    p.ld_kv = p.ld_pe = 576
    for k, v in over.items():
        setattr(p, k, v)
    return p


def test_forward_workspace_size_is_host_logic():
    lib = _abi.load()
    s = _seqs([4096], [4096], [0])
    p = _problem()
    ws = lib.dsa_forward_workspace_size(ctypes.byref(p), s.ref())
    assert ws > 0 and ws % 256 == 0
    # the selection lives in the workspace unless the caller gives idx_out
    p2 = _problem(idx_out=8192)
    assert lib.dsa_forward_workspace_size(ctypes.byref(p2), s.ref()) == ws - 4096 * 2048 * 4
    # FP8 indexer adds the quantised copies
    p3 = _problem(idx_fp8=1)
    assert lib.dsa_forward_workspace_size(ctypes.byref(p3), s.ref()) > ws
    # unsupported dtype -> 0
    assert lib.dsa_forward_workspace_size(ctypes.byref(_problem(dtype=_abi.DSA_E4M3)), s.ref()) == 0


def test_forward_rejects_small_workspace():
    lib = _abi.load()
    s = _seqs([16], [16], [0])
    p = _problem()
    need = lib.dsa_forward_workspace_size(ctypes.byref(p), s.ref())
    st = lib.dsa_forward(ctypes.byref(p), s.ref(), ctypes.c_void_p(1 << 20), need - 256, None)
    assert st == _abi.DSA_ERR_WORKSPACE
    st = lib.dsa_forward(ctypes.byref(p), s.ref(), ctypes.c_void_p((1 << 20) + 8), need, None)  # misaligned
    assert st == _abi.DSA_ERR_WORKSPACE


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _abi.load(str(tmp_path / "libdsa.so"))


def test_bounded_wait_selftest_rejects_out_of_range_limits():
    lib = _abi.load()
    assert lib.dsa_selftest_bounded_wait(0, None, None) == _abi.DSA_ERR_INVALID_ARG
    assert lib.dsa_selftest_bounded_wait((1 << 32) + 1, None, None) == _abi.DSA_ERR_INVALID_ARG


def test_noalloc_scratch_holds_the_documented_batch():
    """dsa_sparse_mla_fwd_noalloc accepts a call while the attention scratch
    (dsa_sparse_mla_workspace_size) fits DSA_NOALLOC_SCRATCH_BYTES; the header
    promises every decode batch of up to 128 query rows at the 671B head shapes.
    Host-side sizes only, so a later change of the scratch layout or of the key
    split count that breaks the promise fails here."""
    lib = _abi.load()

    def need(rows):
        s = _seqs([1] * rows, [4096] * rows, [4095] * rows)
        return lib.dsa_sparse_mla_workspace_size(_abi.DSA_BF16, 128, 128, 64, 512, 128, 2048, s.ref())

    for rows in range(1, 129):
        assert 0 < need(rows) <= _abi.DSA_NOALLOC_SCRATCH_BYTES, rows
    assert need(129) > _abi.DSA_NOALLOC_SCRATCH_BYTES


def test_wait_limit_range():
    lib = _abi.load()
    assert lib.dsa_set_wait_limit(-1) == _abi.DSA_ERR_INVALID_ARG
    assert lib.dsa_set_wait_limit((1 << 32) + 1) == _abi.DSA_ERR_INVALID_ARG
    assert lib.dsa_set_wait_limit(1000) == _abi.DSA_OK
    assert lib.dsa_set_wait_limit(0) == _abi.DSA_OK  # back to the default


def test_fused_topk_modes():
    lib = _abi.load()
    for m in (1, 0, -1):
        assert lib.dsa_set_fused_topk(m) == _abi.DSA_OK
    assert lib.dsa_set_fused_topk(2) == _abi.DSA_ERR_INVALID_ARG
    assert lib.dsa_set_fused_topk(-2) == _abi.DSA_ERR_INVALID_ARG


def test_forward_host_validates_before_any_copy():
    """dsa_forward_host checks its host/device pairing and the appended-row
    ranges on the host and returns before enqueueing a copy (no GPU here)."""
    lib = _abi.load()
    H = ctypes.c_void_p(1 << 16)
    s = _seqs([4], [8], [4])
    p = _problem()
    assert lib.dsa_forward_host(ctypes.byref(p), s.ref(), None, None, 0, None) == _abi.DSA_ERR_INVALID_ARG
    # an lse or idx copy-back needs the device buffer it reads
    io = _abi.dsa_host_io(lse=H.value)
    assert lib.dsa_forward_host(ctypes.byref(p), s.ref(), ctypes.byref(io), None, 0, None) == _abi.DSA_ERR_INVALID_ARG
    io = _abi.dsa_host_io(idx=H.value)
    assert lib.dsa_forward_host(ctypes.byref(p), s.ref(), ctypes.byref(io), None, 0, None) == _abi.DSA_ERR_INVALID_ARG
    # scales only for an e4m3 latent cache
    io = _abi.dsa_host_io(kv_scale_new=H.value)
    assert lib.dsa_forward_host(ctypes.byref(p), s.ref(), ctypes.byref(io), None, 0, None) == _abi.DSA_ERR_INVALID_ARG
    # appended rows start_pos .. S-1 need start_pos <= S
    bad = _seqs([1], [3], [5])
    io = _abi.dsa_host_io(kv_new=H.value)
    assert lib.dsa_forward_host(ctypes.byref(p), bad.ref(), ctypes.byref(io), None, 0, None) == _abi.DSA_ERR_INVALID_ARG
    # the problem itself is checked as dsa_forward checks it
    io = _abi.dsa_host_io()
    p_bad = _problem(dtype=_abi.DSA_E4M3)
    assert lib.dsa_forward_host(ctypes.byref(p_bad), s.ref(), ctypes.byref(io), None, 0, None) != _abi.DSA_OK


def test_batch_of_max_sequences_accepted_one_more_rejected():
    """A launch carries up to DSA_MAX_SEQS sequences in its parameters: a decode batch of exactly that
    many is sized, one more is refused (workspace size 0, INVALID_ARG from the call)."""
    lib = _abi.load()
    p = _problem(idx_out=8192)
    for B, ok in ((_abi.DSA_MAX_SEQS, True), (_abi.DSA_MAX_SEQS + 1, False)):
        s = _seqs([1] * B, [4096] * B, [4095] * B)
        ws = lib.dsa_forward_workspace_size(ctypes.byref(p), s.ref())
        assert (ws > 0) == ok, (B, ws)
        if not ok:
            assert lib.dsa_forward(ctypes.byref(p), s.ref(), ctypes.c_void_p(1 << 20), 1 << 30, None) == \
                _abi.DSA_ERR_INVALID_ARG


def test_forward_host_refuses_a_short_workspace_before_copying():
    """The forward's own checks (here: no workspace) run before the first copy, so the refusal needs no
    GPU and leaves the device buffers as they were."""
    lib = _abi.load()
    s = _seqs([4], [8], [4])
    p = _problem()
    io = _abi.dsa_host_io(q_nope=1 << 16)
    assert lib.dsa_forward_host(ctypes.byref(p), s.ref(), ctypes.byref(io), None, 0, None) == _abi.DSA_ERR_WORKSPACE


def test_ctypes_structs_match_the_header_layout(tmp_path):
    """The binding's ctypes structures have the size and field offsets that a C
    compiler gives the header's structures (a field added to one side only, or in
    another order, fails here)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    structs = [_abi.dsa_seqs, _abi.dsa_problem, _abi.dsa_host_io]
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "dsa.h"', "int main(void) {"]
    for st in structs:
        n = st.__name__
        lines.append(f'    printf("{n} size %zu\\n", sizeof({n}));')
        for f, _ in st._fields_:
            lines.append(f'    printf("{n} {f} %zu\\n", offsetof({n}, {f}));')
    lines += ["    return 0;", "}"]
    src, exe = tmp_path / "layout.c", tmp_path / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([gcc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        n, f, v = line.split()
        got[(n, f)] = int(v)
    for st in structs:
        n = st.__name__
        assert got[(n, "size")] == ctypes.sizeof(st), n
        for f, _ in st._fields_:
            assert got[(n, f)] == getattr(st, f).offset, (n, f)


def test_binding_constants_match_the_header():
    """The status codes, dtype codes, limits, stage count and kernel bits the
    binding uses are the values include/dsa.h defines (compiled, not parsed)."""
    import shutil
    import subprocess
    import tempfile

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    header = open(os.path.join(ROOT, "include", "dsa.h")).read()
    bits = re.findall(r"#define (DSA_KERNEL_[A-Z0-9_]+)\s", header)
    consts = ["DSA_OK", "DSA_ERR_INVALID_ARG", "DSA_ERR_UNSUPPORTED", "DSA_ERR_CUDA", "DSA_ERR_TIMEOUT",
              "DSA_ERR_WORKSPACE", "DSA_F32", "DSA_BF16", "DSA_E4M3", "DSA_MAX_SEQS", "DSA_NOALLOC_SCRATCH_BYTES",
              "DSA_STAGE_EVENTS"] + bits
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "c.c"), os.path.join(d, "c")
        with open(src, "w") as f:
            f.write('#include <stdio.h>\n#include "dsa.h"\nint main(void) {\n')
            for c in consts:
                f.write(f'    printf("{c} %llu\\n", (unsigned long long)({c}));\n')
            f.write("    return 0;\n}\n")
        subprocess.run([gcc, "-std=c11", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        got = dict(line.split() for line in subprocess.run([exe], check=True, capture_output=True,
                                                           text=True).stdout.splitlines())
    for c in consts[:12]:
        assert int(got[c]) == getattr(_abi, c), c
    named = {f"DSA_KERNEL_{k.upper()}": v for k, v in _abi.KERNEL_BITS.items()}
    assert {b: int(got[b]) for b in bits} == named
