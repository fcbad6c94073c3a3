"""dsa_forward_host: one step from host buffers.  The step's queries and the
cache rows it appends are copied in from pinned host memory, the forward runs,
and the outputs come back to host memory.  On the same inputs the host outputs
must equal, bit for bit, the outputs of dsa_forward on device-resident inputs,
and the appended rows must land in the device caches at rows
cu_k[b] + start_pos[b] .. cu_k[b+1] - 1 while the rows before them (the cache
earlier steps left) are untouched."""
import pytest
import torch

import dsa_inputs as di
import sparse_latent_attention_indexer_gb300 as dsa
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _appended(wl, x):
    """The rows start_pos[b] .. S_b - 1 of every sequence of a [sum S, ...] host tensor, in order."""
    return torch.cat([x[wl.cu_k[b] + wl.start_pos[b]:wl.cu_k[b + 1]] for b in range(wl.B)]).contiguous()


@pytest.mark.parametrize("fp8", [False, True])
def test_forward_from_host_buffers_equals_device_forward(fp8):
    shape = di.Shape(k=128, idx_fp8=fp8)
    # chunked prefill: three sequences with resident prefixes and new rows; one decode-like row
    wl = di.generate(f"host-io-{fp8}", shape, 71, [300, 96, 1], [1500, 96, 2200], [1200, 0, 2199])
    sh = wl.shape
    ref = H.to_device(wl)
    out_r, lse_r, idx_r = H.gpu_forward(wl, ref)
    assert dsa.dsa_check_device_error() == (0, 0)

    host = wl.tensors
    # device buffers: the cache rows before start_pos are resident, the appended rows and the
    # queries hold garbage until the call copies them in
    dev = {k: torch.full_like(ref[k], 7.0) for k in ("qI", "w", "q_nope", "q_pe")}
    for k in ("kv_cache", "kI"):
        buf = ref[k].clone()
        for b in range(wl.B):
            buf[wl.cu_k[b] + wl.start_pos[b]:wl.cu_k[b + 1]] = -3.0
        dev[k] = buf
    d_c = sh.d_c
    pinned = {
        "q_idx": host["qI"].pin_memory(), "w": host["w"].pin_memory(), "q_nope": host["q_nope"].pin_memory(),
        "q_pe": host["q_pe"].pin_memory(),
        "kv_new": _appended(wl, host["kv_cache"]).pin_memory(),  # k_pe is inside the latent rows
        "k_idx_new": _appended(wl, host["kI"]).pin_memory(),
        "out": torch.empty(out_r.shape, dtype=out_r.dtype).pin_memory(),
        "lse": torch.empty(lse_r.shape, dtype=lse_r.dtype).pin_memory(),
        "idx": torch.empty(idx_r.shape, dtype=idx_r.dtype).pin_memory(),
    }
    out_d = torch.empty_like(out_r)
    lse_d = torch.empty_like(lse_r)
    idx_d = torch.empty_like(idx_r)
    stream = torch.cuda.current_stream()
    dsa.dsa_forward_host(pinned, dev["qI"], dev["kI"], dev["w"], dev["q_nope"], dev["q_pe"],
                         dev["kv_cache"][:, :d_c], dev["kv_cache"][:, d_c:], ref["W_UK"], ref["W_UV"], H.seqs_of(wl),
                         sh.k, sh.softmax_scale, idx_fp8=sh.idx_fp8, out=out_d, lse=lse_d, idx_out=idx_d,
                         stream=stream)
    stream.synchronize()
    assert dsa.dsa_check_device_error() == (0, 0)
    # the copies filled the device buffers: queries and appended rows as on the host, resident rows kept
    for k in ("qI", "w", "q_nope", "q_pe", "kv_cache", "kI"):
        assert torch.equal(dev[k], ref[k]), k
    # the host outputs are the device forward's, bit for bit
    assert torch.equal(pinned["idx"], idx_r.cpu())
    assert torch.equal(pinned["out"], out_r.cpu())
    assert torch.equal(pinned["lse"], lse_r.cpu())
    assert torch.equal(out_d, out_r)


def test_forward_from_host_pageable_and_partial_copies():
    """Pageable host tensors work too (the copies then block), and an input left out
    (NULL) is read from the device buffer as it stands."""
    wl = di.generate("host-io-pageable", di.Shape(k=64), 72, [40, 9], [300, 9], [260, 0])
    sh = wl.shape
    ref = H.to_device(wl)
    out_r, lse_r, idx_r = H.gpu_forward(wl, ref)
    dev_q = torch.zeros_like(ref["q_nope"])
    host = {"q_nope": wl.tensors["q_nope"].contiguous(), "out": torch.empty(out_r.shape, dtype=out_r.dtype)}
    dsa.dsa_forward_host(host, ref["qI"], ref["kI"], ref["w"], dev_q, ref["q_pe"], ref["ckv"], ref["kpe"],
                         ref["W_UK"], ref["W_UV"], H.seqs_of(wl), sh.k, sh.softmax_scale,
                         out=torch.empty_like(out_r), lse=torch.empty_like(lse_r), idx_out=torch.empty_like(idx_r))
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_error() == (0, 0)
    assert torch.equal(host["out"], out_r.cpu())


@pytest.mark.parametrize("chain_copies", [False, True])
def test_two_streams_chained_by_compute_events(chain_copies):
    """Two calls per slot on two streams, each forward waiting for the previous
    step's (compute_after / compute_done), and with chain_copies each call's input
    copies waiting for the previous call's (copy_after / copy_done): every host
    output still equals the device forward's, bit for bit."""
    wl = di.generate("host-io-chain", di.Shape(k=64), 73, [70, 30], [500, 30], [430, 0])
    sh = wl.shape
    ref = H.to_device(wl)
    out_r, lse_r, idx_r = H.gpu_forward(wl, ref)
    torch.cuda.synchronize()
    host_in = {"q_idx": wl.tensors["qI"].pin_memory(), "w": wl.tensors["w"].pin_memory(),
               "q_nope": wl.tensors["q_nope"].pin_memory(), "q_pe": wl.tensors["q_pe"].pin_memory()}
    slots = []
    for _ in range(2):
        dev = {k: ref[k].clone() for k in ("qI", "kI", "w", "q_nope", "q_pe", "kv_cache")}
        # device outputs kept for the whole test: the calls run on side streams
        slots.append({"dev": dev, "stream": torch.cuda.Stream(), "o": torch.empty_like(out_r),
                      "l": torch.empty_like(lse_r), "i": torch.empty_like(idx_r),
                      "outs": [torch.empty(out_r.shape, dtype=out_r.dtype).pin_memory() for _ in range(2)]})
    done = [torch.cuda.Event(), torch.cuda.Event()]
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    for i in range(4):
        chain = {"copy_done": copied[i % 2], "copy_after": copied[(i + 1) % 2] if i else None} if chain_copies else {}
        sl = slots[i % 2]
        d = sl["dev"]
        dsa.dsa_forward_host(dict(host_in, out=sl["outs"][i // 2]), d["qI"], d["kI"], d["w"], d["q_nope"],
                             d["q_pe"], d["kv_cache"][:, :sh.d_c], d["kv_cache"][:, sh.d_c:], ref["W_UK"],
                             ref["W_UV"], H.seqs_of(wl), sh.k, sh.softmax_scale, out=sl["o"], lse=sl["l"],
                             idx_out=sl["i"], stream=sl["stream"],
                             compute_done=done[i % 2], compute_after=done[(i + 1) % 2] if i else None, **chain)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_error() == (0, 0)
    for sl in slots:
        for o in sl["outs"]:
            assert torch.equal(o, out_r.cpu())


@pytest.mark.parametrize("many_rows", [False, True])
def test_appended_rows_staged_or_per_sequence(many_rows):
    """Appended rows land in their cache rows both ways: staged through the workspace and put in place
    by a kernel (decode: one row per sequence), and copied per sequence when the staging does not fit
    the workspace (a query at position 10 of a 20000-key cache appends 19990 rows, more bytes than its
    forward's workspace)."""
    if many_rows:
        T, S, P = [1, 2], [20000, 40], [10, 38]
    else:
        T, S, P = [1] * 40, [300 + 37 * i for i in range(40)], [299 + 37 * i for i in range(40)]
    wl = di.generate(f"host-io-append-{many_rows}", di.Shape(k=64), 74, T, S, P)
    sh = wl.shape
    ref = H.to_device(wl)
    out_r, lse_r, idx_r = H.gpu_forward(wl, ref)
    dev = {k: ref[k].clone() for k in ("kv_cache", "kI")}
    for k in dev:
        for b in range(wl.B):
            dev[k][wl.cu_k[b] + wl.start_pos[b]:wl.cu_k[b + 1]] = 5.0
    host = {"kv_new": _appended(wl, wl.tensors["kv_cache"]).pin_memory(),
            "k_idx_new": _appended(wl, wl.tensors["kI"]).pin_memory(),
            "out": torch.empty(out_r.shape, dtype=out_r.dtype).pin_memory()}
    dsa.dsa_forward_host(host, ref["qI"], dev["kI"], ref["w"], ref["q_nope"], ref["q_pe"],
                         dev["kv_cache"][:, :sh.d_c], dev["kv_cache"][:, sh.d_c:], ref["W_UK"], ref["W_UV"],
                         H.seqs_of(wl), sh.k, sh.softmax_scale, out=torch.empty_like(out_r),
                         lse=torch.empty_like(lse_r), idx_out=torch.empty_like(idx_r))
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_error() == (0, 0)
    staged = "append" in dsa.last_kernels()
    assert staged != many_rows, dsa.last_kernels()
    for k in dev:
        assert torch.equal(dev[k], ref[k]), k
    assert torch.equal(host["out"], out_r.cpu())


def test_forward_from_host_with_fp8_latent_cache():
    """The e4m3 latent cache through the host-buffer call: the appended rows of all four arrays (latent
    codes, k_pe, k^I, block scales; four row sizes) land in place, and the outputs equal the device
    forward's bit for bit."""
    wl = di.generate("host-io-fp8kv", di.Shape(k=64), 75, [120, 1, 30], [900, 1500, 30], [780, 1499, 0])
    sh = wl.shape
    ref = H.to_device(wl)
    lat = ref["kv_cache"][:, :sh.d_c].contiguous()
    codes, scales = dsa.dsa_quant_e4m3_ue8m0(lat)
    codes = codes.view(-1, sh.d_c)
    scales = scales.view(-1, sh.d_c // 128).contiguous()
    kpe = ref["kv_cache"][:, sh.d_c:].contiguous()  # k_pe in a buffer of its own
    out_r, lse_r, idx_r = dsa.dsa_forward(ref["qI"], ref["kI"], ref["w"], ref["q_nope"], ref["q_pe"], codes, kpe,
                                          ref["W_UK"], ref["W_UV"], H.seqs_of(wl), sh.k, sh.softmax_scale,
                                          kv_scale=scales)
    torch.cuda.synchronize()
    dev = {"codes": codes.clone(), "kpe": kpe.clone(), "kI": ref["kI"].clone(), "scales": scales.clone()}
    for k, v in dev.items():
        for b in range(wl.B):
            v[wl.cu_k[b] + wl.start_pos[b]:wl.cu_k[b + 1]] = 3 if v.dtype == torch.uint8 else 3.0
    host = {"kv_new": _appended(wl, codes.cpu()).pin_memory(), "k_pe_new": _appended(wl, kpe.cpu()).pin_memory(),
            "k_idx_new": _appended(wl, ref["kI"].cpu()).pin_memory(),
            "kv_scale_new": _appended(wl, scales.cpu()).pin_memory(),
            "out": torch.empty(out_r.shape, dtype=out_r.dtype).pin_memory()}
    dsa.dsa_forward_host(host, ref["qI"], dev["kI"], ref["w"], ref["q_nope"], ref["q_pe"], dev["codes"], dev["kpe"],
                         ref["W_UK"], ref["W_UV"], H.seqs_of(wl), sh.k, sh.softmax_scale,
                         out=torch.empty_like(out_r), lse=torch.empty_like(lse_r), idx_out=torch.empty_like(idx_r),
                         kv_scale=dev["scales"])
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_error() == (0, 0)
    assert "append" in dsa.last_kernels()
    assert torch.equal(dev["codes"], codes) and torch.equal(dev["kpe"], kpe) and torch.equal(dev["kI"], ref["kI"])
    assert torch.equal(dev["scales"], scales)
    assert torch.equal(host["out"], out_r.cpu())


@pytest.mark.parametrize("slots", [1, 2])
def test_consecutive_calls_with_different_queries(slots):
    """Three calls in a row without a synchronisation between them, each with its
    own queries (with two slots: alternating device buffers and streams, forwards
    and input copies chained).  q_nope and q_pe travel on the library's side
    stream, and no call may read another call's queries: every host output equals
    the device forward of its own inputs, bit for bit."""
    shape = di.Shape(k=64)
    T, S, P = [50, 1], [400, 300], [350, 299]
    base = di.generate("host-io-seq-0", shape, 90, T, S, P)
    sh = base.shape
    dev0 = H.to_device(base)
    names = ("qI", "w", "q_nope", "q_pe")
    queries = [{k: di.generate(f"host-io-seq-{j}", shape, 90 + j, T, S, P).tensors[k] for k in names}
               for j in range(3)]
    refs = []
    for q in queries:
        t = dict(dev0)
        t.update({k: v.cuda() for k, v in q.items()})
        refs.append(H.gpu_forward(base, t)[0])
    torch.cuda.synchronize()
    assert not torch.equal(refs[0], refs[1]) and not torch.equal(refs[1], refs[2])
    host_in = [{"q_idx": q["qI"].pin_memory(), "w": q["w"].pin_memory(), "q_nope": q["q_nope"].pin_memory(),
                "q_pe": q["q_pe"].pin_memory()} for q in queries]
    outs = [torch.empty(refs[0].shape, dtype=refs[0].dtype).pin_memory() for _ in range(3)]
    bufs = [{k: torch.zeros_like(dev0[k]) for k in names} for _ in range(slots)]
    streams = [torch.cuda.Stream() for _ in range(slots)]
    dev_out = [torch.empty_like(refs[0]) for _ in range(slots)]
    lse = [torch.empty((base.total_q, sh.H), dtype=torch.float32, device="cuda") for _ in range(slots)]
    idx = [torch.empty((base.total_q, sh.k), dtype=torch.int32, device="cuda") for _ in range(slots)]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    for i in range(3):
        s = i % slots
        b = bufs[s]
        chain = {}
        if slots == 2:
            chain = {"compute_done": done[i % 2], "compute_after": done[(i + 1) % 2] if i else None,
                     "copy_done": copied[i % 2], "copy_after": copied[(i + 1) % 2] if i else None}
        dsa.dsa_forward_host(dict(host_in[i], out=outs[i]), b["qI"], dev0["kI"], b["w"], b["q_nope"], b["q_pe"],
                             dev0["ckv"], dev0["kpe"], dev0["W_UK"], dev0["W_UV"], H.seqs_of(base), sh.k,
                             sh.softmax_scale, out=dev_out[s], lse=lse[s], idx_out=idx[s], stream=streams[s], **chain)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_error() == (0, 0)
    for i in range(3):
        assert torch.equal(outs[i], refs[i].cpu()), i
