"""CPU checks of bench.py's host-side logic: the per-stage algorithmic work
(against closed forms on hand-countable batches), the roofline classification,
the indexer's computed-pair count, the score chunking, the row cuts used for
profiling, and the rule that a stored ncu traffic figure is used only while
the kernel sources it was taken on are unchanged."""
import json
import os

import pytest
import torch

import bench
import dsa_inputs as di

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def _wl(T, S, P, **shape):
    return di.generate("bench-host", di.Shape(**shape), 5, T, S, P)


def test_stage_work_closed_forms():
    # one sequence, rows at positions 2, 3, 4 of a 5-key cache, top-2
    wl = _wl([3], [5], [2], k=2)
    sh = wl.shape
    flops, hbm = bench.stage_work(wl)
    causal = 3 + 4 + 5  # each row sees p + 1 keys
    selected = 2 + 2 + 2  # min(k, p + 1)
    assert flops["indexer+topk"] == 2 * 64 * 128 * causal
    assert flops["sparse_mla"] == 2 * 128 * (512 + 512 + 64) * selected == 278_528 * selected
    assert flops["absorb_q"] == 2 * 3 * 128 * 128 * 512
    assert flops["absorb_v"] == 2 * 3 * 128 * 512 * 128
    # bf16: W_UK, q_nope in, q~ out
    assert hbm["absorb_q"] == 2 * (128 * 128 * 512 + 3 * 128 * 128 + 3 * 128 * 512)
    # the attention reads each distinct selected latent row at most once (here 5 cached rows < 6 pairs)
    assert hbm["sparse_mla"] == 5 * 576 * 2 + 3 * 128 * 576 * 2 + 3 * 128 * 512 * 2 + 4 * 3 * sh.k
    assert all(v > 0 for v in hbm.values())


def test_stage_work_fp8_indexer_bytes():
    wl16 = _wl([4], [300], [296], k=64)
    wl8 = _wl([4], [300], [296], k=64, idx_fp8=True)
    _, h16 = bench.stage_work(wl16)
    _, h8 = bench.stage_work(wl8)
    # k^I at 1 byte per value instead of 2; q^I likewise for the 4 scored rows
    assert h16["indexer+topk"] - h8["indexer+topk"] == 300 * 128 + 4 * 64 * 128


def test_indexer_pairs_computed_counts_blocks_of_groups():
    # 6 rows at positions 200..205 with k = 64: groups (200..203) and (204, 205)
    wl = _wl([6], [206], [200], k=64)
    per_group = [(203 // 128 + 1) * 128 * 4, (205 // 128 + 1) * 128 * 2]
    assert bench.indexer_pairs_computed(wl) == sum(per_group)
    # rows that see at most k keys are skipped by the forward, counted when asked
    wl2 = _wl([8], [8], [0], k=64)
    assert bench.indexer_pairs_computed(wl2) == 0
    assert bench.indexer_pairs_computed(wl2, skip_dense=False) == 2 * 128 * 4


def test_roofline_classification():
    wl = _wl([3], [5], [2], k=2)
    # far above the ridge point: tensor-bound, achieved = flops / time
    r = bench.roofline_of("sparse_mla", 2.0, 4e12, 1e6, PEAKS, "measured", wl.name)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(4e12 / 2e9) and r["frac"] == pytest.approx(r["achieved"] / 1900.0)
    # far below it: HBM-bound, against the copy bandwidth; FP8 doubles the tensor peak
    r = bench.roofline_of("indexer+topk", 0.1, 1e9, 6e8, PEAKS, "measured", wl.name, fp8=True)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(6e8 / 1e5) and r["peak"] == 6800.0
    assert r["traffic"] is None  # no capture for this workload


def test_score_chunks_partition_rows_under_one_gib():
    wl = _wl([5, 7], [70000, 9], [69995, 2], k=64)
    chunks = bench.score_chunks(wl)
    ld = (70000 + 3) // 4 * 4
    assert chunks[0][0] == 0 and chunks[-1][1] == wl.total_q
    assert all(a[1] == b[0] for a, b in zip(chunks, chunks[1:]))
    assert all((r1 - r0) * ld * 4 <= 1 << 30 for r0, r1 in chunks)


def test_row_cuts_keep_positions_and_caches():
    wl = _wl([4, 6, 3], [10, 40, 20], [6, 34, 17], k=8)
    f = bench.first_rows(wl, 7)
    assert f.T == [4, 3] and f.S == [10, 40] and f.start_pos == [6, 34]
    assert torch.equal(f.tensors["q_nope"], wl.tensors["q_nope"][:7])
    assert torch.equal(f.tensors["kv_cache"], wl.tensors["kv_cache"][:50])
    last = bench.last_rows(wl, 2)  # the longest sequence is the second: its rows at 38, 39
    assert last.T == [2] and last.S == [40] and last.start_pos == [38]
    assert torch.equal(last.tensors["q_pe"], wl.tensors["q_pe"][8:10])
    assert torch.equal(last.tensors["kI"], wl.tensors["kI"][10:50])


def test_stored_traffic_follows_the_sources(tmp_path, monkeypatch):
    """profiles/traffic.json figures are reported only while the sources they
    were captured on hash to the stored sha256; otherwise the figure is null."""
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    for stage, entries in table.items():
        for e in entries:
            got = bench.ncu_traffic(stage, e["workload"])
            fresh = bench.source_digest(e["sources"]) == e["sha256"]
            assert got == (e["dram_bytes"] if fresh else None), (stage, e["workload"])
    # a copy of the tree with one source changed: the same entry reads as null
    stage, e = next((s, x) for s, xs in table.items() for x in xs)
    before = bench.ncu_traffic(stage, e["workload"])
    root = tmp_path / "tree"
    (root / "profiles").mkdir(parents=True)
    (root / "profiles" / "traffic.json").write_text(json.dumps({stage: [e]}))
    for rel in e["sources"]:
        dst = root / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        dst.write_bytes(open(os.path.join(bench.ROOT, rel), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.ncu_traffic(stage, e["workload"]) == before  # an identical copy reads the same
    with open(root / e["sources"][0], "ab") as f:
        f.write(b"\n// changed\n")
    assert bench.ncu_traffic(stage, e["workload"]) is None


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.25, 1) == 3.25
