"""Host planner (fd_plan / fd_plan_work_items): runs on the CPU, no GPU calls.

Pinned to the grid arithmetic the FlashDecoding++ sequence-split article
(techknowgenie.com) prints in §2 (1 x 32 x 256 = 8192 blocks, about 62 per SM
on 132 SMs) and §1 (a batch x heads grid at batch 1 leaves 100 of 132 SMs
idle, 124 with 8 KV heads), plus coverage invariants on random batches.
"""
import json
import os

import numpy as np
import pytest

import split_kv_flashdecoding_gb300 as fd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def indptr_of(lengths):
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    return ip


def test_article_split_grid_example():
    ex = json.load(open(os.path.join(GOLDEN, "page3_split_grid_example.json")))["split_grid"]
    H = ex["heads"]
    # MHA: every head is its own KV head, so the grid is batch x heads x chunks.
    info = fd.plan(ex["batch"], H, H, 128, [0, ex["seq_len"]], num_sms=ex["sms"],
                   chunk=ex["chunk"])
    assert info.total_splits == ex["chunks"]
    assert info.num_work == ex["blocks"]
    assert info.num_work // ex["sms"] == ex["blocks_per_sm_approx"]


def test_article_unsplit_grid_example():
    ex = json.load(open(os.path.join(GOLDEN, "page3_split_grid_example.json")))["unsplit_grid"]
    L = 65536
    # one chunk covering the whole request = no sequence split
    mha = fd.plan(ex["batch"], ex["heads"], ex["heads"], 128, [0, L], num_sms=ex["sms"], chunk=L)
    assert ex["sms"] - mha.num_work == ex["idle_sms"]
    gqa = fd.plan(ex["batch"], ex["heads"], ex["kv_heads"], 128, [0, L], num_sms=ex["sms"], chunk=L)
    assert ex["sms"] - gqa.num_work == ex["idle_sms_kv_heads"]


def _check_cover(info, ip):
    items = fd.plan_work_items(info, ip)
    assert items.shape == (info.num_work, 5)
    B, Hkv = info.batch, info.num_kv_heads
    seen = {}
    for b, h, s, t0, t1 in items:
        assert 0 <= b < B and 0 <= h < Hkv
        assert ip[b] <= t0 < t1 <= ip[b + 1], "split inside its request and non-empty"
        assert t1 - t0 <= info.chunk
        seen.setdefault((b, h), []).append((s, t0, t1))
    for b in range(B):
        L = ip[b + 1] - ip[b]
        for h in range(Hkv):
            parts = sorted(seen.get((b, h), []))
            if L == 0:
                assert not parts
                continue
            assert [p[0] for p in parts] == list(range(len(parts)))
            assert parts[0][1] == ip[b] and parts[-1][2] == ip[b + 1]
            for (_, _, e), (_, s2, _) in zip(parts[:-1], parts[1:]):
                assert e == s2, "splits tile the request with no gap or overlap"
            for _, t0, t1 in parts[:-1]:
                assert (t1 - t0) % fd.TILE_TOKENS == 0
    # launch order: global split j = w // Hkv, KV head = w % Hkv
    assert np.array_equal(items[:, 1], np.arange(info.num_work) % Hkv)
    return items


@pytest.mark.parametrize("seed", range(6))
def test_random_batches_are_covered_exactly(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    lengths = rng.integers(0, 5000, size=B)
    lengths[rng.random(B) < 0.2] = 0
    ip = indptr_of(lengths)
    for Hq, Hkv in [(8, 8), (32, 8), (64, 8), (4, 2)]:
        for chunk in [0, 32, 96, 1024]:
            info = fd.plan(B, Hq, Hkv, 128, ip, num_sms=152, chunk=chunk)
            assert info.chunk % fd.TILE_TOKENS == 0
            assert info.group_size == Hq // Hkv
            assert info.num_partial_rows == info.total_splits * Hq
            _check_cover(info, ip)


def test_auto_chunk_targets_ctas_per_sm():
    # B=1, 64k keys, 8 KV heads, 152 SMs, 2 CTAs per SM -> 38 splits x 8 heads = 304 CTAs
    info = fd.plan(1, 32, 8, 128, [0, 65536], num_sms=152, ctas_per_sm=2)
    assert info.num_work == 304 and info.chunk == 1728
    info = fd.plan(1, 32, 8, 128, [0, 131072], num_sms=152, ctas_per_sm=2)
    assert info.num_work == 304
    # tiny requests never go below the minimum chunk
    info = fd.plan(1, 8, 8, 128, [0, 2048], num_sms=152)
    assert info.chunk == 128 and info.num_work == 16 * 8
    # more CTAs per SM -> smaller chunks
    a = fd.plan(1, 32, 8, 128, [0, 65536], num_sms=152, ctas_per_sm=1)
    b = fd.plan(1, 32, 8, 128, [0, 65536], num_sms=152, ctas_per_sm=4)
    assert a.num_work < b.num_work


def test_forced_split_counts_one_to_max():
    L = 1000
    ip = [0, L]
    one = fd.plan(1, 4, 4, 128, ip, num_sms=152, chunk=1024)
    assert one.max_splits == 1
    most = fd.plan(1, 4, 4, 128, ip, num_sms=152, chunk=32)
    assert most.max_splits == (L + 31) // 32
    for chunk in range(32, 1025, 32):
        info = fd.plan(1, 4, 4, 128, ip, num_sms=152, chunk=chunk)
        assert info.max_splits == -(-L // chunk)
        _check_cover(info, np.array(ip))


def test_workspace_bytes():
    info = fd.plan(3, 16, 4, 128, [0, 10, 10, 300], num_sms=10, chunk=64)
    rows = info.num_partial_rows
    group = -(-3 * 4 * 4 // 256) * 256             # one int32 per (request, KV head)
    flags = -(-info.num_work * 4 // 256) * 256      # one int32 per split item
    # header | merge tickets | partial LSE | partial O | publication flags
    assert info.workspace_bytes == (256 + group + -(-rows * 4 // 256) * 256 + rows * 128 * 4 +
                                    flags)


def _makespan(info, ip, slots, overhead=3):
    """Independent re-simulation of the block dispatch (heap of slot free times)."""
    import heapq
    items = fd.plan_work_items(info, ip)
    heap = [0] * slots
    end = 0
    for _, _, _, t0, t1 in items:
        start = heapq.heappop(heap)
        fin = start + -(-(t1 - t0) // 32) + overhead
        heapq.heappush(heap, fin)
        end = max(end, fin)
    return end


def test_ragged_batches_get_more_waves_than_even_ones():
    """The planner simulates the block dispatch: a batch-1 request that splits
    evenly gets one wave of resident CTAs, a ragged batch smaller chunks that
    balance the slots."""
    slots = 152 * 2
    one = fd.plan(1, 32, 8, 128, indptr_of([65536]), num_sms=152, ctas_per_sm=2)
    assert one.num_work == slots
    rng = np.random.default_rng(3)
    ragged_len = rng.integers(512, 16385, size=64)
    ragged = fd.plan(64, 32, 8, 128, indptr_of(ragged_len), num_sms=152, ctas_per_sm=2)
    one_wave_chunk = -(-int(ragged_len.sum()) * 8 // slots)
    assert ragged.chunk < one_wave_chunk
    assert ragged.num_work > slots


@pytest.mark.parametrize("lengths", [[65536], [131072], [32768] * 16, [2048], [5000, 300, 70000],
                                     list(np.random.default_rng(5).integers(512, 16385, 64))])
def test_chosen_chunk_is_best_of_the_candidates(lengths):
    """The chunk the planner picks has the shortest re-simulated makespan among
    the 1/2/4/8-wave candidates (ties go to fewer waves)."""
    ip = indptr_of(lengths)
    slots = 152 * 2
    chosen = fd.plan(len(lengths), 32, 8, 128, ip, num_sms=152, ctas_per_sm=2)
    best = _makespan(chosen, ip, slots)
    for waves in (1, 2, 4, 8):
        c = max(128, -(-(-(-int(ip[-1]) * 8 // (slots * waves))) // 32) * 32)
        cand = fd.plan(len(lengths), 32, 8, 128, ip, num_sms=152, chunk=c)
        assert best <= _makespan(cand, ip, slots)


def test_empty_batch_and_empty_requests():
    info = fd.plan(0, 8, 8, 128, [0], num_sms=152)
    assert info.num_work == 0 and info.total_splits == 0
    info = fd.plan(3, 8, 8, 128, [0, 0, 0, 0], num_sms=152)
    assert info.num_work == 0 and info.num_partial_rows == 0
    assert fd.plan_work_items(info, [0, 0, 0, 0]).shape == (0, 5)


@pytest.mark.parametrize("args,code", [
    ((1, 8, 3, 128, [0, 5]), -1),        # Hq % Hkv != 0
    ((1, 8, 8, 64, [0, 5]), -2),         # unsupported head_dim
    ((1, 48, 3, 128, [0, 5]), -2),       # unsupported group size 16
    ((2, 8, 8, 128, [1, 5, 9]), -1),     # indptr[0] != 0
    ((2, 8, 8, 128, [0, 9, 5]), -1),     # decreasing indptr
    ((1, 0, 8, 128, [0, 5]), -1),        # no heads
])
def test_plan_rejects_bad_arguments(args, code):
    with pytest.raises(fd.FdError) as e:
        fd.plan(*args, num_sms=152)
    assert e.value.code == code


def test_plan_rejects_bad_chunk():
    with pytest.raises(fd.FdError) as e:
        fd.plan(1, 8, 8, 128, [0, 100], num_sms=152, chunk=48)
    assert e.value.code == -1


@pytest.mark.parametrize("num_sms", [152, 132, 7, 3, 1])
def test_bench_host_plan_rule_matches_fd_plan(num_sms):
    """bench.py's reference arm counts the partial bytes of fd_plan's plan
    without loading the library, from the rule include/fd.h documents: the
    same chunk on the five workloads and on random ragged batches, including
    plans with more KV heads than resident-CTA slots."""
    import bench
    from workloads import WORKLOADS
    rng = np.random.default_rng(num_sms)
    cases = []
    for w in WORKLOADS:
        lengths = (np.random.default_rng(42 + w.index).integers(w.ragged[0], w.ragged[1] + 1, w.batch)
                   if w.ragged else [w.kv_len] * w.batch)
        cases.append(([int(x) for x in lengths], w.num_qo_heads, w.num_kv_heads))
    for _ in range(60):
        B = int(rng.integers(1, 70))
        lengths = rng.integers(0, 40000, B) * (rng.random(B) > 0.1)
        hkv = int(rng.choice([1, 2, 8]))
        cases.append(([int(x) for x in lengths], hkv * int(rng.choice([1, 2, 4, 8])), hkv))
    for lengths, hq, hkv in cases:
        ip = np.zeros(len(lengths) + 1, dtype=np.int32)
        ip[1:] = np.cumsum(lengths)
        info = fd.plan(len(lengths), hq, hkv, 128, ip, num_sms=num_sms)
        assert bench.plan_chunk(lengths, hkv, num_sms) == info.chunk
        assert bench.plan_partial_rows(lengths, hq, hkv, num_sms) == info.num_partial_rows
