"""Paged KV cache, host side: the oracle's page-table gather (pinned to a hand
example and to the paged layout the generator builds) and fd_plan_paged.

FD++ §6 (vLLM integration): the engine's page table maps each request's keys
onto fixed-size physical pages; a split chunk reads the pages its keys fall in.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_flashdecoding_gb300 as fd
from workloads import make_small, to_paged


def test_gather_hand_example():
    # page p, row r holds the value 10*p + r (one KV head, D = 1)
    P, num_pages = 2, 5
    pool = torch.tensor([[[[10.0 * p + r]] for r in range(P)] for p in range(num_pages)])
    indptr = [0, 2, 2, 3]            # request 0: 2 pages, request 1: none, request 2: 1 page
    indices = [3, 1, 0]
    last = [1, 0, 2]
    K, V, ip = oracle.gather_paged(pool, pool * 2, indptr, indices, last)
    assert K.reshape(-1).tolist() == [30.0, 31.0, 10.0, 0.0, 1.0]
    assert V.reshape(-1).tolist() == [60.0, 62.0, 20.0, 0.0, 2.0]
    assert list(ip) == [0, 3, 3, 5]


@pytest.mark.parametrize("page_size", [16, 32, 48, 64])
def test_paged_layout_reads_back_as_the_ragged_one(page_size):
    inp = make_small(5, 8, 2, 128, [100, 0, 33, 64, 1], seed=4)
    pg = to_paged(inp, page_size, seed=page_size)
    K, V, ip = oracle.gather_paged(pg["k_pages"], pg["v_pages"], pg["kv_page_indptr"],
                                   pg["kv_page_indices"], pg["kv_last_page_len"])
    assert torch.equal(K, inp["k"]) and torch.equal(V, inp["v"])
    assert list(ip) == inp["kv_indptr"].tolist()
    # pages are scattered, not laid out in request order
    assert pg["kv_page_indices"].tolist() != sorted(pg["kv_page_indices"].tolist())


def test_plan_paged_equals_plan_on_key_counts():
    page_indptr = np.array([0, 3, 3, 10, 11], dtype=np.int32)
    last = np.array([5, 0, 16, 1], dtype=np.int32)
    lens = [2 * 16 + 5, 0, 6 * 16 + 16, 1]
    ip = np.zeros(5, dtype=np.int32)
    ip[1:] = np.cumsum(lens)
    for chunk in (0, 32, 64):
        a = fd.plan_paged(4, 32, 8, 128, 16, page_indptr, last, num_sms=152, chunk=chunk)
        b = fd.plan(4, 32, 8, 128, ip, num_sms=152, chunk=chunk)
        assert a.as_dict() == b.as_dict()


@pytest.mark.parametrize("page_size,last,code", [
    (24, [3], -2),          # not a multiple of 16
    (0, [3], -2),
    (16, [0], -1),          # a non-empty request must hold 1..page_size keys in its last page
    (16, [17], -1),
])
def test_plan_paged_rejects_bad_layouts(page_size, last, code):
    with pytest.raises(fd.FdError) as e:
        fd.plan_paged(1, 8, 8, 128, page_size, [0, 2], last, num_sms=152)
    assert e.value.code == code


@pytest.mark.parametrize("page_size", [16, 32, 48, 64, 256])
def test_paged_tiles_never_straddle_a_page(page_size):
    # The paged kernels copy a tile as TMA boxes of 32 rows (P a multiple of
    # 32) or 16 rows (otherwise), each addressed through one page-table entry,
    # which is only right if no box crosses a page boundary: every split, and
    # so every tile, must start at a key offset that is a multiple of the box.
    rng = np.random.default_rng(page_size)
    box = 32 if page_size % 32 == 0 else 16
    for _ in range(20):
        B = int(rng.integers(1, 12))
        pages = rng.integers(0, 40, size=B)
        last = np.where(pages > 0, rng.integers(1, page_size + 1, size=B), 0).astype(np.int32)
        page_indptr = np.zeros(B + 1, dtype=np.int32)
        page_indptr[1:] = np.cumsum(pages)
        lens = np.where(pages > 0, (pages - 1) * page_size + last, 0)
        ip = np.zeros(B + 1, dtype=np.int32)
        ip[1:] = np.cumsum(lens)
        for chunk in (0, 32, 96, 160):
            info = fd.plan_paged(B, 32, 8, 128, page_size, page_indptr, last, num_sms=152,
                                 chunk=chunk)
            for b, _, _, t0, t1 in fd.plan_work_items(info, ip):
                off = t0 - ip[b]
                assert off % fd.TILE_TOKENS == 0
                for k in range(off, t1 - ip[b], box):
                    assert k % page_size + box <= page_size, "a box crosses into the next page"
