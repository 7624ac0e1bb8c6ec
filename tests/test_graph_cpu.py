"""fd_plan_graph (host only): the capacity it plans for covers every batch of at
most max_total_tokens keys under the device-side split rule, and it keeps the
chunk it is given.  FD++ §6 (integration: decode steps run as CUDA graphs with
a fixed batch)."""
import numpy as np
import pytest

import split_kv_flashdecoding_gb300 as fd


def device_rule_splits(lengths, chunk):
    """The device-side plan: ceil(L / chunk) splits, one for an empty request."""
    return sum(max(1, -(-int(L) // chunk)) for L in lengths)


@pytest.mark.parametrize("seed", range(5))
def test_capacity_covers_every_batch_within_it(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 50))
    T = int(rng.integers(1, 200000))
    info = fd.plan_graph(B, 32, 8, 128, T, num_sms=152)
    C = info.chunk
    assert info.total_splits == T // C + B
    assert info.num_work == info.total_splits * 8 and info.num_partial_rows == info.total_splits * 32
    for _ in range(20):
        # random lengths summing to at most T, with empty requests
        cuts = np.sort(rng.integers(0, T + 1, size=B))
        lengths = np.diff(np.concatenate([[0], cuts]))
        lengths[rng.random(B) < 0.2] = 0
        assert device_rule_splits(lengths, C) <= info.total_splits
    # the worst case: every request one key past a chunk boundary
    worst = [C + 1] * min(B, T // (C + 1)) + [0] * (B - min(B, T // (C + 1)))
    assert device_rule_splits(worst, C) <= info.total_splits


def test_given_chunk_and_workspace():
    info = fd.plan_graph(4, 16, 4, 128, 10000, num_sms=152, chunk=256)
    assert info.chunk == 256
    rows = info.num_partial_rows
    assert info.workspace_bytes == 256 + 256 + -(-rows * 4 // 256) * 256 + rows * 128 * 4
    assert info.total_tokens == 10000


def test_rejects_bad_arguments():
    with pytest.raises(fd.FdError):
        fd.plan_graph(4, 16, 4, 128, -1, num_sms=152)
    with pytest.raises(fd.FdError):
        fd.plan_graph(4, 16, 4, 128, 1000, num_sms=152, chunk=48)   # not a multiple of 32
