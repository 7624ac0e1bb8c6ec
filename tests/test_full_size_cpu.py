"""The full-size GPU tests compute the FP8 and INT4 oracle one block of whole
requests at a time (tests/full_size.py).  Attention of a row only reads its
own request's keys, so the blocks must give exactly the numbers of one oracle
call over the whole batch; checked here on a small ragged batch cut into many
blocks, with an empty request and a request longer than a block."""
import numpy as np
import pytest

import oracle
from tests import full_size
from workloads import make_small, to_fp8, to_int4


@pytest.mark.parametrize("block_rows", [1, 300, 1000, 1 << 20])
def test_blockwise_oracle_equals_one_call(monkeypatch, block_rows):
    monkeypatch.setattr(full_size, "_BLOCK_ROWS", block_rows)
    inp = make_small(6, 16, 4, 128, [130, 0, 700, 2, 400, 1500], seed=3)
    ip = inp["kv_indptr"].numpy()
    blocks = full_size._request_blocks(ip)
    assert blocks[0][0] == 0 and blocks[-1][1] == 6
    assert all(a[1] == b[0] for a, b in zip(blocks, blocks[1:]))

    f = to_fp8(inp)
    o, lse = full_size._blockwise(f, lambda q, r0, r1, sub: oracle.decode_fp8(
        q, f["k_fp8"][r0:r1], f["v_fp8"][r0:r1], f["k_scale"], f["v_scale"], sub, f["scale"]))
    o1, l1 = oracle.decode_fp8(f["q"], f["k_fp8"], f["v_fp8"], f["k_scale"], f["v_scale"],
                               f["kv_indptr"], f["scale"])
    assert np.array_equal(o, o1) and np.array_equal(lse, l1)

    g = to_int4(inp)
    o, lse = full_size._blockwise(g, lambda q, r0, r1, sub: oracle.decode_int4(
        q, g["k_int4"][r0:r1], g["v_int4"][r0:r1], g["k_scale_int4"][:, r0:r1],
        g["v_scale_int4"][:, r0:r1], sub, g["scale"]))
    o1, l1 = oracle.decode_int4(g["q"], g["k_int4"], g["v_int4"], g["k_scale_int4"],
                                g["v_scale_int4"], g["kv_indptr"], g["scale"])
    assert np.array_equal(o, o1) and np.array_equal(lse, l1)
