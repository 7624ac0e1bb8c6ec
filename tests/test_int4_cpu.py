"""INT4 KV, host side: the oracle's decoding of the packed codes and its
dequantised decode, pinned to the two's-complement definition, hand-packed
bytes and closed forms.

FD++ §4 (quantisation-friendly fusion) names INT4 beside FP8: the packed cache
stays in HBM and is dequantised in registers.  The format (two codes per byte,
low nibble first; one fp32 scale per key row and KV head, head-major) is the
one include/fd.h documents.
"""
import math

import numpy as np
import torch

import oracle
from workloads import make_small, random_int4, to_int4, to_paged_int4


def test_every_byte_decodes_to_its_two_nibbles():
    b = np.arange(256, dtype=np.uint8)
    got = oracle.int4_codes(b.reshape(256, 1))                 # [256, 2]
    lo, hi = b.astype(np.int64) % 16, b.astype(np.int64) // 16
    # two's complement of a 4-bit field: (n + 8) mod 16 - 8
    assert np.array_equal(got[:, 0], (lo + 8) % 16 - 8)
    assert np.array_equal(got[:, 1], (hi + 8) % 16 - 8)


def test_hand_packed_bytes():
    got = oracle.int4_codes(np.array([[0x00, 0x7F, 0x80, 0x88, 0xFF, 0x21, 0x43]], dtype=np.uint8))
    assert got.tolist() == [[0, 0, -1, 7, 0, -8, -8, -8, -1, -1, 1, 2, 3, 4]]


def test_dequant_takes_each_rows_and_heads_own_scale():
    T, H = 5, 3
    codes = np.full((T, H, 4), 0x11, dtype=np.uint8)            # every code is 1
    sc = (np.arange(H * T, dtype=np.float32).reshape(H, T) + 1) * 0.25
    out = oracle.dequant_int4(codes, sc)
    assert out.shape == (T, H, 8)
    for t in range(T):
        for h in range(H):
            assert np.all(out[t, h] == sc[h, t])


def test_quantisation_error_is_within_half_a_step():
    f = to_int4(make_small(2, 8, 2, 128, [70, 33], seed=3))
    for name in ("k", "v"):
        x = f[name].double().numpy()
        deq = oracle.dequant_int4(f[name + "_int4"], f[name + "_scale_int4"])
        s = f[name + "_scale_int4"].double().numpy().T[:, :, None]
        assert np.all(np.abs(deq - x) <= s / 2 * (1 + 1e-6))
        # each row's largest magnitude maps to code +-7 exactly
        assert np.allclose(np.abs(deq).max(axis=2), 7 * s[:, :, 0], rtol=1e-6)


def test_decode_int4_is_decode_on_the_dequantised_values():
    f = random_int4(make_small(2, 8, 2, 128, [70, 33], seed=4))
    o, lse = oracle.decode_int4(f["q"], f["k_int4"], f["v_int4"], f["k_scale_int4"],
                                f["v_scale_int4"], f["kv_indptr"], f["scale"])
    k = torch.from_numpy(oracle.dequant_int4(f["k_int4"], f["k_scale_int4"]))
    v = torch.from_numpy(oracle.dequant_int4(f["v_int4"], f["v_scale_int4"]))
    o2, lse2 = oracle.decode(f["q"].double(), k, v, f["kv_indptr"], f["scale"])
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_equal_keys_give_the_mean_of_the_dequantised_values():
    """Every K code 1 with one K scale c: all logits are s = scale * c * sum(q),
    so O is the plain mean of V's rows (each code times its own row scale) and
    LSE = s + ln L.  A wrong nibble order, sign or scale index fails this."""
    L, H, D = 9, 1, 128
    base = make_small(1, 1, 1, D, [L], seed=8)
    g = torch.Generator().manual_seed(5)
    k = np.full((L, H, D // 2), 0x11, dtype=np.uint8)
    v = torch.randint(0, 256, (L, H, D // 2), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    c = np.float32(0.375)
    ks = np.full((H, L), c, dtype=np.float32)
    vs = (torch.rand((H, L), generator=g) + 0.5).numpy().astype(np.float32)
    o, lse = oracle.decode_int4(base["q"], k, v, ks, vs, base["kv_indptr"], base["scale"])
    q = base["q"].double().numpy().reshape(D)
    s = float(np.float32(base["scale"])) * float(c) * q.sum()
    # V by hand: low nibble = even dim, high = odd, two's complement, times vs[0, j]
    vv = np.zeros((L, D))
    for j in range(L):
        for byte in range(D // 2):
            x = int(v[j, 0, byte])
            lo, hi = x & 15, x >> 4
            vv[j, 2 * byte] = (lo - 16 if lo >= 8 else lo) * float(vs[0, j])
            vv[j, 2 * byte + 1] = (hi - 16 if hi >= 8 else hi) * float(vs[0, j])
    assert np.allclose(o.reshape(D), vv.mean(axis=0), rtol=0, atol=1e-12)
    assert math.isclose(float(lse.reshape(())), s + math.log(L), rel_tol=0, abs_tol=1e-12)


def test_paged_layout_gathers_back_to_the_ragged_values():
    f = random_int4(make_small(3, 8, 2, 128, [40, 0, 75], seed=6))
    for P in (16, 32, 48):
        pg = to_paged_int4(f, P, seed=P)
        n = pg["k_pages_int4"].shape[0]
        for name in ("k", "v"):
            pool = oracle.dequant_int4(pg[name + "_pages_int4"].reshape(n * P, 2, 64),
                                       pg[name + "_scale_pages"]).reshape(n, P, 2, 128)
            x, _, ip = oracle.gather_paged(torch.from_numpy(pool), torch.from_numpy(pool),
                                           pg["kv_page_indptr"], pg["kv_page_indices"],
                                           pg["kv_last_page_len"])
            ref = oracle.dequant_int4(f[name + "_int4"], f[name + "_scale_int4"])
            assert np.array_equal(x.numpy(), ref) and ip.tolist() == [0, 40, 40, 115]
