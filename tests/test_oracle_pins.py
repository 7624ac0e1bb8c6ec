"""Pins for the fp64 oracle: each one checks it against something other than
itself (closed forms, a brute-force Python loop, a library routine, the
article's own printed check, invariances), so that a dropped term, a wrong
sign, a wrong index or head mapping, or a transposed operand fails a test.

Article: "FlashDecoding++: sequence-dimension KV split parallelism for LLM
serving" (techknowgenie.com), §3 (two-stage reduction) and §5 (equivalence
check).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import fp32_scale, make_small

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RTOL, ATOL = 1e-12, 1e-13


def f64(t):
    return t.detach().to(torch.float64).numpy()


def _rows_of(kv_indptr, b):
    ip = np.asarray(kv_indptr)
    return int(ip[b]), int(ip[b + 1])


# ---------------------------------------------------------------- closed forms

def test_identical_keys_give_mean_of_v():
    """All keys of a request equal => uniform softmax: O = mean_j V_j, LSE = s + ln L."""
    inp = make_small(2, 8, 2, 128, [5, 13], seed=1)
    q, k, v, ip, sc = inp["q"], inp["k"].clone(), inp["v"], inp["kv_indptr"], inp["scale"]
    for b in range(2):
        j0, j1 = _rows_of(ip, b)
        k[j0:j1] = k[j0].unsqueeze(0)
    o, lse = oracle.decode(q, k, v, ip, sc)
    qd, kd, vd = f64(q), f64(k), f64(v)
    G = 4
    for b in range(2):
        j0, j1 = _rows_of(ip, b)
        for hq in range(8):
            kvh = hq // G
            s = sc * math.fsum(qd[b, hq, d] * kd[j0, kvh, d] for d in range(128))
            row = b * 8 + hq
            np.testing.assert_allclose(o[row], vd[j0:j1, kvh].mean(axis=0), rtol=RTOL, atol=ATOL)
            assert abs(lse[row] - (s + math.log(j1 - j0))) < 1e-12


def test_dominant_score_selects_that_value_row():
    """One key k* = 32 q far above the others: O = V_{j*}, LSE = s* (to e^-50)."""
    D, L = 16, 11
    inp = make_small(1, 4, 4, D, [L], seed=2)
    q, k, v, ip = inp["q"], inp["k"].clone(), inp["v"], inp["kv_indptr"]
    sc = fp32_scale(D)
    jstar = 7
    k[jstar] = (q[0] * 32).to(torch.bfloat16)   # exact: power-of-two multiple
    qd, kd, vd = f64(q), f64(k), f64(v)
    o, lse = oracle.decode(q, k, v, ip, sc)
    for h in range(4):
        s = [sc * math.fsum(qd[0, h, d] * kd[j, h, d] for d in range(D)) for j in range(L)]
        gap = s[jstar] - max(s[j] for j in range(L) if j != jstar)
        assert gap >= 50.0
        np.testing.assert_allclose(o[h], vd[jstar, h], rtol=0, atol=1e-15 + L * math.exp(-50) * 10)
        assert abs(lse[h] - s[jstar]) < 1e-12


def test_lse_is_log_sum_exp_without_max_shift():
    """LSE against ln(fsum(exp(s_j))) computed directly (no max subtraction)."""
    inp = make_small(2, 4, 2, 8, [9, 17], seed=3)
    q, k, v, ip, sc = inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"]
    _, lse = oracle.decode(q, k, v, ip, sc)
    qd, kd = f64(q), f64(k)
    for b in range(2):
        j0, j1 = _rows_of(ip, b)
        for hq in range(4):
            s = [sc * math.fsum(qd[b, hq, d] * kd[j, hq // 2, d] for d in range(8))
                 for j in range(j0, j1)]
            assert max(abs(x) for x in s) <= 20.0
            ref = math.log(math.fsum(math.exp(x) for x in s))
            assert abs(lse[b * 4 + hq] - ref) < 1e-12


def test_zero_query_gives_mean_v_and_log_length():
    inp = make_small(3, 4, 4, 32, [1, 6, 10], seed=4)
    q = torch.zeros_like(inp["q"])
    o, lse = oracle.decode(q, inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    vd = f64(inp["v"])
    for b in range(3):
        j0, j1 = _rows_of(inp["kv_indptr"], b)
        for h in range(4):
            np.testing.assert_allclose(o[b * 4 + h], vd[j0:j1, h].mean(axis=0), rtol=RTOL, atol=ATOL)
            assert abs(lse[b * 4 + h] - math.log(j1 - j0)) < 1e-14


def test_empty_request_gives_zero_and_minus_inf():
    inp = make_small(3, 2, 1, 8, [4, 0, 3], seed=5)
    o, lse = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    assert np.all(o[2:4] == 0.0) and np.all(np.isneginf(lse[2:4]))
    assert np.all(np.isfinite(lse[:2])) and np.all(np.isfinite(lse[4:]))


# ------------------------------------------------------------- brute force

def _brute_force(q, k, v, kv_indptr, scale):
    """Independent pure-Python loops: softmax weights from exp(s_j)/sum exp(s)."""
    qd, kd, vd = f64(q), f64(k), f64(v)
    B, Hq, D = qd.shape
    Hkv = kd.shape[1]
    G = Hq // Hkv
    O = np.zeros((B * Hq, D))
    LSE = np.zeros(B * Hq)
    for b in range(B):
        j0, j1 = _rows_of(kv_indptr, b)
        for hq in range(Hq):
            h = hq // G
            s = [scale * math.fsum(qd[b, hq, d] * kd[j, h, d] for d in range(D)) for j in range(j0, j1)]
            top = max(s)
            w = [math.exp(x - top) for x in s]
            z = math.fsum(w)
            for d in range(D):
                O[b * Hq + hq, d] = math.fsum(w[i] * vd[j0 + i, h, d] for i in range(len(s))) / z
            LSE[b * Hq + hq] = top + math.log(z)
    return O, LSE


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [4, 128])
def test_brute_force_tiny(G, D):
    Hkv = 2
    lengths = [1, 17, 6]
    inp = make_small(3, Hkv * G, Hkv, D, lengths, seed=10 * G + D)
    o, lse = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    O, LSE = _brute_force(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    np.testing.assert_allclose(o, O, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(lse, LSE, rtol=RTOL, atol=ATOL)


@pytest.mark.parametrize("G", [1, 4, 8])
def test_matches_torch_sdpa_fp64(G):
    """Library special case: torch's fp64 scaled_dot_product_attention with K/V
    repeated per query head (repeat_interleave by G), and torch.logsumexp."""
    Hkv, D = 2, 64
    lengths = [3, 12]
    inp = make_small(2, Hkv * G, Hkv, D, lengths, seed=20 + G)
    o, lse = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    sc = inp["scale"]
    for b in range(2):
        j0, j1 = _rows_of(inp["kv_indptr"], b)
        qb = inp["q"][b].to(torch.float64).unsqueeze(1)                     # [Hq,1,D]
        kb = inp["k"][j0:j1].to(torch.float64).transpose(0, 1)              # [Hkv,L,D]
        vb = inp["v"][j0:j1].to(torch.float64).transpose(0, 1)
        kb = kb.repeat_interleave(G, dim=0)
        vb = vb.repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, scale=sc)[:, 0]
        ref_lse = torch.logsumexp((qb @ kb.transpose(1, 2))[:, 0] * sc, dim=-1)
        Hq = Hkv * G
        np.testing.assert_allclose(o[b * Hq:(b + 1) * Hq], ref.numpy(), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[b * Hq:(b + 1) * Hq], ref_lse.numpy(), rtol=1e-12, atol=1e-13)


# -------------------------------------------------------------- invariances

def test_joint_permutation_of_keys_and_values():
    inp = make_small(2, 8, 4, 32, [9, 14], seed=6)
    q, k, v, ip, sc = inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"]
    o, lse = oracle.decode(q, k, v, ip, sc)
    g = torch.Generator().manual_seed(7)
    perm = torch.cat([torch.randperm(9, generator=g), 9 + torch.randperm(14, generator=g)])
    o2, lse2 = oracle.decode(q, k[perm], v[perm], ip, sc)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-13)


def test_value_shift_shifts_output():
    inp = make_small(2, 4, 2, 16, [5, 8], seed=8)
    q, ip, sc = inp["q"], inp["kv_indptr"], inp["scale"]
    k64, v64 = inp["k"].to(torch.float64), inp["v"].to(torch.float64)
    o, lse = oracle.decode(q.to(torch.float64), k64, v64, ip, sc)
    o2, lse2 = oracle.decode(q.to(torch.float64), k64, v64 + 0.75, ip, sc)
    np.testing.assert_allclose(o2, o + 0.75, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(lse2, lse)


def test_gqa_equals_mha_with_repeated_kv_heads():
    """Query head hq reads KV head hq // G: the same as MHA over K/V whose heads
    are repeated G times (a hq % Hkv mapping fails this)."""
    G, Hkv = 4, 3
    inp = make_small(2, G * Hkv, Hkv, 32, [7, 10], seed=9)
    o, lse = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    kr = inp["k"].repeat_interleave(G, dim=1)
    vr = inp["v"].repeat_interleave(G, dim=1)
    o2, lse2 = oracle.decode(inp["q"], kr, vr, inp["kv_indptr"], inp["scale"])
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(lse2, lse)
    # and the mapping is not the identity: swapping two KV heads changes the output
    ks = inp["k"][:, [1, 0, 2]]
    o3, _ = oracle.decode(inp["q"], ks, inp["v"], inp["kv_indptr"], inp["scale"])
    assert np.abs(o3 - o).max() > 1e-3


def test_scale_enters_logits_linearly():
    """scale*2 on q is the same as doubling the scale (scale multiplies q.k)."""
    inp = make_small(1, 2, 2, 16, [12], seed=11)
    q64 = inp["q"].to(torch.float64)
    k64, v64 = inp["k"].to(torch.float64), inp["v"].to(torch.float64)
    sc = inp["scale"]
    a = oracle.decode(q64 * 2.0, k64, v64, inp["kv_indptr"], sc)
    b = oracle.decode(q64, k64, v64, inp["kv_indptr"], 2.0 * sc)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------ split / merge (§3)

def _random_items(kv_indptr, Hkv, rng, mode):
    ip = np.asarray(kv_indptr)
    items, seg_rows = [], []
    for b in range(ip.size - 1):
        j0, j1 = int(ip[b]), int(ip[b + 1])
        L = j1 - j0
        if L == 0:
            cuts = [j0, j1]
        elif mode == "one":
            cuts = [j0, j1]
        elif mode == "singletons":
            cuts = list(range(j0, j1 + 1))
        else:
            n = int(rng.integers(1, L + 1))
            inner = sorted(rng.choice(np.arange(j0 + 1, j1), size=min(n - 1, L - 1), replace=False)) if L > 1 else []
            cuts = [j0, *[int(c) for c in inner], j1]
        for h in range(Hkv):
            for c0, c1 in zip(cuts[:-1], cuts[1:]):
                if c1 > c0:
                    items.append((b, h, c0, c1))
    return np.array(items, dtype=np.int64).reshape(-1, 4)


def _seg_for(items, B, Hq, Hkv):
    """Group partial rows (item, g) by output row b*Hq + hq."""
    G = Hq // Hkv
    buckets = [[] for _ in range(B * Hq)]
    for i, (b, h, _, _) in enumerate(items):
        for g in range(G):
            buckets[b * Hq + h * G + g].append(i * G + g)
    order = [r for bucket in buckets for r in bucket]
    seg = np.zeros(B * Hq + 1, dtype=np.int64)
    seg[1:] = np.cumsum([len(bk) for bk in buckets])
    return np.array(order, dtype=np.int64), seg


@pytest.mark.parametrize("mode", ["one", "singletons", "random"])
@pytest.mark.parametrize("G", [1, 4])
def test_merge_of_any_partition_equals_unsplit(mode, G):
    Hkv, D = 2, 64
    inp = make_small(3, Hkv * G, Hkv, D, [1, 23, 40], seed=30 + G)
    q, k, v, ip, sc = inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"]
    rng = np.random.default_rng(G)
    items = _random_items(ip, Hkv, rng, mode)
    acc, m, l = oracle.split_partials(q, k, v, ip, sc, items)
    order, seg = _seg_for(items, 3, Hkv * G, Hkv)
    o, lse = oracle.merge(acc.reshape(-1, D)[order], m.reshape(-1)[order], l.reshape(-1)[order], seg)
    o_ref, lse_ref = oracle.decode(q, k, v, ip, sc)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)
    # the normalised form (O_i, LSE_i) merged with l = 1 is the same partial
    On, Ln = oracle.normalised(acc, m, l)
    o2, lse2 = oracle.merge(On.reshape(-1, D)[order], Ln.reshape(-1)[order],
                            np.ones(order.size), seg)
    np.testing.assert_allclose(o2, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse_ref, rtol=1e-12, atol=1e-13)


def test_single_chunk_partial_is_the_decode_row():
    """One chunk per request: acc/l and m + ln l are O and LSE of the definition."""
    inp = make_small(2, 4, 4, 16, [6, 9], seed=12)
    items = _random_items(inp["kv_indptr"], 4, None, "one")
    acc, m, l = oracle.split_partials(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"], items)
    On, Ln = oracle.normalised(acc, m, l)
    o, lse = oracle.decode(inp["q"], inp["k"], inp["v"], inp["kv_indptr"], inp["scale"])
    # items are ordered (b, h); with G = 1 the row is b*4 + h
    np.testing.assert_allclose(On.reshape(-1, 16), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Ln.reshape(-1), lse, rtol=1e-12, atol=1e-13)


def test_local_stats_closed_form():
    """Stage 1 on identical keys: m = s, l = chunk length, acc = sum of V."""
    inp = make_small(1, 1, 1, 8, [10], seed=13)
    k = inp["k"].clone()
    k[:] = k[0]
    acc, m, l = oracle.split_partials(inp["q"], k, inp["v"], inp["kv_indptr"], inp["scale"],
                                      [(0, 0, 2, 9)])
    qd, kd, vd = f64(inp["q"]), f64(k), f64(inp["v"])
    s = inp["scale"] * math.fsum(qd[0, 0, d] * kd[0, 0, d] for d in range(8))
    assert abs(m[0, 0] - s) < 1e-14
    assert l[0, 0] == 7.0
    np.testing.assert_allclose(acc[0, 0], vd[2:9, 0].sum(axis=0), rtol=1e-13, atol=1e-14)


def test_merge_ignores_empty_partials_and_handles_empty_rows():
    acc = np.array([[1.0, 2.0], [0.0, 0.0], [3.0, -1.0]])
    m = np.array([0.5, -np.inf, 0.5])
    l = np.array([2.0, 0.0, 2.0])
    o, lse = oracle.merge(acc, m, l, [0, 3, 3])
    np.testing.assert_allclose(o[0], [1.0, 0.25], rtol=1e-15)
    assert abs(lse[0] - (0.5 + math.log(4.0))) < 1e-15
    assert np.all(o[1] == 0.0) and np.isneginf(lse[1])


def test_merge_rescaling_sign():
    """Two chunks with different local maxima: the larger max gets factor 1,
    the other exp(m_i - M) < 1 (a sign error would weight it e^{+gap})."""
    acc = np.array([[1.0], [1.0]])
    m = np.array([0.0, -3.0])
    l = np.array([1.0, 1.0])
    o, lse = oracle.merge(acc, m, l, [0, 2])
    w = math.exp(-3.0)
    assert abs(o[0, 0] - 1.0) < 1e-15
    assert abs(lse[0] - math.log(1.0 + w)) < 1e-15
    acc2 = np.array([[2.0], [0.0]])
    o2, _ = oracle.merge(acc2, m, l, [0, 2])
    assert abs(o2[0, 0] - 2.0 / (1.0 + w)) < 1e-15


# ------------------------------------------------------ the article's check

def test_article_equivalence_check_setting():
    """§5's check: seed 42, B=1, H=32, D=128, S=8192, chunk 512, fp32 N(0,1);
    chunked split/merge vs unsplit stays under the printed bound."""
    cfg = json.load(open(os.path.join(GOLDEN, "page3_equivalence_check.json")))
    H, D, S, C = cfg["heads"], cfg["head_dim"], cfg["seq_len"], cfg["chunk"]
    g = torch.Generator().manual_seed(cfg["seed"])
    q = torch.randn(1, H, D, generator=g)
    k = torch.randn(S, H, D, generator=g)
    v = torch.randn(S, H, D, generator=g)
    ip = [0, S]
    sc = 1.0 / math.sqrt(D)
    items = np.array([(0, h, c, min(c + C, S)) for h in range(H) for c in range(0, S, C)])
    assert items.shape[0] == H * (S // C)
    acc, m, l = oracle.split_partials(q, k, v, ip, sc, items)
    order, seg = _seg_for(items, 1, H, H)
    o, _ = oracle.merge(acc.reshape(-1, D)[order], m.reshape(-1)[order], l.reshape(-1)[order], seg)
    o_ref, _ = oracle.decode(q, k, v, ip, sc)
    assert np.abs(o - o_ref).max() < cfg["max_abs_bound"]
