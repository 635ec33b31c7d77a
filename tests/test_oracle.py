"""Pins for the fp64 oracle against things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a wrong index or stride, a transposed operand, a missing max
subtraction, a wrong log base, a broken 16-bit decode) fails at least one:

* hand-worked examples (tests/golden/hand_worked.json, derivations inside);
* brute force with math.fsum on tiny asymmetric shapes (b, sq, sk, h, d all
  different), written from the definition without the max subtraction;
* a library special case: torch's CPU float64 scaled_dot_product_attention
  and logsumexp;
* closed forms and invariants: equal V rows, sk = 1, Q = 0, equal K rows,
  LSE bounds, joint permutation of K and V, V = identity (O = P, rows sum to
  1), scale = 0;
* the split-KV reduce: any split of the keys, empty splits included,
  combines back to the unsplit result;
* every fp16 and bf16 bit pattern decodes like numpy / torch do.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _rand(shape, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape)


# ---------------------------------------------------------------- golden
def _load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load_golden()["attention"], ids=lambda c: c["name"])
def test_hand_worked_attention(oracle_mod, case):
    q = np.array(case["q"], dtype=np.float64)
    k = np.array(case["k"], dtype=np.float64)
    v = np.array(case["v"], dtype=np.float64)
    assert q.shape == (case["b"], case["sq"], case["h"], case["d"])
    o, lse = oracle_mod.attention(q, k, v, case["scale"])
    np.testing.assert_allclose(o, np.array(case["o"]), rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, np.array(case["lse"]), rtol=0, atol=1e-11)


@pytest.mark.parametrize("case", _load_golden()["combine"], ids=lambda c: c["name"])
def test_hand_worked_combine(oracle_mod, case):
    lp = np.array([[float(x) for x in row] for row in case["lse_parts"]], dtype=np.float64)
    op = np.array(case["o_parts"], dtype=np.float64)
    o, lse = oracle_mod.combine(op, lp)
    np.testing.assert_allclose(o, np.array(case["o"]), rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, np.array(case["lse"]), rtol=0, atol=1e-11)


# ---------------------------------------------------------------- brute force
def _brute(q, k, v, scale):
    """Straight from the definition with exact sums; no max subtraction
    (inputs are small, so exp cannot overflow)."""
    b, sq, h, d = q.shape
    sk = k.shape[1]
    o = np.zeros((b, sq, h, d))
    lse = np.zeros((b, h, sq))
    for bb in range(b):
        for hh in range(h):
            for i in range(sq):
                s = [scale * math.fsum(q[bb, i, hh, t] * k[bb, j, hh, t] for t in range(d))
                     for j in range(sk)]
                e = [math.exp(x) for x in s]
                z = math.fsum(e)
                for t in range(d):
                    o[bb, i, hh, t] = math.fsum(e[j] / z * v[bb, j, hh, t] for j in range(sk))
                lse[bb, hh, i] = math.log(z)
    return o, lse


@pytest.mark.parametrize("shape,scale", [((2, 3, 5, 3, 4), 0.37), ((1, 4, 1, 2, 3), -1.3),
                                         ((3, 1, 7, 2, 5), 1.0), ((2, 6, 4, 1, 2), 0.0)])
def test_brute_force(oracle_mod, shape, scale):
    b, sq, sk, h, d = shape
    q = _rand((b, sq, h, d), 1)
    k = _rand((b, sk, h, d), 2)
    v = _rand((b, sk, h, d), 3)
    o, lse = oracle_mod.attention(q, k, v, scale)
    ob, lb = _brute(q, k, v, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_torch_sdpa_special_case(oracle_mod):
    b, sq, sk, h, d = 2, 9, 13, 3, 8
    scale = 0.29
    q = _rand((b, sq, h, d), 4)
    k = _rand((b, sk, h, d), 5)
    v = _rand((b, sk, h, d), 6)
    o, lse = oracle_mod.attention(q, k, v, scale)
    tq, tk, tv = (torch.from_numpy(x).transpose(1, 2) for x in (q, k, v))  # (b, h, s, d)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), rtol=0, atol=1e-12)
    ref_lse = torch.logsumexp(scale * tq @ tk.transpose(-1, -2), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- invariants
def test_equal_v_rows_give_that_row(oracle_mod):
    b, sq, sk, h, d = 2, 5, 11, 2, 6
    q, k = _rand((b, sq, h, d), 7) * 3, _rand((b, sk, h, d), 8) * 3
    c = _rand((b, 1, h, d), 9)
    v = np.broadcast_to(c, (b, sk, h, d)).copy()
    o, _ = oracle_mod.attention(q, k, v, 0.7)
    np.testing.assert_allclose(o, np.broadcast_to(c, (b, sq, h, d)), rtol=0, atol=1e-13)


def test_single_key(oracle_mod):
    b, sq, h, d = 2, 4, 3, 5
    q, k, v = _rand((b, sq, h, d), 10), _rand((b, 1, h, d), 11), _rand((b, 1, h, d), 12)
    o, lse = oracle_mod.attention(q, k, v, 0.45)
    np.testing.assert_allclose(o, np.broadcast_to(v, (b, sq, h, d)), rtol=0, atol=1e-14)
    expect = 0.45 * np.einsum("bihd,bhd->bhi", q, k[:, 0])
    np.testing.assert_allclose(lse, expect, rtol=0, atol=1e-13)


def test_zero_query_is_uniform(oracle_mod):
    b, sq, sk, h, d = 1, 3, 10, 2, 4
    q = np.zeros((b, sq, h, d))
    k, v = _rand((b, sk, h, d), 13), _rand((b, sk, h, d), 14)
    o, lse = oracle_mod.attention(q, k, v, 1.0)
    mean = v.mean(axis=1, keepdims=True)
    np.testing.assert_allclose(o, np.broadcast_to(mean, o.shape), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(sk), rtol=0, atol=1e-13)


def test_equal_k_rows_is_uniform(oracle_mod):
    b, sq, sk, h, d = 2, 3, 9, 1, 4
    q = _rand((b, sq, h, d), 15)
    krow = _rand((b, 1, h, d), 16)
    k = np.broadcast_to(krow, (b, sk, h, d)).copy()
    v = _rand((b, sk, h, d), 17)
    o, lse = oracle_mod.attention(q, k, v, 0.8)
    mean = v.mean(axis=1, keepdims=True)
    np.testing.assert_allclose(o, np.broadcast_to(mean, o.shape), rtol=0, atol=1e-13)
    s0 = 0.8 * np.einsum("bihd,bhd->bhi", q, krow[:, 0])
    np.testing.assert_allclose(lse, s0 + math.log(sk), rtol=0, atol=1e-13)


def test_lse_bounds_and_permutation(oracle_mod):
    b, sq, sk, h, d = 2, 6, 17, 3, 8
    q, k, v = _rand((b, sq, h, d), 18) * 2, _rand((b, sk, h, d), 19), _rand((b, sk, h, d), 20)
    scale = 0.6
    o, lse = oracle_mod.attention(q, k, v, scale)
    s = scale * np.einsum("bihd,bjhd->bhij", q, k)
    smax = s.max(axis=-1)
    assert np.all(lse >= smax - 1e-12)
    assert np.all(lse <= smax + math.log(sk) + 1e-12)
    perm = np.random.default_rng(21).permutation(sk)
    o2, lse2 = oracle_mod.attention(q, k[:, perm], v[:, perm], scale)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


def test_identity_v_exposes_probabilities(oracle_mod):
    """With V = I (sk = d) row i of O is the softmax row P_i: non-negative,
    summing to one, and proportional to exp(s_ij) with LSE as the log of the
    normaliser."""
    b, sq, h = 1, 5, 2
    sk = d = 7
    q, k = _rand((b, sq, h, d), 22) * 2, _rand((b, sk, h, d), 23)
    v = np.zeros((b, sk, h, d))
    for j in range(sk):
        v[:, j, :, j] = 1.0
    scale = 0.9
    o, lse = oracle_mod.attention(q, k, v, scale)
    p = o.transpose(0, 2, 1, 3)  # (b, h, sq, sk)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
    s = scale * np.einsum("bihd,bjhd->bhij", q, k)
    np.testing.assert_allclose(np.log(p), s - lse[..., None], rtol=0, atol=1e-12)


def test_rows_subset_and_key_range(oracle_mod):
    b, sq, sk, h, d = 2, 9, 12, 2, 4
    q, k, v = _rand((b, sq, h, d), 24), _rand((b, sk, h, d), 25), _rand((b, sk, h, d), 26)
    o, lse = oracle_mod.attention(q, k, v, 0.5)
    rows = [8, 0, 3]
    o_r, lse_r = oracle_mod.attention(q, k, v, 0.5, rows=rows)
    np.testing.assert_array_equal(o_r, o[:, rows])
    np.testing.assert_array_equal(lse_r, lse[:, :, rows])
    o_k, lse_k = oracle_mod.attention(q, k, v, 0.5, key_range=(3, 10))
    o_s, lse_s = oracle_mod.attention(q, k[:, 3:10].copy(), v[:, 3:10].copy(), 0.5)
    np.testing.assert_array_equal(o_k, o_s)
    np.testing.assert_array_equal(lse_k, lse_s)
    o_e, lse_e = oracle_mod.attention(q, k, v, 0.5, key_range=(4, 4))
    assert np.all(o_e == 0) and np.all(np.isneginf(lse_e))


@pytest.mark.parametrize("bounds", [
    [(0, 13)],
    [(0, 5), (5, 13)],
    [(0, 1), (1, 2), (2, 7), (7, 13)],
    [(0, 4), (4, 4), (4, 13), (13, 13)],  # empty splits
    [(0, 0), (0, 13)],
])
def test_split_combine_equals_unsplit(oracle_mod, bounds):
    b, sq, sk, h, d = 2, 3, 13, 2, 5
    q, k, v = _rand((b, sq, h, d), 27) * 2, _rand((b, sk, h, d), 28), _rand((b, sk, h, d), 29)
    o, lse = oracle_mod.attention(q, k, v, 0.77)
    o2, lse2 = oracle_mod.split_attention(q, k, v, 0.77, bounds)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)


def test_combine_weights_are_the_formula_not_uniform(oracle_mod):
    """Unequal split sizes make a plain average of O_i wrong; the reduce must
    weight each split by exp(LSE_i - LSE)."""
    b, sq, sk, h, d = 1, 2, 40, 1, 3
    q, k, v = _rand((b, sq, h, d), 30) * 3, _rand((b, sk, h, d), 31), _rand((b, sk, h, d), 32)
    parts = [oracle_mod.attention(q, k, v, 1.0, key_range=r) for r in [(0, 3), (3, 40)]]
    o, _ = oracle_mod.attention(q, k, v, 1.0)
    avg = 0.5 * (parts[0][0] + parts[1][0])
    assert np.abs(avg - o).max() > 1e-3
    o2, _ = oracle_mod.split_attention(q, k, v, 1.0, [(0, 3), (3, 40)])
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- 16-bit decode
def test_every_f16_pattern(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.decode_f16(int(x)) for x in bits])
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_every_bf16_pattern(oracle_mod):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.decode_bf16(int(x) & 0xFFFF) for x in bits.tolist()])
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_narrow_inputs_match_widened(oracle_mod, dtype):
    b, sq, sk, h, d = 2, 5, 7, 3, 16
    g = torch.Generator().manual_seed(0)
    q, k, v = (torch.randn(s, generator=g).to(dtype) for s in
               [(b, sq, h, d), (b, sk, h, d), (b, sk, h, d)])
    o, lse = oracle_mod.attention(q, k, v, 0.25)
    o64, lse64 = oracle_mod.attention(q.double(), k.double(), v.double(), 0.25)
    np.testing.assert_array_equal(o, o64)
    np.testing.assert_array_equal(lse, lse64)


# ---------------------------------------------------------------- causal mask
# Not on the pages; the reading is the bottom-right-aligned mask: query row i
# (of sq) sees key j (of sk) only if j <= i + sk - sq. Rows left with no key
# give O = 0 and LSE = -inf (the empty-range convention of the combine).
def _bottom_right_mask(sq, sk):
    i = np.arange(sq)[:, None]
    j = np.arange(sk)[None, :]
    return j <= i + (sk - sq)


def _torch_masked(q, k, v, scale, mask):
    tq, tk, tv = (torch.from_numpy(x).transpose(1, 2) for x in (q, k, v))  # (b, h, s, d)
    m = torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, scale=scale)
    sc = (scale * tq @ tk.transpose(-1, -2)).masked_fill(~m, float("-inf"))
    return o.transpose(1, 2).numpy(), torch.logsumexp(sc, dim=-1).numpy()


def test_causal_square_is_torch_is_causal(oracle_mod):
    b, s, h, d, scale = 2, 11, 3, 8, 0.41
    q, k, v = _rand((b, s, h, d), 21), _rand((b, s, h, d), 22), _rand((b, s, h, d), 23)
    o, lse = oracle_mod.attention(q, k, v, scale, causal=True)
    tq, tk, tv = (torch.from_numpy(x).transpose(1, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), rtol=0, atol=1e-12)
    _, ref_lse = _torch_masked(q, k, v, scale, _bottom_right_mask(s, s))
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("sq,sk", [(5, 13), (1, 7), (13, 13), (9, 4), (4, 1)])
def test_causal_rectangular_is_torch_bottom_right_mask(oracle_mod, sq, sk):
    b, h, d, scale = 2, 2, 6, 0.7
    q, k, v = _rand((b, sq, h, d), 24), _rand((b, sk, h, d), 25), _rand((b, sk, h, d), 26)
    o, lse = oracle_mod.attention(q, k, v, scale, causal=True)
    mask = _bottom_right_mask(sq, sk)
    seen = mask.any(axis=1)  # rows with at least one key
    ro, rl = _torch_masked(q, k, v, scale, mask)
    np.testing.assert_allclose(o[:, seen], ro[:, seen], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[:, :, seen], rl[:, :, seen], rtol=0, atol=1e-12)
    # rows with no key: the empty-range convention
    assert np.all(o[:, ~seen] == 0.0)
    assert np.all(np.isneginf(lse[:, :, ~seen]))
    assert (~seen).sum() == max(0, sq - sk)


def _brute_causal(q, k, v, scale):
    b, sq, h, d = q.shape
    sk = k.shape[1]
    o = np.zeros((b, sq, h, d))
    lse = np.full((b, h, sq), -np.inf)
    for bb in range(b):
        for hh in range(h):
            for i in range(sq):
                keys = [j for j in range(sk) if j - i <= sk - sq]
                if not keys:
                    continue
                e = [math.exp(scale * math.fsum(q[bb, i, hh, t] * k[bb, j, hh, t] for t in range(d)))
                     for j in keys]
                z = math.fsum(e)
                for t in range(d):
                    o[bb, i, hh, t] = math.fsum(e[n] / z * v[bb, j, hh, t] for n, j in enumerate(keys))
                lse[bb, hh, i] = math.log(z)
    return o, lse


@pytest.mark.parametrize("shape,scale", [((1, 3, 6, 2, 4), 0.5), ((2, 6, 3, 1, 3), -0.8),
                                         ((1, 4, 4, 2, 2), 1.1)])
def test_causal_brute_force(oracle_mod, shape, scale):
    b, sq, sk, h, d = shape
    q, k, v = _rand((b, sq, h, d), 27), _rand((b, sk, h, d), 28), _rand((b, sk, h, d), 29)
    o, lse = oracle_mod.attention(q, k, v, scale, causal=True)
    ob, lb = _brute_causal(q, k, v, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_causal_single_query_row_sees_every_key(oracle_mod):
    b, sk, h, d = 2, 17, 3, 5
    q, k, v = _rand((b, 1, h, d), 30), _rand((b, sk, h, d), 31), _rand((b, sk, h, d), 32)
    o0, l0 = oracle_mod.attention(q, k, v, 0.3)
    o1, l1 = oracle_mod.attention(q, k, v, 0.3, causal=True)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


@pytest.mark.parametrize("bounds", [[(0, 5), (5, 12), (12, 20)], [(0, 20), (20, 20)],
                                    [(0, 1), (1, 2), (2, 20)]])
def test_causal_split_combine_equals_unsplit(oracle_mod, bounds):
    b, sq, sk, h, d = 1, 8, 20, 2, 4
    q, k, v = _rand((b, sq, h, d), 33), _rand((b, sk, h, d), 34), _rand((b, sk, h, d), 35)
    o, lse = oracle_mod.attention(q, k, v, 0.6, causal=True)
    o2, l2 = oracle_mod.split_attention(q, k, v, 0.6, bounds, causal=True)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- paged KV cache
# The paged reference gathers each sequence's keys through its page table and
# calls the pinned `attention`; these pins tie the gather to layouts whose
# answer is known without it.
def _paged_from_contiguous(k, v, page_size, perm_seed=None):
    """Cut contiguous [b, sk, h, d] caches into pages of one pool (optionally
    in a shuffled pool order) and return (k_pages, v_pages, table)."""
    b, sk, h, d = k.shape
    npg = sk // page_size
    kp = k.reshape(b * npg, page_size, h, d)
    vp = v.reshape(b * npg, page_size, h, d)
    order = np.arange(b * npg)
    if perm_seed is not None:
        order = np.random.default_rng(perm_seed).permutation(b * npg)
    # pool slot order[j] holds logical page j
    kpool = np.empty_like(kp)
    vpool = np.empty_like(vp)
    kpool[order] = kp
    vpool[order] = vp
    table = order.reshape(b, npg)
    return kpool, vpool, table


@pytest.mark.parametrize("perm_seed", [None, 5])
def test_paged_equals_contiguous_cache(oracle_mod, perm_seed):
    b, sk, h, d, ps = 3, 12, 2, 4, 4
    q, k, v = _rand((b, 1, h, d), 40), _rand((b, sk, h, d), 41), _rand((b, sk, h, d), 42)
    kp, vp, table = _paged_from_contiguous(k, v, ps, perm_seed)
    o, lse = oracle_mod.paged_attention(q, kp, vp, table, np.full(b, sk), 0.5)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 0.5)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_paged_lengths_are_key_prefixes(oracle_mod):
    b, sk, h, d, ps = 3, 12, 2, 4, 4
    q, k, v = _rand((b, 1, h, d), 43), _rand((b, sk, h, d), 44), _rand((b, sk, h, d), 45)
    kp, vp, table = _paged_from_contiguous(k, v, ps, 7)
    lens = np.array([5, 12, 1])
    o, lse = oracle_mod.paged_attention(q, kp, vp, table, lens, 0.8)
    for i, n in enumerate(lens):
        o_ref, lse_ref = oracle_mod.attention(q[i:i + 1], k[i:i + 1], v[i:i + 1], 0.8, key_range=(0, n))
        np.testing.assert_allclose(o[i:i + 1], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[i:i + 1], lse_ref, rtol=0, atol=1e-12)


def test_paged_empty_sequence(oracle_mod):
    b, sk, h, d, ps = 2, 8, 1, 3, 4
    q, k, v = _rand((b, 1, h, d), 46), _rand((b, sk, h, d), 47), _rand((b, sk, h, d), 48)
    kp, vp, table = _paged_from_contiguous(k, v, ps)
    o, lse = oracle_mod.paged_attention(q, kp, vp, table, np.array([0, 8]), 1.0)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    o_ref, lse_ref = oracle_mod.attention(q[1:], k[1:], v[1:], 1.0)
    np.testing.assert_allclose(o[1:], o_ref, rtol=0, atol=1e-12)


def test_paged_several_rows_equal_contiguous_cache(oracle_mod):
    b, sq, sk, h, d, ps = 2, 5, 12, 2, 4, 4
    q, k, v = _rand((b, sq, h, d), 49), _rand((b, sk, h, d), 50), _rand((b, sk, h, d), 51)
    kp, vp, table = _paged_from_contiguous(k, v, ps, 3)
    o, lse = oracle_mod.paged_attention(q, kp, vp, table, np.full(b, sk), 0.6)
    tq, tk, tv = (torch.from_numpy(x).transpose(1, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.6)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), rtol=0, atol=1e-12)


def test_paged_causal_is_torch_bottom_right_mask_per_sequence(oracle_mod):
    """Several new rows per sequence under the causal mask, each sequence's
    mask aligned to its own key count (torch fp64 SDPA with the explicit
    bottom-right mask on the sequence's keys); rows that see no key (length
    below sq) give O = 0 and LSE = -inf."""
    b, sq, sk, h, d, ps = 4, 6, 16, 2, 5, 4
    q, k, v = _rand((b, sq, h, d), 52), _rand((b, sk, h, d), 53), _rand((b, sk, h, d), 54)
    kp, vp, table = _paged_from_contiguous(k, v, ps, 9)
    lens = np.array([16, 7, 3, 0])
    o, lse = oracle_mod.paged_attention(q, kp, vp, table, lens, 0.45, causal=True)
    for i, n in enumerate(lens):
        if n == 0:
            assert np.all(o[i] == 0.0) and np.all(np.isneginf(lse[i]))
            continue
        mask = _bottom_right_mask(sq, n)
        seen = mask.any(axis=1)
        ro, rl = _torch_masked(q[i:i + 1], k[i:i + 1, :n], v[i:i + 1, :n], 0.45, mask)
        np.testing.assert_allclose(o[i:i + 1, seen], ro[:, seen], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[i:i + 1, :, seen], rl[:, :, seen], rtol=0, atol=1e-12)
        assert np.all(o[i, ~seen] == 0.0) and np.all(np.isneginf(lse[i, :, ~seen]))
        assert (~seen).sum() == max(0, sq - n)


# ---------------------------------------------------------------- backward pass
# The gradients by the chain rule; pinned to torch's fp64 autograd (a library
# special case), to finite differences of the oracle's own forward, and to
# identities that hold for any input.
def _loss_grads_torch(q, k, v, do, scale, causal):
    tq, tk, tv = (torch.from_numpy(x).transpose(1, 2).requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale, is_causal=causal)
    o.backward(torch.from_numpy(do).transpose(1, 2))
    return tuple(t.grad.transpose(1, 2).numpy() for t in (tq, tk, tv))


@pytest.mark.parametrize("shape,scale,causal", [((2, 7, 11, 3, 5), 0.45, False),
                                                ((1, 9, 9, 2, 4), 0.8, True),
                                                ((1, 1, 6, 2, 3), -0.6, False)])
def test_backward_is_torch_autograd(oracle_mod, shape, scale, causal):
    b, sq, sk, h, d = shape
    q, k, v = _rand((b, sq, h, d), 50), _rand((b, sk, h, d), 51), _rand((b, sk, h, d), 52)
    do = _rand((b, sq, h, d), 53)
    dq, dk, dv = oracle_mod.attention_backward(q, k, v, do, scale, causal=causal)
    rq, rk, rv = _loss_grads_torch(q, k, v, do, scale, causal)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_backward_finite_differences(oracle_mod, which):
    """<grad, E> equals the central difference of L = sum(O * G) along E."""
    b, sq, sk, h, d, scale = 1, 3, 4, 1, 2, 0.7
    x = [_rand((b, sq, h, d), 54), _rand((b, sk, h, d), 55), _rand((b, sk, h, d), 56)]
    G = _rand((b, sq, h, d), 57)
    E = _rand(x[which].shape, 58)
    grads = oracle_mod.attention_backward(x[0], x[1], x[2], G, scale)
    eps = 1e-5

    def loss(t):
        y = list(x)
        y[which] = x[which] + t * E
        o, _ = oracle_mod.attention(y[0], y[1], y[2], scale)
        return float((o * G).sum())

    fd = (loss(eps) - loss(-eps)) / (2 * eps)
    assert abs(float((grads[which] * E).sum()) - fd) < 1e-8


def test_backward_identities(oracle_mod):
    """dS rows sum to 0, so dK sums to 0 over the keys; every column of P
    sums the upstream gradient into dV: sum_j dV_j = sum_i dO_i."""
    b, sq, sk, h, d = 2, 6, 9, 2, 4
    q, k, v = _rand((b, sq, h, d), 59), _rand((b, sk, h, d), 60), _rand((b, sk, h, d), 61)
    do = _rand((b, sq, h, d), 62)
    dq, dk, dv = oracle_mod.attention_backward(q, k, v, do, 0.5)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), atol=1e-12)
