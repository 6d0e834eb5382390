"""Pins for the oracle's dense form (O1) against what the pages and plain
mathematics fix: closed forms, hand-worked values, invariants, and special
cases that reduce to library routines.  No GPU."""
import math

import numpy as np
import pytest
import scipy.special

from conftest import read_golden

import oracle
import rsa_inputs


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --- closed forms ---------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_its_value_and_score(causal):
    # T = 1: the only probability is 1, so o = v_0 and lse = s_0 = q.k_0/sqrt(d).
    B, H, d = 2, 3, 5
    q, k, v = rnd((B, H, 1, d), 1), rnd((B, H, 1, d), 2), rnd((B, H, 1, d), 3)
    out, lse = oracle.attention(q, k, v, causal)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-14)
    s0 = (q * k).sum(-1) / math.sqrt(d)
    np.testing.assert_allclose(lse, s0, rtol=0, atol=1e-14)


def test_two_keys_logistic_closed_form():
    # T = 2, full row: p_1 = sigma(s_1 - s_0), o = (1 - p_1) v_0 + p_1 v_1,
    # lse = s_0 + log1p(e^{s_1 - s_0}).
    B, H, d = 1, 2, 7
    q, k, v = rnd((B, H, 2, d), 4), rnd((B, H, 2, d), 5), rnd((B, H, 2, d), 6)
    out, lse = oracle.attention(q, k, v, causal=False)
    for b in range(B):
        for h in range(H):
            for t in range(2):
                s0 = q[b, h, t] @ k[b, h, 0] / math.sqrt(d)
                s1 = q[b, h, t] @ k[b, h, 1] / math.sqrt(d)
                p1 = scipy.special.expit(s1 - s0)
                np.testing.assert_allclose(out[b, h, t], (1 - p1) * v[b, h, 0] + p1 * v[b, h, 1],
                                           rtol=0, atol=1e-14)
                assert abs(lse[b, h, t] - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-14
    # causal: row 0 sees only key 0, row 1 sees both
    outc, lsec = oracle.attention(q, k, v, causal=True)
    np.testing.assert_array_equal(outc[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(outc[:, :, 1], out[:, :, 1], rtol=0, atol=1e-15)


def test_hand_worked_d1_values():
    q = np.ones((1, 1, 3, 1))
    k = np.array([0.0, math.log(2.0), math.log(4.0)]).reshape(1, 1, 3, 1)
    v = np.array([7.0, 14.0, 0.0]).reshape(1, 1, 3, 1)
    res = {c: oracle.attention(q, k, v, bool(c)) for c in (0, 1)}
    rows = read_golden("hand_d1.txt")
    assert len(rows) == 6
    for causal, t, num, den, lse_of in (map(int, r) for r in rows):
        out, lse = res[causal]
        assert abs(out[0, 0, t, 0] - num / den) < 1e-13
        assert abs(lse[0, 0, t] - math.log(lse_of)) < 1e-14


# --- invariants -------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_sum_to_one_and_match_scipy_softmax(causal):
    # With V = I (T = d) the output row is the probability row itself.
    B, H, T = 1, 2, 48
    d = T
    q, k = rnd((B, H, T, d), 7), rnd((B, H, T, d), 8)
    v = np.broadcast_to(np.eye(T), (B, H, T, d)).copy()
    P, lse = oracle.attention(q, k, v, causal)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
    s = np.einsum("bhtx,bhjx->bhtj", q, k) / math.sqrt(d)
    if causal:
        s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
    np.testing.assert_allclose(P, scipy.special.softmax(s, axis=-1), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(s, axis=-1), rtol=0, atol=1e-12)


def test_causal_pattern_matches_printed_figure():
    # V = I makes out[t, j] = p_j for query t; p_j > 0 exactly where allowed.
    T = 5
    q, k = rnd((1, 1, T, T), 9), rnd((1, 1, T, T), 10)
    v = np.eye(T).reshape(1, 1, T, T)
    P, _ = oracle.attention(q, k, v, causal=True)
    pattern = [["X" if P[0, 0, t, j] > 0 else "." for j in range(T)] for t in range(T)]
    assert pattern == read_golden("causal_pattern_5.txt")


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(causal):
    # All scores equal => p = 1/n: out = mean(V) (prefix mean if causal),
    # lse = s + ln n.
    B, H, T, d = 2, 2, 33, 16
    q = rnd((B, H, T, d), 11)
    k = np.broadcast_to(rnd((B, H, 1, d), 12), (B, H, T, d)).copy()
    v = rnd((B, H, T, d), 13)
    out, lse = oracle.attention(q, k, v, causal)
    s = (q * k).sum(-1) / math.sqrt(d)
    n = np.arange(1, T + 1) if causal else np.full(T, T)
    if causal:
        want = np.cumsum(v, axis=2) / n[:, None]
    else:
        want = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, s + np.log(n), rtol=0, atol=1e-12)


def test_causal_row0_is_exactly_v0_and_chunk0_ignores_later_chunks():
    B, H, T, d, N = 1, 2, 64, 8, 4
    q, k, v = rnd((B, H, T, d), 14), rnd((B, H, T, d), 15), rnd((B, H, T, d), 16)
    out, lse = oracle.attention(q, k, v, causal=True)
    np.testing.assert_array_equal(out[:, :, 0], v[:, :, 0])
    Tc = T // N
    k2, v2 = k.copy(), v.copy()
    k2[:, :, Tc:] = rnd((B, H, T - Tc, d), 17)
    v2[:, :, Tc:] = rnd((B, H, T - Tc, d), 18)
    out2, lse2 = oracle.attention(q, k2, v2, causal=True)
    np.testing.assert_array_equal(out2[:, :, :Tc], out[:, :, :Tc])
    np.testing.assert_array_equal(lse2[:, :, :Tc], lse[:, :, :Tc])
    assert not np.array_equal(out2[:, :, Tc:], out[:, :, Tc:])


def test_causal_row_ignores_future_keys():
    B, H, T, d = 1, 1, 40, 8
    q, k, v = rnd((B, H, T, d), 19), rnd((B, H, T, d), 20), rnd((B, H, T, d), 21)
    out, _ = oracle.attention(q, k, v, causal=True)
    t = 17
    k2, v2 = k.copy(), v.copy()
    k2[:, :, t + 1:] *= -3.0
    v2[:, :, t + 1:] += 5.0
    out2, _ = oracle.attention(q, k2, v2, causal=True)
    np.testing.assert_array_equal(out2[:, :, :t + 1], out[:, :, :t + 1])


def test_heads_are_independent():
    # Each (b, h) slice is its own attention problem.
    B, H, T, d = 2, 3, 20, 8
    q, k, v = rnd((B, H, T, d), 22), rnd((B, H, T, d), 23), rnd((B, H, T, d), 24)
    out, lse = oracle.attention(q, k, v, causal=True)
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            o1, l1 = oracle.attention(q[sl], k[sl], v[sl], causal=True)
            np.testing.assert_array_equal(o1[0, 0], out[b, h])
            np.testing.assert_array_equal(l1[0, 0], lse[b, h])


def test_key_permutation_invariance_noncausal():
    # Without a mask the keys form a set: permuting (k_j, v_j) together
    # leaves every output unchanged.
    B, H, T, d = 1, 2, 30, 8
    q, k, v = rnd((B, H, T, d), 25), rnd((B, H, T, d), 26), rnd((B, H, T, d), 27)
    perm = np.random.default_rng(28).permutation(T)
    o1, l1 = oracle.attention(q, k, v, causal=False)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], causal=False)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


def test_scale_uses_per_head_dk():
    # Doubling d with a zero-padded q and k keeps q.k but divides the scores
    # by sqrt(2) more: lse of one key moves from s to s/sqrt(2).
    q, k, v = rnd((1, 1, 1, 4), 29), rnd((1, 1, 1, 4), 30), rnd((1, 1, 1, 4), 31)
    pad = lambda a: np.concatenate([a, np.zeros_like(a)], axis=-1)
    _, l4 = oracle.attention(q, k, v, False)
    _, l8 = oracle.attention(pad(q), pad(k), pad(v), False)
    assert abs(l8[0, 0, 0] - l4[0, 0, 0] / math.sqrt(2.0)) < 1e-14


def test_bf16_inputs_are_widened_exactly():
    import torch
    g = torch.Generator().manual_seed(3)
    x = [torch.randn(1, 2, 24, 16, generator=g).to(torch.bfloat16) for _ in range(3)]
    o_bf, l_bf = oracle.attention(*x, causal=True)
    o_64, l_64 = oracle.attention(*[t.double().numpy() for t in x], causal=True)
    np.testing.assert_array_equal(o_bf, o_64)
    np.testing.assert_array_equal(l_bf, l_64)


def test_sampled_rows_equal_dense_rows():
    B, H, T, d = 2, 2, 50, 8
    q, k, v = rnd((B, H, T, d), 32), rnd((B, H, T, d), 33), rnd((B, H, T, d), 34)
    out, lse = oracle.attention(q, k, v, causal=True)
    rows = np.array([[0, 0, 0], [1, 1, 49], [0, 1, 25], [1, 0, 7]])
    o_s, l_s = oracle.sampled(q, k, v, rows, causal=True)
    for r, (b, h, t) in enumerate(rows):
        np.testing.assert_array_equal(o_s[r], out[b, h, t])
        assert l_s[r] == lse[b, h, t]


def test_block_with_no_allowed_key_is_empty():
    q, k, v = rnd((1, 1, 8, 4), 35), rnd((1, 1, 8, 4), 36), rnd((1, 1, 8, 4), 37)
    o, l = oracle.block(q, k, v, q_off=0, q_len=4, kv_off=4, kv_len=4, causal=True)
    assert np.all(o == 0) and np.all(np.isneginf(l))


# --- page arithmetic ----------------------------------------------------------

def test_page_size_arithmetic():
    g = {r[0]: int(r[1]) for r in read_golden("sizes.txt")}
    assert g["B"] * g["T"] * g["d"] * g["bytes_per_elem"] == g["hidden_bytes"] == 4 * 2**30
    assert g["hidden_bytes"] // g["gpus"] == g["per_gpu_bytes"] == 2**30
    w = rsa_inputs.WORKLOADS["page1_causal_bf16"]
    assert w.H * w.d == g["d"] and w.B == g["B"] and w.T == g["T"] and w.N == g["gpus"]
    q_bytes = w.B * w.H * w.T * w.d * 2
    assert q_bytes == g["hidden_bytes"]
    assert q_bytes // w.N == g["per_gpu_bytes"]
    # the query at token 30,000 (1-based) lives on GPU 3 and sees 30,000 keys
    t = g["query_token"] - 1
    lo, hi = oracle.chunk_range(w.T, w.N, g["query_gpu"])
    assert lo <= t < hi
    rows = np.array([[0, 0, t]])
    assert oracle.rows_flops(rows, w.T, w.d, True) == 4.0 * w.d * g["query_keys"]


@pytest.mark.parametrize("fname,T", [("chunks_t32768_n4.txt", 32768), ("chunks_t100000_n4.txt", 100000)])
def test_chunk_ranges_match_pages(fname, T):
    for i, first, last in (map(int, r) for r in read_golden(fname)):
        lo, hi = oracle.chunk_range(T, 4, i)
        assert (lo + 1, hi) == (first, last)


def test_useful_flops_formula():
    # causal: T(T+1)/2 allowed pairs per head, 4d FLOPs each
    assert oracle.flops_useful(1, 1, 3, 2, True) == 4 * 2 * 6
    assert oracle.flops_useful(2, 1, 3, 2, False) == 4 * 2 * 2 * 9
    # page-1 shape
    assert oracle.flops_useful(8, 64, 32768, 128, True) == pytest.approx(1.4074e14, rel=1e-4)
