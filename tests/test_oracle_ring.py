"""Pins for the oracle's ring forms: O3 (online-softmax merging in ring order)
and O2 (two-pass Ring Self-Attention) must both reproduce the dense
definition O1, for any number of chunks and any order of KV chunks.  No GPU."""
import itertools

import numpy as np
import pytest

from conftest import read_golden

import oracle


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --- ring order against the printed tables -----------------------------------

def test_ring_rounds_match_printed_table():
    want = {}
    for rnd1, gpu, kv in (map(int, r) for r in read_golden("ring_table_n4.txt")):
        want.setdefault(rnd1 - 1, []).append((gpu, kv))
    for r, pairs in want.items():
        assert oracle.ring_round(4, r, causal=False) == sorted(pairs)


def test_librarian_boxes_follow_the_same_ring():
    # box b (0-based) is with librarian (b + r) mod N in round r; equivalently
    # librarian i holds box (i - r) mod N.
    for box1, visit1, lib in (map(int, r) for r in read_golden("librarian_boxes_n4.txt")):
        r = visit1 - 1
        assert (lib, box1 - 1) in oracle.ring_round(4, r, causal=False)


def test_causal_chunk_needs_match_page():
    pairs = oracle.ring_pairs(4, causal=True)
    for row in read_golden("causal_chunk_needs_n4.txt"):
        i = int(row[0])
        need = sorted(int(x) for x in row[1].split(","))
        assert sorted(j for (ii, j) in pairs if ii == i) == need


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 16])
def test_pair_counts(N):
    assert len(oracle.ring_pairs(N, causal=True)) == N * (N + 1) // 2
    assert len(oracle.ring_pairs(N, causal=False)) == N * N
    # every allowed pair exactly once; round 0 is the diagonal
    assert sorted(oracle.ring_pairs(N, True)) == sorted((i, j) for i in range(N) for j in range(i + 1))
    assert oracle.ring_round(N, 0, True) == [(i, i) for i in range(N)]


# --- merge identities -----------------------------------------------------------

def test_merge_empty_is_identity_and_two_empties_stay_empty():
    o = rnd((3, 4), 1)
    l = rnd((3,), 2)
    o2, l2 = oracle.merge_lse(o, l, np.zeros_like(o), np.full(3, -np.inf))
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(l2, l)
    o3, l3 = oracle.merge_lse(np.zeros_like(o), np.full(3, -np.inf), np.zeros_like(o), np.full(3, -np.inf))
    assert np.all(o3 == 0) and np.all(np.isneginf(l3)) and not np.any(np.isnan(o3))


def test_merge_is_commutative():
    oa, la, ob, lb = rnd((5, 4), 3), rnd((5,), 4, 5.0), rnd((5, 4), 5), rnd((5,), 6, 5.0)
    o1, l1 = oracle.merge_lse(oa, la, ob, lb)
    o2, l2 = oracle.merge_lse(ob, lb, oa, la)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-14)


def test_merging_two_key_halves_gives_the_whole():
    B, H, T, d = 1, 2, 24, 8
    q, k, v = rnd((B, H, T, d), 7), rnd((B, H, T, d), 8), rnd((B, H, T, d), 9)
    o1, l1 = oracle.block(q, k, v, 0, T, 0, 10, causal=False)
    o2, l2 = oracle.block(q, k, v, 0, T, 10, T - 10, causal=False)
    om, lm = oracle.merge_lse(o1, l1, o2, l2)
    ow, lw = oracle.attention(q, k, v, causal=False)
    np.testing.assert_allclose(om, ow, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lm, lw, rtol=0, atol=1e-13)


# --- O3 and O2 against O1 -------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
def test_online_ring_and_two_pass_equal_dense(N, causal):
    B, H, T, d = 2, 2, 48, 16
    q, k, v = rnd((B, H, T, d), 10 + N), rnd((B, H, T, d), 20 + N, 2.0), rnd((B, H, T, d), 30 + N)
    ow, lw = oracle.attention(q, k, v, causal)
    o3, l3 = oracle.ring_online(q, k, v, N, causal, check_mlo=True)
    np.testing.assert_allclose(o3, ow, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l3, lw, rtol=0, atol=1e-12)
    o2, l2 = oracle.rsa_two_pass(q, k, v, N, causal)
    np.testing.assert_allclose(o2, ow, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lw, rtol=0, atol=1e-12)


@pytest.mark.parametrize("N", [2, 3, 4])
def test_online_ring_is_order_independent_all_orders(N):
    B, H, T, d = 1, 1, 12 * N, 8
    q, k, v = rnd((B, H, T, d), 40), rnd((B, H, T, d), 41, 3.0), rnd((B, H, T, d), 42)
    ow, lw = oracle.attention(q, k, v, causal=False)
    for perm in itertools.permutations(range(N)):
        order = [(i, perm[(i + r) % N]) for r in range(N) for i in range(N)]
        o, l = oracle.ring_online(q, k, v, N, causal=False, order=order)
        np.testing.assert_allclose(o, ow, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lw, rtol=0, atol=1e-12)


def test_online_ring_random_orders_n8_causal():
    N, B, H, T, d = 8, 1, 2, 64, 8
    q, k, v = rnd((B, H, T, d), 43), rnd((B, H, T, d), 44, 3.0), rnd((B, H, T, d), 45)
    ow, lw = oracle.attention(q, k, v, causal=True)
    pairs = oracle.ring_pairs(N, causal=True)
    rng = np.random.default_rng(46)
    for _ in range(5):
        order = [pairs[i] for i in rng.permutation(len(pairs))]
        o, l = oracle.ring_online(q, k, v, N, causal=True, order=order)
        np.testing.assert_allclose(o, ow, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lw, rtol=0, atol=1e-12)


def test_outlier_keys_wide_scores():
    # Scores spanning hundreds (the stress pattern with sharp outlier keys)
    # still merge to the dense result.
    B, H, T, d, N = 1, 1, 64, 16, 4
    q, k, v = rnd((B, H, T, d), 47, 4.0), rnd((B, H, T, d), 48, 4.0), rnd((B, H, T, d), 49)
    k[:, :, ::16] *= 8.0
    ow, lw = oracle.attention(q, k, v, causal=True)
    o3, l3 = oracle.ring_online(q, k, v, N, causal=True)
    o2, l2 = oracle.rsa_two_pass(q, k, v, N, causal=True)
    scale = max(1.0, np.abs(lw).max())
    np.testing.assert_allclose(o3, ow, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l3, lw, rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(o2, ow, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lw, rtol=0, atol=1e-12 * scale)
