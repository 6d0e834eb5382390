"""Randomised GPU parity: shapes, offsets, chunk counts, masks and dtypes drawn
from a seeded generator, each case compared with the oracle through the C ABI.
The fixed cases elsewhere cover the edges by design; these cover the
combinations nobody listed (odd chunk lengths against tile boundaries, pairs
whose rows and keys straddle each other, both block kernels, both ring forms,
decode shard counts, two-pass chunk counts)."""
import numpy as np
import pytest
import torch

import oracle
import rsa_inputs
import context_attention_rsa_gb300 as rsa
from gpu_helpers import assert_close, need_cuda

pytestmark = pytest.mark.gpu

N_CASES = 24


def _divisors(T, cap):
    return [n for n in range(1, min(T, cap) + 1) if T % n == 0]


def _qkv(B, H, T, d, dtype, seed):
    q, k, v = rsa_inputs.make_qkv(B, H, T, d, dtype, "normal", seed, "cpu")
    return (q, k, v), (q.cuda(), k.cuda(), v.cuda())


def ring_cases():
    rng = np.random.default_rng(20261203)
    out = []
    for i in range(N_CASES):
        d = int(rng.choice([64, 128]))
        dtype = torch.float32 if rng.random() < 0.25 else torch.bfloat16
        T = int(rng.integers(1, 1600))
        N = int(rng.choice(_divisors(T, 24)))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        causal = bool(rng.random() < 0.7)
        fused = bool(rng.random() < 0.5)
        out.append((B, H, T, d, N, causal, dtype, fused, 1000 + i))
    return out


def block_cases():
    rng = np.random.default_rng(4242)
    out = []
    for i in range(N_CASES):
        d = int(rng.choice([64, 128]))
        dtype = torch.float32 if rng.random() < 0.25 else torch.bfloat16
        T = int(rng.integers(2, 1400))
        q_len = int(rng.integers(1, T + 1))
        q_off = int(rng.integers(0, T - q_len + 1))
        kv_len = int(rng.integers(1, T + 1))
        kv_off = int(rng.integers(0, T - kv_len + 1))
        causal = bool(rng.random() < 0.7)
        kernel = str(rng.choice(["one_sm", "two_sm"]))
        out.append((1, int(rng.integers(1, 3)), T, d, q_off, q_len, kv_off, kv_len, causal, dtype, kernel, 2000 + i))
    return out


def decode_cases():
    rng = np.random.default_rng(777)
    out = []
    for i in range(N_CASES // 2):
        T = int(rng.integers(64, 6000))
        N = int(rng.choice(_divisors(T, 64)))
        q_len = int(rng.integers(1, min(T, 9) + 1))
        d = int(rng.choice([64, 128]))
        out.append((int(rng.integers(1, 3)), int(rng.integers(1, 4)), T, d, q_len, N, bool(rng.random() < 0.8),
                    3000 + i))
    return out


def two_pass_cases():
    rng = np.random.default_rng(99)
    out = []
    for i in range(N_CASES // 2):
        N = int(rng.integers(1, 6))
        T = 128 * N * int(rng.integers(1, 4))
        out.append((int(rng.integers(1, 3)), int(rng.integers(1, 3)), T, N, bool(rng.random() < 0.6), 4000 + i))
    return out


def _dt(t):
    return "bf16" if t == torch.bfloat16 else "f32"


@pytest.mark.parametrize("case", ring_cases(), ids=lambda c: "B{}H{}T{}d{}N{}_{}_{}_{}".format(
    *c[:5], "causal" if c[5] else "full", _dt(c[6]), "fused" if c[7] else "merge"))
def test_random_ring_matches_oracle(case):
    need_cuda()
    B, H, T, d, N, causal, dtype, fused, seed = case
    (q, k, v), (qd, kd, vd) = _qkv(B, H, T, d, dtype, seed)
    out, lse = rsa.ring_attn(qd, kd, vd, N, causal, fused=fused)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.attention(q, k, v, causal)
    assert_close(out, lse, ro, rl, dtype, what=str(case))


@pytest.fixture
def block_kernel():
    yield rsa.set_block_kernel
    rsa.set_block_kernel("auto")


@pytest.mark.parametrize("case", block_cases(), ids=lambda c: "T{}d{}_q{}+{}_kv{}+{}_{}_{}_{}".format(
    c[2], c[3], *c[4:8], "causal" if c[8] else "full", _dt(c[9]), c[10]))
def test_random_block_pair_matches_oracle(case, block_kernel):
    need_cuda()
    B, H, T, d, q_off, q_len, kv_off, kv_len, causal, dtype, kernel, seed = case
    block_kernel(kernel)  # the two-SM kernel takes the pairs it applies to
    (q, k, v), (qd, kd, vd) = _qkv(B, H, T, d, dtype, seed)
    o, l = rsa.block_attn_fwd(qd, kd, vd, q_off, q_len, kv_off, kv_len, causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.block(q, k, v, q_off, q_len, kv_off, kv_len, causal)
    assert_close(o, l, ro, rl, dtype, what=str(case))


@pytest.mark.parametrize("case", decode_cases(), ids=lambda c: "B{}H{}T{}d{}_q{}_N{}_{}".format(
    *c[:6], "causal" if c[6] else "full"))
def test_random_decode_matches_oracle(case):
    need_cuda()
    B, H, T, d, ql, N, causal, seed = case
    q_full, k, v = rsa_inputs.make_qkv(B, H, T, d, torch.bfloat16, "normal", seed, "cpu")
    q = q_full[:, :, T - ql:].contiguous()
    out, lse = rsa.decode_attn(q.cuda(), k.cuda(), v.cuda(), N, causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    rows = np.array([[b, h, T - ql + r] for b in range(B) for h in range(H) for r in range(ql)], dtype=np.int64)
    ro, rl = oracle.attend_rows(q.reshape(-1, d), k, v, rows, causal)
    assert_close(out.reshape(-1, d), lse.reshape(-1), ro, rl, torch.bfloat16, what=str(case))


@pytest.mark.parametrize("case", two_pass_cases(), ids=lambda c: "B{}H{}T{}N{}_{}".format(
    *c[:4], "causal" if c[4] else "full"))
def test_random_two_pass_matches_oracle(case):
    need_cuda()
    B, H, T, N, causal, seed = case
    (q, k, v), (qd, kd, vd) = _qkv(B, H, T, 128, torch.bfloat16, seed)
    out, lse = rsa.two_pass_attn(qd, kd, vd, N, causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.attention(q, k, v, causal)
    assert_close(out, lse, ro, rl, torch.bfloat16, what=str(case))


def fold_cases():
    rng = np.random.default_rng(31337)
    out = []
    for i in range(N_CASES // 2):
        d = int(rng.choice([64, 128]))
        dtype = torch.float32 if rng.random() < 0.25 else torch.bfloat16
        T = int(rng.integers(64, 1500))
        q_len = int(rng.integers(1, min(T, 600) + 1))
        q_pos = int(rng.integers(0, T - q_len + 1))
        n_pieces = int(rng.integers(1, 6))
        cuts = sorted(set(int(x) for x in rng.integers(1, T, size=n_pieces - 1))) if n_pieces > 1 else []
        bounds = [0] + cuts + [T]
        pieces = [(bounds[j], bounds[j + 1] - bounds[j]) for j in range(len(bounds) - 1)]
        order = [int(x) for x in rng.permutation(len(pieces))]
        out.append((int(rng.integers(1, 3)), T, d, q_pos, q_len, [pieces[j] for j in order],
                    bool(rng.random() < 0.7), dtype, int(rng.integers(0, 97)), int(rng.integers(0, 53)), 5000 + i))
    return out


@pytest.mark.parametrize("case", fold_cases(), ids=lambda c: "T{}d{}_q{}+{}_{}pieces_{}_{}".format(
    c[1], c[2], c[3], c[4], len(c[5]), "causal" if c[6] else "full", _dt(c[7])))
def test_random_fold_sequences_match_oracle(case):
    # rsa_block_attn_fold as a rank uses it: the query block sits at row
    # q_row0 of its own buffer, each K/V piece at row kv_row0 of a buffer of
    # its own; the pieces (a random cut of the whole key range) are folded in
    # a random order, FIRST .. MERGE .. LAST (ONLY for a single piece), with
    # rows and global positions apart.
    need_cuda()
    from context_attention_rsa_gb300 import rank_ring as rr
    H, T, d, q_pos, q_len, pieces, causal, dtype, q_row0, kv_row0, seed = case
    B = 1
    (q, k, v), _ = _qkv(B, H, T, d, dtype, seed)
    qb = torch.full((B, H, q_row0 + q_len, d), float("nan"), dtype=dtype)
    qb[:, :, q_row0:] = q[:, :, q_pos:q_pos + q_len]
    qb = qb.cuda()
    acc = torch.full((B, H, q_row0 + q_len, d), float("nan"), device="cuda")
    lse = torch.full((B, H, q_row0 + q_len), 7.0, device="cuda")
    out = torch.full((B, H, q_row0 + q_len, d), 3.0, dtype=dtype, device="cuda")
    n = len(pieces)
    for j, (kv_pos, kv_len) in enumerate(pieces):
        fold = rr.FOLD_ONLY if n == 1 else (rr.FOLD_FIRST if j == 0 else (rr.FOLD_LAST if j == n - 1 else rr.FOLD_MERGE))
        kb = torch.zeros((B, H, kv_row0 + kv_len, d), dtype=dtype)
        vb = torch.zeros((B, H, kv_row0 + kv_len, d), dtype=dtype)
        kb[:, :, kv_row0:] = k[:, :, kv_pos:kv_pos + kv_len]
        vb[:, :, kv_row0:] = v[:, :, kv_pos:kv_pos + kv_len]
        step = dict(q_row0=q_row0, q_pos=q_pos, q_len=q_len, kv_row0=kv_row0, kv_pos=kv_pos, kv_len=kv_len,
                    fold=fold)
        rr.block_attn_fold(qb, kb.cuda(), vb.cuda(), step, causal, acc if n > 1 else None, lse, out)
        torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.block(q, k, v, q_pos, q_len, 0, T, causal)
    assert_close(out[:, :, q_row0:], lse[:, :, q_row0:], ro, rl, dtype, what=str(case[:7]))
    assert torch.all(out[:, :, :q_row0] == 3.0) and torch.all(lse[:, :, :q_row0] == 7.0)
