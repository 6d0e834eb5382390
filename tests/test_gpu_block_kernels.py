"""GPU parity of both bf16 tensor-core block kernels, chosen explicitly with
rsa_set_block_kernel: the one-SM kernel (a CTA per 256 query rows) and the
two-SM kernel (a CTA pair per 512 rows sharing each K/V tile through the
paired MMA).  Each is compared with the oracle on single pairs and whole
rings, including the epilogues that fold a pair into the ring accumulator."""
import pytest
import torch

import oracle
import context_attention_rsa_gb300 as rsa
from gpu_helpers import assert_close, need_cuda, qkv_cuda

pytestmark = pytest.mark.gpu

KERNELS = ["one_sm", "two_sm"]


@pytest.fixture
def kernel(request):
    rsa.set_block_kernel(request.param)
    yield request.param
    rsa.set_block_kernel("auto")


PAIR_CASES = [
    # B, H, T, d, q_off, q_len, kv_off, kv_len, causal
    (1, 2, 1024, 128, 0, 512, 0, 512, True),        # one cluster, diagonal
    (1, 2, 2048, 128, 1024, 1024, 0, 1024, True),   # off-diagonal, every key visible
    (2, 3, 1536, 128, 0, 1536, 0, 1536, False),     # three clusters per head, full
    (1, 2, 3000, 128, 1000, 1000, 1000, 1000, True),  # ragged diagonal: 1000 rows, odd key tail
    (1, 1, 2000, 128, 1100, 700, 0, 900, True),     # ragged off-diagonal
    (1, 1, 1200, 128, 100, 600, 650, 500, True),    # rows before the keys see nothing
    (1, 1, 1024, 128, 0, 512, 512, 512, True),      # every row fully masked
    (1, 1, 1100, 128, 0, 1100, 0, 1100, True),      # the last cluster holds 76 rows
]


@pytest.mark.parametrize("kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "B{}H{}T{}_q{}+{}_kv{}+{}_{}".format(
    c[0], c[1], c[2], *c[4:8], "causal" if c[8] else "full"))
def test_pair_matches_oracle(case, kernel):
    need_cuda()
    B, H, T, d, q_off, q_len, kv_off, kv_len, causal = case
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=T + q_off)
    o, l = rsa.block_attn_fwd(qd, kd, vd, q_off, q_len, kv_off, kv_len, causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.block(q, k, v, q_off, q_len, kv_off, kv_len, causal)
    assert_close(o, l, ro, rl, torch.bfloat16, what=f"{kernel} {case}")


RING_CASES = [
    # B, H, T, d, N, causal
    (1, 4, 4096, 128, 4, True),    # chunks of 1024: two clusters per pair
    (2, 2, 3072, 128, 3, False),   # chunks of 1024, every pair full
    (1, 3, 3000, 128, 2, True),    # chunks of 1500: ragged last cluster
]


@pytest.mark.parametrize("kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("fused", [False, True], ids=["merge_kernel", "fused_merge"])
@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: "B{}H{}T{}N{}_{}".format(
    c[0], c[1], c[2], c[4], "causal" if c[5] else "full"))
def test_ring_matches_oracle(case, fused, kernel):
    need_cuda()
    B, H, T, d, N, causal = case
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=7 * T + N)
    out, lse = rsa.ring_attn(qd, kd, vd, N, causal, fused=fused)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.attention(q, k, v, causal)
    assert_close(out, lse, ro, rl, torch.bfloat16, what=f"{kernel} fused={fused} {case}")


def test_kernels_agree_and_each_is_deterministic():
    need_cuda()
    B, H, T, d = 2, 8, 4096, 128
    _, (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=99)
    res = {}
    try:
        for kern in KERNELS:
            rsa.set_block_kernel(kern)
            a = rsa.ring_attn(qd, kd, vd, 4, True)
            b = rsa.ring_attn(qd, kd, vd, 4, True)
            torch.cuda.synchronize()
            rsa.check_device_error()
            assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]), kern
            res[kern] = a
    finally:
        rsa.set_block_kernel("auto")
    (o1, l1), (o2, l2) = res["one_sm"], res["two_sm"]
    # Same arithmetic in the same order per row: only the MMA's internal
    # accumulation order may differ, so the two agree far inside the bf16 bar.
    assert (o1.float() - o2.float()).abs().max().item() <= 8e-3
    assert (l1 - l2).abs().max().item() <= 1e-4

