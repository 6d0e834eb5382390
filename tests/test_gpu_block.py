"""GPU parity of the block-attention step (one (query chunk, KV chunk) pair)
and of the merge step, against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import context_attention_rsa_gb300 as rsa
from gpu_helpers import assert_close, need_cuda, qkv_cuda

pytestmark = pytest.mark.gpu


BLOCK_CASES = [
    # B, H, T, d, q_off, q_len, kv_off, kv_len, causal
    (1, 1, 128, 128, 0, 128, 0, 128, True),     # one tile, diagonal
    (1, 2, 256, 128, 0, 256, 0, 256, True),     # one CTA, two tiles
    (2, 3, 512, 128, 0, 512, 0, 512, False),    # several CTAs and KV tiles
    (1, 2, 1000, 128, 500, 500, 0, 500, True),  # off-diagonal, ragged tiles
    (1, 1, 1000, 128, 250, 250, 250, 250, True),  # ragged diagonal
    (1, 2, 700, 128, 3, 129, 1, 127, True),     # odd offsets, queries ahead of keys
    (1, 1, 300, 128, 0, 1, 0, 300, False),      # a single query row
    (1, 1, 300, 128, 299, 1, 0, 300, True),     # last row sees everything
    (2, 2, 384, 64, 0, 384, 0, 384, True),      # d = 64
    (1, 2, 600, 64, 100, 300, 350, 200, False), # d = 64, ragged
    (1, 1, 512, 128, 0, 256, 256, 256, True),   # every row fully masked
    (1, 1, 512, 128, 100, 200, 150, 300, True), # some rows fully masked
]


@pytest.mark.parametrize("case", BLOCK_CASES, ids=lambda c: "B{}H{}T{}d{}_q{}+{}_kv{}+{}_{}".format(
    *c[:8], "causal" if c[8] else "full"))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_block_attn_matches_oracle(case, dtype):
    need_cuda()
    B, H, T, d, q_off, q_len, kv_off, kv_len, causal = case
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, dtype, seed=hash(case) % 1000)
    o, l = rsa.block_attn_fwd(qd, kd, vd, q_off, q_len, kv_off, kv_len, causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.block(q, k, v, q_off, q_len, kv_off, kv_len, causal)
    assert_close(o, l, ro, rl, dtype, what=str(case))


def test_block_attn_wide_scores_and_outlier_keys():
    need_cuda()
    import rsa_inputs
    for recipe in ("wide", "outlier"):
        (q, k, v), (qd, kd, vd) = qkv_cuda(1, 4, 8192, 128, torch.bfloat16, recipe, seed=3)
        o, l = rsa.block_attn_fwd(qd, kd, vd, 4096, 4096, 0, 8192, True)
        torch.cuda.synchronize()
        rows = rsa_inputs.sample_rows(rsa_inputs.Workload("x", 1, 4, 8192, 128, 2, True, "bf16", recipe,
                                                          "sample"), n=512, seed=5)
        rows[:, 2] = 4096 + rows[:, 2] % 4096
        ro, rl = oracle.sampled(q, k, v, rows, causal=True)
        go = o[rows[:, 0], rows[:, 1], rows[:, 2] - 4096]
        gl = l[rows[:, 0], rows[:, 1], rows[:, 2] - 4096]
        assert_close(go, gl, ro, rl, torch.bfloat16, what=recipe)


@pytest.mark.parametrize("blk_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
def test_merge_matches_oracle(blk_dtype, d):
    need_cuda()
    g = torch.Generator().manual_seed(11)
    rows = 3001
    o_acc = torch.randn(rows, d, generator=g)
    o_blk = torch.randn(rows, d, generator=g).to(blk_dtype)
    lse_acc = torch.randn(rows, generator=g) * 20
    lse_blk = torch.randn(rows, generator=g) * 20
    lse_acc[::7] = -float("inf")
    lse_blk[::11] = -float("inf")
    o_acc[::7] = 0
    o_blk[::11] = 0
    ref_o, ref_l = oracle.merge_lse(o_acc.double().numpy(), lse_acc.double().numpy(),
                                    o_blk.double().numpy(), lse_blk.double().numpy())
    oa, la = o_acc.cuda(), lse_acc.cuda()
    rsa.merge(oa, la, o_blk.cuda(), lse_blk.cuda())
    torch.cuda.synchronize()
    assert_close(oa, la, ref_o, ref_l, torch.float32, what="merge")
    # finalising merge to bf16 leaves the accumulator alone
    oa2, la2 = o_acc.cuda(), lse_acc.cuda()
    out, lse_out = rsa.merge_finalize(oa2, la2, o_blk.cuda(), lse_blk.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(oa2.cpu(), o_acc) and torch.equal(la2.cpu(), lse_acc)
    assert_close(out, lse_out, ref_o, ref_l, torch.bfloat16, what="merge_finalize")


def test_merge_order_independence_through_block_calls():
    # Split one query chunk's keys four ways, merge the four partials in
    # several orders: every order matches the oracle.
    need_cuda()
    B, H, T, d = 1, 4, 2048, 128
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=21)
    ro, rl = oracle.block(q, k, v, 1536, 512, 0, 2048, True)
    parts = [rsa.block_attn_fwd(qd, kd, vd, 1536, 512, j * 512, 512, True) for j in range(4)]
    for order in ([0, 1, 2, 3], [3, 2, 1, 0], [2, 0, 3, 1]):
        o_acc = parts[order[0]][0].float().clone()
        l_acc = parts[order[0]][1].clone()
        for j in order[1:]:
            rsa.merge(o_acc, l_acc, parts[j][0], parts[j][1])
        torch.cuda.synchronize()
        assert_close(o_acc, l_acc, ro, rl, torch.bfloat16, what=str(order))


def test_block_outputs_leave_guard_bytes_alone():
    need_cuda()
    B, H, T, d = 1, 2, 700, 128
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=31)
    q_len = 333
    pad = 4096
    o_buf = torch.full((pad + B * H * q_len * d + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((pad + B * H * q_len + pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + B * H * q_len * d].view(B, H, q_len, d)
    l = l_buf[pad:pad + B * H * q_len].view(B, H, q_len)
    rsa.block_attn_fwd(qd, kd, vd, 367, q_len, 0, 700, True, o_blk=o, lse_blk=l)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7) and torch.all(o_buf[pad + o.numel():] == 7)
    assert torch.all(l_buf[:pad] == 7) and torch.all(l_buf[pad + l.numel():] == 7)
    ro, rl = oracle.block(q, k, v, 367, q_len, 0, 700, True)
    assert_close(o, l, ro, rl, torch.bfloat16)
