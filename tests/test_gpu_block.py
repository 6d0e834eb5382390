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
    # An empty row (lse = -inf) carries no values: the library must not read
    # its o, so the GPU copies hold NaN there (the oracle's hold zeros).
    o_acc_g, o_blk_g = o_acc.clone(), o_blk.clone()
    o_acc_g[::7] = float("nan")
    o_blk_g[::11] = float("nan")
    oa, la = o_acc_g.cuda(), lse_acc.cuda()
    rsa.merge(oa, la, o_blk_g.cuda(), lse_blk.cuda())
    torch.cuda.synchronize()
    assert_close(oa, la, ref_o, ref_l, torch.float32, what="merge")
    # finalising merge to bf16 leaves the accumulator alone
    oa2, la2 = o_acc_g.cuda(), lse_acc.cuda()
    out, lse_out = rsa.merge_finalize(oa2, la2, o_blk_g.cuda(), lse_blk.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(oa2.cpu().nan_to_num(7.0), o_acc_g.nan_to_num(7.0)) and torch.equal(la2.cpu(), lse_acc)
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


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
def test_fold_on_partial_buffers_matches_oracle(dtype, d):
    # rsa_block_attn_fold: the query piece (positions 1024..1535) sits at row
    # 256 of its own buffer and each K/V piece at row 88 of another, so rows
    # and positions differ; FIRST, MERGE, LAST fold three pieces in an order
    # that is not the positions' order.
    need_cuda()
    from context_attention_rsa_gb300 import rank_ring as rr
    B, H, T = 1, 3, 1536
    (q, k, v), _ = qkv_cuda(B, H, T, d, dtype, seed=61)
    ro, rl = oracle.block(q, k, v, 1024, 512, 0, T, True)
    qb = torch.full((B, H, 768, d), float("nan"), dtype=dtype)
    qb[:, :, 256:768] = q[:, :, 1024:1536]
    qb = qb.cuda()
    acc = torch.full((B, H, 768, d), float("nan"), device="cuda")
    lse = torch.full((B, H, 768), 7.0, device="cuda")
    out = torch.full((B, H, 768, d), 3.0, dtype=dtype, device="cuda")
    for kv_pos, fold in ((512, rr.FOLD_FIRST), (0, rr.FOLD_MERGE), (1024, rr.FOLD_LAST)):
        kb = torch.zeros((B, H, 600, d), dtype=dtype)
        vb = torch.zeros((B, H, 600, d), dtype=dtype)
        kb[:, :, 88:600] = k[:, :, kv_pos:kv_pos + 512]
        vb[:, :, 88:600] = v[:, :, kv_pos:kv_pos + 512]
        step = dict(q_row0=256, q_pos=1024, q_len=512, kv_row0=88, kv_pos=kv_pos, kv_len=512, fold=fold)
        rr.block_attn_fold(qb, kb.cuda(), vb.cuda(), step, True, acc, lse, out)
        torch.cuda.synchronize()
    rsa.check_device_error()
    assert_close(out[:, :, 256:], lse[:, :, 256:], ro, rl, dtype, what="fold")
    assert torch.all(out[:, :, :256] == 3.0) and torch.all(lse[:, :, :256] == 7.0)  # other rows untouched
    # a single pair: RSA_FOLD_ONLY writes out and lse directly
    ro2, rl2 = oracle.block(q, k, v, 1024, 512, 1024, 512, True)
    kb = torch.zeros((B, H, 600, d), dtype=dtype)
    vb = torch.zeros((B, H, 600, d), dtype=dtype)
    kb[:, :, 88:600] = k[:, :, 1024:1536]
    vb[:, :, 88:600] = v[:, :, 1024:1536]
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    step = dict(q_row0=256, q_pos=1024, q_len=512, kv_row0=88, kv_pos=1024, kv_len=512, fold=rr.FOLD_ONLY)
    rr.block_attn_fold(qb, kb.cuda(), vb.cuda(), step, True, None, lse2, out2)
    torch.cuda.synchronize()
    assert_close(out2[:, :, 256:], lse2[:, :, 256:], ro2, rl2, dtype, what="fold only")


def test_fold_rejects_bad_rows_and_modes():
    need_cuda()
    from context_attention_rsa_gb300 import rank_ring as rr
    q = torch.zeros((1, 1, 256, 128), dtype=torch.bfloat16, device="cuda")
    acc = torch.zeros((1, 1, 256, 128), device="cuda")
    lse = torch.zeros((1, 1, 256), device="cuda")
    good = dict(q_row0=0, q_pos=0, q_len=256, kv_row0=0, kv_pos=0, kv_len=256, fold=rr.FOLD_FIRST)
    for bad in (dict(q_row0=1), dict(kv_len=257), dict(q_pos=-1), dict(fold=4)):
        with pytest.raises(rsa.RsaError) as e:
            rr.block_attn_fold(q, q, q, dict(good, **bad), True, acc, lse, q)
        assert e.value.status == 1
    with pytest.raises(rsa.RsaError):
        rr.block_attn_fold(q, q, q, good, True, None, lse, q)  # FIRST needs the accumulator
