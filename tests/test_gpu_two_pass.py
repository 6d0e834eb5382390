"""GPU parity of the two-pass Ring Self-Attention (full score rows per query
chunk, softmax over the row, then the value ring) against the oracle's dense
form and its own two-pass form, and agreement with the online ring."""
import numpy as np
import pytest
import torch

import oracle
import rsa_inputs
import context_attention_rsa_gb300 as rsa
from gpu_helpers import assert_close, need_cuda, qkv_cuda

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, T, d, N, causal
    (1, 2, 512, 128, 4, True),
    (2, 1, 1024, 128, 2, False),
    (1, 3, 1024, 128, 8, True),
    (1, 1, 384, 128, 1, True),
    (2, 2, 768, 128, 3, False),
    (1, 1, 8192, 128, 4, True),   # 64 key tiles per row: the row statistics take two strides of a warp
    (2, 3, 2048, 128, 2, True),   # several score tiles per persistent CTA, ranges across query tiles and heads
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}T{}d{}N{}_{}".format(*c[:5], "causal" if c[5] else "full"))
def test_two_pass_matches_oracle(case):
    need_cuda()
    B, H, T, d, N, causal = case
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=T * 7 + N)
    out, lse = rsa.two_pass_attn(qd, kd, vd, N, causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.attention(q, k, v, causal)
    assert_close(out, lse, ro, rl, torch.bfloat16, what=str(case))
    o2, l2 = oracle.rsa_two_pass(q, k, v, N, causal)
    assert_close(out, lse, o2, l2, torch.bfloat16, what="oracle two-pass " + str(case))


def test_two_pass_noncausal_workload_all_rows_and_agrees_with_ring():
    need_cuda()
    w = rsa_inputs.WORKLOADS["noncausal_bf16"]
    q, k, v = rsa_inputs.make_workload(w, seed=0, device="cpu")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = rsa.two_pass_attn(qd, kd, vd, w.N, w.causal)
    o_ring, l_ring = rsa.ring_attn(qd, kd, vd, w.N, w.causal)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, w.causal)
    assert_close(out, lse, ro, rl, torch.bfloat16, what=w.name)
    assert (out.float() - o_ring.float()).abs().max().item() <= 2e-2
    assert (lse - l_ring).abs().max().item() <= 1e-3


def test_two_pass_rejects_unsupported_shapes():
    need_cuda()
    q = torch.zeros(1, 1, 384, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rsa.RsaError):
        rsa.two_pass_attn(q, q, q, 2, True)   # chunks of 192 keys
    qf = torch.zeros(1, 1, 256, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(rsa.RsaError):
        rsa.two_pass_attn(qf, qf, qf, 2, True)
