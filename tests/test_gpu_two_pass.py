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


def test_two_pass_and_decode_capture_into_cuda_graphs_and_replay_bit_exactly():
    # Both calls only enqueue kernels on the caller's stream, so a caller can
    # capture one call and replay it (the benchmark times the two-pass form
    # that way too); the replays must give the plain call's results exactly.
    need_cuda()
    B, H, T, d, N = 1, 2, 1024, 128, 4
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=77)
    ref_o, ref_l = rsa.two_pass_attn(qd, kd, vd, N, True)
    qn = qd[:, :, T - 3:].contiguous()
    ref_do, ref_dl = rsa.decode_attn(qn, kd, vd, N, True)
    out, lse = torch.empty_like(qd), torch.empty((B, H, T), device="cuda")
    ws = torch.empty(rsa.two_pass_workspace_size(qd.dtype, B, H, T, d, N), dtype=torch.uint8, device="cuda")
    dout, dlse = torch.empty_like(qn), torch.empty((B, H, 3), device="cuda")
    dws = torch.empty(max(rsa.decode_workspace_size(qd.dtype, B, H, T, d, 3, N), 1), dtype=torch.uint8,
                      device="cuda")
    rsa.two_pass_attn(qd, kd, vd, N, True, out=out, lse=lse, workspace=ws)  # warm-up outside capture
    rsa.decode_attn(qn, kd, vd, N, True, out=dout, lse=dlse, workspace=dws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rsa.two_pass_attn(qd, kd, vd, N, True, out=out, lse=lse, workspace=ws)
            rsa.decode_attn(qn, kd, vd, N, True, out=dout, lse=dlse, workspace=dws)
    torch.cuda.current_stream().wait_stream(s)
    for t in (out, lse, dout, dlse):
        t.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    rsa.check_device_error()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert torch.equal(dout, ref_do) and torch.equal(dlse, ref_dl)
