"""GPU parity of decode against a sharded KV cache (rsa_decode_attn_fwd): the
newest q_len tokens attend to the whole cache, cut into N shards and split
further, with the split partials folded by the online-softmax rule."""
import numpy as np
import pytest
import torch

import oracle
import rsa_inputs
import context_attention_rsa_gb300 as rsa
from gpu_helpers import assert_close, need_cuda

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, T, d, q_len, N, causal, dtype
    (1, 2, 4096, 128, 1, 4, True, torch.bfloat16),
    (2, 3, 5000, 128, 7, 5, True, torch.bfloat16),      # ragged shards and splits
    (1, 2, 65536, 128, 16, 4, True, torch.bfloat16),    # several splits per shard
    (1, 1, 3000, 128, 300, 3, True, torch.bfloat16),    # two 256-row groups, causal inside the new rows
    (1, 2, 2048, 64, 4, 2, False, torch.bfloat16),
    (1, 2, 1000, 64, 3, 4, True, torch.float32),
    (2, 1, 4096, 128, 1, 1, False, torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}T{}d{}q{}N{}_{}_{}".format(
    *c[:6], "causal" if c[6] else "full", "bf16" if c[7] == torch.bfloat16 else "f32"))
def test_decode_matches_oracle(case):
    need_cuda()
    B, H, T, d, ql, N, causal, dtype = case
    q_full, k, v = rsa_inputs.make_qkv(B, H, T, d, dtype, "normal", seed=T + ql, device="cpu")
    q = q_full[:, :, T - ql:].contiguous()   # the newest tokens
    out, lse = rsa.decode_attn(q.cuda(), k.cuda(), v.cuda(), N, causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    rows = np.array([[b, h, T - ql + r] for b in range(B) for h in range(H) for r in range(ql)], dtype=np.int64)
    ro, rl = oracle.attend_rows(q.reshape(-1, d), k, v, rows, causal)
    assert_close(out.reshape(-1, d), lse.reshape(-1), ro, rl, dtype, what=str(case))


def test_decode_equals_last_rows_of_the_ring():
    # The newest rows of a full causal ring and a decode step see the same keys.
    need_cuda()
    B, H, T, d = 1, 4, 8192, 128
    q, k, v = (t.cuda() for t in rsa_inputs.make_qkv(B, H, T, d, torch.bfloat16, "normal", seed=3))
    o_ring, l_ring = rsa.ring_attn(q, k, v, 4, True)
    o_dec, l_dec = rsa.decode_attn(q[:, :, T - 5:].contiguous(), k, v, 8, True)
    torch.cuda.synchronize()
    assert (o_dec.float() - o_ring[:, :, T - 5:].float()).abs().max().item() <= 2e-2
    assert (l_dec - l_ring[:, :, T - 5:]).abs().max().item() <= 1e-3


def test_decode_million_token_cache_sampled():
    # A million-token cache in 16 shards with outlier keys; one new token per head.
    need_cuda()
    w = rsa_inputs.WORKLOADS["million_causal_bf16"]
    q, k, v = rsa_inputs.make_workload(w, seed=0, device="cuda")
    qd = q[:, :, w.T - 1:].contiguous()
    out, lse = rsa.decode_attn(qd, k, v, w.N, True)
    torch.cuda.synchronize()
    rows = np.array([[0, h, w.T - 1] for h in range(w.H)], dtype=np.int64)
    ro, rl = oracle.attend_rows(qd.reshape(-1, w.d).cpu(), k.cpu(), v.cpu(), rows, True)
    assert_close(out.reshape(-1, w.d), lse.reshape(-1), ro, rl, torch.bfloat16, what="million decode")
