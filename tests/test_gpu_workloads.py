"""GPU parity on the three large workloads at full size, in the launch
configuration the benchmark times, checked on 4096 sampled query rows each
(forced rows at tile, chunk and ragged boundaries and after outlier keys, plus
uniform rows) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import rsa_inputs
import context_attention_rsa_gb300 as rsa
from gpu_helpers import assert_close, need_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True], ids=["merge_kernel", "fused_merge"])
@pytest.mark.parametrize("name", ["page1_causal_bf16", "ragged_causal_bf16", "million_causal_bf16"])
def test_full_size_workload_sampled_rows(name, fused):
    need_cuda()
    w = rsa_inputs.WORKLOADS[name]
    q, k, v = rsa_inputs.make_workload(w, seed=0, device="cuda")
    out, lse = rsa.ring_attn(q, k, v, w.N, w.causal, fused=fused)
    torch.cuda.synchronize()
    rsa.check_device_error()
    rows = rsa_inputs.sample_rows(w, n=4096, seed=1)
    ri = torch.from_numpy(rows).cuda()
    q_rows = q[ri[:, 0], ri[:, 1], ri[:, 2]].cpu()
    g_out = out[ri[:, 0], ri[:, 1], ri[:, 2]].cpu()
    g_lse = lse[ri[:, 0], ri[:, 1], ri[:, 2]].cpu()
    del out, lse, q
    k_h, v_h = k.cpu(), v.cpu()
    del k, v
    torch.cuda.empty_cache()
    ro, rl = oracle.attend_rows(q_rows, k_h, v_h, rows, w.causal)
    stats = assert_close(g_out, g_lse, ro, rl, torch.bfloat16, what=name)
    print(name, 'fused' if fused else 'merge_kernel', stats)


def test_decode_workload_full_size():
    # One new token per sequence against a million-token KV cache in 16 shards,
    # in the launch configuration the benchmark times; every query row checked.
    need_cuda()
    w = rsa_inputs.WORKLOADS["decode_million_bf16"]
    q, k, v = rsa_inputs.make_workload(w, seed=0, device="cuda")
    qd = q[:, :, w.T - w.q_len:].contiguous()
    del q
    out, lse = rsa.decode_attn(qd, k, v, w.N, w.causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    rows = np.array([[b, h, w.T - w.q_len + r] for b in range(w.B) for h in range(w.H) for r in range(w.q_len)],
                    dtype=np.int64)
    ro, rl = oracle.attend_rows(qd.reshape(-1, w.d).cpu(), k.cpu(), v.cpu(), rows, w.causal)
    stats = assert_close(out.reshape(-1, w.d), lse.reshape(-1), ro, rl, torch.bfloat16, what=w.name)
    print(w.name, stats)
