"""The allocation-free ring entry point, rsa_ring_attn_fwd_noalloc.

It serves callers that cannot allocate device memory when they call (their
memory belongs to another allocator, or a cudaMalloc is not allowed where
they run): the library's built-in 64 MiB scratch array replaces the
workspace.  Its results must match the oracle and rsa_ring_attn_fwd on the
same inputs, on two calls in a row (the shared scratch keeps the first call's
contents); the second call must leave the device's free memory unchanged; and
shapes needing more scratch than it has must be rejected.  This file is
collected last on purpose."""
import pytest
import torch

import context_attention_rsa_gb300 as rsa
import oracle
from gpu_helpers import BF16_ATOL, BF16_RFRO, LSE_ATOL, F32_ATOL, assert_close, need_cuda, qkv_cuda

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, q, k, v, N, causal, out, lse):
    B, H, T, d = q.shape
    dt = 1 if q.dtype == torch.bfloat16 else 0
    return lib.rsa_ring_attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), dt, B, H, T, d, N,
                                        int(causal), out.data_ptr(), lse.data_ptr(),
                                        int(torch.cuda.current_stream().cuda_stream))


def _within(a_out, a_lse, b_out, b_lse, dtype):
    da = (a_out.float() - b_out.float()).abs()
    fin = torch.isfinite(b_lse)
    assert torch.equal(torch.isfinite(a_lse), fin)
    dl = (a_lse[fin] - b_lse[fin]).abs().max().item() if fin.any() else 0.0
    if dtype == torch.float32:
        assert da.max().item() <= F32_ATOL and dl <= F32_ATOL
    else:
        rfro = (da.norm() / b_out.float().norm().clamp_min(1e-30)).item()
        assert da.max().item() <= BF16_ATOL and rfro <= BF16_RFRO and dl <= LSE_ATOL


@pytest.mark.parametrize("shape", [(1, 4, 4096, 128, 4, True, torch.bfloat16),
                                   (2, 2, 1000, 64, 8, False, torch.bfloat16),
                                   (1, 1, 256, 64, 4, True, torch.float32)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(shape):
    need_cuda()
    B, H, T, d, N, causal, dtype = shape
    lib = rsa.load()
    for call in range(2):  # the second call reuses the scratch left by the first
        (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, dtype, seed=123 + call)
        ref_out, ref_lse = rsa.ring_attn(qd, kd, vd, N, causal)
        out = torch.full_like(qd, float("nan"))
        lse = torch.full((B, H, T), float("nan"), device="cuda")
        torch.cuda.synchronize()
        free_before, _ = torch.cuda.mem_get_info()
        st = _noalloc_call(lib, qd, kd, vd, N, causal, out, lse)
        assert st == 0, lib.rsa_last_error_string()
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
        rsa.check_device_error()
        if call == 1:  # every kernel is loaded by now: nothing may be allocated
            assert free_after == free_before, (free_before, free_after)
        _within(out, lse, ref_out, ref_lse, dtype)
        oo, ol = oracle.attention(q, k, v, causal)
        assert_close(out, lse, oo, ol, dtype, what=f"noalloc call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    need_cuda()
    lib = rsa.load()
    B, H, T, d, N = 8, 8, 4096, 128, 4   # a 128 MiB accumulator: too big
    assert rsa.workspace_size(torch.bfloat16, B, H, T, d, N, False) > 64 << 20
    q = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    st = _noalloc_call(lib, q, q, q, N, False, out, lse)
    assert st == 1
    assert b"scratch" in lib.rsa_last_error_string()
