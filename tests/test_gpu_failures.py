"""Failure reporting of the C ABI, with the failures made on the host.

rsa_debug_inject_launch_failure makes a chosen launch report a launch
failure instead of launching (no GPU fault is involved): the call must return
RSA_ERR_CUDA with the reason in rsa_last_error_string(), leave every output
it did not reach untouched, switch the injection off, and leave the library
and the CUDA context usable."""
import pytest
import torch

import context_attention_rsa_gb300 as rsa
import oracle
from gpu_helpers import assert_close, need_cuda, qkv_cuda

pytestmark = pytest.mark.gpu

GUARD = 12345.0


def test_injected_first_launch_fails_the_ring_and_touches_nothing():
    need_cuda()
    B, H, T, d, N = 1, 2, 1024, 128, 4
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=71)
    out = torch.full_like(qd, GUARD)
    lse = torch.full((B, H, T), GUARD, device="cuda")
    rsa.inject_launch_failure(0)
    with pytest.raises(rsa.RsaError) as e:
        rsa.ring_attn(qd, kd, vd, N, True, out=out, lse=lse)
    assert e.value.status == 3 and "injected launch failure" in str(e.value)
    torch.cuda.synchronize()
    rsa.check_device_error()
    assert torch.all(out == GUARD) and torch.all(lse == GUARD)
    # the injection switched itself off: the same call now succeeds
    rsa.ring_attn(qd, kd, vd, N, True, out=out, lse=lse)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, True)
    assert_close(out, lse, ro, rl, torch.bfloat16, what="after injection")


def test_injected_later_launch_keeps_earlier_work_only():
    # Launch 0 (round 0: the diagonal pairs) runs, launch 1 (round 1's
    # block launch) fails: chunk 0, visited once, is final; chunks 1-3 of
    # out are untouched.
    need_cuda()
    B, H, T, d, N = 1, 2, 1024, 128, 4
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=72)
    out = torch.full_like(qd, GUARD)
    lse = torch.full((B, H, T), GUARD, device="cuda")
    rsa.inject_launch_failure(1)
    with pytest.raises(rsa.RsaError) as e:
        rsa.ring_attn(qd, kd, vd, N, True, out=out, lse=lse)
    assert e.value.status == 3 and "block attention launch" in str(e.value)
    torch.cuda.synchronize()
    Tc = T // N
    ro, rl = oracle.attention(q, k, v, True)
    assert_close(out[:, :, :Tc], lse[:, :, :Tc], ro[:, :, :Tc], rl[:, :, :Tc], torch.bfloat16, what="chunk 0")
    assert torch.all(out[:, :, Tc:] == GUARD)


def test_injected_failure_through_the_c_abi_and_merge():
    need_cuda()
    lib = rsa.load()
    rows, d = 300, 128
    o_acc = torch.randn(rows, d, device="cuda")
    lse_acc = torch.randn(rows, device="cuda")
    o_blk = torch.randn(rows, d, device="cuda").to(torch.bfloat16)
    lse_blk = torch.randn(rows, device="cuda")
    before = (o_acc.clone(), lse_acc.clone())
    assert lib.rsa_debug_inject_launch_failure(0) == 0
    st = lib.rsa_merge(o_acc.data_ptr(), lse_acc.data_ptr(), o_blk.data_ptr(), 1, lse_blk.data_ptr(), rows, d,
                       int(torch.cuda.current_stream().cuda_stream))
    assert st == 3
    assert b"injected launch failure" in lib.rsa_last_error_string()
    assert lib.rsa_status_string(st) == b"RSA_ERR_CUDA"
    torch.cuda.synchronize()
    assert torch.equal(o_acc, before[0]) and torch.equal(lse_acc, before[1])
    # switched off by a negative countdown before it fires
    lib.rsa_debug_inject_launch_failure(5)
    lib.rsa_debug_inject_launch_failure(-1)
    rsa.merge(o_acc, lse_acc, o_blk, lse_blk)
    torch.cuda.synchronize()
    assert not torch.equal(o_acc, before[0])
