"""GPU parity of the whole ring (rsa_ring_attn_fwd) against the oracle, with
ragged and degenerate shapes, bit-exact invariants from the pages, and the
device-side wait-limit self-test."""
import numpy as np
import pytest
import torch

import oracle
import rsa_inputs
import context_attention_rsa_gb300 as rsa
from gpu_helpers import assert_close, need_cuda, qkv_cuda

pytestmark = pytest.mark.gpu


def test_tiny_fp32_causal_workload_all_rows():
    need_cuda()
    w = rsa_inputs.WORKLOADS["tiny_fp32_causal"]
    q, k, v = rsa_inputs.make_workload(w, seed=0, device="cpu")
    out, lse = rsa.ring_attn(q.cuda(), k.cuda(), v.cuda(), w.N, w.causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.attention(q, k, v, w.causal)
    assert_close(out, lse, ro, rl, torch.float32, what=w.name)


def test_noncausal_bf16_workload_all_rows():
    need_cuda()
    w = rsa_inputs.WORKLOADS["noncausal_bf16"]
    q, k, v = rsa_inputs.make_workload(w, seed=0, device="cpu")
    out, lse = rsa.ring_attn(q.cuda(), k.cuda(), v.cuda(), w.N, w.causal)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.attention(q, k, v, w.causal)
    assert_close(out, lse, ro, rl, torch.bfloat16, what=w.name)


RING_CASES = [
    # B, H, T, d, N, causal, dtype
    (1, 1, 1, 128, 1, True, torch.bfloat16),      # a single token
    (1, 2, 127, 128, 1, True, torch.bfloat16),
    (1, 2, 129, 128, 3, True, torch.bfloat16),    # chunks of 43
    (2, 2, 384, 128, 3, False, torch.bfloat16),
    (1, 3, 1000, 128, 8, True, torch.bfloat16),   # chunks of 125
    (1, 2, 1024, 128, 4, True, torch.bfloat16),
    (1, 1, 2048, 128, 16, True, torch.bfloat16),  # many small chunks
    (1, 1, 96, 128, 96, True, torch.bfloat16),    # chunks of one token
    (2, 2, 768, 64, 3, True, torch.bfloat16),     # d = 64
    (1, 2, 300, 64, 5, False, torch.float32),
    (1, 1, 200, 128, 4, True, torch.float32),
]


@pytest.mark.parametrize("fused", [False, True], ids=["merge_kernel", "fused_merge"])
@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: "B{}H{}T{}d{}N{}_{}_{}".format(
    *c[:5], "causal" if c[5] else "full", "bf16" if c[6] == torch.bfloat16 else "f32"))
def test_ring_matches_oracle(case, fused):
    need_cuda()
    B, H, T, d, N, causal, dtype = case
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, dtype, seed=T + N)
    out, lse = rsa.ring_attn(qd, kd, vd, N, causal, fused=fused)
    torch.cuda.synchronize()
    rsa.check_device_error()
    ro, rl = oracle.attention(q, k, v, causal)
    assert_close(out, lse, ro, rl, dtype, what=str(case))


def test_ring_n1_and_n4_agree_and_row0_is_v0():
    need_cuda()
    B, H, T, d = 1, 4, 4096, 128
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=5)
    o1, l1 = rsa.ring_attn(qd, kd, vd, 1, True)
    o4, l4 = rsa.ring_attn(qd, kd, vd, 4, True)
    torch.cuda.synchronize()
    # row 0 sees only key 0: p = 1 exactly, so out[0] is V[0] to the bit
    assert torch.equal(o1[:, :, 0], vd[:, :, 0])
    assert torch.equal(o4[:, :, 0], vd[:, :, 0])
    diff = (o1.float() - o4.float()).abs().max().item()
    assert diff <= 2e-2
    assert (l1 - l4).abs().max().item() <= 1e-3


def test_chunk0_is_bit_identical_when_later_chunks_change():
    # Causal: chunk 0 only ever meets its own KV chunk.
    need_cuda()
    B, H, T, d, N = 1, 2, 2048, 128, 4
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=6)
    o_a, l_a = rsa.ring_attn(qd, kd, vd, N, True)
    kd2, vd2 = kd.clone(), vd.clone()
    Tc = T // N
    kd2[:, :, Tc:] = torch.randn_like(kd2[:, :, Tc:].float()).to(torch.bfloat16)
    vd2[:, :, Tc:] = torch.randn_like(vd2[:, :, Tc:].float()).to(torch.bfloat16)
    o_b, l_b = rsa.ring_attn(qd, kd2, vd2, N, True)
    torch.cuda.synchronize()
    assert torch.equal(o_a[:, :, :Tc], o_b[:, :, :Tc])
    assert torch.equal(l_a[:, :, :Tc], l_b[:, :, :Tc])
    assert not torch.equal(o_a[:, :, Tc:], o_b[:, :, Tc:])


def test_ring_is_deterministic():
    need_cuda()
    (q, k, v), (qd, kd, vd) = qkv_cuda(2, 2, 1024, 128, torch.bfloat16, seed=7)
    a = rsa.ring_attn(qd, kd, vd, 4, True)
    b = rsa.ring_attn(qd, kd, vd, 4, True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("fused", [True, False], ids=["fused_merge", "merge_kernel"])
def test_ring_outputs_leave_guard_bytes_alone(fused):
    need_cuda()
    B, H, T, d, N = 1, 2, 1000, 128, 8
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=8)
    pad = 8192
    n_o = B * H * T * d
    o_buf = torch.full((pad + n_o + pad,), 3.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((pad + B * H * T + pad,), 3.0, dtype=torch.float32, device="cuda")
    need = rsa.workspace_size(torch.bfloat16, B, H, T, d, N, True, fused=fused)
    ws_buf = torch.full((pad + need + pad,), 0x5a, dtype=torch.uint8, device="cuda")
    out = o_buf[pad:pad + n_o].view(B, H, T, d)
    lse = l_buf[pad:pad + B * H * T].view(B, H, T)
    rsa.ring_attn(qd, kd, vd, N, True, out=out, lse=lse, workspace=ws_buf[pad:pad + need], fused=fused)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 3) and torch.all(o_buf[pad + n_o:] == 3)
    assert torch.all(l_buf[:pad] == 3) and torch.all(l_buf[pad + B * H * T:] == 3)
    assert torch.all(ws_buf[:pad] == 0x5a) and torch.all(ws_buf[pad + need:] == 0x5a)
    ro, rl = oracle.attention(q, k, v, True)
    assert_close(out, lse, ro, rl, torch.bfloat16)


def test_timed_ring_records_every_launch():
    need_cuda()
    B, H, T, d, N = 1, 2, 1024, 128, 4
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=9)
    n = rsa.ring_launch_count(N, True, fused=False)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = torch.empty(rsa.workspace_size(torch.bfloat16, B, H, T, d, N, True, fused=False), dtype=torch.uint8,
                     device="cuda")
    kinds = rsa.ring_attn_timed(qd, kd, vd, N, True, out, lse, ws, ev0, ev1, fused=False)
    torch.cuda.synchronize()
    assert kinds == [0] + [0, 1] * (N - 1)
    assert all(a.elapsed_time(b) >= 0 for a, b in zip(ev0, ev1))
    ro, rl = oracle.attention(q, k, v, True)
    assert_close(out, lse, ro, rl, torch.bfloat16)


def test_wait_limit_selftest_reports_timeout_and_context_survives():
    need_cuda()
    rsa.set_wait_limit_ns(50_000_000)
    try:
        rsa.selftest_wait_timeout()
        with pytest.raises(rsa.RsaError) as ei:
            rsa.check_device_error()
        assert ei.value.status == 4
    finally:
        rsa.set_wait_limit_ns(2_000_000_000)
    rsa.check_device_error()  # cleared
    # the context still works
    (q, k, v), (qd, kd, vd) = qkv_cuda(1, 1, 256, 128, torch.bfloat16, seed=10)
    out, lse = rsa.ring_attn(qd, kd, vd, 2, True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, True)
    assert_close(out, lse, ro, rl, torch.bfloat16)


def test_unsupported_and_invalid_calls_raise():
    need_cuda()
    q = torch.zeros(1, 1, 256, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rsa.RsaError):
        rsa.ring_attn(q, q, q, 4, True)
    q = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rsa.RsaError):
        rsa.ring_attn(q, q, q, 3, True)


def test_fused_and_unfused_rings_agree_and_fused_launches_only_block_kernels():
    need_cuda()
    B, H, T, d, N = 2, 4, 4096, 128, 8
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=12)
    o_a, l_a = rsa.ring_attn(qd, kd, vd, N, True)
    n = rsa.ring_launch_count(N, True, fused=True)
    assert n == N
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = torch.empty(rsa.workspace_size(torch.bfloat16, B, H, T, d, N, True, fused=True), dtype=torch.uint8,
                     device="cuda")
    kinds = rsa.ring_attn_timed(qd, kd, vd, N, True, out, lse, ws, ev0, ev1, fused=True)
    torch.cuda.synchronize()
    assert kinds == [0] * N
    # both orders of folding are the same rounds and the same merge rule
    assert (out.float() - o_a.float()).abs().max().item() <= 2e-2
    assert (lse - l_a).abs().max().item() <= 1e-3
    assert torch.equal(out[:, :, :T // N], o_a[:, :, :T // N])  # chunk 0 is never merged


@pytest.mark.parametrize("mode", ["auto", "engines", "sm"])
@pytest.mark.parametrize("B,H,T,N,dtype", [(2, 5, 1024, 4, torch.bfloat16), (1, 64, 512, 4, torch.bfloat16),
                                             (2, 37, 384, 3, torch.bfloat16), (1, 3, 256, 4, torch.float32),
                                             (1, 6, 130, 2, torch.bfloat16)])
def test_ring_from_host_matches_device_ring(B, H, T, N, dtype, mode):
    # rsa_ring_attn_fwd_host (head slabs streamed through the GPU, copies on
    # the library's streams) gives exactly the device ring's result: every
    # head is its own problem.  64 and 74 heads run ramped plans of slabs of
    # 1 to 7 and 1 to 5 heads; torch-pinned inputs are accepted as well.
    need_cuda()
    # The copy path of each tensor follows the mode: torch-pinned inputs move
    # by the copy kernel in "auto" and "sm", by the copy engines in "engines";
    # rows of 130 x 4 bytes of lse are not 16-byte multiples and fall back to
    # the copy engines.
    d = 64 if dtype == torch.float32 else 128
    q, k, v = (t.pin_memory() for t in qkv_cuda(B, H, T, d, dtype, seed=13)[0])
    ref_o, ref_l = rsa.ring_attn(q.cuda(), k.cuda(), v.cuda(), N, True)
    rsa.set_host_copy_mode(mode)
    try:
        assert rsa.host_copy_path(q) == ("engines" if mode == "engines" else "kernel")
        bufs = {}
        for _ in range(2):  # second call reuses the buffers
            oh, lh, bufs = rsa.ring_attn_from_host(q, k, v, N, True, buffers=bufs)
            torch.cuda.synchronize()
            assert torch.equal(oh, ref_o.cpu()) and torch.equal(lh, ref_l.cpu())
            oh.fill_(float("nan"))
            lh.fill_(float("nan"))
    finally:
        rsa.set_host_copy_mode("auto")


def test_ring_from_host_accepts_pageable_tensors():
    # Pageable host memory moves through the runtime's staged copies (the
    # copy engines); the result is still the device ring's, bit for bit.
    need_cuda()
    B, H, T, d, N = 1, 8, 1024, 128, 4
    (q, k, v), _ = qkv_cuda(B, H, T, d, torch.bfloat16, seed=17)
    assert not q.is_pinned() and rsa.host_copy_path(q) == "engines"
    ref_o, ref_l = rsa.ring_attn(q.cuda(), k.cuda(), v.cuda(), N, True)
    oh, lh, _ = rsa.ring_attn_from_host(q, k, v, N, True)
    torch.cuda.synchronize()
    assert torch.equal(oh, ref_o.cpu()) and torch.equal(lh, ref_l.cpu())


def test_host_empty_is_page_locked_huge_and_streams_bit_exactly():
    need_cuda()
    B, H, T, d, N = 1, 64, 512, 128, 4
    (q, k, v), _ = qkv_cuda(B, H, T, d, torch.bfloat16, seed=21)
    qh, kh, vh = (rsa.host_empty(t.shape, t.dtype) for t in (q, k, v))
    for th, t in ((qh, q), (kh, k), (vh, v)):
        th.copy_(t)
        assert th.is_pinned() and torch.equal(th, t)
        info = rsa.host_info(th)
        assert info["bytes"] >= t.numel() * 2 and info["kind"] in ("registered-huge", "pinned")
        if info["kind"] == "registered-huge":  # rsa_host_alloc kept it only if >= 90% of it is huge
            assert info["huge_bytes"] >= info["bytes"] * 9 // 10
        assert rsa.host_kind(th) == info["kind"]
    ref_o, ref_l = rsa.ring_attn(q.cuda(), k.cuda(), v.cuda(), N, True)
    for th in (qh, kh, vh):  # "auto": copy engines while the block is on huge pages
        info = rsa.host_info(th)
        huge = info["kind"] == "registered-huge" and info["huge_bytes"] >= info["bytes"] * 9 // 10
        assert rsa.host_copy_path(th) == ("engines" if huge else "kernel")
    bufs = {}
    oh, lh, bufs = rsa.ring_attn_from_host(qh, kh, vh, N, True, buffers=bufs)
    torch.cuda.synchronize()
    assert oh.is_pinned() and lh.is_pinned()
    assert torch.equal(oh, ref_o.cpu()) and torch.equal(lh, ref_l.cpu())
    assert rsa.host_kind(q) == "pageable"
    # a block goes back to the system with its last tensor
    addr = qh.untyped_storage().data_ptr()
    del qh
    import gc
    gc.collect()
    assert addr not in rsa._host_blocks


def _huge_page_bytes():
    try:
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            return int(f.read())
    except OSError:
        return 0


def test_ring_from_host_splits_copies_by_huge_page_regions():
    # A block the kernel has split in one place moves by the copy engines
    # where it is still huge and by the copy kernel where it is not, and the
    # call's results stay bit-exact.  The split is made here the way the
    # kernel makes one: changing the protection of one base page inside a
    # huge page (and changing it back) remaps that huge page with base pages.
    need_cuda()
    import ctypes
    import os
    hp = _huge_page_bytes()
    page = os.sysconf("SC_PAGE_SIZE")
    if hp <= 0 or hp > (512 << 20):
        pytest.skip("no transparent huge pages of a usable size")
    T, d, N = 8192, 128, 4
    H = 2 * hp // (T * d * 2)  # each tensor spans two huge pages
    g = torch.Generator(device="cuda").manual_seed(61)
    q, k, v = (torch.randn((1, H, T, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    qh, kh, vh = (rsa.host_empty(t.shape, t.dtype) for t in (q, k, v))
    for th, t in ((qh, q), (kh, k), (vh, v)):
        th.copy_(t)
    info = rsa.host_info(kh)
    if info["kind"] != "registered-huge" or info["huge_bytes"] < 2 * hp:
        pytest.skip("the host block did not get huge pages")
    torch.cuda.synchronize()
    libc = ctypes.CDLL(None, use_errno=True)
    libc.mprotect.argtypes = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int)
    at = kh.data_ptr() + hp + hp // 2  # inside the second huge page
    assert libc.mprotect(at, page, 1) == 0  # PROT_READ
    assert libc.mprotect(at, page, 3) == 0  # PROT_READ | PROT_WRITE
    after = rsa.host_info(kh)
    if after["huge_bytes"] > info["huge_bytes"] - hp:
        pytest.skip("the kernel kept the huge page mapped whole")
    flat = kh.view(-1)
    half = hp // 2 // 2  # bf16 elements in half a huge page
    assert rsa.host_copy_path(flat[:half]) == "engines"  # inside the first, intact huge page
    assert rsa.host_copy_path(flat[2 * half:3 * half]) == "kernel"  # inside the split one
    assert rsa.host_copy_path(kh) == "kernel"  # half of the tensor is on base pages
    ref_o, ref_l = rsa.ring_attn(q, k, v, N, True)
    oh, lh, _ = rsa.ring_attn_from_host(qh, kh, vh, N, True)
    torch.cuda.synchronize()
    assert torch.equal(oh, ref_o.cpu()) and torch.equal(lh, ref_l.cpu())


def test_ring_from_host_waits_for_the_callers_stream():
    # The copies start only after work already enqueued on the caller's
    # stream: inputs written there just before the call are the ones used.
    need_cuda()
    B, H, T, d, N = 1, 16, 1024, 128, 4
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=41)
    qh, kh, vh = (rsa.host_empty(t.shape, t.dtype) for t in (q, k, v))
    for th in (qh, kh, vh):
        th.zero_()
    ref_o, ref_l = rsa.ring_attn(qd, kd, vd, N, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(50_000_000)  # keep the stream busy, then write the inputs on it
        for th, td in ((qh, qd), (kh, kd), (vh, vd)):
            th.copy_(td, non_blocking=True)
        oh, lh, _ = rsa.ring_attn_from_host(qh, kh, vh, N, True, stream=s)
    s.synchronize()
    assert torch.equal(oh, ref_o.cpu()) and torch.equal(lh, ref_l.cpu())


@pytest.mark.parametrize("fused", [False, True], ids=["merge_kernel", "fused_merge"])
def test_ring_captures_into_a_cuda_graph_and_replays(fused):
    # The C ABI only enqueues work on the caller's stream (no synchronisation, no
    # allocation), so a whole ring can be captured once and replayed.
    need_cuda()
    B, H, T, d, N = 1, 4, 2048, 128, 4
    (q, k, v), (qd, kd, vd) = qkv_cuda(B, H, T, d, torch.bfloat16, seed=31)
    ref_o, ref_l = rsa.ring_attn(qd, kd, vd, N, True, fused=fused)
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(rsa.workspace_size(qd.dtype, B, H, T, d, N, True, fused=fused), 1), dtype=torch.uint8,
                     device="cuda")
    rsa.ring_attn(qd, kd, vd, N, True, out=out, lse=lse, workspace=ws, fused=fused)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rsa.ring_attn(qd, kd, vd, N, True, out=out, lse=lse, workspace=ws, fused=fused)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    lse.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    rsa.check_device_error()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
