"""Host-side checks of the C ABI: the library builds and loads, exports every
symbol include/*.h declares, schedules the ring as the pages print it, sizes
its workspace, and rejects bad arguments before touching a GPU.  No GPU."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT, read_golden

import context_attention_rsa_gb300 as rsa

FAKE = 0x10000  # a 16-byte-aligned non-null pointer value; never dereferenced


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(rsa_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_library_loads_and_exports_every_declared_symbol():
    lib = rsa.load()
    names = declared_symbols()
    assert "rsa_ring_attn_fwd" in names and "rsa_block_attn_fwd" in names and "rsa_merge" in names
    for n in names:
        assert hasattr(lib, n), n
    assert rsa.version() == 10000
    assert lib.rsa_status_string(4) == b"RSA_ERR_TIMEOUT"


def test_schedule_matches_printed_ring_table():
    want = {}
    for rnd1, gpu, kv in (map(int, r) for r in read_golden("ring_table_n4.txt")):
        want.setdefault(rnd1 - 1, []).append((gpu, kv))
    for r, pairs in want.items():
        assert rsa.ring_schedule(4, False, r) == sorted(pairs)


def test_schedule_causal_needs_and_counts():
    for row in read_golden("causal_chunk_needs_n4.txt"):
        i = int(row[0])
        need = sorted(int(x) for x in row[1].split(","))
        got = sorted(j for r in range(4) for (ii, j) in rsa.ring_schedule(4, True, r) if ii == i)
        assert got == need
    for N in (1, 2, 3, 4, 7, 16, 64):
        pc = [p for r in range(N) for p in rsa.ring_schedule(N, True, r)]
        pn = [p for r in range(N) for p in rsa.ring_schedule(N, False, r)]
        assert len(pc) == N * (N + 1) // 2 and len(set(pc)) == len(pc)
        assert len(pn) == N * N and len(set(pn)) == len(pn)
        assert rsa.ring_schedule(N, True, 0) == [(i, i) for i in range(N)]


def test_launch_count():
    # default (merge folded into the block epilogue): one block launch per round
    assert rsa.ring_launch_count(1, True) == 1
    assert rsa.ring_launch_count(4, True) == 4
    assert rsa.ring_launch_count(16, True) == 16
    # separate merge kernel: a block and a merge launch per round after the first
    assert rsa.ring_launch_count(4, True, fused=False) == 1 + 2 * 3
    assert rsa.ring_launch_count(16, True, fused=False) == 1 + 2 * 15
    assert rsa.ring_launch_count(4, False, fused=False) == 1 + 2 * 3


def test_workspace_size():
    import torch
    B, H, T, d, N = 8, 64, 32768, 128, 4
    ws = rsa.workspace_size(torch.bfloat16, B, H, T, d, N, True, fused=False)
    acc = B * H * T * d * 4
    Tc = T // N
    blk = (N - 1) * B * H * Tc * d * 4 + (N - 1) * B * H * Tc * 4  # fp32 partials
    assert ws == acc + blk
    assert rsa.workspace_size(torch.bfloat16, 1, 1, 256, 128, 1, True) == 0
    assert rsa.workspace_size(torch.bfloat16, B, H, T, d, N, True) == acc  # the default: the accumulator alone
    lib = rsa.load()
    n = ctypes.c_size_t(0)
    assert lib.rsa_ring_attn_workspace_size(1, B, H, T, d, N, 1, ctypes.byref(n)) == 0 and n.value == acc
    assert lib.rsa_ring_attn_workspace_size_ex(1, B, H, T, d, N, 1, 3, ctypes.byref(n)) == 1  # both flags
    assert lib.rsa_ring_attn_workspace_size_ex(1, B, H, T, d, N, 1, 4, ctypes.byref(n)) == 1  # unknown flag
    # non-causal rounds have N pairs
    ws2 = rsa.workspace_size(torch.float32, 1, 1, 256, 64, 4, False, fused=False)
    assert ws2 == 256 * 64 * 4 + 4 * 64 * 64 * 4 + 4 * 64 * 4


@pytest.mark.parametrize("kwargs,code", [
    (dict(N=3), 1),           # N does not divide T
    (dict(N=0), 1),
    (dict(d=96), 2),          # unsupported head dim
    (dict(T=0), 1),
    (dict(dt=7), 1),
])
def test_ring_rejects_bad_shapes(kwargs, code):
    lib = rsa.load()
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=1, B=1, H=1, T=256, d=128, N=4, causal=1, out=FAKE, lse=FAKE,
             ws=FAKE, ws_bytes=1 << 40, stream=None)
    a.update(kwargs)
    st = lib.rsa_ring_attn_fwd(a["q"], a["k"], a["v"], a["dt"], a["B"], a["H"], a["T"], a["d"], a["N"],
                               a["causal"], a["out"], a["lse"], a["ws"], a["ws_bytes"], a["stream"])
    assert st == code, lib.rsa_last_error_string()


def test_ring_rejects_null_misaligned_and_small_workspace():
    lib = rsa.load()
    args = [FAKE, FAKE, FAKE, 1, 1, 1, 256, 128, 4, 1, FAKE, FAKE, FAKE, 1 << 40, None]
    for idx in (0, 1, 2, 10, 11, 12):
        bad = list(args)
        bad[idx] = None
        assert lib.rsa_ring_attn_fwd(*bad) == 1
        bad[idx] = FAKE + 4
        assert lib.rsa_ring_attn_fwd(*bad) == 1
    small = list(args)
    small[13] = 100
    assert lib.rsa_ring_attn_fwd(*small) == 1
    assert b"workspace" in lib.rsa_last_error_string()


def test_block_rejects_pairs_outside_the_sequence():
    lib = rsa.load()
    base = [FAKE, FAKE, FAKE, 1, 1, 1, 256, 128]
    for q_off, q_len, kv_off, kv_len in [(200, 100, 0, 10), (-1, 10, 0, 10), (0, 0, 0, 10),
                                         (0, 10, 250, 7), (0, 10, 0, 0)]:
        st = lib.rsa_block_attn_fwd(*base, q_off, q_len, kv_off, kv_len, 1, FAKE, FAKE, None)
        assert st == 1


def test_merge_rejects_bad_arguments():
    lib = rsa.load()
    assert lib.rsa_merge(FAKE, FAKE, FAKE, 1, FAKE, 0, 128, None) == 1
    assert lib.rsa_merge(FAKE, FAKE, FAKE, 1, FAKE, 10, 96, None) == 2
    assert lib.rsa_merge(None, FAKE, FAKE, 1, FAKE, 10, 128, None) == 1
    assert lib.rsa_merge_finalize(FAKE, FAKE, FAKE, 1, FAKE, 10, 128, None, 1, FAKE, None) == 1


def test_wait_limit_bounds():
    lib = rsa.load()
    assert lib.rsa_set_wait_limit_ns(10) == 1
    assert lib.rsa_set_wait_limit_ns(2_000_000_000) == 0


def test_decode_workspace_and_validation():
    import torch
    # 4 x 8 heads, million-token cache in 16 shards: 32 x 16 = 512 (head, shard)
    # units, so each shard is cut into 4 splits of 16384 keys (about 2048 CTAs)
    B, H, T, d, N, ql = 4, 8, 1 << 20, 128, 16, 1
    ws = rsa.decode_workspace_size(torch.bfloat16, B, H, T, d, ql, N)
    S = N * 4
    assert ws == (S * B * H * ql * d * 4 + 255) // 256 * 256 + (S * B * H * ql * 4 + 255) // 256 * 256
    lib = rsa.load()
    args = [FAKE, FAKE, FAKE, 1, 1, 1, 256, 128, 1, 4, 1, FAKE, FAKE, FAKE, 1 << 40, None]
    bad = list(args); bad[8] = 0          # q_len 0
    assert lib.rsa_decode_attn_fwd(*bad) == 1
    bad = list(args); bad[8] = 300        # q_len > T
    assert lib.rsa_decode_attn_fwd(*bad) == 1
    bad = list(args); bad[9] = 3          # N does not divide T
    assert lib.rsa_decode_attn_fwd(*bad) == 1
    bad = list(args); bad[14] = 16        # workspace too small
    assert lib.rsa_decode_attn_fwd(*bad) == 1


def test_two_pass_workspace_is_quadratic():
    import torch
    B, H, T, d, N = 2, 8, 4096, 128, 4
    ws = rsa.two_pass_workspace_size(torch.bfloat16, B, H, T, d, N)
    rows = B * H * (T // N)
    # fp32 scores and bf16 probabilities of one chunk, and (max, sum) per row and 64 keys
    assert ws == rows * T * (4 + 2) + rows * (T // 64) * 8
    lib = rsa.load()
    n = ctypes.c_size_t(0)
    assert lib.rsa_two_pass_workspace_size(1, 1, 1, 384, 128, 2, ctypes.byref(n)) == 2  # 192-key chunks
    assert lib.rsa_two_pass_workspace_size(0, 1, 1, 256, 128, 2, ctypes.byref(n)) == 2  # fp32


def test_set_block_kernel_accepts_the_three_choices_only():
    lib = rsa.load()
    assert lib.rsa_set_block_kernel(3) == 1
    assert lib.rsa_set_block_kernel(-1) == 1
    for which in (1, 2, 0):
        assert lib.rsa_set_block_kernel(which) == 0


@pytest.mark.parametrize("BH,groups", [(512, 8), (512, 16), (64, 8), (100, 8), (37, 8), (7, 3), (1, 8), (512, 1)])
def test_slab_plan_covers_every_head_and_ramps_gently(BH, groups):
    plan = rsa.slab_plan(BH, groups)
    assert sum(plan) == BH and all(n >= 1 for n in plan)
    cap = -(-BH // min(groups, BH))
    assert max(plan) <= cap
    # each slab's copy-in must hide under its predecessor's ring: slabs grow by
    # at most 1.6x (+1 for rounding) from one to the next
    for a, b in zip(plan, plan[1:]):
        assert b <= max(a + 1, (a * 8) // 5 + 1), plan
    assert rsa.slab_plan(BH, groups, ramp=False) == [cap] * (BH // cap) + ([BH % cap] if BH % cap else [])


def test_host_streaming_workspace_and_validation():
    lib = rsa.load()
    n = ctypes.c_size_t(0)
    # page-1 shape: 512 heads, largest slab 57 heads (ramped plan of 8 groups)
    assert lib.rsa_ring_attn_host_workspace_size(1, 8, 64, 32768, 128, 4, 1, ctypes.byref(n)) == 0
    hg = max(rsa.slab_plan(512, 8))
    slab = hg * 32768 * 128 * 2
    ring = rsa.workspace_size(__import__("torch").bfloat16, 1, hg, 32768, 128, 4, True)
    assert n.value == 2 * (4 * slab + hg * 32768 * 4) + (ring + 255) // 256 * 256
    assert lib.rsa_ring_attn_host_workspace_size(1, 1, 1, 100, 128, 3, 1, ctypes.byref(n)) == 1  # N does not divide T
    args = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, ws=0x100000, nb=1 << 40)

    def call(**kw):
        a = dict(args, **kw)
        return lib.rsa_ring_attn_fwd_host(a["q"], a["k"], a["v"], 1, 1, 4, 1024, 128, 4, 1, a["out"], a["lse"],
                                          a["ws"], a["nb"], None)
    assert call(q=None) == 1 and b"NULL" in lib.rsa_last_error_string()
    assert call(lse=None) == 1
    assert call(ws=0x100010) == 1 and b"256-byte" in lib.rsa_last_error_string()
    assert call(nb=1024) == 1 and b"needed" in lib.rsa_last_error_string()


def test_host_alloc_rejects_bad_arguments():
    lib = rsa.load()
    p = ctypes.c_void_p(0)
    assert lib.rsa_host_alloc(0, ctypes.byref(p)) == 1 and not p.value
    assert lib.rsa_host_alloc(16, None) == 1
    assert lib.rsa_host_free(FAKE) == 1 and b"rsa_host_alloc" in lib.rsa_last_error_string()
    assert lib.rsa_host_info(FAKE, None, None, None) == 1
    slabs = (ctypes.c_int * 4)()
    cnt = ctypes.c_int(0)
    assert lib.rsa_host_slab_plan(512, 8, 1, slabs, 4, ctypes.byref(cnt)) == 1 and cnt.value == 14
    assert lib.rsa_host_slab_plan(0, 8, 1, slabs, 4, ctypes.byref(cnt)) == 1


def test_host_copy_mode_setter():
    lib = rsa.load()
    assert lib.rsa_set_host_copy_mode(3) == 1 and lib.rsa_set_host_copy_mode(-1) == 1
    for mode in (1, 2, 0):
        assert lib.rsa_set_host_copy_mode(mode) == 0
    path = ctypes.c_int(0)
    assert lib.rsa_host_copy_path(None, 16, ctypes.byref(path)) == 1
