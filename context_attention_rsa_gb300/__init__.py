"""Blockwise ring self-attention (forward) on one NVIDIA GB300.

A thin ctypes binding over ``librsa.so`` (the C ABI in ``include/rsa.h``).  It
only marshals arguments: torch tensors supply device memory and the current
stream; every step of the attention path runs in the library's CUDA kernels.
There is no CPU fallback -- if the library cannot be built or loaded, every
call raises.

Pages: "Sequence parallelism -- splitting the token dimension across GPUs"
(llmdaily, day 58): chunking ("Split tokens across four GPUs"), the ring
("A better mental model: move blocks past the queries"), online softmax ("But
softmax seems to require all attention scores at once") and causal skipping
("Causal attention gives us another optimization").
"""
from __future__ import annotations

import atexit
import ctypes
import mmap
import threading
from typing import List, Optional, Sequence, Tuple

import torch

from . import _build

__all__ = [
    "RsaError", "load", "library_path", "block_attn_fwd", "merge", "merge_finalize",
    "ring_attn", "ring_attn_noalloc", "ring_attn_timed", "decode_attn", "decode_workspace_size",
    "two_pass_attn", "two_pass_workspace_size", "ring_attn_from_host", "slab_plan", "host_empty", "host_kind", "host_free",
    "workspace_size", "ring_schedule", "set_block_kernel",
    "set_wait_limit_ns", "check_device_error", "selftest_wait_timeout", "version",
    "RSA_F32", "RSA_BF16",
]

RSA_F32 = 0
RSA_BF16 = 1
_STATUS = {0: "RSA_OK", 1: "RSA_ERR_INVALID_ARG", 2: "RSA_ERR_UNSUPPORTED", 3: "RSA_ERR_CUDA",
           4: "RSA_ERR_TIMEOUT"}


class RsaError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn}: {_STATUS.get(status, status)}: {detail}")
        self.status = status
        self.fn = fn


_lib = None
_lock = threading.Lock()

_c_void_p = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64

_SIGS = {
    "rsa_block_attn_fwd": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32,
                           _i64, _i64, _i64, _i64, _i32, _c_void_p, _c_void_p, _c_void_p],
    "rsa_merge": [_c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _i64, _i32, _c_void_p],
    "rsa_merge_finalize": [_c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _i64, _i32,
                           _c_void_p, _i32, _c_void_p, _c_void_p],
    "rsa_ring_attn_workspace_size": [_i32, _i32, _i32, _i64, _i32, _i32, _i32,
                                     ctypes.POINTER(ctypes.c_size_t)],
    "rsa_ring_attn_fwd": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                          _c_void_p, _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p],
    "rsa_ring_attn_fwd_noalloc": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32, _i32,
                                  _i32, _c_void_p, _c_void_p, _c_void_p],
    "rsa_ring_attn_fwd_timed": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32, _i32,
                                _i32, _c_void_p, _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p,
                                ctypes.POINTER(_c_void_p), ctypes.POINTER(_c_void_p),
                                ctypes.POINTER(_i32), _i32, ctypes.POINTER(_i32)],
    "rsa_ring_attn_workspace_size_ex": [_i32, _i32, _i32, _i64, _i32, _i32, _i32, ctypes.c_uint,
                                        ctypes.POINTER(ctypes.c_size_t)],
    "rsa_ring_attn_fwd_ex": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                             ctypes.c_uint, _c_void_p, _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p,
                             ctypes.POINTER(_c_void_p), ctypes.POINTER(_c_void_p), ctypes.POINTER(_i32),
                             _i32, ctypes.POINTER(_i32)],
    "rsa_two_pass_workspace_size": [_i32, _i32, _i32, _i64, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)],
    "rsa_two_pass_attn_fwd": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                              _c_void_p, _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p],
    "rsa_decode_workspace_size": [_i32, _i32, _i32, _i64, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_size_t)],
    "rsa_decode_attn_fwd": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32, _i32, _i32, _i32,
                            _c_void_p, _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p],
    "rsa_ring_schedule": [_i32, _i32, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32), _i32,
                          ctypes.POINTER(_i32)],
    "rsa_set_wait_limit_ns": [ctypes.c_uint64],
    "rsa_set_block_kernel": [_i32],
    "rsa_check_device_error": [_c_void_p],
    "rsa_selftest_wait_timeout": [_c_void_p],
    "rsa_status_string": [_i32],
    "rsa_last_error_string": [],
    "rsa_version": [],
}


def library_path(build: bool = True) -> str:
    return _build.build() if build else _build.LIB


def load(build: bool = True):
    """Load librsa.so (building it in-tree first if it is stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path(build)
            lib = ctypes.CDLL(path)
            for name, args in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_char_p if name in ("rsa_status_string", "rsa_last_error_string") \
                    else ctypes.c_int
            _lib = lib
    return _lib


def _call(name: str, *args) -> None:
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        detail = lib.rsa_last_error_string()
        raise RsaError(name, st, detail.decode() if detail else "")


def version() -> int:
    return int(load().rsa_version())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return RSA_F32
    if t.dtype == torch.bfloat16:
        return RSA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _check_qkv(q, k, v) -> Tuple[int, int, int, int]:
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, T, d] tensor")
    if not (q.shape == k.shape == v.shape) or not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share shape and dtype")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must live on one device")
    B, H, T, d = q.shape
    return B, H, T, d


RSA_RING_FUSED_MERGE = 1


def workspace_size(dtype: torch.dtype, B: int, H: int, T: int, d: int, N: int, causal: bool,
                   fused: bool = False) -> int:
    n = ctypes.c_size_t(0)
    dt = RSA_F32 if dtype == torch.float32 else RSA_BF16
    if fused:
        _call("rsa_ring_attn_workspace_size_ex", dt, B, H, T, d, N, int(bool(causal)), RSA_RING_FUSED_MERGE,
              ctypes.byref(n))
    else:
        _call("rsa_ring_attn_workspace_size", dt, B, H, T, d, N, int(bool(causal)), ctypes.byref(n))
    return int(n.value)


def block_attn_fwd(q, k, v, q_off: int, q_len: int, kv_off: int, kv_len: int, causal: bool,
                   o_blk: Optional[torch.Tensor] = None, lse_blk: Optional[torch.Tensor] = None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One (query chunk, KV chunk) pair: (o_blk [B, H, q_len, d], lse_blk [B, H, q_len])."""
    B, H, T, d = _check_qkv(q, k, v)
    if o_blk is None:
        o_blk = torch.empty((B, H, q_len, d), dtype=q.dtype, device=q.device)
    if lse_blk is None:
        lse_blk = torch.empty((B, H, q_len), dtype=torch.float32, device=q.device)
    _call("rsa_block_attn_fwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d,
          q_off, q_len, kv_off, kv_len, int(bool(causal)), o_blk.data_ptr(), lse_blk.data_ptr(),
          _stream(stream))
    return o_blk, lse_blk


def merge(o_acc: torch.Tensor, lse_acc: torch.Tensor, o_blk: torch.Tensor, lse_blk: torch.Tensor,
          stream=None) -> None:
    """In place: (o_acc, lse_acc) <- merge((o_acc, lse_acc), (o_blk, lse_blk))."""
    d = o_acc.shape[-1]
    rows = lse_acc.numel()
    if o_acc.dtype != torch.float32 or lse_acc.dtype != torch.float32 or lse_blk.dtype != torch.float32:
        raise TypeError("o_acc, lse_acc and lse_blk must be float32")
    if o_blk.numel() != rows * d or o_acc.numel() != rows * d or lse_blk.numel() != rows:
        raise ValueError("row counts differ")
    for t in (o_acc, lse_acc, o_blk, lse_blk):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("merge operands must be contiguous CUDA tensors")
    _call("rsa_merge", o_acc.data_ptr(), lse_acc.data_ptr(), o_blk.data_ptr(), _dt(o_blk),
          lse_blk.data_ptr(), rows, d, _stream(stream))


def merge_finalize(o_acc, lse_acc, o_blk, lse_blk, out_dtype=torch.bfloat16, out=None, lse_out=None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    d = o_acc.shape[-1]
    rows = lse_acc.numel()
    if o_blk.numel() != rows * d or o_acc.numel() != rows * d or lse_blk.numel() != rows:
        raise ValueError("row counts differ")
    if out is None:
        out = torch.empty(o_acc.shape, dtype=out_dtype, device=o_acc.device)
    if lse_out is None:
        lse_out = torch.empty(lse_acc.shape, dtype=torch.float32, device=o_acc.device)
    _call("rsa_merge_finalize", o_acc.data_ptr(), lse_acc.data_ptr(), o_blk.data_ptr(), _dt(o_blk),
          lse_blk.data_ptr(), rows, d, out.data_ptr(), _dt(out), lse_out.data_ptr(), _stream(stream))
    return out, lse_out


def ring_attn(q, k, v, N: int, causal: bool, out=None, lse=None, workspace=None,
              stream=None, fused: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """The whole ring: (out [B, H, T, d] in q's dtype, lse [B, H, T] fp32).
    fused=True folds each pair into the accumulator in the block epilogue
    (RSA_RING_FUSED_MERGE) instead of launching the merge kernel."""
    B, H, T, d = _check_qkv(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    need = workspace_size(q.dtype, B, H, T, d, N, causal, fused)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if fused:
        _call("rsa_ring_attn_fwd_ex", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), RSA_RING_FUSED_MERGE, out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream), None, None, None, 0, None)
    else:
        _call("rsa_ring_attn_fwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream))
    return out, lse


def ring_attn_noalloc(q, k, v, N: int, causal: bool, out=None, lse=None,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """ring_attn without a workspace, for callers that cannot allocate device
    memory at call time: the library's built-in 64 MiB scratch array is used
    instead (shapes needing more are rejected).  Calls share that array, so
    calls that could overlap on the GPU must be serialised by the caller."""
    B, H, T, d = _check_qkv(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    _call("rsa_ring_attn_fwd_noalloc", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
          int(bool(causal)), out.data_ptr(), lse.data_ptr(), _stream(stream))
    return out, lse


def ring_attn_timed(q, k, v, N: int, causal: bool, out, lse, workspace, events_start: Sequence,
                    events_stop: Sequence, stream=None, fused: bool = False) -> List[int]:
    """ring_attn that records the given torch.cuda.Event pairs around each
    kernel launch; returns the launch kinds (0 block attention, 1 merge)."""
    B, H, T, d = _check_qkv(q, k, v)
    cap = len(events_start)
    st = torch.cuda.current_stream() if stream is None else stream
    for e in list(events_start) + list(events_stop):
        if not e.cuda_event:  # torch creates the CUDA event on first record
            e.record(st)
    ev_s = (ctypes.c_void_p * cap)(*[int(e.cuda_event) for e in events_start])
    ev_e = (ctypes.c_void_p * cap)(*[int(e.cuda_event) for e in events_stop])
    kinds = (ctypes.c_int * cap)()
    n = ctypes.c_int(0)
    if fused:
        _call("rsa_ring_attn_fwd_ex", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), RSA_RING_FUSED_MERGE, out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream), ev_s, ev_e, kinds, cap,
              ctypes.byref(n))
    else:
        _call("rsa_ring_attn_fwd_timed", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream), ev_s, ev_e, kinds, cap,
              ctypes.byref(n))
    return [kinds[i] for i in range(n.value)]


def ring_launch_count(N: int, causal: bool, fused: bool = False) -> int:
    """Kernel launches one ring makes (block-attention plus merge launches)."""
    n = 0
    for r in range(N):
        np_ = len(ring_schedule(N, causal, r))
        groups = (np_ + 31) // 32
        n += groups if (r == 0 or fused) else 2 * groups
    return n


# Page-locked host blocks made by host_empty: storage address -> (mmap, bytes, base tensor).
_host_blocks = {}
_host_lock = threading.Lock()


def _huge_bytes(addr: int) -> int:
    """Bytes of the mapping that contains addr that sit on transparent huge
    pages (AnonHugePages in /proc/self/smaps); 0 if it cannot be read."""
    try:
        with open("/proc/self/smaps") as f:
            inside = False
            for line in f:
                head = line.split(None, 1)[0]
                if "-" in head and ":" not in head:
                    lo, hi = (int(x, 16) for x in head.split("-"))
                    inside = lo <= addr < hi
                elif inside and head == "AnonHugePages:":
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError):
        pass
    return 0


def host_empty(shape, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """A page-locked host tensor for streaming copies, on transparent huge
    pages where the host can provide them.

    The memory is an anonymous mapping advised for huge pages and touched, so
    that its pages exist.  If at least 90% of it landed on huge pages it is
    registered with cudaHostRegister: a few large pages for the copy engines
    to translate instead of many small ones.  Otherwise (small pages only,
    where a registered block has copied several times slower than a
    driver-pinned one) the tensor comes from torch's pinned allocator.

    A registered block stays registered until host_free() is called on the
    tensor (or a view of its storage), or the process exits."""
    shape = tuple(int(x) for x in shape)
    numel = 1
    for x in shape:
        numel *= x
    nbytes = numel * torch.empty((), dtype=dtype).element_size()
    size = max(1, (nbytes + (2 << 20) - 1) // (2 << 20)) * (2 << 20)
    if hasattr(mmap, "MADV_HUGEPAGE"):
        m = mmap.mmap(-1, size, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS, prot=mmap.PROT_READ | mmap.PROT_WRITE)
        m.madvise(mmap.MADV_HUGEPAGE)
        raw = torch.frombuffer(m, dtype=torch.uint8, count=size)
        raw.fill_(0)
        if _huge_bytes(raw.data_ptr()) >= 0.9 * size:
            err = torch.cuda.cudart().cudaHostRegister(raw.data_ptr(), size, 0)
            if int(err) != 0:
                raise RsaError("host_empty", 3, f"cudaHostRegister of {size} bytes failed: {err}")
            with _host_lock:
                _host_blocks[raw.data_ptr()] = (m, size, raw)
            return raw[:nbytes].view(dtype).view(shape)
        del raw
        try:
            m.close()
        except BufferError:
            pass  # closed when the last reference goes
    return torch.empty(shape, dtype=dtype, pin_memory=True)


def host_kind(t: torch.Tensor) -> str:
    """How a host tensor's memory is held: "registered-huge" (a host_empty
    block on huge pages, registered with cudaHostRegister), "pinned" (torch's
    page-locked allocator) or "pageable"."""
    with _host_lock:
        if t.untyped_storage().data_ptr() in _host_blocks:
            return "registered-huge"
    return "pinned" if t.is_pinned() else "pageable"


def host_free(t: torch.Tensor) -> None:
    """Unregister a block made by host_empty (the memory itself goes away with
    its last tensor).  Tensors not made by host_empty are left alone."""
    ptr = t.untyped_storage().data_ptr()
    with _host_lock:
        blk = _host_blocks.pop(ptr, None)
    if blk is not None:
        torch.cuda.cudart().cudaHostUnregister(ptr)


@atexit.register
def _host_free_all():
    with _host_lock:
        ptrs = list(_host_blocks)
        _host_blocks.clear()
    for ptr in ptrs:
        try:
            torch.cuda.cudart().cudaHostUnregister(ptr)
        except Exception:
            pass


def slab_plan(BH: int, groups: int = 8, ramp: bool = True) -> List[int]:
    """Heads per slab for ring_attn_from_host.

    Without ramp: `groups` equal slabs.  With ramp: slabs of at most
    ceil(BH / groups) heads in the middle, preceded by slabs that grow about
    1.6x at a time from an eighth of that, and followed by slabs that shrink
    back to an eighth.  Copying one head in takes less time than computing it,
    so each slab's copy hides under its predecessor's ring.  What is left
    exposed is the first slab's copy in and the last slab's copy out, and the
    ramps keep those small."""
    if BH <= 0:
        return []
    cap = max(1, -(-BH // max(1, min(int(groups), BH))))
    if not ramp or cap < 8:
        n = -(-BH // cap)
        return [cap] * (BH // cap) + ([BH % cap] if BH % cap else []) if n > 0 else []
    up, x = [], max(1, cap // 8)
    while x < cap:
        up.append(x)
        x = max(x + 1, (x * 8) // 5)
    down = [max(1, cap // 2), max(1, cap // 4), max(1, cap // 8)]
    if sum(up) + sum(down) >= BH:
        return slab_plan(BH, groups, ramp=False)
    mid = BH - sum(up) - sum(down)
    k = -(-mid // cap)  # middle slabs, as equal as possible
    middle = [mid // k + (1 if i < mid % k else 0) for i in range(k)]
    return up + middle + down


def ring_attn_from_host(q_host, k_host, v_host, N: int, causal: bool, device=None, stream=None,
                        buffers=None, groups: int = 8, ramp: bool = True):
    """End-to-end call from host memory: Q, K, V (host tensors, ideally made
    by host_empty) in, out and lse (page-locked host tensors) back.

    Heads are independent problems, so the B*H heads are cut into slabs
    (slab_plan(B*H, groups, ramp)) that stream through three CUDA streams: the
    copy of slab g+1 to the device, the ring on slab g (C ABI, on ``stream``
    or the current stream) and the copy of slab g-1 back to the host all
    overlap.  Device slabs are double-buffered.  The returned host tensors are
    complete once ``stream`` has passed the call (it waits for the last copy
    back).  ``buffers`` (a dict, filled on first use) keeps the device slabs,
    the workspace, the pinned outputs and the copy streams for reuse."""
    dev = torch.device(device) if device is not None else torch.device("cuda")
    b = buffers if buffers is not None else {}
    B, H, T, d = q_host.shape
    BH = B * H
    plan = slab_plan(BH, groups, ramp)
    hg = max(plan)  # heads in the largest slab
    main = torch.cuda.current_stream(dev) if stream is None else stream
    key = (tuple(q_host.shape), q_host.dtype, N, bool(causal), tuple(plan), str(dev))
    if b.get("key") != key:
        for name in ("out_host", "lse_host"):
            if name in b:
                host_free(b[name])
        b.clear()
        b["key"] = key
        mk = lambda *shape, dt=q_host.dtype: torch.empty(shape, dtype=dt, device=dev)
        b["in"] = [[mk(hg, T, d) for _ in range(3)] for _ in range(2)]
        b["out"] = [mk(hg, T, d) for _ in range(2)]
        b["lse"] = [mk(hg, T, dt=torch.float32) for _ in range(2)]
        b["ws"] = mk(max(workspace_size(q_host.dtype, 1, hg, T, d, N, causal), 1), dt=torch.uint8)
        b["out_host"] = host_empty(q_host.shape, q_host.dtype)
        b["lse_host"] = host_empty((B, H, T), torch.float32)
        b["s_in"] = torch.cuda.Stream(dev)
        b["s_out"] = torch.cuda.Stream(dev)
    s_in, s_out = b["s_in"], b["s_out"]
    src = [t.reshape(BH, T, d) for t in (q_host, k_host, v_host)]
    oh = b["out_host"].view(BH, T, d)
    lh = b["lse_host"].view(BH, T)
    s_in.wait_stream(main)
    s_out.wait_stream(main)
    ev_comp, ev_out = [], []
    h0 = 0
    for g, n in enumerate(plan):
        h1 = h0 + n
        slot = g % 2
        with torch.cuda.stream(s_in):
            if g >= 2:
                s_in.wait_event(ev_comp[g - 2])  # ring on slab g-2 has read this slot
            for t_dev, t_host in zip(b["in"][slot], src):
                t_dev[:n].copy_(t_host[h0:h1], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        main.wait_event(ev_in)
        if g >= 2:
            main.wait_event(ev_out[g - 2])  # slab g-2 has been copied out of this slot
        qd, kd, vd = (t[:n].view(1, n, T, d) for t in b["in"][slot])
        ring_attn(qd, kd, vd, N, causal, out=b["out"][slot][:n].view(1, n, T, d),
                  lse=b["lse"][slot][:n].view(1, n, T), workspace=b["ws"], stream=main)
        ev = torch.cuda.Event()
        ev.record(main)
        ev_comp.append(ev)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev)
            oh[h0:h1].copy_(b["out"][slot][:n], non_blocking=True)
            lh[h0:h1].copy_(b["lse"][slot][:n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s_out)
            ev_out.append(ev)
        h0 = h1
    main.wait_event(ev_out[-1])
    return b["out_host"], b["lse_host"], b


def two_pass_workspace_size(dtype: torch.dtype, B: int, H: int, T: int, d: int, N: int) -> int:
    n = ctypes.c_size_t(0)
    dt = RSA_F32 if dtype == torch.float32 else RSA_BF16
    _call("rsa_two_pass_workspace_size", dt, B, H, T, d, N, ctypes.byref(n))
    return int(n.value)


def two_pass_attn(q, k, v, N: int, causal: bool, out=None, lse=None, workspace=None,
                  stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Two-pass Ring Self-Attention (full score rows per query chunk, then
    softmax, then the value ring): (out [B, H, T, d], lse [B, H, T])."""
    B, H, T, d = _check_qkv(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(two_pass_workspace_size(q.dtype, B, H, T, d, N), dtype=torch.uint8, device=q.device)
    _call("rsa_two_pass_attn_fwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
          int(bool(causal)), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return out, lse


def decode_workspace_size(dtype: torch.dtype, B: int, H: int, T: int, d: int, q_len: int, N: int) -> int:
    n = ctypes.c_size_t(0)
    dt = RSA_F32 if dtype == torch.float32 else RSA_BF16
    _call("rsa_decode_workspace_size", dt, B, H, T, d, q_len, N, ctypes.byref(n))
    return int(n.value)


def decode_attn(q, k, v, N: int, causal: bool, out=None, lse=None, workspace=None,
                stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Decode against a KV cache cut into N shards: q [B, H, q_len, d] holds the
    q_len newest tokens (positions T-q_len .. T-1), k and v [B, H, T, d] the
    cache.  Returns (out [B, H, q_len, d], lse [B, H, q_len] fp32)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-d CUDA tensor")
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3] or not (
            q.dtype == k.dtype == v.dtype):
        raise ValueError("q [B, H, q_len, d] and k, v [B, H, T, d] must agree")
    B, H, q_len, d = q.shape
    T = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, q_len), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(decode_workspace_size(q.dtype, B, H, T, d, q_len, N), 1), dtype=torch.uint8,
                                device=q.device)
    _call("rsa_decode_attn_fwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, q_len, N,
          int(bool(causal)), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return out, lse


def ring_schedule(N: int, causal: bool, rnd: int) -> List[Tuple[int, int]]:
    """Pairs (q_chunk, kv_chunk) of round rnd as the library schedules them."""
    cap = max(N, 1)
    qi = (ctypes.c_int * cap)()
    kj = (ctypes.c_int * cap)()
    n = ctypes.c_int(0)
    _call("rsa_ring_schedule", N, int(bool(causal)), rnd, qi, kj, cap, ctypes.byref(n))
    return [(qi[i], kj[i]) for i in range(n.value)]


def set_wait_limit_ns(limit_ns: int) -> None:
    _call("rsa_set_wait_limit_ns", int(limit_ns))


BLOCK_KERNELS = {"auto": 0, "one_sm": 1, "two_sm": 2}


def set_block_kernel(which: str) -> None:
    """Pick the bf16 tensor-core block kernel for later calls: "auto" (the
    one-SM kernel), "one_sm", or "two_sm" (the CTA-pair kernel where it
    applies: d = 128, pairs of at least 512 rows, no key splits)."""
    _call("rsa_set_block_kernel", BLOCK_KERNELS[which])


def check_device_error(stream=None) -> None:
    _call("rsa_check_device_error", _stream(stream))


def selftest_wait_timeout(stream=None) -> None:
    _call("rsa_selftest_wait_timeout", _stream(stream))
