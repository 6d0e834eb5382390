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

import ctypes
import threading
from typing import List, Optional, Sequence, Tuple

import torch

from . import _build

__all__ = [
    "RsaError", "load", "library_path", "block_attn_fwd", "merge", "merge_finalize",
    "ring_attn", "ring_attn_noalloc", "ring_attn_timed", "decode_attn", "decode_workspace_size",
    "two_pass_attn", "two_pass_workspace_size", "ring_attn_from_host", "slab_plan", "host_empty", "host_kind",
    "host_info", "host_workspace_size", "set_host_copy_mode", "host_copy_path",
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
    "rsa_block_attn_fold": [_c_void_p, _i64, _c_void_p, _c_void_p, _i64, _i32, _i32, _i32, _i32, _i64, _i64, _i64,
                            _i64, _i64, _i64, _i32, _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p],
    "rsa_rank_ring_plan": [_i32, _i32, _i64, _i32, _i32, ctypes.POINTER(_i64), _i32, ctypes.POINTER(_i32)],
    "rsa_host_alloc": [ctypes.c_size_t, ctypes.POINTER(_c_void_p)],
    "rsa_host_free": [_c_void_p],
    "rsa_host_info": [_c_void_p, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t),
                      ctypes.POINTER(_i32)],
    "rsa_host_slab_plan": [_i32, _i32, _i32, ctypes.POINTER(_i32), _i32, ctypes.POINTER(_i32)],
    "rsa_set_host_copy_mode": [_i32],
    "rsa_host_copy_path": [_c_void_p, ctypes.c_size_t, ctypes.POINTER(_i32)],
    "rsa_ring_attn_host_workspace_size": [_i32, _i32, _i32, _i64, _i32, _i32, _i32,
                                          ctypes.POINTER(ctypes.c_size_t)],
    "rsa_ring_attn_fwd_host": [_c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                               _c_void_p, _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p],
    "rsa_set_wait_limit_ns": [ctypes.c_uint64],
    "rsa_set_block_kernel": [_i32],
    "rsa_debug_inject_launch_failure": [_i32],
    "rsa_debug_checks": [],
    "rsa_check_device_error": [_c_void_p],
    "rsa_selftest_wait_timeout": [_c_void_p],
    "rsa_status_string": [_i32],
    "rsa_last_error_string": [],
    "rsa_version": [],
}


def debug_variant() -> bool:
    """True when the environment asks for the RSA_DEBUG build (RSA_DEBUG=1):
    kernels with device-side bounds checks, reported by check_device_error."""
    import os
    return os.environ.get("RSA_DEBUG", "0") not in ("", "0")


def library_path(build: bool = True) -> str:
    dbg = debug_variant()
    if build:
        return _build.build(debug=dbg)
    return _build.DEBUG_LIB if dbg else _build.LIB


def load(build: bool = True):
    """Load librsa.so (building it in-tree first if it is stale); the
    RSA_DEBUG variant when the environment sets RSA_DEBUG=1."""
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
            if bool(lib.rsa_debug_checks()) != debug_variant():
                raise RsaError("load", 2, f"{path} does not match RSA_DEBUG={int(debug_variant())}")
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
RSA_RING_SEPARATE_MERGE = 2


def _ring_flags(fused: bool) -> int:
    return RSA_RING_FUSED_MERGE if fused else RSA_RING_SEPARATE_MERGE


def workspace_size(dtype: torch.dtype, B: int, H: int, T: int, d: int, N: int, causal: bool,
                   fused: bool = True) -> int:
    """Workspace bytes of the ring: the fused merge (default) or, with
    fused=False, the separate merge kernel (RSA_RING_SEPARATE_MERGE)."""
    n = ctypes.c_size_t(0)
    dt = RSA_F32 if dtype == torch.float32 else RSA_BF16
    _call("rsa_ring_attn_workspace_size_ex", dt, B, H, T, d, N, int(bool(causal)), _ring_flags(fused),
          ctypes.byref(n))
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
    """The last merge of a ring: merge((o_acc, lse_acc), (o_blk, lse_blk))
    written to (out [o_acc's shape, out_dtype], lse_out fp32); the
    accumulator is only read."""
    d = o_acc.shape[-1]
    rows = lse_acc.numel()
    if o_acc.dtype != torch.float32 or lse_acc.dtype != torch.float32 or lse_blk.dtype != torch.float32:
        raise TypeError("o_acc, lse_acc and lse_blk must be float32")
    if o_blk.numel() != rows * d or o_acc.numel() != rows * d or lse_blk.numel() != rows:
        raise ValueError("row counts differ")
    if out is None:
        out = torch.empty(o_acc.shape, dtype=out_dtype, device=o_acc.device)
    if lse_out is None:
        lse_out = torch.empty(lse_acc.shape, dtype=torch.float32, device=o_acc.device)
    if out.dtype != out_dtype or out.numel() != rows * d:
        raise ValueError("out must hold rows x d values of out_dtype")
    if lse_out.dtype != torch.float32 or lse_out.numel() != rows:
        raise ValueError("lse_out must hold one float32 per row")
    for t in (o_acc, lse_acc, o_blk, lse_blk, out, lse_out):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("merge operands must be contiguous CUDA tensors")
    _call("rsa_merge_finalize", o_acc.data_ptr(), lse_acc.data_ptr(), o_blk.data_ptr(), _dt(o_blk),
          lse_blk.data_ptr(), rows, d, out.data_ptr(), _dt(out), lse_out.data_ptr(), _stream(stream))
    return out, lse_out


def ring_attn(q, k, v, N: int, causal: bool, out=None, lse=None, workspace=None,
              stream=None, fused: bool = True) -> Tuple[torch.Tensor, torch.Tensor]:
    """The whole ring: (out [B, H, T, d] in q's dtype, lse [B, H, T] fp32).
    By default (rsa_ring_attn_fwd) each pair's block epilogue folds it into
    the accumulator; fused=False computes partials and launches the merge
    kernel instead (RSA_RING_SEPARATE_MERGE)."""
    B, H, T, d = _check_qkv(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    need = workspace_size(q.dtype, B, H, T, d, N, causal, fused)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if fused:
        _call("rsa_ring_attn_fwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream))
    else:
        _call("rsa_ring_attn_fwd_ex", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), RSA_RING_SEPARATE_MERGE, out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream), None, None, None, 0, None)
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
                    events_stop: Sequence, stream=None, fused: bool = True) -> List[int]:
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
        _call("rsa_ring_attn_fwd_timed", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream), ev_s, ev_e, kinds, cap,
              ctypes.byref(n))
    else:
        _call("rsa_ring_attn_fwd_ex", q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), B, H, T, d, N,
              int(bool(causal)), RSA_RING_SEPARATE_MERGE, out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), _stream(stream), ev_s, ev_e, kinds, cap,
              ctypes.byref(n))
    return [kinds[i] for i in range(n.value)]


def ring_launch_count(N: int, causal: bool, fused: bool = True) -> int:
    """Kernel launches one ring makes: one block-attention launch per round
    (up to 32 pairs each), plus, with fused=False, one merge launch per round
    after the first."""
    n = 0
    for r in range(N):
        np_ = len(ring_schedule(N, causal, r))
        groups = (np_ + 31) // 32
        n += groups if (r == 0 or fused) else 2 * groups
    return n


# Host blocks made by host_empty: block address -> bytes.  A block is freed
# (rsa_host_free) when the last tensor viewing it is garbage-collected.
_host_blocks = {}
_host_lock = threading.Lock()

RSA_HOST_HUGE = 1
RSA_HOST_PINNED = 2


def _release_host_block(ptr: int) -> None:
    with _host_lock:
        known = _host_blocks.pop(ptr, None) is not None
    if known and _lib is not None:
        _lib.rsa_host_free(ptr)


def host_empty(shape, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """A page-locked host tensor for streaming copies, from rsa_host_alloc:
    memory on transparent huge pages registered with the CUDA driver (or
    driver-pinned memory where huge pages are not to be had).  Copies from
    base-page pinned memory have been measured to slow down after the memory
    sat idle; huge-page memory kept its speed.  The block is released when the
    last tensor viewing it is gone."""
    import weakref
    shape = tuple(int(x) for x in shape)
    numel = 1
    for x in shape:
        numel *= x
    nbytes = max(1, numel * torch.empty((), dtype=dtype).element_size())
    ptr = ctypes.c_void_p(0)
    _call("rsa_host_alloc", nbytes, ctypes.byref(ptr))
    addr = int(ptr.value)
    buf = (ctypes.c_uint8 * nbytes).from_address(addr)
    with _host_lock:
        _host_blocks[addr] = nbytes
    weakref.finalize(buf, _release_host_block, addr)
    raw = torch.frombuffer(buf, dtype=torch.uint8, count=nbytes)
    return raw[:numel * torch.empty((), dtype=dtype).element_size()].view(dtype).view(shape)


def host_info(t: torch.Tensor) -> dict:
    """rsa_host_info of a tensor made by host_empty: usable bytes, bytes the
    kernel backs with huge pages now, and kind ("registered-huge" or
    "pinned")."""
    ptr = t.untyped_storage().data_ptr()
    n, huge, kind = ctypes.c_size_t(0), ctypes.c_size_t(0), ctypes.c_int(0)
    _call("rsa_host_info", ptr, ctypes.byref(n), ctypes.byref(huge), ctypes.byref(kind))
    return {"bytes": int(n.value), "huge_bytes": int(huge.value),
            "kind": "registered-huge" if kind.value == RSA_HOST_HUGE else "pinned"}


def host_kind(t: torch.Tensor) -> str:
    """How a host tensor's memory is held: "registered-huge" or "pinned" (a
    host_empty block), "pinned" (torch's page-locked allocator) or
    "pageable"."""
    with _host_lock:
        ours = t.untyped_storage().data_ptr() in _host_blocks
    if ours:
        return host_info(t)["kind"]
    return "pinned" if t.is_pinned() else "pageable"


HOST_COPY_MODES = {"auto": 0, "engines": 1, "sm": 2}


def set_host_copy_mode(mode: str) -> None:
    """How ring_attn_from_host moves host tensors: "auto" (copy engines for
    library blocks still on huge pages and for pageable memory, a copy kernel
    for other page-locked memory), "engines" or "sm"."""
    _call("rsa_set_host_copy_mode", HOST_COPY_MODES[mode])


def host_copy_path(t: torch.Tensor) -> str:
    """"engines" or "kernel": how ring_attn_from_host would move this host
    tensor now."""
    path = ctypes.c_int(0)
    _call("rsa_host_copy_path", t.data_ptr(), t.numel() * t.element_size(), ctypes.byref(path))
    return "engines" if path.value == 1 else "kernel"


def slab_plan(BH: int, groups: int = 8, ramp: bool = True) -> List[int]:
    """Heads per slab of the host-streaming path (rsa_host_slab_plan): about
    `groups` slabs of at most ceil(BH / groups) heads; with ramp, small slabs
    that grow about 1.6x at a time lead in and shrinking ones lead out, so
    each slab's copy hides under its predecessor's ring."""
    if BH <= 0:
        return []
    cap = max(8, BH)
    slabs = (ctypes.c_int * cap)()
    n = ctypes.c_int(0)
    _call("rsa_host_slab_plan", int(BH), int(groups), int(bool(ramp)), slabs, cap, ctypes.byref(n))
    return [slabs[i] for i in range(n.value)]


def host_workspace_size(dtype: torch.dtype, B: int, H: int, T: int, d: int, N: int, causal: bool) -> int:
    n = ctypes.c_size_t(0)
    dt = RSA_F32 if dtype == torch.float32 else RSA_BF16
    _call("rsa_ring_attn_host_workspace_size", dt, B, H, T, d, N, int(bool(causal)), ctypes.byref(n))
    return int(n.value)


def ring_attn_from_host(q_host, k_host, v_host, N: int, causal: bool, device=None, stream=None,
                        buffers=None):
    """End-to-end call from host memory (rsa_ring_attn_fwd_host): Q, K, V host
    tensors [B, H, T, d] in (ideally made by host_empty), out and lse back in
    page-locked host tensors.  The C library streams slabs of heads through
    the GPU, overlapping the copies in and out with the ring.  The returned
    host tensors are complete once ``stream`` (default: the current stream)
    has passed the call.  ``buffers`` (a dict, filled on first use) keeps the
    device workspace and the host outputs for reuse."""
    dev = torch.device(device) if device is not None else torch.device("cuda")
    b = buffers if buffers is not None else {}
    for name, t in (("q", q_host), ("k", k_host), ("v", v_host)):
        if t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, T, d] host tensor")
    if not (q_host.shape == k_host.shape == v_host.shape and q_host.dtype == k_host.dtype == v_host.dtype):
        raise ValueError("q, k, v must share shape and dtype")
    B, H, T, d = q_host.shape
    key = (tuple(q_host.shape), q_host.dtype, N, bool(causal), str(dev))
    if b.get("key") != key:
        b.clear()
        b["key"] = key
        with torch.cuda.device(dev):
            b["ws"] = torch.empty(host_workspace_size(q_host.dtype, B, H, T, d, N, causal) + 256,
                                  dtype=torch.uint8, device=dev)
        # out and lse share one huge-page block
        esz = q_host.element_size()
        out_bytes = B * H * T * d * esz
        lse_off = (out_bytes + 255) // 256 * 256
        blk = host_empty((lse_off + B * H * T * 4,), torch.uint8)
        b["out_host"] = blk[:out_bytes].view(q_host.dtype).view(B, H, T, d)
        b["lse_host"] = blk[lse_off:].view(torch.float32).view(B, H, T)
    ws = b["ws"]
    ws_ptr = (ws.data_ptr() + 255) // 256 * 256
    st = torch.cuda.current_stream(dev) if stream is None else stream
    with torch.cuda.device(dev):
        _call("rsa_ring_attn_fwd_host", q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), _dt(q_host),
              B, H, T, d, N, int(bool(causal)), b["out_host"].data_ptr(), b["lse_host"].data_ptr(), ws_ptr,
              ws.numel() - (ws_ptr - ws.data_ptr()), _stream(st))
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


def inject_launch_failure(countdown: int) -> None:
    """Make the library's launch after the next `countdown` ones report a
    launch failure (RSA_ERR_CUDA) instead of launching; negative: off."""
    _call("rsa_debug_inject_launch_failure", int(countdown))


def check_device_error(stream=None) -> None:
    _call("rsa_check_device_error", _stream(stream))


def selftest_wait_timeout(stream=None) -> None:
    _call("rsa_selftest_wait_timeout", _stream(stream))
