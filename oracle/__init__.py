"""CPU oracle for blockwise ring self-attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  It shares no
code with the CUDA library and never imports it.

Pages cited (the text of three web pages on sequence parallelism):
  [P1] "Sequence parallelism -- splitting the token dimension across GPUs"
       (llmdaily, day 58)
  [P3] "Sequence Parallelism" (glossary entry, zhongzhoutan-coder terms)

Forms:
  O1  ``attend_rows`` / ``attention`` / ``block`` -- the dense definition in
      fp64 (C, ``rsa_oracle.c``): [P1] "Attention wants keys and values from
      other tokens", softmax(Q K^T / sqrt(d_k)) V; causal mask of [P1]
      "Causal attention gives us another optimization" (j <= t, inclusive).
  O2  ``rsa_two_pass`` -- [P3] "How It Works", steps 1-2: a score pass that
      circulates the K chunks to build each chunk's full score rows, then an
      output pass that circulates the V chunks and sums P^n_j V_j.
  O3  ``ring_online`` -- [P1] "A better mental model: move blocks past the
      queries" (the round table) with the running statistics of [P1] "But
      softmax seems to require all attention scores at once":
      m_new = max(m, m'), old terms scaled by e^{m - m_new}, new ones by
      e^{m' - m_new}.  Kept both as (m, l, o) and as (normalised o, lse).

Every function here is pinned by tests against closed forms, invariants and
library routines; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import itertools
import os
import subprocess
import threading
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DTYPE_CODE = {"f32": 0, "bf16": 1, "f64": 2}


def build(force: bool = False) -> str:
    """Compile rsa_oracle.c with gcc (OpenMP, no fast-math) if it is stale."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or \
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.rsa_oracle_attend.restype = ctypes.c_int
            lib.rsa_oracle_attend.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.rsa_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().rsa_oracle_max_threads())


def as_input(x, tag: Optional[str] = None) -> Tuple[np.ndarray, str]:
    """Accept a numpy array (float32, float64, or uint16 bf16 bits) or a CPU
    torch tensor; return a C-contiguous array and its dtype tag."""
    if not isinstance(x, np.ndarray):
        import torch  # plain CPU plumbing only
        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), "bf16"
        x = t.numpy()
    x = np.ascontiguousarray(x)
    if tag is not None:
        return x, tag
    if x.dtype == np.float32:
        return x, "f32"
    if x.dtype == np.float64:
        return x, "f64"
    if x.dtype == np.uint16:
        return x, "bf16"
    raise TypeError(f"oracle input dtype {x.dtype}")


def to_f64(x, tag: Optional[str] = None) -> np.ndarray:
    """Exact fp64 values of an oracle input (bf16 bits are widened exactly)."""
    a, tg = as_input(x, tag)
    if tg == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def attend_rows(q_rows, k, v, rows, causal: bool, kv_lo: int = 0, kv_hi: Optional[int] = None,
                nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """O1 on listed rows.  q_rows [n, d] are the rows' query vectors, k and v
    are full [B, H, T, d] tensors, rows [n, 3] holds (b, h, t).  Returns
    fp64 (out [n, d], lse [n])."""
    lib = _load()
    qa, tq = as_input(q_rows)
    ka, tk = as_input(k)
    va, tv = as_input(v)
    if not (tq == tk == tv):
        raise TypeError("q, k, v must share a dtype")
    B, H, T, d = ka.shape
    if va.shape != ka.shape or qa.shape[-1] != d:
        raise ValueError("shape mismatch")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    if qa.size != n * d:
        raise ValueError("q_rows must hold one d-vector per listed row")
    kv_hi = T if kv_hi is None else kv_hi
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.rsa_oracle_attend(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, _DTYPE_CODE[tq],
                               B, H, T, d, rows.ctypes.data, n, kv_lo, kv_hi, int(bool(causal)),
                               out.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, lse


def _all_rows(B: int, H: int, t_lo: int, t_hi: int) -> np.ndarray:
    b, h, t = np.meshgrid(np.arange(B), np.arange(H), np.arange(t_lo, t_hi), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), t.ravel()], axis=1).astype(np.int64)


def block(q, k, v, q_off: int, q_len: int, kv_off: int, kv_len: int, causal: bool,
          nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """O1 for one (query chunk, KV chunk) pair: queries [q_off, q_off+q_len)
    against keys [kv_off, kv_off+kv_len), global positions for the mask.
    Returns (o_blk [B, H, q_len, d], lse_blk [B, H, q_len])."""
    qa, tq = as_input(q)
    B, H, T, d = qa.shape
    rows = _all_rows(B, H, q_off, q_off + q_len)
    q_rows = np.ascontiguousarray(qa[:, :, q_off:q_off + q_len, :]).reshape(-1, d)
    out, lse = _attend_tagged(q_rows, tq, k, v, rows, causal, kv_off, kv_off + kv_len, nthreads)
    return out.reshape(B, H, q_len, d), lse.reshape(B, H, q_len)


def _attend_tagged(q_rows, tag, k, v, rows, causal, kv_lo, kv_hi, nthreads):
    lib = _load()
    ka, tk = as_input(k)
    va, tv = as_input(v)
    if not (tag == tk == tv):
        raise TypeError("q, k, v must share a dtype")
    B, H, T, d = ka.shape
    q_rows = np.ascontiguousarray(q_rows)
    n = rows.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.rsa_oracle_attend(q_rows.ctypes.data, ka.ctypes.data, va.ctypes.data,
                               _DTYPE_CODE[tag], B, H, T, d, rows.ctypes.data, n, kv_lo, kv_hi,
                               int(bool(causal)), out.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, lse


def attention(q, k, v, causal: bool, nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """O1 over the whole sequence: (out [B, H, T, d], lse [B, H, T]) in fp64."""
    qa, _ = as_input(q)
    T = qa.shape[2]
    return block(q, k, v, 0, T, 0, T, causal, nthreads)


def sampled(q, k, v, rows, causal: bool, nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """O1 on sampled rows (b, h, t) of full tensors q, k, v."""
    qa, tq = as_input(q)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    q_rows = np.ascontiguousarray(qa[rows[:, 0], rows[:, 1], rows[:, 2], :])
    T = qa.shape[2]
    return _attend_tagged(q_rows, tq, k, v, rows, causal, 0, T, nthreads)


# ---------------------------------------------------------------------------
# Chunks ([P1] "Split tokens across four GPUs") and ring order ([P1] "A better
# mental model: move blocks past the queries")
# ---------------------------------------------------------------------------

def chunk_range(T: int, N: int, i: int) -> Tuple[int, int]:
    """0-based half-open token range [lo, hi) of chunk i: contiguous pieces of
    T/N tokens in order (the page's GPU 0 holds tokens 1-8192 of 32768)."""
    if T % N:
        raise ValueError("N must divide T")
    Tc = T // N
    return i * Tc, (i + 1) * Tc


def ring_round(N: int, r: int, causal: bool) -> List[Tuple[int, int]]:
    """Pairs (query chunk i, KV chunk j) of round r (0-based).  The page's
    table has GPU i seeing KV_{(i - r) mod N} in round r+1; under the causal
    mask chunk i never needs a later chunk ([P1] "Causal attention gives us
    another optimization"), so pairs with j > i are dropped."""
    pairs = []
    for i in range(N):
        j = (i - r) % N
        if causal and j > i:
            continue
        pairs.append((i, j))
    return pairs


def ring_pairs(N: int, causal: bool) -> List[Tuple[int, int]]:
    return [p for r in range(N) for p in ring_round(N, r, causal)]


# ---------------------------------------------------------------------------
# O3: online-softmax merging ([P1] "But softmax seems to require all
# attention scores at once")
# ---------------------------------------------------------------------------

def merge_lse(o_a: np.ndarray, lse_a: np.ndarray, o_b: np.ndarray, lse_b: np.ndarray
              ) -> Tuple[np.ndarray, np.ndarray]:
    """Fold two normalised partial results (o, lse) of disjoint key sets.

    With M = max(lse_a, lse_b): L = M + ln(e^{lse_a - M} + e^{lse_b - M}),
    o = o_a e^{lse_a - L} + o_b e^{lse_b - L}.  Both -inf gives (0, -inf)."""
    o_a = np.asarray(o_a, np.float64)
    o_b = np.asarray(o_b, np.float64)
    lse_a = np.asarray(lse_a, np.float64)
    lse_b = np.asarray(lse_b, np.float64)
    M = np.maximum(lse_a, lse_b)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    with np.errstate(invalid="ignore", over="ignore"):
        wa = np.where(finite, np.exp(lse_a - Ms), 0.0)
        wb = np.where(finite, np.exp(lse_b - Ms), 0.0)
        tot = wa + wb
        L = np.where(finite, Ms + np.log(np.where(finite, tot, 1.0)), -np.inf)
        ca = np.where(finite, wa / np.where(finite, tot, 1.0), 0.0)
        cb = np.where(finite, wb / np.where(finite, tot, 1.0), 0.0)
    o = o_a * ca[..., None] + o_b * cb[..., None]
    return o, L


def merge_mlo(m_a, l_a, o_a, m_b, l_b, o_b):
    """The page's own form: running max m, normaliser l and unnormalised
    accumulator o.  m_new = max(m, m'); old terms x e^{m - m_new}, new terms
    x e^{m' - m_new}.  Rows where both maxima are -inf stay empty."""
    m_new = np.maximum(m_a, m_b)
    finite = np.isfinite(m_new)
    mn = np.where(finite, m_new, 0.0)
    with np.errstate(invalid="ignore"):
        sa = np.where(np.isfinite(m_a), np.exp(np.where(np.isfinite(m_a), m_a, 0.0) - mn), 0.0)
        sb = np.where(np.isfinite(m_b), np.exp(np.where(np.isfinite(m_b), m_b, 0.0) - mn), 0.0)
    l_new = l_a * sa + l_b * sb
    o_new = o_a * sa[..., None] + o_b * sb[..., None]
    return m_new, l_new, o_new


def block_mlo(q, k, v, q_off, q_len, kv_off, kv_len, causal):
    """(m, l, unnormalised o) of one pair, straight from the definition with
    numpy: s = q k^T / sqrt(d), m = row max, l = sum e^{s - m},
    o = sum e^{s - m} v.  Used to hold O3's (m, l, o) form against its lse
    form."""
    Q, K, V = to_f64(q), to_f64(k), to_f64(v)
    d = Q.shape[-1]
    qs = Q[:, :, q_off:q_off + q_len]
    ks = K[:, :, kv_off:kv_off + kv_len]
    vs = V[:, :, kv_off:kv_off + kv_len]
    s = np.einsum("bhtx,bhjx->bhtj", qs, ks) / np.sqrt(d)
    if causal:
        qi = np.arange(q_off, q_off + q_len)[:, None]
        kj = np.arange(kv_off, kv_off + kv_len)[None, :]
        s = np.where(kj <= qi, s, -np.inf)
    m = s.max(axis=-1) if s.shape[-1] else np.full(s.shape[:-1], -np.inf)
    mf = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - mf[..., None])
    l = e.sum(axis=-1)
    o = np.einsum("bhtj,bhjx->bhtx", e, vs)
    return m, l, o


def ring_online(q, k, v, N: int, causal: bool, order: Optional[Sequence[Tuple[int, int]]] = None,
                nthreads: int = 0, check_mlo: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """O3: chunk the sequence into N pieces, compute each pair's (o_blk, lse_blk)
    with O1 restricted to the pair, and fold them per query chunk in ring
    order (or in ``order``, a list of pairs).  If ``check_mlo`` is set the
    (m, l, o) form is folded alongside and must agree."""
    qa, _ = as_input(q)
    B, H, T, d = qa.shape
    if T % N:
        raise ValueError("N must divide T")
    Tc = T // N
    order = list(order) if order is not None else ring_pairs(N, causal)
    out = np.zeros((B, H, T, d))
    lse = np.full((B, H, T), -np.inf)
    mlo = {}
    for (i, j) in order:
        ob, lb = block(q, k, v, i * Tc, Tc, j * Tc, Tc, causal, nthreads)
        sl = slice(i * Tc, (i + 1) * Tc)
        out[:, :, sl], lse[:, :, sl] = merge_lse(out[:, :, sl], lse[:, :, sl], ob, lb)
        if check_mlo:
            m2, l2, o2 = block_mlo(q, k, v, i * Tc, Tc, j * Tc, Tc, causal)
            if i not in mlo:
                mlo[i] = (np.full(m2.shape, -np.inf), np.zeros(l2.shape), np.zeros(o2.shape))
            mlo[i] = merge_mlo(*mlo[i], m2, l2, o2)
    if check_mlo:
        for i, (m, l, o) in mlo.items():
            sl = slice(i * Tc, (i + 1) * Tc)
            with np.errstate(invalid="ignore", divide="ignore"):
                lse_f = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
                o_f = np.where((l > 0)[..., None], o / np.where(l > 0, l, 1.0)[..., None], 0.0)
            if not (np.allclose(lse_f, lse[:, :, sl], rtol=0, atol=1e-12)
                    and np.allclose(o_f, out[:, :, sl], rtol=0, atol=1e-12)):
                raise AssertionError("(m, l, o) and (o, lse) forms of the merge disagree")
    return out, lse


# ---------------------------------------------------------------------------
# O2: two-pass Ring Self-Attention ([P3] "How It Works")
# ---------------------------------------------------------------------------

def rsa_two_pass(q, k, v, N: int, causal: bool) -> Tuple[np.ndarray, np.ndarray]:
    """Score pass: chunk n's queries meet K chunk (n - r) mod N in round r, so
    after N - 1 transfers plus its own chunk it holds the full score rows
    S^n (L/N x L).  Softmax is taken over each full row.  Output pass: the V
    chunks go round the same ring and O^n accumulates P^n_j V_j, where P^n_j
    is the block of probabilities against chunk j's keys.  Returns fp64
    (out, lse)."""
    Q, K, V = to_f64(q), to_f64(k), to_f64(v)
    B, H, T, d = Q.shape
    if T % N:
        raise ValueError("N must divide T")
    Tc = T // N
    out = np.zeros((B, H, T, d))
    lse = np.zeros((B, H, T))
    for n in range(N):
        qn = Q[:, :, n * Tc:(n + 1) * Tc]
        S = np.full((B, H, Tc, T), -np.inf)
        for r in range(N):                      # score pass
            j = (n - r) % N
            blk = np.einsum("bhtx,bhjx->bhtj", qn, K[:, :, j * Tc:(j + 1) * Tc]) / np.sqrt(d)
            if causal:
                qi = np.arange(n * Tc, (n + 1) * Tc)[:, None]
                kj = np.arange(j * Tc, (j + 1) * Tc)[None, :]
                blk = np.where(kj <= qi, blk, -np.inf)
            S[..., j * Tc:(j + 1) * Tc] = blk
        m = S.max(axis=-1, keepdims=True)
        E = np.exp(S - m)
        Z = E.sum(axis=-1, keepdims=True)
        P = E / Z
        lse[:, :, n * Tc:(n + 1) * Tc] = (m + np.log(Z))[..., 0]
        On = np.zeros((B, H, Tc, d))
        for r in range(N):                      # output pass
            j = (n - r) % N
            On += np.einsum("bhtj,bhjx->bhtx", P[..., j * Tc:(j + 1) * Tc],
                            V[:, :, j * Tc:(j + 1) * Tc])
        out[:, :, n * Tc:(n + 1) * Tc] = On
    return out, lse


def flops_useful(B: int, H: int, T: int, d: int, causal: bool) -> float:
    """Useful forward FLOPs: 2d for q.k and 2d for p.v per allowed
    (query, key) pair; T(T+1)/2 pairs per head when causal, T^2 otherwise."""
    pairs = T * (T + 1) // 2 if causal else T * T
    return 4.0 * B * H * d * pairs


def rows_flops(rows: np.ndarray, T: int, d: int, causal: bool) -> float:
    """Useful FLOPs of attending the listed rows (b, h, t) over the sequence."""
    rows = np.asarray(rows).reshape(-1, 3)
    keys = (rows[:, 2] + 1).sum() if causal else rows.shape[0] * T
    return 4.0 * d * float(keys)
