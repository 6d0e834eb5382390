"""Ring attention across ranks: each rank keeps its query tokens while the
K/V blocks travel round the ranks.

Page: "Sequence parallelism -- splitting the token dimension across GPUs"
(llmdaily, day 58).  "A better mental model: move blocks past the queries":
in round r+1 GPU i holds the K/V block that started on GPU (i - r) mod N,
computes against it, and passes it on.  "Causal attention gives us another
optimization": pairs whose keys all lie after their queries are skipped; the
zigzag layout (rank i owns pieces i and 2N-1-i of 2N) gives every rank the
same work in every round after the first.

What runs where:
  - the pair list of this rank: ``rsa_rank_ring_plan`` (C, host);
  - every pair: ``rsa_block_attn_fold`` (the library's CUDA kernels), folding
    straight into this rank's fp32 accumulator, the last pair of a query
    piece writing out and lse;
  - the exchange: torch.distributed point-to-point sends and receives of one
    packed [2, B, H, T/N, d] K/V block per round into a second landing buffer,
    issued before the round's pairs so that the transfer overlaps them.
    exchange="device" sends device tensors (an NCCL group: one GPU per rank);
    exchange="host" sends page-locked host copies (a gloo group), each
    received block being copied to a device landing buffer on the compute
    stream.  The kernels read only this rank's own device memory.
"""
from __future__ import annotations

import ctypes
from typing import Dict, Iterator, List, Tuple

import torch

from . import _call, _dt, _stream

LAYOUTS = {"contiguous": 0, "zigzag": 1}
FOLD_FIRST, FOLD_MERGE, FOLD_LAST, FOLD_ONLY = 0, 1, 2, 3


def rank_ring_plan(N: int, rank: int, T: int, causal: bool, layout: str = "zigzag") -> List[Dict[str, int]]:
    """This rank's steps, in execution order (rsa_rank_ring_plan): dicts with
    round, src (whose K/V block), q_row0, q_pos, q_len, kv_row0, kv_pos,
    kv_len and fold."""
    cap = 4 * N + 4
    buf = (ctypes.c_int64 * (9 * cap))()
    n = ctypes.c_int(0)
    _call("rsa_rank_ring_plan", N, rank, T, int(bool(causal)), LAYOUTS[layout], buf, cap, ctypes.byref(n))
    keys = ("round", "src", "q_row0", "q_pos", "q_len", "kv_row0", "kv_pos", "kv_len", "fold")
    return [dict(zip(keys, (int(buf[9 * i + j]) for j in range(9)))) for i in range(n.value)]


def owned_positions(N: int, rank: int, T: int, layout: str = "zigzag") -> torch.Tensor:
    """Global token positions of this rank's rows, in buffer order."""
    if layout == "contiguous":
        Tc = T // N
        return torch.arange(rank * Tc, (rank + 1) * Tc)
    S = T // (2 * N)
    return torch.cat([torch.arange(rank * S, (rank + 1) * S),
                      torch.arange((2 * N - 1 - rank) * S, (2 * N - rank) * S)])


def shard(x: torch.Tensor, N: int, rank: int, layout: str = "zigzag") -> torch.Tensor:
    """This rank's rows of a full [B, H, T, ...] tensor, in buffer order."""
    return x[:, :, owned_positions(N, rank, x.shape[2], layout).to(x.device)].contiguous()


def block_attn_fold(q, k, v, step: Dict[str, int], causal: bool, acc, lse, out, stream=None) -> None:
    """One planned pair through rsa_block_attn_fold: q [B, H, q_rows, d] this
    rank's queries, k and v [B, H, kv_rows, d] the block held this round."""
    B, H, q_rows, d = q.shape
    kv_rows = k.shape[2]
    _call("rsa_block_attn_fold", q.data_ptr(), q_rows, k.data_ptr(), v.data_ptr(), kv_rows, _dt(q), B, H, d,
          step["q_row0"], step["q_pos"], step["q_len"], step["kv_row0"], step["kv_pos"], step["kv_len"],
          int(bool(causal)), step["fold"], acc.data_ptr() if acc is not None else None, lse.data_ptr(),
          out.data_ptr(), _stream(stream))


class KVRing:
    """Rotates a packed K/V block round the ranks of a process group: in round
    r this rank holds the block that started on rank (rank - r) mod N.  Two
    buffers: while the caller works on the current one, the next round's
    block is already being received into the other and the current one sent
    on (torch.distributed.batch_isend_irecv)."""

    def __init__(self, block: torch.Tensor, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.N = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.bufs = [block, torch.empty_like(block)]

    def _peer(self, r: int) -> int:
        # global rank of group rank r (point-to-point calls take global ranks)
        if self.group is None:
            return r
        return self.dist.get_global_rank(self.group, r)

    def rounds(self) -> Iterator[Tuple[int, int, torch.Tensor]]:
        """Yields (round, source rank, block).  The block must not be written,
        and is only valid until the generator resumes (the next receive reuses
        its buffer two rounds later; resume waits for this round's transfers)."""
        dist, N, i = self.dist, self.N, self.rank
        for r in range(N):
            cur = self.bufs[r % 2]
            nxt = self.bufs[(r + 1) % 2]
            works = []
            if r < N - 1:
                ops = [dist.P2POp(dist.isend, cur, self._peer((i + 1) % N), self.group),
                       dist.P2POp(dist.irecv, nxt, self._peer((i - 1) % N), self.group)]
                works = dist.batch_isend_irecv(ops)
            yield r, (i - r) % N, cur
            for w in works:
                w.wait()


def rank_ring_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, T: int, causal: bool,
                   layout: str = "zigzag", group=None, exchange: str = "device",
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """This rank's part of ring attention over a sequence of T tokens.

    q, k, v: [B, H, T/N, d] CUDA tensors holding this rank's tokens in buffer
    order (``shard``).  Returns (out [B, H, T/N, d] in q's dtype, lse
    [B, H, T/N] fp32) for the same rows.  Every rank of ``group`` calls it
    with the same T, causal and layout."""
    import torch.distributed as dist
    N = dist.get_world_size(group)
    rank = dist.get_rank(group)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, T/N, d] CUDA tensor")
    B, H, Tl, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or Tl * N != T:
        raise ValueError(f"q, k, v must be [B, H, T/N, d] with T/N = {T // N}")
    if exchange not in ("device", "host"):
        raise ValueError("exchange is 'device' or 'host'")
    plan = rank_ring_plan(N, rank, T, causal, layout)
    by_round: Dict[int, List[Dict[str, int]]] = {}
    for s in plan:
        by_round.setdefault(s["round"], []).append(s)
    st = torch.cuda.current_stream(q.device) if stream is None else stream
    with torch.cuda.stream(st):
        acc = torch.empty((B, H, Tl, d), dtype=torch.float32, device=q.device)
        lse = torch.empty((B, H, Tl), dtype=torch.float32, device=q.device)
        out = torch.empty_like(q)
        kv = torch.stack([k, v])
        if exchange == "device":
            ring = KVRing(kv, group)
            for r, _, blk in ring.rounds():
                for s in by_round.get(r, []):
                    block_attn_fold(q, blk[0], blk[1], s, causal, acc, lse, out, st)
        else:
            host = torch.empty(kv.shape, dtype=kv.dtype, pin_memory=True)
            host.copy_(kv)
            ring = KVRing(host, group)
            dev = [kv, torch.empty_like(kv)]
            for r, _, blk in ring.rounds():
                cur = dev[r % 2]
                if r > 0:
                    cur.copy_(blk, non_blocking=True)
                    # the host block is received into again two rounds on:
                    # the copy must be done before the generator resumes
                    done = torch.cuda.Event()
                    done.record(st)
                for s in by_round.get(r, []):
                    block_attn_fold(q, cur[0], cur[1], s, causal, acc, lse, out, st)
                if r > 0:
                    done.synchronize()
    return out, lse
