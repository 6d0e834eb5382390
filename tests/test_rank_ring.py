"""Host logic of the multi-rank ring (no GPU): each rank's pair list from
rsa_rank_ring_plan, and the rotation of K/V blocks round gloo ranks.

Pages: "Sequence parallelism -- splitting the token dimension across GPUs"
(llmdaily, day 58), "A better mental model: move blocks past the queries"
(GPU i holds the block of GPU (i - r) mod N in round r+1) and "Causal
attention gives us another optimization" (blocks of keys that all come
after their queries are skipped)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT, read_golden

from context_attention_rsa_gb300 import rank_ring as rr


def coverage(N, T, causal, layout):
    """How often each (query position, key position) is computed over all ranks."""
    cov = np.zeros((T, T), dtype=np.int64)
    for rank in range(N):
        mine = rr.owned_positions(N, rank, T, layout).numpy()
        for s in rr.rank_ring_plan(N, rank, T, causal, layout):
            theirs = rr.owned_positions(N, s["src"], T, layout).numpy()
            qp = mine[s["q_row0"]:s["q_row0"] + s["q_len"]]
            kp = theirs[s["kv_row0"]:s["kv_row0"] + s["kv_len"]]
            # rows and positions agree, and pieces are contiguous in position
            assert np.array_equal(qp, np.arange(s["q_pos"], s["q_pos"] + s["q_len"]))
            assert np.array_equal(kp, np.arange(s["kv_pos"], s["kv_pos"] + s["kv_len"]))
            if causal:
                assert kp[0] <= qp[-1], "a block with every key after every query was kept"
                sub = np.less_equal.outer(kp, qp).T
            else:
                sub = np.ones((len(qp), len(kp)), dtype=bool)
            cov[np.ix_(qp, kp)] += sub
    return cov


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
def test_plans_cover_every_allowed_pair_once(N, causal, layout):
    T = 2 * N * 4
    cov = coverage(N, T, causal, layout)
    want = np.tril(np.ones((T, T), dtype=np.int64)) if causal else np.ones((T, T), dtype=np.int64)
    np.testing.assert_array_equal(cov, want)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_rounds_follow_the_printed_ring_table(layout):
    # the page's table: in round r+1 GPU i holds the KV block of GPU (i - r) mod N
    want = {}
    for rnd1, gpu, kv in (map(int, r) for r in read_golden("ring_table_n4.txt")):
        want[(rnd1 - 1, gpu)] = kv
    checked = set()
    for rank in range(4):
        for s in rr.rank_ring_plan(4, rank, 64, False, layout):
            if (s["round"], rank) in want:  # the page prints rounds 1-3
                assert s["src"] == want[(s["round"], rank)]
                checked.add((s["round"], rank))
    assert checked == set(want)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("N", [1, 2, 4, 7])
def test_fold_modes_and_round_order(N, layout):
    for rank in range(N):
        plan = rr.rank_ring_plan(N, rank, 2 * N * 8, True, layout)
        rounds = [s["round"] for s in plan]
        assert rounds == sorted(rounds)
        for s in plan:
            assert s["src"] == (rank - s["round"]) % N
        for q0 in sorted({s["q_row0"] for s in plan}):
            folds = [s["fold"] for s in plan if s["q_row0"] == q0]
            if len(folds) == 1:
                assert folds == [rr.FOLD_ONLY]
            else:
                assert folds[0] == rr.FOLD_FIRST and folds[-1] == rr.FOLD_LAST
                assert all(f == rr.FOLD_MERGE for f in folds[1:-1])


@pytest.mark.parametrize("N", [2, 4, 8])
def test_zigzag_balances_causal_work_and_contiguous_does_not(N):
    T = 2 * N * 16

    def work(layout):
        # allowed (query, key) pairs per rank and round
        w = np.zeros((N, N), dtype=np.int64)
        for rank in range(N):
            mine = rr.owned_positions(N, rank, T, layout).numpy()
            for s in rr.rank_ring_plan(N, rank, T, True, layout):
                theirs = rr.owned_positions(N, s["src"], T, layout).numpy()
                qp = mine[s["q_row0"]:s["q_row0"] + s["q_len"]]
                kp = theirs[s["kv_row0"]:s["kv_row0"] + s["kv_len"]]
                w[rank, s["round"]] += np.less_equal.outer(kp, qp).sum()
        return w
    z = work("zigzag")
    assert (z == z[0]).all(), z                      # every rank, every round: the same work
    assert (z[:, 1:] == 2 * (T // (2 * N)) ** 2).all()  # two full S x S blocks after round 0
    c = work("contiguous").sum(axis=1)
    Tc = T // N
    # contiguous chunks: rank i needs i full blocks and one diagonal block
    assert c.tolist() == [i * Tc * Tc + Tc * (Tc + 1) // 2 for i in range(N)]
    assert z.sum() == c.sum() == T * (T + 1) // 2


def test_plan_rejects_bad_arguments():
    lib = __import__("context_attention_rsa_gb300").load()
    import ctypes
    n = ctypes.c_int(0)
    buf = (ctypes.c_int64 * 90)()
    assert lib.rsa_rank_ring_plan(4, 0, 100, 1, 1, buf, 10, ctypes.byref(n)) == 1  # 2N does not divide T
    assert lib.rsa_rank_ring_plan(4, 4, 64, 1, 1, buf, 10, ctypes.byref(n)) == 1   # rank out of range
    assert lib.rsa_rank_ring_plan(4, 0, 64, 1, 2, buf, 10, ctypes.byref(n)) == 1   # unknown layout
    assert lib.rsa_rank_ring_plan(4, 3, 64, 1, 1, buf, 1, ctypes.byref(n)) == 1 and n.value == 9  # cap too small
    assert lib.rsa_rank_ring_plan(4, 3, 64, 1, 0, buf, 10, ctypes.byref(n)) == 0 and n.value == 4


# --- the rotation of K/V blocks on gloo ranks -----------------------------------------

def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rotate_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    from context_attention_rsa_gb300 import rank_ring
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # a packed [2, B, H, T/N, d] block whose every value names its origin
        blk = torch.full((2, 1, 2, 8, 4), float(rank)) + torch.arange(8.0).view(1, 1, 1, 8, 1) * 1000
        seen = []
        for r, src, cur in rank_ring.KVRing(blk, None).rounds():
            vals = (cur - torch.arange(8.0).view(1, 1, 1, 8, 1) * 1000).unique().tolist()
            seen.append((r, src, vals))
        out[rank] = seen
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_kv_blocks_rotate_round_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rotate_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn",
                           join=True)
        res = dict(out)
    for rank in range(world):
        assert [r for r, _, _ in res[rank]] == list(range(world))
        for r, src, vals in res[rank]:
            assert src == (rank - r) % world
            assert vals == [float(src)]  # the block held is exactly the source rank's, untouched
