"""The multi-rank ring on the GPU (rsa_block_attn_fold per planned pair, K/V
blocks exchanged between ranks), checked against the oracle.

Every rank here runs as its own process on the one GPU of the box, and the
blocks travel through gloo as page-locked host copies (exchange="host"): the
ranks' kernels never wait on one another, only their host threads wait for
the exchange.  On a node with one GPU per rank the same code sends device
tensors through NCCL (exchange="device"); that transport, and its NVLink
throughput, are not measured here."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT

pytestmark = pytest.mark.gpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, case, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import rsa_inputs
    from context_attention_rsa_gb300 import rank_ring
    B, H, T, d, causal, layout, dtype = case
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        q, k, v = rsa_inputs.make_qkv(B, H, T, d, dtype, "normal", 7, "cpu")
        ql, kl, vl = (rank_ring.shard(t, world, rank, layout).cuda() for t in (q, k, v))
        o, l = rank_ring.rank_ring_attn(ql, kl, vl, T, causal, layout=layout, exchange="host")
        torch.cuda.synchronize()
        o2, l2 = rank_ring.rank_ring_attn(ql, kl, vl, T, causal, layout=layout, exchange="host")  # again: same
        torch.cuda.synchronize()
        out[rank] = (o.float().cpu(), l.cpu(), bool(torch.equal(o, o2) and torch.equal(l, l2)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


CASES = [
    (2, (1, 4, 2048, 128, True, "zigzag", torch.bfloat16)),
    (2, (1, 4, 2048, 128, True, "contiguous", torch.bfloat16)),
    (3, (2, 2, 1536, 128, False, "zigzag", torch.bfloat16)),
    (3, (1, 2, 768, 64, True, "zigzag", torch.bfloat16)),
    (2, (1, 2, 512, 64, True, "zigzag", torch.float32)),
    (1, (1, 2, 1000, 128, True, "contiguous", torch.bfloat16)),
]


@pytest.mark.parametrize("world,case", CASES, ids=[f"n{w}-{c[5]}-{'causal' if c[4] else 'full'}-{str(c[6])[6:]}-d{c[3]}"
                                                   for w, c in CASES])
def test_rank_ring_matches_oracle(world, case):
    import oracle
    import rsa_inputs
    from context_attention_rsa_gb300 import rank_ring
    from gpu_helpers import assert_close, need_cuda
    need_cuda()
    B, H, T, d, causal, layout, dtype = case
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), case, out), nprocs=world, start_method="spawn",
                           join=True)
        res = dict(out)
    q, k, v = rsa_inputs.make_qkv(B, H, T, d, dtype, "normal", 7, "cpu")
    ro, rl = oracle.attention(q, k, v, causal)
    o = np.zeros((B, H, T, d))
    l = np.zeros((B, H, T))
    for rank in range(world):
        pos = rank_ring.owned_positions(world, rank, T, layout).numpy()
        o[:, :, pos] = res[rank][0].double().numpy()
        l[:, :, pos] = res[rank][1].double().numpy()
        assert res[rank][2], "a second call gave a different result"
    assert_close(o, l, ro, rl, dtype, what=f"rank ring {world} {layout}")
