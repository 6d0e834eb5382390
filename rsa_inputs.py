"""Seeded synthetic inputs for blockwise ring self-attention.

This module only draws random tensors and picks query rows to check.  It holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle can
take their inputs from it without sharing any of the method.

Workloads (the five shapes the library is measured and checked on):

  tiny_fp32_causal     B=1 H=1 T=256     d=64  N=4  causal  fp32
  noncausal_bf16       B=2 H=8 T=4096    d=128 N=4  full    bf16
  page1_causal_bf16    B=8 H=64 T=32768  d=128 N=4  causal  bf16
  ragged_causal_bf16   B=1 H=32 T=100000 d=128 N=4  causal  bf16  (chunks of 25000)
  million_causal_bf16  B=1 H=8 T=1048576 d=128 N=16 causal  bf16
  decode_million_bf16  B=4 H=8 T=1048576 d=128 N=16 shards, 1 new token per
                       sequence against a million-token KV cache (decode)

The page-1 shape is the hidden state of "Sequence parallelism -- splitting
the token dimension across GPUs" (llmdaily day 58, section "Start with the
hidden-state tensor"): B=8, T=32768, hidden 8192 = 64 heads x 128.

Value recipes (drawn in fp32, then rounded to the tensor dtype):
  normal   Q, K, V ~ N(0, 1)
  wide     Q = 4 N(0,1), K = 4 N(0,1), V ~ U(-1, 1)     (score std ~16)
  outlier  Q, K, V ~ N(0, 1), then every key with index j % 4096 == 0 is
           multiplied by 8 (exact in bf16), key 0 included
Draw order is Q, K, V; each tensor is drawn one batch entry at a time so that
no single draw exceeds 2**31 elements.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    N: int
    causal: bool
    dtype: str          # "f32" or "bf16"
    recipe: str         # "normal", "wide" or "outlier"
    check: str          # "all" rows or "sample" rows
    q_len: int = 0      # decode: the newest q_len tokens query the whole cache (0: every token)

    @property
    def Tc(self) -> int:
        return self.T // self.N

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_fp32_causal", 1, 1, 256, 64, 4, True, "f32", "normal", "all"),
        Workload("noncausal_bf16", 2, 8, 4096, 128, 4, False, "bf16", "normal", "all"),
        Workload("page1_causal_bf16", 8, 64, 32768, 128, 4, True, "bf16", "normal", "sample"),
        Workload("ragged_causal_bf16", 1, 32, 100000, 128, 4, True, "bf16", "wide", "sample"),
        Workload("million_causal_bf16", 1, 8, 1048576, 128, 16, True, "bf16", "outlier", "sample"),
        Workload("decode_million_bf16", 4, 8, 1048576, 128, 16, True, "bf16", "normal", "sample", q_len=1),
    ]
}

OUTLIER_PERIOD = 4096
OUTLIER_SCALE = 8.0


def _draw(kind: str, shape, gen: torch.Generator, device) -> torch.Tensor:
    if kind == "randn":
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if kind == "rand":
        return torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    raise ValueError(kind)


def make_qkv(B: int, H: int, T: int, d: int, dtype: torch.dtype = torch.bfloat16,
             recipe: str = "normal", seed: int = 0, device="cpu"
             ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Draw contiguous [B, H, T, d] tensors Q, K, V with the given recipe."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    shape = (H, T, d)
    out = []
    for name in ("q", "k", "v"):
        t = torch.empty((B, H, T, d), dtype=dtype, device=dev)
        for b in range(B):
            if recipe == "normal":
                x = _draw("randn", shape, gen, dev)
            elif recipe == "wide":
                x = _draw("rand", shape, gen, dev) * 2.0 - 1.0 if name == "v" \
                    else _draw("randn", shape, gen, dev) * 4.0
            elif recipe == "outlier":
                x = _draw("randn", shape, gen, dev)
                if name == "k":
                    x[:, ::OUTLIER_PERIOD, :] *= OUTLIER_SCALE
            else:
                raise ValueError(f"unknown recipe {recipe!r}")
            t[b].copy_(x)
            del x
        out.append(t)
    return out[0], out[1], out[2]


def make_workload(w: Workload, seed: int = 0, device="cpu"):
    return make_qkv(w.B, w.H, w.T, w.d, w.torch_dtype, w.recipe, seed, device)


def sample_rows(w: Workload, n: int = 4096, seed: int = 1) -> np.ndarray:
    """Pick n query rows (b, h, t) to check on a workload too large for the oracle.

    Forced rows come first: t = 0, 1, 127, 128, every chunk start and end +-1,
    T-1, the ragged tails of 25000-token chunks, and the rows just after each
    outlier key; each forced t gets a random (b, h).  The rest are uniform.
    """
    rng = np.random.default_rng(seed)
    forced = {0, 1, 127, 128, w.T - 1}
    for i in range(w.N + 1):
        for dt in (-1, 0, 1):
            t = i * w.Tc + dt
            if 0 <= t < w.T:
                forced.add(t)
    if w.recipe == "outlier":
        for j in range(0, w.T, OUTLIER_PERIOD):
            for dt in (0, 1):
                if j + dt < w.T:
                    forced.add(j + dt)
    forced = sorted(forced)
    if len(forced) > n:
        forced = list(rng.choice(np.array(forced), size=n, replace=False))
    rows = np.empty((n, 3), dtype=np.int64)
    nf = len(forced)
    rows[:nf, 2] = forced
    rows[nf:, 2] = rng.integers(0, w.T, size=n - nf)
    rows[:, 0] = rng.integers(0, w.B, size=n)
    rows[:, 1] = rng.integers(0, w.H, size=n)
    return rows


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a bf16 CPU tensor, as a numpy uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def host_array(t: torch.Tensor):
    """(numpy array, dtype tag) of a CPU tensor as the oracle takes it."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return bf16_bits(t), "bf16"
    if t.dtype == torch.float32:
        return t.numpy(), "f32"
    if t.dtype == torch.float64:
        return t.numpy(), "f64"
    raise TypeError(t.dtype)
