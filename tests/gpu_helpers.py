"""Shared pieces of the GPU parity tests: tolerances and comparisons against
the oracle.  The bars are the ones the library is built to: fp32 max abs
error 1e-4; bf16 max abs 2e-2, relative Frobenius 5e-3, |lse| 1e-3."""
import numpy as np
import pytest
import torch

F32_ATOL = 1e-4
BF16_ATOL = 2e-2
BF16_RFRO = 5e-3
LSE_ATOL = 1e-3


def need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy() if t.dtype != torch.float64 else t.cpu().numpy()


def assert_close(out, lse, ref_out, ref_lse, dtype, what=""):
    """Compare GPU (out, lse) with the oracle's fp64 (ref_out, ref_lse)."""
    o = to64(out) if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    l = to64(lse) if isinstance(lse, torch.Tensor) else np.asarray(lse, np.float64)
    ro = np.asarray(ref_out, np.float64)
    rl = np.asarray(ref_lse, np.float64)
    assert o.shape == ro.shape, (o.shape, ro.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite outputs"
    # -inf lse (rows with no visible key) must agree exactly, with o = 0
    empty = np.isneginf(rl)
    np.testing.assert_array_equal(np.isneginf(l), empty, err_msg=f"{what}: empty rows differ")
    if empty.any():
        assert np.all(o[empty] == 0), f"{what}: empty rows must be zero"
    fin = ~empty
    err = np.abs(o - ro)
    if dtype == torch.float32:
        assert err.max(initial=0) <= F32_ATOL, f"{what}: max abs {err.max():.3e} > {F32_ATOL}"
        lerr = np.abs(l[fin] - rl[fin]).max(initial=0)
        assert lerr <= F32_ATOL, f"{what}: lse err {lerr:.3e}"
        return dict(max_abs=float(err.max(initial=0)), lse=float(lerr))
    rfro = np.linalg.norm(o - ro) / max(np.linalg.norm(ro), 1e-30)
    lerr = np.abs(l[fin] - rl[fin]).max(initial=0)
    assert err.max(initial=0) <= BF16_ATOL, f"{what}: max abs {err.max():.3e} > {BF16_ATOL}"
    assert rfro <= BF16_RFRO, f"{what}: rel Frobenius {rfro:.3e} > {BF16_RFRO}"
    assert lerr <= LSE_ATOL, f"{what}: lse err {lerr:.3e} > {LSE_ATOL}"
    return dict(max_abs=float(err.max(initial=0)), rel_fro=float(rfro), lse=float(lerr))


def qkv_cuda(B, H, T, d, dtype, recipe="normal", seed=0):
    """Seeded inputs drawn on the CPU (so the oracle sees the same values) and
    copied to the GPU."""
    import rsa_inputs
    q, k, v = rsa_inputs.make_qkv(B, H, T, d, dtype, recipe, seed, "cpu")
    return (q, k, v), (q.cuda(), k.cuda(), v.cuda())
