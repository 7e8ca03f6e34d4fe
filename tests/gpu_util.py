"""Helpers for the GPU parity tests: move seeded inputs to the device, call the library through its binding,
compare against the oracle with the tolerances stated below.

Tolerances (derived from the arithmetic; the kernels compute in fp32, the oracle in fp64):

* fp32 values (state, cache, o in fp32):  max|x - ref| <= 1e-4 * max|ref| over the compared tensor.
* bf16 values stored from fp32 (o, or a bf16 cache / pool) against the oracle's fp64 value rounded the same
  way: |x - ref| <= 1 bf16 ulp(ref) + 1e-4 * max|ref| element-wise (a 1-ulp flip happens where the fp32 and
  fp64 values straddle a rounding midpoint), max|x - ref| <= 2e-2, and at least 95 % bit-identical (a
  rounding mode other than nearest-even would fail this).
* bf16 o against the oracle's unrounded fp64 o: |x - ref| <= 2^-8 |ref| + 1e-4 * max|ref|, max <= 2e-2.
* indexing, padding skip and commit: bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_linear_mtp_gb300 as gdn

CANARY_F32 = 0x7FC0DEAD
CANARY_BF16 = 0x7FDE


def dev(x: np.ndarray, dtype: str = None) -> torch.Tensor:
    """numpy storage array -> CUDA tensor (uint16 = bf16 bits)."""
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy storage array (bf16 as uint16 bits)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def storage_to_f64(x: np.ndarray) -> np.ndarray:
    return bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def canary(shape, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.full(shape, CANARY_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return torch.full(shape, CANARY_F32, dtype=torch.int32, device="cuda").view(torch.float32)


def is_canary(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return x == CANARY_BF16
    return x.view(np.uint32) == CANARY_F32


class Dev:
    """Device copies of one workload's arrays."""

    def __init__(self, x: dict):
        self.t = {k: dev(v) for k, v in x.items()}

    def __getitem__(self, k):
        return self.t[k]


def run_verify(w, t: Dev, cache: bool, err=None, o=None, cache_buf=None, stream=None):
    B, T, HV, DV, DK = t["q"].shape[0], w.T, w.HV, w.DV, w.DK
    if o is None:
        o = canary((B, T, HV, DV), w.out_dtype)
    if cache and cache_buf is None:
        cache_buf = canary((B, T, HV, DV, DK), w.state_dtype)
    gdn.gdn_mtp_verify(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"], o,
                       cache_buf if cache else None, err, scale=w.scale, l2_eps=w.l2_eps, stream=stream)
    return o, (cache_buf if cache else None)


def run_decode(w, t: Dev, pool: torch.Tensor, err=None, o=None):
    B, T, HV, DV = t["q"].shape[0], w.T, w.HV, w.DV
    if o is None:
        o = canary((B, T, HV, DV), w.out_dtype)
    gdn.gdn_decode(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], pool, t["indices"], o, err,
                   scale=w.scale, l2_eps=w.l2_eps)
    return o


# ---- comparisons ------------------------------------------------------------------------------------------
def assert_f32_close(x, ref, what="", rel=1e-4):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, (what, x.shape, ref.shape)
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    scale = max(np.abs(ref).max(), 1e-30)
    err = np.abs(x - ref).max()
    assert err <= rel * scale, f"{what}: max|x-ref| = {err:.3e} > {rel:g} * {scale:.3e}"
    return err / scale


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits; subnormal spacing 2^-133)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def assert_bf16_stored_close(x_bits, ref_bits, what="", min_exact=0.95):
    """bf16 result vs the oracle's fp64 value rounded to bf16 (both as bit patterns)."""
    x_bits = np.asarray(x_bits)
    ref_bits = np.asarray(ref_bits)
    assert x_bits.shape == ref_bits.shape, (what, x_bits.shape, ref_bits.shape)
    x, ref = bf16_to_f64(x_bits), bf16_to_f64(ref_bits)
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    scale = np.abs(ref).max()
    d = np.abs(x - ref)
    bound = bf16_ulp(ref) + 1e-4 * scale
    bad = d > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1 ulp + 1e-4*max (worst {d.max():.3e})"
    assert d.max() <= 2e-2, f"{what}: max-abs {d.max():.3e} > 2e-2"
    exact = float((x_bits == ref_bits).mean()) if x_bits.size else 1.0
    assert exact >= min_exact, f"{what}: only {exact:.4f} bit-identical"
    return exact


def assert_bf16_out_close(x_bits, ref, what=""):
    """bf16 result vs the oracle's unrounded fp64 value."""
    x = bf16_to_f64(np.asarray(x_bits))
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    scale = np.abs(ref).max()
    d = np.abs(x - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * scale
    bad = d > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond the bf16 rounding bound (worst {d.max():.3e})"
    assert d.max() <= 2e-2, f"{what}: max-abs {d.max():.3e} > 2e-2"
    return float(d.max())


def check_o(w, o_gpu: np.ndarray, o_ref: np.ndarray, what="o"):
    if w.out_dtype == "bf16":
        return assert_bf16_out_close(o_gpu, o_ref, what)
    return assert_f32_close(o_gpu, o_ref, what)


def check_state(w, s_gpu: np.ndarray, s_ref: np.ndarray, what="state"):
    """Stored states (cache / pool) in the state dtype, both sides rounded at the same point."""
    if w.state_dtype == "bf16":
        return assert_bf16_stored_close(s_gpu, s_ref, what)
    return assert_f32_close(s_gpu, s_ref, what)
