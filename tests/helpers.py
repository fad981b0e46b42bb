"""Shared test helpers: device transfer of storage-bit arrays and the parity tolerances.

Tolerances (the accuracy bar of this path):
  * hash ids, table rows: bit-exact;
  * kv (the projection alone): within 1 bf16 ulp of the correctly rounded value, plus the f32
    accumulation bound K * 2^-24 * sum_k |a_k w_k| (an f32 sum of K terms in any order is within
    that of the exact sum; it only matters where the sum cancels);
  * gate: within 2e-4 absolute;
  * out: |out - ref| <= ulp_bf16(ref) + 2e-4 * |value|, value being the shared value element
    added to that output (a 2e-4 gate error moves h + gate * value by at most 2e-4 * |value|,
    and the final bf16 rounding by at most one ulp).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle.numerics import bf16_to_f64, bf16_ulp, f64_to_bf16

GATE_ATOL = 2e-4
OUT_VALUE_RTOL = 2e-4


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy storage bits -> CUDA tensor with the same bytes (uint16 -> int16, uint64 -> int64)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint64:
        a = a.view(np.int64)
    elif a.dtype == np.bool_:
        a = a.astype(np.uint8)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    elif a.dtype == np.int16:
        a = a.view(np.uint16)
    return a


def empty_bf16(*shape) -> torch.Tensor:
    """bf16 buffer pre-filled with NaN bits, so an element the kernel never wrote shows up."""
    return torch.full(shape, 0x7FC1, dtype=torch.int16, device="cuda")


def kv_tolerance(kv_ref: np.ndarray, a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """ulp_bf16(ref) + K 2^-24 sum_k |a_k||w_k| for kv = a @ w^T (a: [M,K], w: [N,K] bits)."""
    K = a.shape[-1]
    mag = np.abs(bf16_to_f64(a)) @ np.abs(bf16_to_f64(w)).T
    return bf16_ulp(bf16_to_f64(kv_ref)) + K * 2.0 ** -24 * mag


def assert_kv_close(kv_gpu: np.ndarray, kv_ref: np.ndarray, a: np.ndarray, w: np.ndarray,
                    min_exact: float = 0.999):
    g, r = bf16_to_f64(kv_gpu), bf16_to_f64(kv_ref)
    assert not np.isnan(g).any(), "kv has unwritten / NaN elements"
    bad = np.abs(g - r) > kv_tolerance(kv_ref, a, w)
    assert not bad.any(), f"{bad.sum()} kv elements beyond 1 ulp; first {np.argwhere(bad)[:5]}"
    exact = (g == r).mean()
    assert exact >= min_exact, f"only {exact:.6f} of kv elements equal the correctly rounded value"


def assert_gate_close(g_gpu: np.ndarray, g_ref: np.ndarray):
    d = np.abs(g_gpu.astype(np.float64) - g_ref)
    assert d.max() <= GATE_ATOL, f"gate error {d.max():.3e} > {GATE_ATOL}"


def out_violations(out_gpu: np.ndarray, out_ref: np.ndarray, value: np.ndarray) -> np.ndarray:
    """Boolean mask of outputs beyond ulp(ref) + 2e-4 |value|. value: [M, dim] bits."""
    o, r = bf16_to_f64(out_gpu), bf16_to_f64(out_ref)
    v = np.abs(bf16_to_f64(value))[:, None, :]
    return ~(np.abs(o - r) <= bf16_ulp(r) + OUT_VALUE_RTOL * v)


def assert_out_close(out_gpu, out_ref, value):
    bad = out_violations(out_gpu, out_ref, value)
    assert not bad.any(), f"{bad.sum()} outputs beyond tolerance; first {np.argwhere(bad)[:5]}"


def kv_flips(kv_gpu: np.ndarray, a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Boolean mask of the kv elements where the GPU's bf16 value is not the correctly rounded
    one, after checking that each of them is a legitimate consequence of f32 accumulation: the
    GPU's value is the bf16 rounding of a sum within the f32-order bound K 2^-24 sum_k |a_k w_k|
    of the exact one, i.e. |gpu - exact| <= ulp(gpu) / 2 + that bound. Where the sum does not
    cancel this is a one-ulp flip at a rounding boundary; where it cancels, the bound (and the
    flip) can be a few ulps."""
    A, W = bf16_to_f64(a), bf16_to_f64(w)
    exact = A @ W.T
    ref = f64_to_bf16(exact)
    g = np.asarray(kv_gpu, dtype=np.uint16)
    flip = g != ref
    if flip.any():
        gv = bf16_to_f64(g[flip])
        bound = a.shape[-1] * 2.0 ** -24 * (np.abs(A) @ np.abs(W).T)[flip]
        far = np.abs(gv - exact[flip]) > bf16_ulp(gv) / 2 + bound
        assert not far.any(), f"{far.sum()} kv values not explained by f32 accumulation"
    return flip
