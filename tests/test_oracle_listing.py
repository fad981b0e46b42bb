"""Pin of the oracle's gate-and-add against the Engram listing's own arithmetic, run in torch.

The Engram listing (page "DeepSeek V4.1", class Engram, forward) is the one literal definition of
stage 4 on the pages. Its steps after the projection are evaluated here with torch CPU operations
in the precision the listing uses (key, value, weight and h in float32; the result cast back to
bf16), on generic data, and compared with the oracle's float64 gate_and_add. One comparison on
generic inputs checks together what the closed-form pins check one at a time on special inputs:
where eps enters (inside each rsqrt, beside the mean), that the norm is the mean over dim and
per (token, stream), the dim^-1/2 factor, the product q * k, the signed square root with its
1e-6 clamp, the mask, and that the value row is shared by the streams.

The torch evaluation below is written from what the listing computes, step by step, not copied
from it.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import engram as E
from oracle.numerics import bf16_to_f64, bf16_ulp


def _bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def listing_gate_and_add_torch(x_bits, kv_bits, q_bits, k_bits, mask, eps):
    """Stage 4 as the listing states it, in torch float32 (Engram listing, forward after wkv).

    x: bf16 bits [M, hc, dim]; kv: bf16 bits [M, dim * (hc + 1)]; q, k: bf16 bits [hc, dim];
    mask: bool [M] or None. Returns (out bf16 bits [M, hc, dim], gate float32 [M, hc]).
    """
    x = _bf16(x_bits)
    M, hc, dim = x.shape
    kv = _bf16(kv_bits).reshape(M, dim * (hc + 1))
    # split into hc keys and one value; keys as f32 [M, hc, dim]
    keys = kv[:, : hc * dim].float().reshape(M, hc, dim)
    val = kv[:, hc * dim:].float()
    wgt = _bf16(q_bits).float() * _bf16(k_bits).float()          # the learned product
    hf = x.float()
    # per (token, stream) reciprocal rms of the stream and of its key, eps inside each root
    inv_rms = torch.rsqrt(torch.mean(hf * hf, dim=-1) + eps) * \
        torch.rsqrt(torch.mean(keys * keys, dim=-1) + eps)
    a = torch.sum(hf * wgt * keys, dim=-1) * inv_rms * (dim ** -0.5)
    signed_root = torch.copysign(torch.sqrt(torch.clamp(torch.abs(a), min=1e-6)), a)
    g = torch.sigmoid(signed_root)
    if mask is not None:
        g = torch.where(torch.from_numpy(np.asarray(mask, dtype=bool))[:, None], g,
                        torch.zeros((), dtype=g.dtype))
    res = (hf + g[:, :, None] * val[:, None, :]).to(torch.bfloat16)
    return res.view(torch.int16).numpy().view(np.uint16), g.numpy()


def generic_inputs(geom, M, seed, x_dist):
    rng = np.random.default_rng(seed)
    x = synth.make_x((M, geom.hc_mult, geom.dim), rng, dist=x_dist)
    # a generic kv: bf16 values of a few magnitudes (not the projection of anything)
    kv = synth.f32_to_bf16_bits(
        (rng.standard_normal((M, geom.N)) * rng.choice([0.05, 0.5, 3.0], size=(M, 1)))
        .astype(np.float32))
    q, k = synth.make_qk(geom, rng)
    mask = rng.random(M) > 0.25
    mask[0] = True
    return x, kv, q, k, mask


@pytest.mark.parametrize("geom", [synth.TINY, synth.FULL], ids=["dim256", "dim5120"])
@pytest.mark.parametrize("eps", [1e-6, 1e-2])
@pytest.mark.parametrize("x_dist", ["normal", "student_t3"])
def test_oracle_gate_and_add_equals_the_listing_run_in_torch(geom, eps, x_dist):
    M = 40 if geom is synth.TINY else 6
    x, kv, q, k, mask = generic_inputs(geom, M, 901 + geom.dim + int(eps * 1e6), x_dist)
    out_t, gate_t = listing_gate_and_add_torch(x, kv, q, k, mask, eps)
    out_o, gate_o = E.gate_and_add(x, kv, q, k, mask, eps)
    # the listing's f32 sums over dim differ from the oracle's f64 ones by rounding only
    np.testing.assert_allclose(gate_o, gate_t.astype(np.float64), rtol=0, atol=1e-6)
    # both round h + gate * value to bf16 once at the end. Before that, the listing's f32
    # evaluation rounds the product and the sum (2^-24 each, relative) and carries its gate's
    # difference from the f64 one; these only show where h + gate * value cancels to far below
    # |h|, and otherwise move a result that sits at a rounding boundary by one ulp
    o, t = bf16_to_f64(out_o), bf16_to_f64(out_t)
    h = bf16_to_f64(x)
    v = bf16_to_f64(kv)[:, geom.hc_mult * geom.dim:][:, None, :]
    dg = np.abs(gate_o - gate_t.astype(np.float64))[:, :, None]
    bound = bf16_ulp(t) + dg * np.abs(v) + 2.0 ** -23 * (np.abs(h) + np.abs(gate_o)[:, :, None]
                                                         * np.abs(v))
    assert (np.abs(o - t) <= bound).all()
    assert (o == t).mean() > 0.999
    # masked tokens: gate exactly 0 on both sides
    assert (gate_t[~mask] == 0).all() and (gate_o[~mask] == 0).all()


def test_listing_run_catches_eps_outside_the_root():
    """The comparison above is sharp enough to see eps moved outside the mean (a plausible
    misreading of rsqrt(mean + eps)): the gates then differ by far more than 1e-6."""
    geom = synth.TINY
    x, kv, q, k, mask = generic_inputs(geom, 16, 77, "normal")
    eps = 1e-2
    _, gate_t = listing_gate_and_add_torch(x, kv, q, k, None, eps)
    h = bf16_to_f64(x)
    kvf = bf16_to_f64(kv)
    key = kvf[:, : geom.hc_mult * geom.dim].reshape(16, geom.hc_mult, geom.dim)
    w = bf16_to_f64(q) * bf16_to_f64(k)
    # the misreading, evaluated in f64: eps added to the rms instead of the mean square
    rstd = 1.0 / (np.sqrt((h * h).mean(-1)) + eps) / (np.sqrt((key * key).mean(-1)) + eps)
    a = (h * w * key).sum(-1) * rstd * geom.dim ** -0.5
    g_wrong = 1 / (1 + np.exp(-np.copysign(np.sqrt(np.maximum(np.abs(a), 1e-6)), a)))
    assert np.abs(g_wrong - gate_t).max() > 1e-4
