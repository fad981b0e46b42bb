"""Pins for oracle.numerics: bf16 / e4m3 / e8m0 against library casts, closed forms, page facts."""
import numpy as np
import pytest
import torch

from oracle.numerics import (bf16_to_f64, bf16_ulp, e4m3_to_f64, e8m0_to_f64, f32_to_e4m3_rne,
                             f32_to_e8m0_rne, f64_to_bf16)


def torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    ours = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    ref = torch_e4m3_values()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    assert np.isnan(ours[[0x7F, 0xFF]]).all() and np.isnan(ours).sum() == 2


def test_e4m3_decode_landmarks(page_facts):
    v = e4m3_to_f64(np.array([0x7E, 0xFE, 0x01, 0x08, 0x38, 0x00, 0x80], dtype=np.uint8))
    assert v[0] == page_facts["e4m3_saturation"] == 448.0 and v[1] == -448.0
    assert v[2] == 2.0 ** -9 and v[3] == 2.0 ** -6 and v[4] == 1.0
    assert v[5] == 0.0 and not np.signbit(v[5]) and np.signbit(v[6])


def test_e4m3_values_exact_in_bf16_under_block_scales():
    # "e4m3 values are exactly representable in bf16" (Module engram, stage 2), also after a
    # power-of-two block scale in 2^[-4, 4]
    vals = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    vals = vals[~np.isnan(vals)]
    for s in range(-4, 5):
        x = vals * 2.0 ** s
        np.testing.assert_array_equal(bf16_to_f64(f64_to_bf16(x)), x)


def test_f64_to_bf16_matches_torch_on_binary32_values():
    # For values exact in binary32, a single rounding to bf16 is what torch's cast computes.
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),     # subnormal range
        np.clip(rng.standard_normal(20000) * 3e38, -3.4e38, 3.4e38).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf], dtype=np.float32),
    ])
    # exact ties: bf16 value + half a bf16 step
    t = bf16_to_f64(rng.integers(0, 0x7F00, size=20000).astype(np.uint16))
    x = np.concatenate([x, (t + bf16_ulp(t) / 2).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(f64_to_bf16(x.astype(np.float64)), ref)


def test_f64_to_bf16_rounds_once():
    # 1 + 2^-8 + 2^-40 lies just above the tie between 1 and 1 + 2^-7: the single rounding goes
    # up; a detour through binary32 would have dropped 2^-40 and tied to even (1.0).
    assert f64_to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert f64_to_bf16(np.array([1 + 2.0 ** -8]))[0] == 0x3F80          # tie -> even
    assert f64_to_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82      # tie -> even (up)
    assert f64_to_bf16(np.array([-(1 + 2.0 ** -8 + 2.0 ** -40)]))[0] == 0xBF81
    assert f64_to_bf16(np.array([np.nan]))[0] & 0x7FFF == 0x7FC0


def test_bf16_ulp_closed_form():
    assert bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([1.99]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([-3.0]))[0] == 2.0 ** -6
    assert bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133


def test_f32_to_e4m3_matches_torch_inside_range():
    # torch's cast is RNE; inside [-448, 448] it must agree with ours code for code.
    rng = np.random.default_rng(2)
    vals = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    vals = np.sort(vals[~np.isnan(vals)])
    mids = (vals[1:] + vals[:-1]) / 2                     # exact ties between neighbours
    x = np.concatenate([vals, mids, rng.uniform(-448, 448, 100000),
                        rng.standard_normal(100000) * 0.01]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = f32_to_e4m3_rne(x)
    # +-0 may differ only in the sign of zero; compare values plus the sign bit
    np.testing.assert_array_equal(ours, ref)


def test_f32_to_e4m3_saturates_and_hand_cases(page_facts):
    sat = page_facts["e4m3_saturation"]
    x = np.array([449.0, 464.0, 465.0, 1e6, np.inf, -500.0], dtype=np.float64)
    np.testing.assert_array_equal(e4m3_to_f64(f32_to_e4m3_rne(x)), [sat, sat, sat, sat, sat, -sat])
    # 2^-10 is the tie between 0 and 2^-9 -> even code 0; 1.5*2^-9 ties 2^-9 / 2^-8 -> code 2
    y = e4m3_to_f64(f32_to_e4m3_rne(np.array([2.0 ** -10, 1.5 * 2.0 ** -9, 0.75 * 2.0 ** -9])))
    np.testing.assert_array_equal(y, [0.0, 2.0 ** -8, 2.0 ** -9])
    assert f32_to_e4m3_rne(np.array([np.nan]))[0] == 0x7F


def test_f32_to_e8m0_ties_to_even_exponent(page_facts):
    # "nearest exponent, ties (exactly 1.5 * 2^e) to the even exponent"
    x = np.array([1.5, 3.0, 0.75, 6.0, 12.0, 0.375, 1.5 * 2.0 ** 20, 1.5 * 2.0 ** -21])
    want = np.array([1.0, 4.0, 1.0, 4.0, 16.0, 0.25, 2.0 ** 20, 2.0 ** -20])
    np.testing.assert_array_equal(e8m0_to_f64(f32_to_e8m0_rne(x)), want)


def test_f32_to_e8m0_matches_torch_off_ties():
    # Off the ties torch's float8_e8m0fnu cast is the nearest power of two; it rounds ties up,
    # which the page's rule overrides, so ties are excluded here.
    rng = np.random.default_rng(3)
    x = np.exp2(rng.uniform(-40, 40, 200000)).astype(np.float32).astype(np.float64)
    m, _ = np.frexp(x)
    x = x[2 * m != 1.5]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e8m0fnu).view(torch.uint8).numpy()
    np.testing.assert_array_equal(f32_to_e8m0_rne(x), ref)


def test_e8m0_decode():
    np.testing.assert_array_equal(e8m0_to_f64(np.array([127, 128, 123, 131, 0], dtype=np.uint8)),
                                  [1.0, 2.0, 1 / 16, 16.0, 2.0 ** -127])
    assert np.isnan(e8m0_to_f64(np.array([255], dtype=np.uint8)))[0]
