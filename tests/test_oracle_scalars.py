"""Pins of the oracle's scalar conversions against library routines.

bf16 rounding and the OCP e4m3 codec are checked against torch's CPU casts
(exhaustively for e4m3), SiLU against torch.nn.functional.silu in float64,
and the greedy argmax against planted maxima.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_round_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(7)
    vals = torch.cat([
        torch.randn(20000, generator=g),
        torch.randn(2000, generator=g) * 1e-38,      # bf16 subnormals
        torch.randn(2000, generator=g) * 1e30,
        torch.tensor([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-45]),
    ]).to(torch.float32)
    # exact halfway cases: 1 + 2^-8 (tie -> even 1.0), 1 + 3*2^-8 (-> up)
    ties = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8),
                         2 + 2 ** -7], dtype=torch.float32)
    vals = torch.cat([vals, ties])
    want = _bf16_bits(vals)
    got = oracle.bf16_from_double(vals.double().numpy())
    assert np.array_equal(got, want)


def test_bf16_specials():
    assert oracle.bf16_from_double(np.array([math.inf]))[0] == 0x7F80
    assert oracle.bf16_from_double(np.array([-math.inf]))[0] == 0xFF80
    assert oracle.bf16_from_double(np.array([1e39]))[0] == 0x7F80  # overflow
    nan = oracle.bf16_from_double(np.array([math.nan]))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


def test_bf16_to_double_exact_roundtrip():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_double(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double()
    both_nan = np.isnan(vals) & np.isnan(want.numpy())
    assert np.all((vals == want.numpy()) | both_nan)


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9                # smallest subnormal
    assert got[0x08] == 2.0 ** -6                # smallest normal


def test_e4m3_encode_every_bf16_value_in_range():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_double(bits)
    finite = np.isfinite(vals) & (np.abs(vals) < 448.0)
    v = vals[finite]
    got = oracle.e4m3_encode(v)
    want = torch.from_numpy(v).float().to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    # -0.0 and +0.0 both decode to zero; compare decoded values for zeros
    same = (got == want) | ((v == 0) & ((got & 0x7F) == 0) & ((want & 0x7F) == 0))
    assert same.all(), (v[~same][:5], got[~same][:5], want[~same][:5])


def test_e4m3_encode_saturates_and_rounds_half_even():
    assert oracle.e4m3_encode(np.array([448.0]))[0] == 0x7E
    assert oracle.e4m3_encode(np.array([1e6]))[0] == 0x7E
    assert oracle.e4m3_encode(np.array([-1e6]))[0] == 0xFE
    assert oracle.e4m3_encode(np.array([math.nan]))[0] == 0x7F
    # 1.0625 is halfway between 1.0 (mantissa 0, even) and 1.125 -> 1.0
    assert oracle.e4m3_decode(oracle.e4m3_encode(np.array([1.0625])))[0] == 1.0
    # 1.1875 is halfway between 1.125 (odd) and 1.25 (even) -> 1.25
    assert oracle.e4m3_decode(oracle.e4m3_encode(np.array([1.1875])))[0] == 1.25
    # subnormal halfway: 1.5 * 2^-9 -> 2 * 2^-9 (even)
    assert oracle.e4m3_decode(oracle.e4m3_encode(np.array([1.5 * 2 ** -9])))[0] == 2 * 2 ** -9
    # rounding up across the subnormal/normal boundary
    assert oracle.e4m3_encode(np.array([7.6 * 2 ** -9]))[0] == 0x08


def test_silu_matches_torch():
    z = np.concatenate([np.linspace(-30, 30, 1001), [0.0, 1e-300, 700.0]])
    want = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    got = oracle.silu(z)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([50.0]))[0] - 50.0) < 1e-15


def test_argmax_planted_and_ties():
    rng = np.random.default_rng(3)
    for n in (1, 2, 17, 151936):
        x = rng.standard_normal(n).astype(np.float32)
        i = int(rng.integers(0, n))
        x[i] = 100.0
        assert oracle.argmax(x) == i
    x = np.zeros(10, np.float32)
    x[[3, 7]] = 5.0
    assert oracle.argmax(x) == 3            # ties -> lowest index
    x = np.full(8, -np.inf, np.float32)
    x[5] = -1e30
    assert oracle.argmax(x) == 5
