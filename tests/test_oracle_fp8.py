"""Pins of the oracle's fp8 input decoding (OCP 8-bit floating point, E4M3):
every one of the 256 codes against torch's float8_e4m3fn conversion (an
independent library routine), closed-form values of the format, the bf16
rounding against torch's float32 -> bfloat16 conversion, and a planted
wrong exponent bias that the library pin must catch."""
import math

import numpy as np
import torch

from oracle import csbp_oracle as O


def test_all_256_codes_match_the_library_decoding():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([O.e4m3_value(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2                      # S.1111.111 only
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))  # -0.0 at 0x80


def test_closed_form_values_of_the_format():
    want = {0x00: 0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0,
            0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0xB8: -1.0,
            0x30: 0.5,
            0x4B: 5.5}  # 0 1001 011: exponent 9 - 7 = 2, mantissa 3/8 -> 1.375 * 4
    for code, v in want.items():
        assert O.e4m3_value(code) == v, hex(code)
    assert math.copysign(1.0, O.e4m3_value(0x80)) == -1.0 and O.e4m3_value(0x80) == 0.0
    assert math.isnan(O.e4m3_value(0x7F)) and math.isnan(O.e4m3_value(0xFF))


def test_bf16_rounding_matches_the_library_conversion():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(100000, generator=g) * torch.exp(4 * torch.randn(100000, generator=g))
    # exact ties: values halfway between two bf16 numbers
    base = torch.randn(1000, generator=g).to(torch.bfloat16).to(torch.float32)
    ties = base * (1 + 2.0 ** -8 * torch.sign(base).abs())
    x = torch.cat([x, ties, torch.tensor([0.0, -0.0, float("inf"), float("-inf"), 3.4e38])])
    want = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_bf16(x.numpy())
    assert np.array_equal(got, want)


def test_scaled_decoding_rounds_the_fp32_product_once_more_to_bf16():
    codes = np.arange(256, dtype=np.uint8)
    for scale in (1.0, 2.0 ** -5, 128.0, 0.3, -1.7):
        got = O.e4m3_to_bf16(codes, scale)
        lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
        want = (lib.to(torch.float32) * torch.tensor(scale, dtype=torch.float32)).to(
            torch.bfloat16).to(torch.float64).numpy()
        nan = np.isnan(want)
        assert np.array_equal(nan, np.isnan(got))
        assert np.array_equal(got[~nan], want[~nan]), scale


def test_pin_catches_a_planted_exponent_bias(monkeypatch):
    good = O.e4m3_value

    def bias8(code):
        v = good(code)
        return v if math.isnan(v) else v / 2.0  # bias 8 instead of 7

    monkeypatch.setattr(O, "e4m3_value", bias8)
    try:
        test_all_256_codes_match_the_library_decoding()
    except AssertionError:
        return
    raise AssertionError("a wrong exponent bias passed the library pin")
