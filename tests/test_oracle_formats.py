"""Pins for the oracle's number-format conversions.

The oracle writes fp16/bf16 rounding from the IEEE definitions; here it is held
against two independent implementations: numpy's float16 conversion and
torch's bfloat16 conversion, on every 16-bit pattern (widening) and on
millions of fp32 patterns chosen to hit every rounding case (narrowing)."""
import numpy as np
import pytest
import torch

import oracle


def _fp32_probe_patterns(n_random=1 << 20, seed=0):
    rng = np.random.default_rng(seed)
    pats = [rng.integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32)]
    # every fp16 value and the midpoints to both neighbours (ties), in fp32
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    hv = h.view(np.float16).astype(np.float32)
    hv = hv[np.isfinite(hv)]
    with np.errstate(over="ignore"):
        nxt = np.nextafter(hv.astype(np.float16), np.float16(np.inf)).astype(np.float32)
    mid = (hv.astype(np.float64) + nxt.astype(np.float64)) / 2
    mid = mid[np.isfinite(mid)].astype(np.float32)  # exact: midpoints of fp16 fit fp32
    pats.append(hv.view(np.uint32))
    pats.append(mid.view(np.uint32))
    pats.append(np.nextafter(mid, np.float32(np.inf)).view(np.uint32))
    pats.append(np.nextafter(mid, np.float32(-np.inf)).view(np.uint32))
    # every bf16 value and the fp32 patterns around bf16 ties
    b = (np.arange(1 << 16, dtype=np.uint32) << 16)
    pats.append(b)
    pats.append(b | 0x8000)
    pats.append(b | 0x7fff)
    pats.append(b | 0x8001)
    # specials
    pats.append(np.array([0, 0x80000000, 0x7f800000, 0xff800000, 0x7fc00000, 0x477fefff,
                          0x477ff000, 0x477fe000, 0x38800000, 0x33000000, 0x33000001,
                          0x00000001, 0x007fffff, 0x7f7fffff], np.uint32))
    return np.concatenate(pats).view(np.float32)


def test_f32_to_f16_matches_numpy():
    x = _fp32_probe_patterns()
    got = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    # NaN stays NaN with the sign kept
    g = got[nan]
    assert np.all((g & 0x7c00) == 0x7c00) and np.all((g & 0x3ff) != 0)


def test_f32_to_bf16_matches_torch():
    x = _fp32_probe_patterns(seed=1)
    got = oracle.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    g = got[nan]
    assert np.all((g & 0x7f80) == 0x7f80) and np.all((g & 0x7f) != 0)


def test_f16_widening_all_patterns():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_f64(h)
    ref = h.view(np.float16).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_widening_all_patterns():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_bits_to_f64(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("x,bits", [(65504.0, 0x7bff), (65519.99, 0x7bff), (65520.0, 0x7c00),
                                    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),
                                    (1.5 * 2.0 ** -24, 0x0002), (1.0 + 2.0 ** -11, 0x3c00),
                                    (1.0 + 3 * 2.0 ** -11, 0x3c02), (-2.0, 0xc000)])
def test_f16_rounding_worked_cases(x, bits):
    """Round-half-to-even at the overflow edge, in the subnormal range and at ties."""
    assert int(oracle.f32_to_f16_bits(np.array([x], np.float32))[0]) == bits
