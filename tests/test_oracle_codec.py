"""Pins for the oracle's block codec and fp16 conversion (CPU only).

Each test checks the oracle against something other than itself: the byte
table printed on the reference page, hand-derived blocks, numpy's IEEE fp16
conversion, a brute-force search over the integer codes, or the error bound
that follows from the format definition.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

FMT = {"f16": oracle.FMT_F16, "q8_0": oracle.FMT_Q8_0, "q4_0": oracle.FMT_Q4_0}


def _parse(s: str) -> float:
    s = s.strip()
    if s == "-0":
        return -0.0
    if "*2^" in s:
        a, e = s.split("*2^")
        return float(Fraction(int(a)) * Fraction(2) ** int(e))
    return float(Fraction(s))


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_block_sizes_match_the_modes_table():
    # "Blocked 8-bit, one f16 scale per 32 elements (34 bytes)"; 4-bit packs into 18 bytes.
    assert oracle.block_bytes(oracle.FMT_Q8_0) == 34
    assert oracle.block_bytes(oracle.FMT_Q4_0) == 18
    assert oracle.block_bytes(oracle.FMT_F16) == 64


def test_bytes_per_position_and_session_totals(golden_dir):
    g = _golden(golden_dir, "kv_bytes_per_position.json")
    n = g["elements_per_tensor_per_layer"]
    for m in g["modes"]:
        per_pos = n // 32 * (oracle.block_bytes(FMT[m["k"]]) + oracle.block_bytes(FMT[m["v"]]))
        assert per_pos == m["bytes_per_position"], m
        gb = per_pos * g["layers"] * g["session_tokens"] / 1e9
        assert round(gb, 2) == m["session_gb"], (m, gb)
    # ratio fp16 : Q8_0 : Q4_0 per element = 2 : 1.0625 : 0.5625
    per_elem = [oracle.block_bytes(f) / 32 for f in (oracle.FMT_F16, oracle.FMT_Q8_0, oracle.FMT_Q4_0)]
    assert per_elem == [2.0, 1.0625, 0.5625]


def _cases(golden_dir, fmt_name):
    return _golden(golden_dir, "codec_blocks.json")[fmt_name]


def _block_input(case):
    if "fill" in case:
        xs = [_parse(case["fill"])] * 32
        q = [case["q_fill"]] * 32
    else:
        xs = [_parse(s) for s in case["x"]]
        q = case["q"]
    assert len(xs) == 32 and len(q) == 32
    x16 = np.array(xs, dtype=np.float16)
    # every fixture value must be exactly representable in fp16
    assert np.array_equal(x16.astype(np.float64), np.array(xs, dtype=np.float64))
    assert np.array_equal(np.signbit(x16), np.signbit(np.array(xs)))
    return x16, np.array(q, dtype=np.int64)


@pytest.mark.parametrize("name", ["zeros", "power_of_two_scale_ties_away", "fp16_rounding_of_scale",
                                  "scale_underflows_to_zero", "subnormal_scale"])
def test_q8_0_hand_derived_blocks(golden_dir, name):
    case = next(c for c in _cases(golden_dir, "q8_0") if c["name"] == name)
    x16, q = _block_input(case)
    blk = oracle.quantize(oracle.FMT_Q8_0, x16[None, :])[0, 0]
    assert blk.shape == (34,)
    scale_bits = int(blk[0]) | (int(blk[1]) << 8)
    assert scale_bits == int(case["scale_bits"], 16), hex(scale_bits)
    got_q = blk[2:].view(np.int8).astype(np.int64)
    assert np.array_equal(got_q, q), (got_q, q)
    # dequantised value = fp16(scale) * q, the scale read by numpy's fp16 decoder
    d = np.array([scale_bits], dtype=np.uint16).view(np.float16).astype(np.float64)[0]
    assert np.array_equal(oracle.dequantize(oracle.FMT_Q8_0, blk[None, :]), d * q)


@pytest.mark.parametrize("name", ["zeros", "negative_max_first_trunc_and_clamp", "positive_max_first",
                                  "negative_max_first_mirror", "scale_underflows_to_negative_zero",
                                  "subnormal_scale"])
def test_q4_0_hand_derived_blocks(golden_dir, name):
    case = next(c for c in _cases(golden_dir, "q4_0") if c["name"] == name)
    x16, q = _block_input(case)
    blk = oracle.quantize(oracle.FMT_Q4_0, x16[None, :])[0, 0]
    assert blk.shape == (18,)
    scale_bits = int(blk[0]) | (int(blk[1]) << 8)
    assert scale_bits == int(case["scale_bits"], 16), hex(scale_bits)
    packed = blk[2:].astype(np.int64)
    # byte k holds element k in the low nibble and element k+16 in the high nibble
    assert np.array_equal(packed, q[:16] | (q[16:] << 4)), (packed, q)
    d = np.array([scale_bits], dtype=np.uint16).view(np.float16).astype(np.float64)[0]
    deq = oracle.dequantize(oracle.FMT_Q4_0, blk[None, :])
    assert np.array_equal(deq, (q - 8) * d)


def test_f16_mode_is_identity():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 128), dtype=np.float32).astype(np.float16)
    blk = oracle.quantize(oracle.FMT_F16, x)
    assert blk.shape == (5, 4, 64)
    assert np.array_equal(blk.reshape(5, 256).view(np.uint16), x.view(np.uint16))
    assert np.array_equal(oracle.dequantize(oracle.FMT_F16, blk), x.astype(np.float64))


# ---------------------------------------------------------------------------
# fp16 conversion against numpy's IEEE binary16 conversion
# ---------------------------------------------------------------------------

def test_f16_to_f32_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = oracle.f16_bits_to_f32(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_matches_numpy_rne():
    rng = np.random.default_rng(11)
    parts = [
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(200000) * 1e-5).astype(np.float32),   # subnormal range
        (rng.standard_normal(200000) * 1e-8).astype(np.float32),   # underflow
        (rng.standard_normal(50000) * 3e4).astype(np.float32),     # near overflow
        np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, np.inf, -np.inf], dtype=np.float32),
    ]
    # exact halfway points between consecutive fp16 values (ties to even)
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    parts.append(mid[(mid.astype(np.float64) == (lo + hi) / 2)])
    x = np.concatenate(parts)
    x = np.concatenate([x, -x])
    ref = x.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16_bits(x)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Brute force over the integer codes and the format's error bounds
# ---------------------------------------------------------------------------

def _random_blocks(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 32)).astype(np.float32)
    scale = np.exp2(rng.integers(-26, 10, size=(n, 1))).astype(np.float32)
    x = (x * scale).astype(np.float16)
    # make some magnitude ties and exact zeros
    x[::7, 5] = -x[::7, 3]
    x[::11] = np.float16(0)
    x[::13, :16] = np.float16(0)
    return x


def test_q8_0_codes_by_brute_force():
    x16 = _random_blocks(3000, 1)
    blocks = oracle.quantize(oracle.FMT_Q8_0, x16).reshape(-1, 34)
    q = blocks[:, 2:].view(np.int8).astype(np.int64)
    x = x16.astype(np.float32)
    amax = np.abs(x).max(axis=1, keepdims=True)
    d = amax / np.float32(127)
    with np.errstate(divide="ignore"):
        idv = np.where(d != 0, np.float32(1) / d, np.float32(0)).astype(np.float32)
    v = (x * idv).astype(np.float64)  # fp32 product, then exact in fp64
    cand = np.arange(-127, 128)
    dist = np.abs(v[..., None] - cand)  # [n, 32, 255]
    best = dist.min(axis=-1, keepdims=True)
    ties = dist == best
    # nearest integer; on an exact tie the one of larger magnitude (away from zero)
    mag = np.where(ties, np.abs(cand), -1)
    pick = cand[np.argmax(mag, axis=-1)]
    assert np.array_equal(q, pick)


def test_q4_0_codes_by_brute_force():
    x16 = _random_blocks(3000, 2)
    blocks = oracle.quantize(oracle.FMT_Q4_0, x16).reshape(-1, 18)
    packed = blocks[:, 2:].astype(np.int64)
    q = np.concatenate([packed & 15, packed >> 4], axis=1)
    x = x16.astype(np.float32)
    # signed value of largest magnitude, lowest index on ties (searched directly)
    m = np.empty((x.shape[0], 1), dtype=np.float32)
    for i in range(x.shape[0]):
        a = np.abs(x[i])
        m[i, 0] = x[i][np.flatnonzero(a == a.max())[0]]
    d = m / np.float32(-8)
    with np.errstate(divide="ignore"):
        idv = np.where(d != 0, np.float32(1) / d, np.float32(0)).astype(np.float32)
    s = ((x * idv).astype(np.float32) + np.float32(8.5)).astype(np.float64)
    # largest code c in 0..15 with c <= s (truncation of a positive value), clamped at 15
    cand = np.arange(16)
    pick = np.where(cand <= s[..., None], cand, -1).max(axis=-1)
    assert (pick >= 0).all()
    assert np.array_equal(q, pick)


def test_error_bounds_follow_from_the_format():
    x16 = _random_blocks(2000, 3)
    x = x16.astype(np.float64)
    for fmt in (oracle.FMT_Q8_0, oracle.FMT_Q4_0):
        blocks = oracle.quantize(fmt, x16)
        xh = oracle.dequantize(fmt, blocks).reshape(x.shape)
        bb = blocks.reshape(-1, oracle.block_bytes(fmt))
        dh = bb[:, :2].copy().view(np.float16).astype(np.float64)  # [n, 1]
        if fmt == oracle.FMT_Q8_0:
            d = np.abs(x).max(axis=1, keepdims=True) / 127.0
            bound = d / 2 + 127 * np.abs(d - dh)
        else:
            i = np.argmax(np.abs(x), axis=1)
            mm = x[np.arange(len(x)), i][:, None]
            d = np.abs(mm) / 8.0
            # half a step, a full step at the clamp (q = 15), plus the fp16 scale error
            bound = d + 8 * np.abs(np.abs(d) - np.abs(dh))
        err = np.abs(x - xh)
        assert (err <= bound * (1 + 1e-4) + 1e-30).all()
    # the element of largest magnitude comes back as +-127 d_h (Q8_0) / exactly -8 d_h (Q4_0)
    b8 = oracle.quantize(oracle.FMT_Q8_0, x16).reshape(-1, 34)
    q8 = b8[:, 2:].view(np.int8)
    nz = np.abs(x).max(axis=1) > 0
    i = np.argmax(np.abs(x), axis=1)
    assert (np.abs(q8[np.arange(len(x)), i][nz]) == 127).all()
    b4 = oracle.quantize(oracle.FMT_Q4_0, x16).reshape(-1, 18)
    p = b4[:, 2:].astype(np.int64)
    q4 = np.concatenate([p & 15, p >> 4], axis=1)
    assert (q4[np.arange(len(x)), i][nz] == 0).all()
