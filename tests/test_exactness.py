"""Arithmetic facts the CUDA path relies on, checked on the CPU by emulating
each rounding step in numpy (IEEE binary16 round-to-nearest-even from exact
fp64 values).  These are not oracle pins: they establish that the kernels'
operand encodings are exact, so that the parity bar of the GPU tests leaves
room only for accumulation order and the final rounding.

* Chunk tiles feed every dequantised value d * q to the tensor cores as two fp16
  halves, hi = fp16(d * q) (clamped to +-65504 for Q8_0) and lo = fp16(d * q - hi).
  hi + lo must equal d * q exactly for every code and every finite fp16 scale
  the format can produce (Q8_0: 0 <= d <= fp16(65504 / 127) = 516; Q4_0:
  |d| <= 65504 / 8 = 8188).
* Decode tiles feed codes as fp16 subnormals: the 16-bit pattern of an unsigned
  integer u < 1024 is the fp16 number u * 2^-24.
"""
import numpy as np


def _finite_f16(lo, hi):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    keep = np.isfinite(vals) & (vals >= lo) & (vals <= hi)
    return np.unique(vals[keep])


def _split(prod, clamp):
    hi = prod.astype(np.float16).astype(np.float64)  # round to nearest even (inf beyond 65520)
    if clamp:
        hi = np.clip(hi, -65504.0, 65504.0)
    lo = (prod - hi).astype(np.float16).astype(np.float64)  # fma: exact difference, one rounding
    return hi, lo


def test_q8_0_hi_lo_split_is_exact_for_every_code_and_scale():
    d = _finite_f16(0.0, 516.0)
    assert d.max() == 516.0
    q = np.arange(-127, 128, dtype=np.float64)
    prod = q[:, None] * d[None, :]  # exact in fp64 (<= 18 significant bits)
    hi, lo = _split(prod, clamp=True)
    assert np.isfinite(hi).all() and np.isfinite(lo).all()
    assert np.array_equal(hi + lo, prod)
    # without the clamp the largest codes of the largest scale overflow
    hi_raw = prod.astype(np.float16).astype(np.float64)
    assert np.isinf(hi_raw).any() and np.isinf(hi_raw[np.abs(prod) >= 65520]).all()


def test_q4_0_hi_lo_split_is_exact_without_a_clamp():
    d = _finite_f16(-8188.0, 8188.0)
    q = np.arange(-8, 8, dtype=np.float64)  # q - 8 for the stored nibble q = 0..15
    prod = q[:, None] * d[None, :]
    hi, lo = _split(prod, clamp=False)
    assert np.isfinite(hi).all() and np.isfinite(lo).all()
    assert np.array_equal(hi + lo, prod)


def test_small_unsigned_integers_are_exact_fp16_subnormals():
    u = np.arange(0, 1024, dtype=np.uint16)
    assert np.array_equal(u.view(np.float16).astype(np.float64), u.astype(np.float64) * 2.0 ** -24)
