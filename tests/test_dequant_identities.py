"""The arithmetic identities the kernels' dequantisation rests on, checked exhaustively
on the CPU with IEEE binary16 / bfloat16 rounding (numpy float16 rounds each
operation; an FMA is an exact FP64 evaluation rounded once).

Each packed code reaches a 16-bit lane by OR-ing it into the fraction of a constant,
so a single subtraction (or FMA) gives the integer q - z exactly, and the only
rounding of the dequantised weight is that of the product with the scale. These
tests pin those claims for every code and zero-point the formats allow; they do not
run the CUDA code."""
import numpy as np


def f16(bits):
    return np.array(bits, dtype=np.uint16).view(np.float16)


def bf16(bits):
    return float((np.array(bits, dtype=np.uint32) << 16).view(np.float32))


def round_bf16(v):
    b = np.array(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return bf16(int((b + 0x7FFF + ((b >> 16) & 1)) >> 16))


def test_four_bit_low_nibble_identity():
    # 0x6400 | q is 1024 + q; minus (1024 + z), the constant 0x6400 | z, is q - z exactly
    for q in range(16):
        for z in range(16):
            v = np.float16(f16(0x6400 | q)) - np.float16(f16(0x6400 | z))
            assert float(v) == q - z, (q, z)


def test_four_bit_high_nibble_identity():
    # 0x6400 | (q << 4) is 1024 + 16q; FMA with 1/16 (0x2C00) and -(64 + z) (0xD400 | 16z)
    # gives q - z exactly (the FMA rounds once, and the exact result is a small integer)
    assert float(f16(0x2C00)) == 1.0 / 16
    for q in range(16):
        for z in range(16):
            assert float(f16(0x6400 | (q << 4))) == 1024 + 16 * q
            assert float(f16(0xD400 | (z << 4))) == -(64 + z)
            exact = float(f16(0x6400 | (q << 4))) * (1.0 / 16) + float(f16(0xD400 | (z << 4)))
            assert float(np.float16(exact)) == q - z, (q, z)


def test_eight_bit_identity():
    # 0x6400 | q is 1024 + q for q < 256 (the ulp at 1024 is 1); minus 1152 (0x6480) is q - 128
    assert float(f16(0x6480)) == 1152
    for q in range(256):
        v = np.float16(f16(0x6400 | q)) - np.float16(f16(0x6480))
        assert float(v) == q - 128, q


def test_bfloat16_identity():
    # 0x4300 | q is 128 + q in bfloat16 (7 fraction bits, ulp 1 at 128); minus 136 (0x4308)
    assert bf16(0x4300) == 128 and bf16(0x4308) == 136
    for q in range(16):
        assert bf16(0x4300 | q) == 128 + q
        assert round_bf16(bf16(0x4300 | q) - bf16(0x4308)) == q - 8


def test_single_rounding_at_the_scale():
    # (q - z) exact, then one FP16 product: equal to the exact product rounded once
    rng = np.random.default_rng(0)
    scales = np.abs(rng.standard_normal(4000)).astype(np.float16)
    scales = np.concatenate([scales, f16(np.arange(1, 1024, 37)), f16([0x7BFF, 0x0400, 0x0001])])
    for d in range(-15, 16):
        with np.errstate(over="ignore"):   # the largest scales overflow: both sides give inf
            prod = (np.float16(d) * scales).astype(np.float64)
            exact = np.float16(d * scales.astype(np.float64)).astype(np.float64)
        ok = np.isfinite(exact)
        assert np.array_equal(prod[ok], exact[ok]), d
