"""Seeded synthetic inputs for the W4A16 matmul (no arithmetic of the method here).

Both the CUDA path and the CPU oracle are fed from these generators, so they see
identical bits. Every tensor draws from its own PCG64 stream keyed by
(seed, stream id): activations 0, codes 1, scales 2, outlier mask 3, zero-points 4,
2:4 sparsity pattern 5.

Distributions follow the workloads the pages measure (a layer sweep over batch
sizes on Llama-2-like shapes, a 72k x 18k layer, prefill shapes):
  * activations x ~ N(0, 1) rounded to FP16 (round-to-nearest-even); the
    prefill workload multiplies an independent 1% of entries by 20 (outliers);
  * codes q ~ uniform on {0..15};
  * scales s = FP16(|N(0,1)| * c) per (group, column) with c = 0.02 (0.01 for
    the 72k x 18k layer), or FP16(10^U(-4,-1)) for the edge sweep;
  * zero-points z ~ uniform on {0..15} per (group, column) for the asymmetric
    format (every value, the extremes 0 and 15 included, is exercised);
  * for BF16 activations, the same x and s distributions rounded to bfloat16
    (round-to-nearest-even of the float32 draw), passed as bit patterns;
  * 2:4 sparse codes: in each aligned group of four k of a column one of the six
    position pairs, uniformly, keeps its uniform code and the other two are 8.
"""
import numpy as np

X_STREAM, CODE_STREAM, SCALE_STREAM, OUTLIER_STREAM, ZERO_STREAM, SPARSITY_STREAM = 0, 1, 2, 3, 4, 5


def rng(seed, stream):
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def activations(M, K, seed=0, outlier_frac=0.0, outlier_mult=20.0):
    """x[M][K] as float16."""
    x = rng(seed, X_STREAM).standard_normal((M, K), dtype=np.float32)
    if outlier_frac > 0.0:
        mask = rng(seed, OUTLIER_STREAM).random((M, K), dtype=np.float32) < outlier_frac
        x = np.where(mask, x * np.float32(outlier_mult), x)
    return x.astype(np.float16)


def to_bf16_bits(a):
    """float32 array -> bfloat16 bit patterns (uint16), round to nearest even (finite values)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def activations_bf16(M, K, seed=0):
    """x[M][K] ~ N(0, 1) as bfloat16 bit patterns (uint16), from the same stream as activations()."""
    return to_bf16_bits(rng(seed, X_STREAM).standard_normal((M, K), dtype=np.float32))


def codes(K, N, seed=0):
    """q[K][N] uniform on 0..15 as uint8."""
    return rng(seed, CODE_STREAM).integers(0, 16, size=(K, N), dtype=np.uint8)


def codes_2to4(K, N, seed=0):
    """q[K][N] 2:4 sparse along k: in every aligned group of four k of a column, two
    positions (one of the six pairs, uniformly) hold codes uniform on 0..15 and the
    other two hold 8 (weight 0). K must be a multiple of 4."""
    assert K % 4 == 0
    r = rng(seed, SPARSITY_STREAM)
    pairs = np.array([(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)])
    choice = pairs[r.integers(0, 6, size=(K // 4, N))]            # [K/4][N][2]
    keep = np.zeros((K // 4, N, 4), bool)
    np.put_along_axis(keep, choice, True, axis=2)
    keep = keep.transpose(0, 2, 1).reshape(K, N)
    return np.where(keep, codes(K, N, seed), np.uint8(8)).astype(np.uint8)


def n_groups(K, group_size):
    return -(-K // group_size)


def scales(K, N, group_size, seed=0, kind="halfnormal", mult=0.02):
    """s[ceil(K/G)][N] as float16."""
    ng = n_groups(K, group_size)
    r = rng(seed, SCALE_STREAM)
    if kind == "halfnormal":
        s = np.abs(r.standard_normal((ng, N), dtype=np.float32)) * np.float32(mult)
    elif kind == "loguniform":
        s = np.power(10.0, r.uniform(-4.0, -1.0, size=(ng, N))).astype(np.float32)
    else:
        raise ValueError(kind)
    return s.astype(np.float16)


def scales_bf16(K, N, group_size, seed=0, mult=0.02):
    """s[ceil(K/G)][N] = |N(0,1)| * mult as bfloat16 bit patterns (uint16)."""
    s = np.abs(rng(seed, SCALE_STREAM).standard_normal((n_groups(K, group_size), N), dtype=np.float32))
    return to_bf16_bits(s * np.float32(mult))


def zeros(K, N, group_size, seed=0):
    """z[ceil(K/G)][N] uniform on 0..15 as uint8."""
    return rng(seed, ZERO_STREAM).integers(0, 16, size=(n_groups(K, group_size), N), dtype=np.uint8)


def problem(M, K, N, group_size, seed=0, scale_kind="halfnormal", scale_mult=0.02,
            outlier_frac=0.0):
    """(x, q, s) for one matmul."""
    return (activations(M, K, seed, outlier_frac),
            codes(K, N, seed),
            scales(K, N, group_size, seed, scale_kind, scale_mult))


# The workloads: shapes and value distributions, named by what they are.
LLAMA2_7B_LAYERS = [(4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096)]  # (K, N)
LLAMA2_13B_LAYERS = [(5120, 15360), (5120, 5120), (5120, 27648), (13824, 5120)]
DECODE_M = [1, 2, 4, 8, 16, 32, 64, 128]
LARGE_LAYER = (18432, 73728)
LARGE_LAYER_M = [1, 16, 32, 64, 128]
PREFILL_M = [256, 512, 1024, 2048, 4096]
EDGE_M = [1, 3, 17, 127]

WORKLOADS = {
    "single_m16_4096x4096": dict(
        cases=[(16, 4096, 4096)], group_size=128, scale_mult=0.02),
    "llama2_7b_decode_sweep": dict(
        cases=[(m, k, n) for m in DECODE_M for (k, n) in LLAMA2_7B_LAYERS],
        group_size=128, scale_mult=0.02),
    "large_layer_18432x73728": dict(
        cases=[(m,) + LARGE_LAYER for m in LARGE_LAYER_M], group_size=128, scale_mult=0.01),
    "llama2_13b_prefill": dict(
        cases=[(m, k, n) for m in PREFILL_M for (k, n) in LLAMA2_13B_LAYERS],
        group_size=128, scale_mult=0.02, outlier_frac=0.01),
}
