"""Pins for the CPU oracle: each check ties it to something other than itself.

* the binary16 decoder against numpy's float16 over all 65536 bit patterns;
* brute force in exact rational arithmetic on tiny inputs (all group sizes,
  K not a multiple of G, subnormal scales);
* the hand-worked 1x8x8 example in tests/golden/hand_1x8x8.txt;
* invariants: zero scales, all codes 8, a single nonzero code, linearity in x,
  doubling the scales, one-hot rows of x;
* mutants: a copy of the oracle with one planted mistake must fail a pin;
* per-group zero-points: brute force in exact rationals, zero-points of 8 equal
  the symmetric form bit for bit, codes equal to their zero-points give 0, the
  closed form of a unit step in one zero-point, numpy's matmul on the expanded
  weights, the hand example with zero-point n in column n;
* 8-bit codes (W8A16, zero-point 128): brute force in exact rationals, codes 128
  give 0, 8-bit codes 16*q equal 16 times the 4-bit result for codes q, numpy's
  matmul on the expanded weights, the 8-bit layout (bijection, round trip, the
  pair (k, k+1) in bytes 0 and 2 of a word);
* BF16 activations: the bfloat16 decoder against numpy's float32 reading of the
  same bits over all 65536 patterns, brute force in exact rationals on bfloat16
  inputs, and equality with the FP16 form on values exact in both formats;
* 2:4 sparse layout: round trip of 2:4 codes, the fill rule and the bits of a
  hand-worked chunk, violations counted, the generator's 2:4 structure.
"""
import os
import re
import shutil
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

from weight_only_int4_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_1x8x8.txt")


def read_golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = np.array([float(v) for v in vals.split()])
    return out


def hand_inputs(G):
    x = np.array([1, -1, 2, -2, 0.5, -0.5, 1, 0], np.float16).reshape(1, 8)
    q = np.array([[(3 * k + n) % 16 for n in range(8)] for k in range(8)], np.uint8)
    base = np.array([0.25 * (1 + n % 4) for n in range(8)])
    if G == 4:
        s = np.stack([base, base / 2]).astype(np.float16)
    else:
        s = base.reshape(1, 8).astype(np.float16)
    return x, q, s


def test_half_decoder_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # a few fixed points of the format
    named = {0x3C00: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14,
             0x7BFF: 65504.0, 0x6400: 1024.0, 0x8000: -0.0}
    for b, v in named.items():
        assert oracle_mod.half_to_double(np.array([b], np.uint16))[0] == v


def exact_reference(x, q, s, G, z=None, zdef=8):
    """Exact rationals: each FP16 value converts to Fraction without rounding.
    z: integer zero-points [ceil(K/G)][N], or None for the fixed zdef."""
    M, K = x.shape
    N = q.shape[1]
    xf = [[Fraction(float(v)) for v in row] for row in x.astype(np.float64)]
    sf = [[Fraction(float(v)) for v in row] for row in s.astype(np.float64)]
    y = [[Fraction(0)] * N for _ in range(M)]
    a = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc, acc_abs = Fraction(0), Fraction(0)
            for k in range(K):
                zero = zdef if z is None else int(z[k // G][n])
                t = xf[m][k] * (int(q[k][n]) - zero) * sf[k // G][n]
                acc += t
                acc_abs += abs(t)
            y[m][n], a[m][n] = acc, acc_abs
    return y, a


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_exact(oracle_mod, seed):
    r = np.random.default_rng(1000 + seed)
    M, K, N = (int(v) for v in r.integers(1, 9, size=3))
    G = int(r.choice([1, 2, 3, 4, K]))
    x = (r.standard_normal((M, K)) * 4).astype(np.float16)
    q = r.integers(0, 16, size=(K, N)).astype(np.uint8)
    ng = -(-K // G)
    s = np.abs(r.standard_normal((ng, N))).astype(np.float16)
    if seed % 3 == 0:   # subnormal scales: multiples of 2^-24 below 2^-14
        s = (r.integers(1, 1024, size=(ng, N)) * 2.0 ** -24).astype(np.float16)
    y, a = oracle_mod.gemm(x, q, s, G)
    ye, ae = exact_reference(x, q, s, G)
    for m in range(M):
        for n in range(N):
            bound = (K * 2.0 ** -53) * float(ae[m][n])
            assert abs(Fraction(y[m][n]) - ye[m][n]) <= Fraction(bound)
            assert abs(Fraction(a[m][n]) - ae[m][n]) <= Fraction(bound)


def test_hand_example(oracle_mod):
    g = read_golden()
    for G, key in ((4, "G4"), (8, "G8")):
        x, q, s = hand_inputs(G)
        assert np.array_equal(x[0].astype(np.float64), g["x"])
        y, a = oracle_mod.gemm(x, q, s, G)
        assert np.array_equal(y[0], g[key + "_y"]), (G, y[0])
        assert np.array_equal(a[0], g[key + "_abs"]), (G, a[0])


def small_problem(M=5, K=96, N=24, G=32, seed=7):
    return inputs.problem(M, K, N, G, seed=seed)


def test_zero_scales_give_zero(oracle_mod):
    x, q, s = small_problem()
    y, _ = oracle_mod.gemm(x, q, np.zeros_like(s), 32)
    assert np.all(y == 0)


def test_all_codes_eight_give_zero(oracle_mod):
    x, q, s = small_problem()
    y, _ = oracle_mod.gemm(x, np.full_like(q, 8), s, 32)
    assert np.all(y == 0)


def test_single_code_gives_single_column(oracle_mod):
    x, q, s = small_problem()
    K, N = q.shape
    G = 32
    k0, n0, code = 45, 17, 3
    q1 = np.full_like(q, 8)
    q1[k0, n0] = code
    y, _ = oracle_mod.gemm(x, q1, s, G)
    expect = x[:, k0].astype(np.float64) * (code - 8) * float(s[k0 // G, n0])
    assert np.array_equal(y[:, n0], expect)
    others = np.delete(y, n0, axis=1)
    assert np.all(others == 0)


def test_linearity_in_x(oracle_mod):
    x, q, s = small_problem()
    M, K = x.shape
    x1 = x.copy()
    x1[:, 1::2] = 0      # disjoint supports keep 2*x1 + 0.5*x2 exact in FP16
    x2 = x.copy()
    x2[:, 0::2] = 0
    xs = (2 * x1.astype(np.float32) + 0.5 * x2.astype(np.float32)).astype(np.float16)
    assert np.array_equal(xs.astype(np.float32), 2 * x1.astype(np.float32) + 0.5 * x2.astype(np.float32))
    y, a = oracle_mod.gemm(xs, q, s, 32)
    y1, _ = oracle_mod.gemm(x1, q, s, 32)
    y2, _ = oracle_mod.gemm(x2, q, s, 32)
    assert np.all(np.abs(y - (2 * y1 + 0.5 * y2)) <= 4 * K * 2.0 ** -53 * a)


def test_doubling_scales_doubles_output(oracle_mod):
    x, q, s = small_problem()
    y, _ = oracle_mod.gemm(x, q, s, 32)
    y2, _ = oracle_mod.gemm(x, q, (s.astype(np.float32) * 2).astype(np.float16), 32)
    assert np.array_equal(y2, 2 * y)


def test_one_hot_rows_return_dequantised_rows(oracle_mod):
    _, q, s = small_problem()
    K, N = q.shape
    rows = [0, 31, 32, 95]
    x = np.zeros((len(rows), K), np.float16)
    for i, k in enumerate(rows):
        x[i, k] = 1.0
    y, _ = oracle_mod.gemm(x, q, s, 32)
    w = oracle_mod.dequant(q, s, 32)
    for i, k in enumerate(rows):
        assert np.array_equal(y[i], w[k])
        assert np.array_equal(w[k], (q[k].astype(np.float64) - 8) * s[k // 32].astype(np.float64))


def test_per_column_group_equals_single_group(oracle_mod):
    x, q, _ = small_problem(K=64)
    s1 = inputs.scales(64, q.shape[1], 64, seed=3)
    y_a, _ = oracle_mod.gemm(x, q, s1, 64)
    s_rep = np.repeat(s1, 2, axis=0)
    y_b, _ = oracle_mod.gemm(x, q, s_rep, 32)
    assert np.array_equal(y_a, y_b)


def test_sample_matches_full_and_threads_do_not_matter(oracle_mod):
    x, q, s = inputs.problem(9, 200, 70, 64, seed=11)
    y, a = oracle_mod.gemm(x, q, s, 64, threads=1)
    y4, a4 = oracle_mod.gemm(x, q, s, 64, threads=4)
    assert np.array_equal(y, y4) and np.array_equal(a, a4)
    rows, cols = [8, 0, 3], [69, 1, 33, 34]
    ys, as_ = oracle_mod.gemm_sample(x, q, s, 64, rows, cols, threads=3)
    assert np.array_equal(ys, y[np.ix_(rows, cols)])
    assert np.array_equal(as_, a[np.ix_(rows, cols)])


@pytest.mark.parametrize("K,N", [(64, 128), (200, 130), (8, 8), (4040, 256)])
def test_layout_is_a_bijection_and_round_trips(oracle_mod, K, N):
    KC, NT = -(-(-(-K // 64)) // 4) * 4, -(-N // 128)
    total = oracle_mod.packed_words(K, N)
    assert total == KC * NT * 1024
    if K * N <= 64 * 1024:
        seen = set()
        for k in range(KC * 64):
            for n in range(NT * 128):
                w, i = oracle_mod.locate(K, k, n)
                assert 0 <= w < total and 0 <= i < 8
                seen.add((w, i))
        assert len(seen) == total * 8
    q = inputs.codes(K, N, seed=5)
    p = oracle_mod.pack(q)
    q2, bad = oracle_mod.unpack(p, K, N)
    assert bad == 0 and np.array_equal(q, q2)
    for pattern in (0, 15):
        qq = np.full((K, N), pattern, np.uint8)
        q3, bad = oracle_mod.unpack(oracle_mod.pack(qq), K, N)
        assert bad == 0 and np.array_equal(q3, qq)


def test_layout_pairs_adjacent_k_in_nibbles_i_and_i_plus_4(oracle_mod):
    # nibble i of a word holds k0 + 2*(i mod 4) + i//4: the two halves of a
    # 16-bit lane pair hold k and k+1.
    for k in range(64):
        w, i = oracle_mod.locate(64, k, 0)
        assert (k % 8) == 2 * (i % 4) + i // 4
        w2, i2 = oracle_mod.locate(64, k, 1)
        assert w2 == w + 4 and i2 == i


def test_scales_unpack(oracle_mod):
    N, ng = 200, 3
    s = inputs.scales(3 * 32, N, 32, seed=2)
    sp = np.zeros(-(-N // 128) * ng * 128, np.uint16)
    for g in range(ng):
        for n in range(N):
            sp[((n // 128) * ng + g) * 128 + n % 128] = s.view(np.uint16)[g, n]
    s2, bad = oracle_mod.unpack_scales(sp, ng, N)
    assert bad == 0 and np.array_equal(s2, s.view(np.uint16))


MUTANTS = {
    "zero_point_7": ("return gemm_sample_any(x, q, s, z, 8,", "return gemm_sample_any(x, q, s, z, 7,"),
    "zero_points_ignored": ("int zero = z ? z[(size_t)g * N + n] : zdef;", "int zero = zdef;"),
    "zero_point_of_first_group": ("int zero = z ? z[(size_t)g * N + n] : zdef;",
                                  "int zero = z ? z[n] : zdef;"),
    "zero_point_of_mirrored_column": ("int zero = z ? z[(size_t)g * N + n] : zdef;",
                                      "int zero = z ? z[(size_t)g * N + (N - 1 - n)] : zdef;"),
    "zero_point_sign": ("(double)(code - zero)", "(double)(zero - code)"),
    "bf16_exponent_bias": ("ldexp((double)(128 + f), e - 134)", "ldexp((double)(128 + f), e - 133)"),
    "bf16_x_read_as_fp16": ("xd[(size_t)r * K + k] = dec(x[(size_t)rows[r] * K + k]);",
                            "xd[(size_t)r * K + k] = w4o_half_to_double(x[(size_t)rows[r] * K + k]);"),
    "sp_nibble_order": ("int nib = (o % 2) * 4 + o / 2;     /* o = 2*(nib mod 4) + nib/4 */",
                        "int nib = o;"),
    "sp_position_field": ("mw[L * 4 + mm] |= (uint32_t)(pos[0] | (pos[1] << 2)) << (4 * u);",
                          "mw[L * 4 + mm] |= (uint32_t)(pos[1] | (pos[0] << 2)) << (4 * u);"),
    "sp_position_lane": ("*lane = 16 * (n_in / 16) + 8 * (t / 4) + n_in % 8;", "*lane = n_in;"),
    "w8_zero_point_127": ("return gemm_sample_any(x, q, s, NULL, 128,", "return gemm_sample_any(x, q, s, NULL, 127,"),
    "w8_byte_order": ("slot_of_offset[4] = {0, 2, 1, 3}", "slot_of_offset[4] = {0, 1, 2, 3}"),
    "no_groups": ("static int group_of(int k, int G) { return k / G; }",
                  "static int group_of(int k, int G) { (void)k; (void)G; return 0; }"),
    "transposed_weights": ("int code = q[(size_t)k * N + n];", "int code = q[(size_t)n * N + k];"),
    "exponent_bias": ("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
    "subnormal_scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "dropped_abs": ("acc_abs += fabs(t);", "acc_abs += t;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(oracle_mod, name):
    """Each planted mistake in a copy of the oracle must break a pin above."""
    import importlib.util
    src_dir = os.path.dirname(oracle_mod.__file__)
    old, new = MUTANTS[name]
    text = open(os.path.join(src_dir, "w4a16_oracle.c")).read()
    assert old in text
    with tempfile.TemporaryDirectory() as d:
        mdir = os.path.join(d, "oracle_mutant")
        os.mkdir(mdir)
        shutil.copy(os.path.join(src_dir, "__init__.py"), mdir)
        with open(os.path.join(mdir, "w4a16_oracle.c"), "w") as f:
            f.write(text.replace(old, new))
        spec = importlib.util.spec_from_file_location("oracle_mutant", os.path.join(mdir, "__init__.py"))
        mut = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mut)
        mut.build(force=True)
        failures = 0
        for check in (test_hand_example, test_half_decoder_all_patterns,
                      test_all_codes_eight_give_zero, test_per_column_group_equals_single_group,
                      lambda o: test_brute_force_exact(o, 0), lambda o: test_brute_force_exact(o, 1),
                      lambda o: test_zero_points_brute_force_exact(o, 0),
                      lambda o: test_zero_points_brute_force_exact(o, 1),
                      lambda o: test_w8_brute_force_exact(o, 0),
                      test_bf16_decoder_all_patterns, lambda o: test_bf16_brute_force_exact(o, 0),
                      test_sp_hand_worked_chunk, lambda o: test_sp_round_trip(o, 512, 256),
                      test_w8_layout_pairs_adjacent_k_in_bytes_0_and_2):
            try:
                check(mut)
            except AssertionError:
                failures += 1
                break
        assert failures > 0, name


# --------------------------------------------------------------------------- per-group zero-points
# w = (q - z[g][n]) * s[g][n] with an integer zero-point 0..15 per (group, column):
# the asymmetric 4-bit format of AWQ checkpoints, which "Low-Precision
# Quantization Kernels in Production" (llms.blog), section 1, lists among those the
# Marlin kernel family serves.
@pytest.mark.parametrize("seed", range(8))
def test_zero_points_brute_force_exact(oracle_mod, seed):
    r = np.random.default_rng(2000 + seed)
    M, K, N = (int(v) for v in r.integers(1, 9, size=3))
    G = int(r.choice([1, 2, 3, 4, K]))
    ng = -(-K // G)
    x = (r.standard_normal((M, K)) * 4).astype(np.float16)
    q = r.integers(0, 16, size=(K, N)).astype(np.uint8)
    z = r.integers(0, 16, size=(ng, N)).astype(np.uint8)
    s = np.abs(r.standard_normal((ng, N))).astype(np.float16)
    y, a = oracle_mod.gemm(x, q, s, G, z=z)
    ye, ae = exact_reference(x, q, s, G, z)
    for m in range(M):
        for n in range(N):
            bound = (K * 2.0 ** -53) * float(ae[m][n])
            assert abs(Fraction(y[m][n]) - ye[m][n]) <= Fraction(bound)
            assert abs(Fraction(a[m][n]) - ae[m][n]) <= Fraction(bound)


def test_zero_points_of_eight_equal_the_symmetric_form(oracle_mod):
    x, q, s = small_problem()
    z = np.full((3, q.shape[1]), 8, np.uint8)
    y, a = oracle_mod.gemm(x, q, s, 32)
    yz, az = oracle_mod.gemm(x, q, s, 32, z=z)
    assert np.array_equal(y, yz) and np.array_equal(a, az)
    assert np.array_equal(oracle_mod.dequant(q, s, 32), oracle_mod.dequant(q, s, 32, z=z))


def test_codes_equal_to_their_zero_points_give_zero(oracle_mod):
    x, _, s = small_problem()
    z = inputs.zeros(96, 24, 32, seed=4)
    q = np.repeat(z, 32, axis=0)
    y, a = oracle_mod.gemm(x, q, s, 32, z=z)
    assert np.all(y == 0) and np.all(a == 0)


def test_unit_step_in_one_zero_point(oracle_mod):
    """Raising z[g][n] by one lowers column n by s[g][n] * sum of x over group g and
    leaves every other column alone. Integer x and power-of-two scales keep every
    sum exact, so the step is compared exactly."""
    r = np.random.default_rng(5)
    M, K, N, G = 4, 96, 24, 32
    x = r.integers(-8, 9, size=(M, K)).astype(np.float16)
    q = inputs.codes(K, N, seed=6)
    s = (2.0 ** r.integers(-6, 0, size=(3, N))).astype(np.float16)
    z = np.minimum(inputs.zeros(K, N, G, seed=6), 14)
    y, _ = oracle_mod.gemm(x, q, s, G, z=z)
    for g, n in ((0, 0), (1, 17), (2, 23)):
        z1 = z.copy()
        z1[g, n] += 1
        y1, _ = oracle_mod.gemm(x, q, s, G, z=z1)
        step = -float(s[g, n]) * x[:, g * G:(g + 1) * G].astype(np.float64).sum(axis=1)
        assert np.array_equal(y1[:, n] - y[:, n], step)
        assert np.array_equal(np.delete(y1, n, axis=1), np.delete(y, n, axis=1))


def test_zero_points_against_numpy_matmul(oracle_mod):
    x, q, s = inputs.problem(17, 300, 200, 64, seed=9)
    z = inputs.zeros(300, 200, 64, seed=9)
    w = (q.astype(np.float64) - np.repeat(z, 64, axis=0)[:300]) * np.repeat(s.astype(np.float64), 64, axis=0)[:300]
    ref = x.astype(np.float64) @ w
    y, a = oracle_mod.gemm(x, q, s, 64, z=z)
    assert np.all(np.abs(y - ref) <= 2 * 300 * 2.0 ** -53 * a)
    assert np.array_equal(oracle_mod.dequant(q, s, 64, z=z), w)
    rows, cols = [16, 0, 7], [199, 3, 128]
    ys, as_ = oracle_mod.gemm_sample(x, q, s, 64, rows, cols, z=z)
    assert np.array_equal(ys, y[np.ix_(rows, cols)]) and np.array_equal(as_, a[np.ix_(rows, cols)])


def test_zero_points_on_the_hand_example(oracle_mod):
    """Hand example, one group (G = K = 8), zero-point n in column n: sum_k x_k = 1,
    so y[n] = y_8[n] + (8 - n) * s[n] with y_8 the golden symmetric result."""
    g = read_golden()
    x, q, s = hand_inputs(8)
    z = np.arange(8, dtype=np.uint8).reshape(1, 8)
    y, _ = oracle_mod.gemm(x, q, s, 8, z=z)
    assert float(x.astype(np.float64).sum()) == 1.0
    assert np.array_equal(y[0], g["G8_y"] + (8 - np.arange(8)) * s[0].astype(np.float64))


def test_zeros_unpack(oracle_mod):
    N, ng = 200, 3
    z = inputs.zeros(3 * 32, N, 32, seed=2)
    zp = np.zeros(-(-N // 128) * ng * 64, np.uint8)
    for g in range(ng):
        for n in range(-(-N // 128) * 128):
            v = int(z[g, n]) if n < N else 8
            zp[((n // 128) * ng + g) * 64 + (n % 128) // 2] |= v << (4 * (n % 2))
    z2, bad = oracle_mod.unpack_zeros(zp, ng, N)
    assert bad == 0 and np.array_equal(z2, z)
    zp[-1] = 0   # a padding column that does not hold 8
    assert oracle_mod.unpack_zeros(zp, ng, N)[1] == 2


# --------------------------------------------------------------------------- 8-bit codes (W8A16)
# w = (q - 128) * s with q 0..255: the 8-bit checkpoints that "Low-Precision
# Quantization Kernels in Production" (llms.blog), section 1, says the Marlin
# kernel family serves beside the 4-bit ones; 128 is the symmetric zero-point of
# unsigned 8-bit codes.
@pytest.mark.parametrize("seed", range(8))
def test_w8_brute_force_exact(oracle_mod, seed):
    r = np.random.default_rng(3000 + seed)
    M, K, N = (int(v) for v in r.integers(1, 9, size=3))
    G = int(r.choice([1, 2, 3, 4, K]))
    ng = -(-K // G)
    x = (r.standard_normal((M, K)) * 4).astype(np.float16)
    q = r.integers(0, 256, size=(K, N)).astype(np.uint8)
    s = np.abs(r.standard_normal((ng, N))).astype(np.float16)
    if seed % 3 == 0:
        s = (r.integers(1, 1024, size=(ng, N)) * 2.0 ** -24).astype(np.float16)
    y, a = oracle_mod.gemm_w8(x, q, s, G)
    ye, ae = exact_reference(x, q, s, G, zdef=128)
    for m in range(M):
        for n in range(N):
            bound = (K * 2.0 ** -53) * float(ae[m][n])
            assert abs(Fraction(y[m][n]) - ye[m][n]) <= Fraction(bound)
            assert abs(Fraction(a[m][n]) - ae[m][n]) <= Fraction(bound)


def test_w8_codes_128_give_zero(oracle_mod):
    x, q, s = small_problem()
    y, a = oracle_mod.gemm_w8(x, np.full_like(q, 128), s, 32)
    assert np.all(y == 0) and np.all(a == 0)


def test_w8_codes_16q_equal_16_times_the_4bit_result(oracle_mod):
    """(16q - 128) = 16 (q - 8): 8-bit codes 16q give exactly 16 times the 4-bit
    result for codes q (a power-of-two factor is exact in FP64)."""
    x, q, s = small_problem()
    y4, a4 = oracle_mod.gemm(x, q, s, 32)
    y8, a8 = oracle_mod.gemm_w8(x, (q.astype(np.uint16) * 16).astype(np.uint8), s, 32)
    assert np.array_equal(y8, 16 * y4) and np.array_equal(a8, 16 * a4)


def test_w8_against_numpy_matmul(oracle_mod):
    x, _, s = inputs.problem(17, 300, 200, 64, seed=9)
    q = np.random.default_rng(9).integers(0, 256, size=(300, 200)).astype(np.uint8)
    w = (q.astype(np.float64) - 128) * np.repeat(s.astype(np.float64), 64, axis=0)[:300]
    ref = x.astype(np.float64) @ w
    y, a = oracle_mod.gemm_w8(x, q, s, 64)
    assert np.all(np.abs(y - ref) <= 2 * 300 * 2.0 ** -53 * a)
    assert np.array_equal(oracle_mod.dequant_w8(q, s, 64), w)


@pytest.mark.parametrize("K,N", [(64, 128), (200, 130), (8, 8)])
def test_w8_layout_is_a_bijection_and_round_trips(oracle_mod, K, N):
    KC, NT = -(-(-(-K // 64)) // 4) * 4, -(-N // 128)
    total = oracle_mod.packed_bytes_w8(K, N)
    assert total == KC * NT * 8192
    seen = set()
    for k in range(KC * 64):
        for n in range(NT * 128):
            b = oracle_mod.locate_w8(K, k, n)
            assert 0 <= b < total
            seen.add(b)
    assert len(seen) == total
    q = np.random.default_rng(5).integers(0, 256, size=(K, N)).astype(np.uint8)
    q2, bad = oracle_mod.unpack_w8(oracle_mod.pack_w8(q), K, N)
    assert bad == 0 and np.array_equal(q, q2)


def test_w8_layout_pairs_adjacent_k_in_bytes_0_and_2(oracle_mod):
    # a word holds k0 .. k0+3 as bytes (k0, k0+2, k0+1, k0+3): masking bytes 0 and 2
    # (or 1 and 3) of the word gives the 16-bit pair (k, k+1) of one TMEM column
    for k0 in range(0, 64, 4):
        b = [oracle_mod.locate_w8(64, k0 + i, 5) for i in range(4)]
        assert b[0] % 4 == 0 and b[1] == b[0] + 2 and b[2] == b[0] + 1 and b[3] == b[0] + 3
    # adjacent columns' 16-byte blocks are adjacent; quarters of 16 k are 2 KB apart
    assert oracle_mod.locate_w8(64, 0, 1) == oracle_mod.locate_w8(64, 0, 0) + 16
    assert oracle_mod.locate_w8(64, 16, 0) == oracle_mod.locate_w8(64, 0, 0) + 2048


# --------------------------------------------------------------------------- BF16 activations
# x and s as bfloat16 ("Low-Precision Quantization Kernels in Production"
# (llms.blog), introduction: FP16 and BF16 are the 16-bit types the weights are
# quantised from and the tensor cores run).
def bf16_values(bits):
    """numpy's reading of bfloat16 bits: the upper half of a float32."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def test_bf16_decoder_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.bf16_to_double(bits)
    with np.errstate(invalid="ignore"):   # signalling-NaN patterns
        ref = bf16_values(bits).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    named = {0x3F80: 1.0, 0xC000: -2.0, 0x4300: 128.0, 0x4308: 136.0, 0x0001: 2.0 ** -133,
             0x0080: 2.0 ** -126, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127}
    for b, v in named.items():
        assert oracle_mod.bf16_to_double(np.array([b], np.uint16))[0] == v


@pytest.mark.parametrize("seed", range(6))
def test_bf16_brute_force_exact(oracle_mod, seed):
    r = np.random.default_rng(4000 + seed)
    M, K, N = (int(v) for v in r.integers(1, 9, size=3))
    G = int(r.choice([1, 2, 3, 4, K]))
    ng = -(-K // G)
    x = inputs.to_bf16_bits((r.standard_normal((M, K)) * 4).astype(np.float32))
    q = r.integers(0, 16, size=(K, N)).astype(np.uint8)
    s = inputs.to_bf16_bits(np.abs(r.standard_normal((ng, N))).astype(np.float32))
    y, a = oracle_mod.gemm_bf16(x, q, s, G)
    ye, ae = exact_reference(bf16_values(x), q, bf16_values(s), G)
    for m in range(M):
        for n in range(N):
            bound = (K * 2.0 ** -53) * float(ae[m][n])
            assert abs(Fraction(y[m][n]) - ye[m][n]) <= Fraction(bound)
            assert abs(Fraction(a[m][n]) - ae[m][n]) <= Fraction(bound)


def test_bf16_equals_fp16_on_values_exact_in_both(oracle_mod):
    r = np.random.default_rng(6)
    M, K, N, G = 4, 96, 24, 32
    xv = (r.integers(-64, 65, size=(M, K)) / 16.0).astype(np.float32)   # 8 significant bits at most
    sv = (2.0 ** r.integers(-12, 0, size=(3, N))).astype(np.float32)
    q = inputs.codes(K, N, seed=6)
    y16, a16 = oracle_mod.gemm(xv.astype(np.float16), q, sv.astype(np.float16), G)
    yb, ab = oracle_mod.gemm_bf16(inputs.to_bf16_bits(xv), q, inputs.to_bf16_bits(sv), G)
    assert np.array_equal(bf16_values(inputs.to_bf16_bits(xv)), xv)
    assert np.array_equal(y16, yb) and np.array_equal(a16, ab)


# --------------------------------------------------------------------------- 2:4 sparse 4-bit layout
# Sparse-MARLIN ("MARLIN: Mixed-Precision Auto-Regressive Parallel Inference on
# Large Language Models" note, key results: INT4 with 2:4 sparsity): at most two
# codes other than 8 in every aligned group of four k; the GEMM is the dense one.
@pytest.mark.parametrize("K,N", [(256, 8), (200, 130), (512, 256)])
def test_sp_round_trip(oracle_mod, K, N):
    q = inputs.codes_2to4(K, N, seed=7)
    packed, violations = oracle_mod.sp_pack(q)
    assert violations == 0 and packed.size == oracle_mod.sp_packed_bytes(K, N)
    q2, bad = oracle_mod.sp_unpack(packed, K, N)
    assert bad == 0 and np.array_equal(q2, q)


def test_sp_generator_is_2to4(oracle_mod):
    q = inputs.codes_2to4(64, 40, seed=3)
    nonzero = (q != 8).reshape(16, 4, 40).sum(axis=1)
    assert nonzero.max() <= 2 and (q != 8).mean() > 0.4


def test_sp_hand_worked_chunk(oracle_mod):
    """Column 0, k 0..3 = [8, 3, 8, 8], k 4..7 = [5, 8, 8, 2]; column 8, k 0..3 =
    [8, 8, 6, 7]; column 0, k 16..19 = [9, 8, 8, 1]; all else 8.
    Positions: (0, 1) (3 kept, filled with position 0), (0, 3), (2, 3), (0, 3).
    Code word (b 0, column 0, word 0): stored value o in nibble (o%2)*4 + o/2, so
    nibbles 0..7 = 8, 5, 8, 8, 3, 2, 8, 8 -> 0x88238858.
    Position words in tensor-memory lane order: lane 0 holds groups 0..3 of column 0
    in nibbles 0..3 and of column 8 in nibbles 4..7 -> 0x444E44C4; lane 8 holds
    groups 4..7 of column 0 (nibble 0: group 4 = (0, 3) -> 0xC) -> 0x4444444C."""
    q = np.full((256, 16), 8, np.uint8)
    q[1, 0], q[4, 0], q[7, 0] = 3, 5, 2
    q[2, 8], q[3, 8] = 6, 7
    q[16, 0], q[19, 0] = 9, 1
    packed, violations = oracle_mod.sp_pack(q)
    assert violations == 0
    words = packed.view(np.uint32)
    meta = words[4096 // 4:]
    assert words[0] == 0x88238858
    assert meta[0 * 4 + 0] == 0x444E44C4
    assert meta[8 * 4 + 0] == 0x4444444C
    assert meta[0 * 4 + 1] == 0x44444444      # MMA 1 (k 32..63): empty groups
    assert words[4] == 0x88888888             # column 1, word 0


def test_sp_violations_are_counted(oracle_mod):
    q = np.full((256, 8), 8, np.uint8)
    q[0:3, 0] = [1, 2, 3]             # three codes other than 8 in one group
    q[8:12, 5] = [4, 5, 6, 7]         # four
    packed, violations = oracle_mod.sp_pack(q)
    assert violations == 2
    q2, bad = oracle_mod.sp_unpack(packed, 256, 8)
    assert bad == 0 and list(q2[0:4, 0]) == [1, 2, 8, 8] and list(q2[8:12, 5]) == [4, 5, 8, 8]


# --------------------------------------------------------------------------- fused epilogue
def test_epilogue_bias_and_residual_are_exact_adds(oracle_mod):
    rng = np.random.default_rng(7)
    z = rng.integers(-1000, 1000, size=(5, 24)).astype(np.float64) / 8.0       # exact in any order
    b = (rng.integers(-64, 64, size=24) / 4.0).astype(np.float16)
    r = (rng.integers(-64, 64, size=(5, 24)) / 2.0).astype(np.float16)
    assert np.array_equal(oracle_mod.epilogue(z, bias=b) - z, np.broadcast_to(b.astype(np.float64), z.shape))
    assert np.array_equal(oracle_mod.epilogue(z, residual=r) - z, r.astype(np.float64))
    assert np.array_equal(oracle_mod.epilogue(z), z)


def test_epilogue_silu_matches_library_logistic(oracle_mod):
    scipy_special = pytest.importorskip("scipy.special")
    z = np.linspace(-40.0, 40.0, 4001)
    got = oracle_mod.epilogue(z[None, :], activation="silu")[0]
    want = z * scipy_special.expit(z)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-300)
    # special values and the reflection identity SiLU(-z) = SiLU(z) - z
    assert oracle_mod.epilogue(np.zeros((1, 1)), activation="silu")[0, 0] == 0.0
    assert np.allclose(oracle_mod.epilogue(-z[None, :], activation="silu")[0], got - z, rtol=1e-12, atol=1e-12)
    big = oracle_mod.epilogue(np.array([[-1000.0, 1000.0]]), activation="silu")[0]
    assert big[0] == 0.0 and big[1] == 1000.0


def test_epilogue_relu_and_order_of_operations(oracle_mod):
    z = np.array([[-3.0, -0.5, 0.0, 0.5, 3.0]])
    b = np.array([1.0, 1.0, -1.0, -1.0, 0.0], np.float16)
    r = np.array([[0.25, 0.25, 0.25, 0.25, 0.25]], np.float16)
    # bias before the activation, residual after it
    assert np.array_equal(oracle_mod.epilogue(z, bias=b, residual=r, activation="relu"),
                          np.array([[0.25, 0.75, 0.25, 0.25, 3.25]]))


def test_epilogue_on_the_hand_example(oracle_mod):
    """The 1x8x8 hand example with G = K: y = [-4.125, -3.75, -4.875, -5.5, -3.125,
    -5.75, -7.875, 22.5]; with bias b[n] = n/2 and ReLU every value is exact."""
    x, q, s = hand_inputs(8)
    y, _ = oracle_mod.gemm(x, q, s, 8)
    b = (np.arange(8) / 2.0).astype(np.float16)
    got = oracle_mod.epilogue(y, bias=b, activation="relu")[0]
    want = np.maximum(np.array([-4.125, -3.75, -4.875, -5.5, -3.125, -5.75, -7.875, 22.5]) + np.arange(8) / 2.0, 0.0)
    assert np.array_equal(got, want)


def test_epilogue_bf16_decodes_bias_and_residual_as_bfloat16(oracle_mod):
    z = np.array([[1.0, -2.0, 0.5]])
    b = np.array([0x3F80, 0xC000, 0x4300], np.uint16)          # 1, -2, 128 in bfloat16
    r = np.array([[0x3F00, 0x0000, 0xBF80]], np.uint16)        # 0.5, 0, -1
    got = oracle_mod.epilogue(z, bias=b, residual=r, activation="relu", dtype="bf16")
    assert np.array_equal(got, np.array([[2.5, 0.0, 127.5]]))


def test_epilogue_sampled_matches_full(oracle_mod):
    rng = np.random.default_rng(3)
    z = rng.standard_normal((6, 40))
    b = rng.standard_normal(40).astype(np.float16)
    r = rng.standard_normal((6, 40)).astype(np.float16)
    rows, cols = np.array([0, 5, 2]), np.array([39, 0, 17, 8])
    full = oracle_mod.epilogue(z, bias=b, residual=r, activation="silu")
    part = oracle_mod.epilogue(z[np.ix_(rows, cols)], bias=b, residual=r, activation="silu", rows=rows, cols=cols)
    assert np.array_equal(part, full[np.ix_(rows, cols)])
