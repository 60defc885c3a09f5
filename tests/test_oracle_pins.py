"""Pins for the CPU oracle: each check ties it to something other than itself
(exhaustive code tables, a brute-force search, a library routine on a special
case, exact rational arithmetic on tiny inputs, or an invariant of the math),
so that a dropped term, a wrong sign or index or a transposed operand fails."""
from fractions import Fraction
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import quantize as Q
from oracle import linear as L
from oracle import probe as P
from oracle import dispatch as D


# ---------------------------------------------------------------- E4M3 codes
def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan], lib[~nan])
    # sign of zero
    assert math.copysign(1.0, ours[0x80]) == -1.0 and math.copysign(1.0, ours[0x00]) == 1.0


def test_e4m3_named_values():
    golden = {}
    with open(__file__.replace("test_oracle_pins.py", "golden/e4m3_named_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                golden[int(c, 16)] = float(Fraction(v))
    assert len(golden) >= 8
    for c, v in golden.items():
        assert F.e4m3_decode_code(c) == v, hex(c)


def test_e4m3_round_trip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    back = F.e4m3_encode(vals)
    finite = ~np.isnan(vals)
    assert np.array_equal(back[finite], codes[finite])
    assert back[0x7F] == 0x7F and back[0xFF] == 0xFF


def _brute_force_encode(v: np.ndarray) -> np.ndarray:
    """Nearest of all 254 finite codes by exhaustive distance, ties -> even
    mantissa bit, magnitudes beyond 448 -> 448.  Independent of the table
    search in the oracle."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.int64)
    vals = np.array([F.e4m3_decode_code(int(c)) for c in codes])
    out = np.empty(v.shape, dtype=np.uint8)
    for i, x in enumerate(v.astype(np.float64)):
        if np.isnan(x):
            out[i] = 0xFF if np.signbit(x) else 0x7F
            continue
        xc = np.clip(x, -448.0, 448.0)
        d = np.abs(vals - xc)
        best = np.nonzero(d == d.min())[0]
        cand = codes[best]
        # same magnitude twice only for +-0: keep the sign of x
        if len(cand) > 1:
            even = [c for c in cand if (c & 1) == 0]
            if len(even) > 1:
                even = [c for c in even if ((c >> 7) & 1) == int(np.signbit(x))]
            cand = even
        out[i] = cand[0]
    return out


def test_e4m3_encode_all_bf16_patterns_vs_brute_force():
    v = W.all_bf16_patterns().to(torch.float32).numpy()
    ours = F.e4m3_encode(v)
    # brute force on every pattern whose magnitude is within 2x of the code
    # range plus a spread sample of the rest (the rest saturates or flushes)
    sel = np.nonzero((np.abs(v) < 1024) & (np.abs(v) > 2.0 ** -12) | np.isnan(v))[0]
    rest = np.setdiff1d(np.arange(v.size), sel)[::97]
    idx = np.concatenate([sel, rest])
    assert np.array_equal(ours[idx], _brute_force_encode(v[idx]))


def test_e4m3_encode_matches_torch_cast_in_range():
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest even; it does not
    # saturate (it gives NaN from 480 up), so compare below that.
    v = W.all_bf16_patterns().to(torch.float32)
    keep = torch.isfinite(v) & (v.abs() < 464)
    v = v[keep]
    lib = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.e4m3_encode(v.numpy())
    assert np.array_equal(ours, lib)


@pytest.mark.parametrize("x,code", [
    (448.0, 0x7E), (449.0, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (480.0, 0x7E), (1e30, 0x7E),
    (float("inf"), 0x7E), (-448.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE),
    (432.0, 0x7E),             # midpoint 416|448 -> even code 0x7E
    (1.0625, 0x38),            # midpoint 1|1.125 -> even code 0x38 (1.0)
    (1.1875, 0x3A),            # midpoint 1.125|1.25 -> even code 0x3A (1.25)
    (2.0 ** -10, 0x00),        # midpoint 0|2^-9 -> 0
    (-(2.0 ** -10), 0x80),
    (3 * 2.0 ** -10, 0x02),    # midpoint 2^-9|2^-8 -> code 2
    (2.0 ** -11, 0x00), (0.0, 0x00), (-0.0, 0x80),
    (0.875 * 2.0 ** -6, 0x07), (2.0 ** -6, 0x08),
])
def test_e4m3_saturation_and_ties(x, code):
    assert int(F.e4m3_encode(np.float32(x))) == code


# --------------------------------------------------------------- E8M0 / MX
def test_e8m0_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    ours = F.e8m0_decode(codes)
    assert np.isnan(ours[255]) and np.isnan(lib[255])
    assert np.array_equal(ours[:255], lib[:255])


def test_mx_exponent_brackets_block_amax():
    rng = np.random.default_rng(1)
    am = np.abs(rng.standard_normal(20000).astype(np.float32)) * np.float32(2.0) ** rng.integers(-100, 100, 20000).astype(np.float32)
    am = am[(am > 0) & np.isfinite(am)]
    e = Q.mx_exponent(am)
    scaled = am.astype(np.float64) * np.ldexp(1.0, -e)
    inside = (e > -127) & (e < 127)
    assert np.all((scaled[inside] >= 256.0) & (scaled[inside] < 512.0))
    # an independent formula on exact powers of two
    for p in range(-119, 128):
        assert Q.mx_exponent(np.float32(2.0 ** p)) == p - 8
        if p < 127:
            assert Q.mx_exponent(np.float32(2.0 ** p * 1.999)) == p - 8


def test_mx_exponent_clamp_and_zero():
    assert Q.mx_exponent(np.float32(0.0)) == -127
    assert Q.mx_exponent(np.float32(2.0 ** -130)) == -127      # subnormal
    assert Q.mx_exponent(np.float32(3.0e38)) == 127 - 8
    q, s = Q.quantize_mx(np.zeros((2, 64), np.float32))
    assert np.all(q == 0) and np.all(s == 0)


def test_mx_quantize_small_block_by_hand():
    # one block: amax 3.0 -> floor(log2 3) = 1 -> e = -7 -> code 120, x * 2^7
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 3.0
    x[0, 1] = -0.01
    x[0, 2] = 1.0
    q, s = Q.quantize_mx(x)
    assert int(s[0, 0]) == 120
    assert F.e4m3_decode_code(int(q[0, 0])) == 384.0                # 3 * 128
    assert F.e4m3_decode_code(int(q[0, 2])) == 128.0
    # -0.01 * 128 = -1.28 -> nearest E4M3 is -1.25
    assert F.e4m3_decode_code(int(q[0, 1])) == -1.25


# ------------------------------------------------ square 32x32 block scales
def test_block32_is_transpose_invariant():
    # GEM "Low Precision Flash Attention": one scale per 32x32 block, so
    # quantizing X^T gives the transposed codes and scales of X
    x = W.random_bf16((96, 160), seed=12, dist="laplace", outlier_frac=0.02)
    q, s = Q.quantize_block32(x)
    qt, st = Q.quantize_block32(x.t().contiguous())
    assert s.shape == (3, 5) and st.shape == (5, 3)
    assert np.array_equal(q.T, qt) and np.array_equal(s.T, st)


def test_block32_codes_by_brute_force_and_frexp():
    x = W.random_bf16((70, 64), seed=13, outlier_frac=0.05)      # a ragged last block row
    q, s = Q.quantize_block32(x)
    xf = Q.as_f32(x).astype(np.float64)
    assert s.shape == (3, 2)
    for rb in range(3):
        for cb in range(2):
            blk = xf[rb * 32:(rb + 1) * 32, cb * 32:(cb + 1) * 32]
            _, p = np.frexp(np.abs(blk).max())
            e = p - 1 - 8
            assert int(s[rb, cb]) == e + 127
            prod = np.ldexp(blk, -e).astype(np.float32)
            assert np.array_equal(q[rb * 32:(rb + 1) * 32, cb * 32:(cb + 1) * 32].ravel(),
                                  _brute_force_encode(prod.ravel()))


def test_block32_equals_mx_when_every_row_holds_the_block_amax():
    # when each row of a 32x32 block reaches the block's amax, the per-row
    # 1x32 (MX) exponents are the block's: the two quantizations coincide
    rng = np.random.default_rng(14)
    xf = rng.standard_normal((64, 96)).astype(np.float32)
    for rb in range(2):
        for cb in range(3):
            a = np.float32(2.0 ** rng.integers(-6, 6) * 1.5)
            xf[rb * 32:(rb + 1) * 32, cb * 32] = a
            xf[rb * 32:(rb + 1) * 32, cb * 32 + 1:(cb + 1) * 32] = np.clip(
                xf[rb * 32:(rb + 1) * 32, cb * 32 + 1:(cb + 1) * 32], -a, a)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    qb, sb = Q.quantize_block32(x)
    qm, sm = Q.quantize_mx(x)
    assert np.array_equal(qb, qm)
    assert np.array_equal(np.repeat(sb, 32, axis=0), sm)


def test_block32_layer_dequantizes_with_block_row_scales():
    # prenorm with square blocks equals the float64 product of the
    # dequantized operands, each element scaled by its block's 2^e
    inp = W.make_layer(70, 128, 64, mode=4, norm=L.NORM_NONE, seed=15)
    v, ops = L.prenorm(inp.x, inp.w, None, 4)
    qx, sx, qw, sw = ops.get("qx"), ops.get("sx"), ops.get("qw"), ops.get("sw")
    if qx is None:
        qx, sx = Q.quantize_block32(inp.x)
        qw, sw = Q.quantize_block32(inp.w)
    dx = F.e4m3_decode(qx) * np.ldexp(1.0, np.repeat(np.repeat(sx.astype(np.int64) - 127, 32, 0)[:70], 32, 1))
    dw = F.e4m3_decode(qw) * np.ldexp(1.0, np.repeat(np.repeat(sw.astype(np.int64) - 127, 32, 0)[:64], 32, 1))
    assert np.allclose(v, dx @ dw.T, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------- tensor / row scales
def test_rowwise_amax_element_maps_to_448_and_error_bound():
    x = W.random_bf16((64, 256), seed=3, outlier_frac=0.02)
    q, s = Q.quantize_rows(x)
    xf = Q.as_f32(x).astype(np.float64)
    vals = F.e4m3_decode(q)
    assert np.all(np.max(np.abs(vals), axis=1) == 448.0)
    # per element: |decode(q) - x*inv| <= half the E4M3 spacing at that size
    inv = 448.0 / np.max(np.abs(xf), axis=1)
    y = xf * inv[:, None]
    a = np.abs(y)
    _, p = np.frexp(np.maximum(a, 2.0 ** -6))
    spacing = np.ldexp(1.0, p - 1 - 3)
    assert np.all(np.abs(vals - y) <= spacing / 2 * (1 + 1e-6))
    # scale is amax / 448 in float32
    am = np.max(np.abs(Q.as_f32(x)), axis=1)
    assert np.array_equal(s, (am / np.float32(448.0)).astype(np.float32))


def test_tensorwise_matches_torch_e4m3_cast():
    x = W.random_bf16((96, 128), seed=5)
    q, s = Q.quantize_tensor(x)
    xf = x.to(torch.float32)
    am = xf.abs().max()
    inv = torch.tensor(448.0, dtype=torch.float32) / am
    lib = (xf * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, lib)
    assert s == np.float32(am.item() / np.float32(448.0))


def test_zero_rows_get_unit_scale():
    x = torch.zeros((3, 64), dtype=torch.bfloat16)
    q, s = Q.quantize_rows(x)
    assert np.all(q == 0) and np.all(s == 1.0)
    q, s = Q.quantize_tensor(x)
    assert np.all(q == 0) and s == 1.0


# ----------------------------------------------------------------- GEMM
def _fraction_gemm(qx, qw):
    dx = [[Fraction(F.e4m3_decode_code(int(c))) for c in row] for row in qx]
    dw = [[Fraction(F.e4m3_decode_code(int(c))) for c in row] for row in qw]
    return [[sum(a * b for a, b in zip(rx, rw)) for rw in dw] for rx in dx]


def test_gemm_exact_vs_rational_brute_force():
    rng = np.random.default_rng(7)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qx = rng.choice(finite, size=(5, 37))
    qw = rng.choice(finite, size=(3, 37))
    got = L.gemm_exact(qx, qw)
    want = _fraction_gemm(qx, qw)
    assert got.shape == (5, 3)
    for m in range(5):
        for n in range(3):
            assert Fraction(got[m, n]) == want[m][n]


def test_gemm_identity_weight():
    x = W.random_bf16((8, 32), seed=9)
    qx, _ = Q.quantize_rows(x)
    eye = np.zeros((32, 32), np.uint8)
    eye[np.arange(32), np.arange(32)] = 0x38     # 1.0
    assert np.array_equal(L.gemm_exact(qx, eye), F.e4m3_decode(qx))


def test_prenorm_rowwise_vs_rational_brute_force():
    inp = W.make_layer(4, 64, 5, mode=W.SCALE_ROW, norm=W.NORM_NONE, seed=11, bias_var=0.5, outlier_frac=0.05)
    v, ops = L.prenorm(inp.x, inp.w, inp.bias, W.SCALE_ROW)
    acc = _fraction_gemm(ops["qx"], ops["qw"])
    b = Q.as_f32(inp.bias)
    for m in range(4):
        for n in range(5):
            want = acc[m][n] * Fraction(float(ops["sx"][m])) * Fraction(float(ops["sw"][n])) + Fraction(float(b[n]))
            assert abs(Fraction(v[m, n]) - want) <= abs(want) * Fraction(1, 2 ** 50)


def test_prenorm_mx_vs_rational_brute_force():
    inp = W.make_layer(3, 96, 4, mode=W.SCALE_MX32, norm=W.NORM_NONE, seed=12, x_dist="laplace")
    v, ops = L.prenorm(inp.x, inp.w, None, W.SCALE_MX32)
    for m in range(3):
        for n in range(4):
            want = Fraction(0)
            for k in range(96):
                ex = int(ops["sx"][m, k // 32]) - 127
                ew = int(ops["sw"][n, k // 32]) - 127
                want += Fraction(F.e4m3_decode_code(int(ops["qx"][m, k]))) * Fraction(2) ** ex \
                    * Fraction(F.e4m3_decode_code(int(ops["qw"][n, k]))) * Fraction(2) ** ew
            assert abs(Fraction(v[m, n]) - want) <= abs(want) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 200)


def test_prenorm_bf16_matches_torch_double_linear():
    inp = W.make_layer(16, 64, 24, mode=W.SCALE_BF16, norm=W.NORM_NONE, seed=13, bias_var=0.1)
    v, _ = L.prenorm(inp.x, inp.w, inp.bias, W.SCALE_BF16)
    lib = torch.nn.functional.linear(inp.x.double(), inp.w.double(), inp.bias.double()).numpy()
    np.testing.assert_allclose(v, lib, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------ normalization
def test_layernorm_matches_torch_and_invariants():
    rng = np.random.default_rng(15)
    v = rng.standard_normal((32, 256)) * 3 + 1
    g = rng.uniform(0.5, 1.5, 256)
    b = rng.standard_normal(256)
    ours = L.layernorm(v, g, b, 1e-5)
    lib = torch.nn.functional.layer_norm(torch.from_numpy(v), (256,), torch.from_numpy(g), torch.from_numpy(b), 1e-5).numpy()
    np.testing.assert_allclose(ours, lib, rtol=1e-12, atol=1e-12)
    plain = L.layernorm(v, np.ones(256), np.zeros(256), 1e-5)
    var = v.var(axis=1)
    assert np.all(np.abs(plain.mean(axis=1)) < 1e-12)
    np.testing.assert_allclose((plain ** 2).mean(axis=1), var / (var + 1e-5), rtol=1e-12)


def test_rmsnorm_matches_torch_and_invariants():
    rng = np.random.default_rng(16)
    v = rng.standard_normal((32, 256)) * 2 + 0.5
    g = rng.uniform(0.5, 1.5, 256)
    ours = L.rmsnorm(v, g, 1e-6)
    lib = torch.nn.functional.rms_norm(torch.from_numpy(v), (256,), torch.from_numpy(g), 1e-6).numpy()
    np.testing.assert_allclose(ours, lib, rtol=1e-12, atol=1e-12)
    plain = L.rmsnorm(v, np.ones(256), 1e-6)
    m2 = (v * v).mean(axis=1)
    np.testing.assert_allclose((plain ** 2).mean(axis=1), m2 / (m2 + 1e-6), rtol=1e-12)


def test_layernorm_degenerate_rows():
    v = np.full((2, 8), 3.25)
    beta = np.arange(8, dtype=np.float64)
    np.testing.assert_array_equal(L.layernorm(v, np.ones(8), beta, 1e-5), np.tile(beta, (2, 1)))
    np.testing.assert_array_equal(L.layernorm(np.ones((1, 1)), np.ones(1), np.full(1, 0.5), 1e-5), [[0.5]])


def test_linear_norm_end_to_end_vs_library_composition():
    """Per-row FP8 layer composed from torch's own E4M3 cast, float64 matmul
    and layer_norm; agrees with the oracle to float64 rounding."""
    inp = W.make_layer(24, 128, 32, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=17, bias_var=0.02, outlier_frac=0.01)
    y, yb, _ = L.linear_norm_inputs(inp)
    xf, wf = inp.x.float(), inp.w.float()
    ax = xf.abs().amax(dim=1, keepdim=True)
    aw = wf.abs().amax(dim=1, keepdim=True)
    qx = (xf * (torch.tensor(448.0) / ax)).to(torch.float8_e4m3fn).double()
    qw = (wf * (torch.tensor(448.0) / aw)).to(torch.float8_e4m3fn).double()
    v = (qx @ qw.T) * (ax / torch.tensor(448.0)).double() * (aw / torch.tensor(448.0)).double().T + inp.bias.double()
    lib = torch.nn.functional.layer_norm(v, (32,), eps=inp.eps).numpy()
    np.testing.assert_allclose(y, lib, rtol=1e-11, atol=1e-11)
    # the bf16 output is the nearest bf16 of the exact value
    assert np.all(np.abs(yb - y) <= F.bf16_ulp(y) / 2)


# ------------------------------------------------------------- bf16 rounding
# ------------------------------------- probe: online input statistics, sampler
from oracle import probe_stats as PS


def test_chan_merge_equals_two_pass_statistics_of_all_rows():
    # merging batches of any sizes gives the mean and scatter of the
    # concatenated rows, computed directly in two passes (closed form)
    rng = np.random.default_rng(20)
    K = 24
    batches = [rng.standard_normal((b, K)) * rng.uniform(0.5, 3.0, K) + rng.uniform(-2, 2, K)
               for b in (7, 1, 64, 129, 3)]
    n, mu, S = 0, np.zeros(K), np.zeros((K, K))
    for xb in batches:
        n, mu, S = PS.stats_update(n, mu, S, xb)
    allx = np.concatenate(batches)
    m = allx.mean(axis=0)
    assert n == allx.shape[0]
    assert np.allclose(mu, m, rtol=0, atol=1e-13)
    assert np.allclose(S, (allx - m).T @ (allx - m), rtol=1e-12, atol=1e-11)
    # the unbiased covariance is numpy's (a library routine)
    assert np.allclose(PS.covariance(n, S), np.cov(allx, rowvar=False), rtol=1e-12, atol=1e-12)


def test_chan_merge_first_batch_and_empty_batch():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((10, 5))
    n, mu, S = PS.stats_update(0, np.zeros(5), np.zeros((5, 5)), x)
    assert n == 10 and np.allclose(mu, x.mean(0)) and np.allclose(S, (x - x.mean(0)).T @ (x - x.mean(0)))
    n2, mu2, S2 = PS.stats_update(n, mu, S, np.zeros((0, 5)))
    assert n2 == n and np.array_equal(mu2, mu) and np.array_equal(S2, S)


def test_stream_normals_have_normal_moments_and_uniform_bits():
    # invariants of the generator: the 24-bit uniforms are uniform (chi-square
    # over 64 bins) and the Box-Muller pairs have N(0,1) moments
    r = PS.splitmix64(7, np.arange(1 << 18, dtype=np.uint64))
    bins = np.bincount((r >> np.uint64(58)).astype(np.int64), minlength=64)
    chi2 = ((bins - bins.mean()) ** 2 / bins.mean()).sum()
    assert chi2 < 63 + 5 * np.sqrt(2 * 63)
    z = PS.normals(7, 1 << 18)
    n = z.size
    assert abs(z.mean()) < 4 / np.sqrt(n)
    assert abs(z.var() - 1) < 4 * np.sqrt(2 / n)
    assert abs((z ** 4).mean() - 3) < 4 * np.sqrt(96 / n)
    assert abs(np.corrcoef(z[0::2], z[1::2])[0, 1]) < 4 / np.sqrt(n / 2)
    # different seeds give different streams; a seed's stream is reproducible
    assert not np.array_equal(PS.normals(8, 64), PS.normals(7, 64))
    assert np.array_equal(PS.normals(7, 64), z[:64])


def test_cholesky_factor_reproduces_the_regularized_covariance():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((50, 12)) @ rng.standard_normal((12, 12))
    n, mu, S = PS.stats_update(0, np.zeros(12), np.zeros((12, 12)), x)
    L = PS.cholesky_factor(n, S, 1e-3)
    sigma = np.cov(x, rowvar=False)
    assert np.allclose(np.triu(L, 1), 0) and (np.diag(L) > 0).all()
    assert np.allclose(L @ L.T, sigma + 1e-3 * np.trace(sigma) / 12 * np.eye(12), rtol=1e-12, atol=1e-12)


def test_sampler_reproduces_mean_and_covariance():
    rng = np.random.default_rng(22)
    K = 16
    A = rng.standard_normal((K, K))
    sigma = A @ A.T / K + 0.1 * np.eye(K)
    L = np.linalg.cholesky(sigma)
    mu = rng.uniform(-1, 1, K)
    Z, T = PS.sample_inputs(mu, L, 40000, seed=3)
    assert np.allclose(T - mu, Z @ L.T)
    assert np.allclose(T.mean(0), mu, atol=5 * np.sqrt(np.diag(sigma).max() / 40000))
    assert np.allclose(np.cov(T, rowvar=False), sigma, atol=0.05 * np.abs(sigma).max())


# ------------------------------------------------- BlockNorm and Hard Swish
@pytest.mark.parametrize("block", [32, 64, 128, 256])
def test_blocknorm_is_rms_norm_of_the_blocked_view(block):
    # LoKA III-B 2: RMSNorm((Wx + b).view(-1, BlockN)).view(B, N); torch's
    # rms_norm on that view is an independent library routine
    rng = np.random.default_rng(block)
    M, N, eps = 6, 512, 1e-6
    v = rng.standard_normal((M, N)) * rng.uniform(0.1, 10.0, (M, 1))
    g = rng.uniform(0.5, 1.5, N)
    ours = L.blocknorm(v, g, eps, block)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(v).view(-1, block), (block,), eps=eps).view(M, N).numpy()
    assert np.allclose(ours, ref * g[None, :], rtol=1e-13, atol=1e-13)
    # gamma = 1: every block's mean square is ms / (ms + eps)
    y = L.blocknorm(v, np.ones(N), eps, block).reshape(M, N // block, block)
    ms = (v.reshape(M, N // block, block) ** 2).mean(axis=2)
    assert np.allclose((y ** 2).mean(axis=2), ms / (ms + eps), rtol=1e-12)


def test_blocknorm_over_the_whole_row_is_rmsnorm():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((4, 256))
    g = rng.uniform(0.5, 1.5, 256)
    assert np.allclose(L.blocknorm(v, g, 1e-6, 256), L.rmsnorm(v, g, 1e-6), rtol=0, atol=0)


def test_hardswish_matches_torch_and_known_points():
    x = np.concatenate([np.linspace(-8, 8, 4001), [-3.0, -1.5, 0.0, 3.0, -3.0000001, 2.9999999]])
    ref = torch.nn.functional.hardswish(torch.from_numpy(x)).numpy()
    assert np.allclose(L.hardswish(x), ref, rtol=1e-15, atol=1e-15)
    assert L.hardswish(np.array([-3.0]))[0] == 0.0 and L.hardswish(np.array([3.0]))[0] == 3.0
    assert L.hardswish(np.array([-1.5]))[0] == -0.375              # the minimum
    assert np.all(L.hardswish(np.array([-5.0, -100.0])) == 0.0)
    assert np.all(L.hardswish(np.array([4.0, 50.0])) == np.array([4.0, 50.0]))


def test_layer_applies_hard_swish_after_the_norm():
    inp = W.make_layer(16, 128, 256, mode=L.SCALE_ROW, norm=L.NORM_BLOCK_RMS, seed=9, gamma_uniform=True)
    inp.norm_block = 64
    y0, _, _ = L.linear_norm_inputs(inp)
    inp.act = L.ACT_HARDSWISH
    y1, _, _ = L.linear_norm_inputs(inp)
    assert np.array_equal(y1, L.hardswish(y0))


# ------------------------------------- quantized output for the next layer
def test_quantized_output_rowwise_is_the_quantized_bf16_output():
    # per row: the largest |bf16 output| maps to 448, the scale is amax/448,
    # and every code is the nearest E4M3 value (brute force) of the fp32
    # product bf16(y) * fl32(448/amax)
    M, N = 40, 64
    inp = W.make_layer(M, 128, N, mode=L.SCALE_ROW, norm=L.NORM_LAYER, seed=21, bias_var=0.02, gamma_uniform=True)
    inp.beta = W.random_bf16((N,), seed=22, var=0.1)
    y, yb, q, s = L.linear_norm_quantized_inputs(inp, L.SCALE_ROW)
    assert q.shape == (M, N) and s.shape == (M,)
    _, yb_plain, _ = L.linear_norm_inputs(inp)
    assert np.array_equal(yb, yb_plain)
    vals = F.e4m3_decode(q)
    assert np.all(np.max(np.abs(vals), axis=1) == 448.0)
    am = np.max(np.abs(yb), axis=1).astype(np.float32)
    inv = np.array([np.float32(448.0) / a for a in am], dtype=np.float32)
    assert np.array_equal(s, np.array([a / np.float32(448.0) for a in am], dtype=np.float32))
    prod = (yb.astype(np.float32) * inv[:, None]).astype(np.float32)
    assert np.array_equal(q.ravel(), _brute_force_encode(prod.ravel()))
    # the codes are those of bf16(y), not of the unrounded y: some differ
    prod_exact = (y.astype(np.float32) * inv[:, None]).astype(np.float32)
    assert not np.array_equal(q.ravel(), _brute_force_encode(prod_exact.ravel()))


def test_quantized_output_mx_blocks_run_along_the_output_row():
    # one E8M0 exponent per 32 consecutive output columns of a row, from
    # frexp (amax = f 2^p, f in [0.5, 1), so floor(log2 amax) = p - 1)
    M, N = 24, 96
    inp = W.make_layer(M, 128, N, mode=L.SCALE_MX32, norm=L.NORM_RMS, seed=23, gamma_uniform=True, eps=1e-6)
    y, yb, q, s = L.linear_norm_quantized_inputs(inp, L.SCALE_MX32)
    assert s.shape == (M, N // 32) and s.dtype == np.uint8
    blocks = yb.reshape(M, N // 32, 32)
    _, p = np.frexp(np.abs(blocks).max(axis=2))
    e = p - 1 - 8
    assert np.array_equal(s.astype(np.int64), e + 127)
    prod = np.ldexp(blocks, -e[:, :, None]).astype(np.float32)     # exact: a power of two
    assert np.array_equal(q.ravel(), _brute_force_encode(prod.ravel()))


def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(18)
    v = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(F.bf16_round(v.astype(np.float64)), lib)


def test_bf16_round_ties_and_near_ties():
    one_ulp = 2.0 ** -7
    assert F.bf16_round(np.float64(1.0 + one_ulp / 2))[()] == 1.0                       # tie -> even
    assert F.bf16_round(np.float64(1.0 + 3 * one_ulp / 2))[()] == 1.0 + 2 * one_ulp     # tie -> even
    assert F.bf16_round(np.float64(1.0 + one_ulp / 2 + 2.0 ** -40))[()] == 1.0 + one_ulp


# ------------------------------------------------------------------ MERE
def test_mere_hand_vectors():
    ref = np.array([[1.0, -2.0, 4.0, 0.0]])
    out = ref * 1.1
    m, z = P.mere(out, ref)
    assert z == 1 and abs(m - 0.1) < 1e-15
    out2 = ref + np.array([[0.5, 0.0, 0.0, 7.0]])
    m2, _ = P.mere(out2, ref)
    assert abs(m2 - (0.5 / 1.0) / 3) < 1e-15
    assert abs(P.normwise(ref * 1.25, ref) - 0.25) < 1e-15
    assert P.max_abs(out2, ref) == 7.0
    # scale invariance
    assert abs(P.mere(out * 1e-7, ref * 1e-7)[0] - m) < 1e-12


def test_quant_error_bf16_is_zero_and_fp8_is_small():
    inp = W.make_layer(32, 128, 16, mode=W.SCALE_ROW, norm=W.NORM_NONE, seed=19)
    s = P.quant_error(inp.x, inp.w, None, W.SCALE_BF16)
    assert s["mere"] == 0.0 and s["rel_err_fro"] == 0.0
    s = P.quant_error(inp.x, inp.w, None, W.SCALE_ROW)
    assert 0.0 < s["rel_err_fro"] < 0.1
    assert s["max_abs_post_norm"] == s["max_abs"]      # no norm, no activation


def test_quant_error_post_norm_against_torch_layer_norm():
    # the post-norm error is the largest difference of the two outputs after
    # the layer's LayerNorm: recomputed here from the pre-norm outputs with
    # torch's own layer_norm (an independent library routine, float64)
    import torch
    inp = W.make_layer(40, 128, 64, mode=W.SCALE_ROW, norm=W.NORM_LAYER, seed=23, bias_var=0.02,
                       gamma_uniform=True)
    beta = W.random_bf16((64,), seed=2, var=0.1)
    s = P.quant_error(inp.x, inp.w, inp.bias, W.SCALE_ROW, norm=W.NORM_LAYER, gamma=inp.gamma, beta=beta, eps=1e-5)
    out, _ = L.prenorm(inp.x, inp.w, inp.bias, W.SCALE_ROW)
    ref, _ = L.prenorm(inp.x, inp.w, inp.bias, W.SCALE_BF16)
    g = inp.gamma.to(torch.float64)
    b = beta.to(torch.float64)
    ln = lambda v: torch.nn.functional.layer_norm(torch.from_numpy(v), (64,), g, b, eps=1e-5).numpy()
    want = float(np.max(np.abs(ln(out) - ln(ref))))
    assert abs(s["max_abs_post_norm"] - want) <= 1e-12 * max(1.0, want)
    assert s["max_abs_post_norm"] > 0.0
    # RMSNorm with an activation after it: the same definition
    s2 = P.quant_error(inp.x, inp.w, inp.bias, W.SCALE_ROW, norm=W.NORM_RMS, gamma=inp.gamma, eps=1e-6, act=1)
    rms = lambda v: torch.nn.functional.rms_norm(torch.from_numpy(v), (64,), g, eps=1e-6)
    hs = lambda v: torch.nn.functional.hardswish(rms(v)).numpy()
    want2 = float(np.max(np.abs(hs(out) - hs(ref))))
    assert abs(s2["max_abs_post_norm"] - want2) <= 1e-12 * max(1.0, want2)


# --------------------------------------------------------------- dispatch
def _e(M, variant, t, rel=1e-3, mere=0.05, N=256, K=512, norm=1, o=0.0):
    return D.Entry(M, N, K, norm, o, variant, t, rel, mere)


def test_dispatch_picks_fastest_within_budget():
    tab = [_e(65536, 0, 10.0, rel=0.02), _e(65536, 1, 12.0), _e(65536, 2, 11.0), _e(65536, 3, 20.0)]
    assert D.select(tab, 65536, 256, 512, 1, 0.0) == 2          # 0 fails rel_err
    assert D.select(tab, 65536, 256, 512, 1, 0.0, D.Policy(max_rel_err=0.05)) == 0


def test_dispatch_speedup_and_mere_filters_and_fallback():
    tab = [_e(4096, 1, 9.8), _e(4096, 2, 9.0, mere=0.3), _e(4096, 3, 10.0)]
    # row 1: speedup 10/9.8 = 1.02 < 1.05 ; row 2: MERE 0.3 >= 0.2
    assert D.select(tab, 4096, 256, 512, 1, 0.0, D.Policy(min_speedup=1.05)) == 3
    assert D.select(tab, 4096, 256, 512, 1, 0.0, D.Policy(min_speedup=1.0)) == 1
    assert D.select(tab, 4096, 256, 512, 1, 0.0, D.Policy(max_mere=-1)) == 2
    assert D.select([], 4096, 256, 512, 1, 0.0) == 3
    assert D.select(tab, 4096, 128, 512, 1, 0.0) == 3           # no row for N


def test_dispatch_bucket_and_ties():
    tab = [_e(4096, 1, 5.0), _e(16384, 2, 5.0), _e(16384, 1, 6.0),
           _e(16384, 0, 5.0, rel=5e-4), _e(16384, 2, 5.0, o=0.01)]
    # M=8192 is equidistant in log2 from 4096 and 16384 -> larger M bucket
    assert D.select(tab, 8192, 256, 512, 1, 0.0) == 0            # tie on time -> smaller rel_err
    assert D.select(tab, 5000, 256, 512, 1, 0.0) == 1
    assert D.select(tab, 16384, 256, 512, 1, 0.02) == 2          # nearest outlier regime


def test_dispatch_brute_force_random_tables():
    rng = np.random.default_rng(21)
    for trial in range(200):
        tab = [_e(4096, int(v), float(rng.uniform(1, 3)), rel=float(rng.uniform(0, 0.02)),
                  mere=float(rng.uniform(0, 0.3))) for v in rng.permutation(4)]
        pol = D.Policy(max_rel_err=0.01, max_mere=0.2, min_speedup=1.05)
        got = D.select(tab, 4096, 256, 512, 1, 0.0, pol)
        t_ref = [e.time_us for e in tab if e.variant == 3][0]
        ok = [e for e in tab if e.variant != 3 and e.rel_err <= 0.01 and e.mere < 0.2 and t_ref / e.time_us > 1.05]
        want = min(ok, key=lambda e: e.time_us).variant if ok else 3
        assert got == want


# ------------------------------------------------- probe: weight model
from oracle import probe_weights as PW


def _spd(n, seed, cond=5.0):
    rng = np.random.default_rng(seed)
    q, _ = np.linalg.qr(rng.standard_normal((n, n)))
    return (q * np.linspace(1.0, cond, n)) @ q.T


def test_weight_model_second_update_closed_form():
    # After the first update (M = W1, U = I, V = I) and with no jitter, the
    # second update is: Wc = W2 - W1, U' = Wc Wc^T / C, V' = Wc^T Wc / R,
    # U = m I + (1-m) U', V = m I + (1-m) V' (already symmetric), then
    # s = trace(U) / R, U / s, V * s, M = m W1 + (1-m) W2.  Written out here
    # element by element.
    rng = np.random.default_rng(3)
    R, C, m = 4, 3, 0.9
    W1, W2 = rng.standard_normal((R, C)), rng.standard_normal((R, C))
    st = PW.weight_update(None, W1, m, 0.0)
    assert st.n == 1 and np.array_equal(st.M, W1) and np.array_equal(st.U, np.eye(R))
    st = PW.weight_update(st, W2, m, 0.0)
    d = W2 - W1
    U = np.array([[m * (i == j) + (1 - m) * sum(d[i, k] * d[j, k] for k in range(C)) / C for j in range(R)]
                  for i in range(R)])
    V = np.array([[m * (i == j) + (1 - m) * sum(d[k, i] * d[k, j] for k in range(R)) / R for j in range(C)]
                  for i in range(C)])
    s = sum(U[i, i] for i in range(R)) / R
    assert np.allclose(st.U, U / s, rtol=1e-12, atol=1e-14)
    assert np.allclose(st.V, V * s, rtol=1e-12, atol=1e-14)
    assert np.allclose(st.M, m * W1 + (1 - m) * W2, rtol=0, atol=1e-15)


def test_weight_model_invariants_every_update():
    rng = np.random.default_rng(4)
    st = None
    for t in range(20):
        st = PW.weight_update(st, rng.standard_normal((6, 5)) * (1 + t % 3), 0.9, 1e-6)
        assert abs(np.trace(st.U) - 6) < 1e-9                      # the scale renormalization
        assert np.array_equal(st.U, st.U.T) and np.array_equal(st.V, st.V.T)
        assert np.linalg.eigvalsh(st.U).min() > 0 and np.linalg.eigvalsh(st.V).min() > 0


def test_weight_model_recovers_a_known_kronecker_covariance():
    # weights drawn from MN(M0, U0, V0): the tracked V (x) U approaches
    # V0 (x) U0 (the pair itself is defined up to (cU, V/c)) and M
    # approaches M0
    R, C = 6, 5
    U0, V0 = _spd(R, 11), _spd(C, 12)
    LU0, LV0 = np.linalg.cholesky(U0), np.linalg.cholesky(V0)
    rng = np.random.default_rng(13)
    M0 = rng.standard_normal((R, C))
    st = None
    for _ in range(3000):
        st = PW.weight_update(st, M0 + LU0 @ rng.standard_normal((R, C)) @ LV0.T, 0.995, 1e-6)
    want = np.kron(V0, U0)
    got = np.kron(st.V, st.U)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 0.15
    assert np.abs(st.M - M0).max() < 0.5
    # a transposed Kronecker order (U (x) V) is far off
    assert np.linalg.norm(np.kron(st.U, st.V) - want) / np.linalg.norm(want) > 0.3


def test_weight_sampler_has_the_kronecker_covariance():
    # vec(W') of the sampler: mean vec(M), covariance V (x) U (plus the
    # jitter), checked on the sample moments of many seeds
    R, C = 4, 3
    st = PW.WeightStats(5, np.arange(R * C, dtype=np.float64).reshape(R, C) / 7.0, _spd(R, 21), _spd(C, 22))
    samples = np.stack([PW.weight_sample(st, 1e-6, seed)[1].T.reshape(-1) for seed in range(6000)])
    mean = samples.mean(axis=0)
    cov = np.cov(samples.T)
    assert np.abs(mean - st.M.T.reshape(-1)).max() < 0.15
    want = np.kron(st.V, st.U)
    assert np.linalg.norm(cov - want) / np.linalg.norm(want) < 0.06


def test_forward_solve_residual():
    rng = np.random.default_rng(5)
    L = np.tril(rng.standard_normal((7, 7))) + 7 * np.eye(7)
    B = rng.standard_normal((7, 4))
    X = PW.forward_solve(L, B)
    assert np.abs(L @ X - B).max() < 1e-12
