"""The FMA-pipe exponential of the tensor-core softmax (ex2_fma2 in
csrc/common.cuh): its cubic is re-derived here from its stated method, and
the device steps, restated in numpy with fp32 rounding, stay within the
stated error bound over the whole range the softmax feeds it, with masked
scores (-inf) giving exactly 0."""
import os
import re

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
COMMON = os.path.join(HERE, "..", "varlen_flashattention_causal_gb300", "csrc", "common.cuh")


def constants():
    src = open(COMMON).read()
    out = {}
    for k in "ABC":
        m = re.search(r"constexpr float kEx2Poly%s = ([0-9.eE+-]+)f;" % k, src)
        assert m, k
        out[k] = float(m.group(1))
    return out


def lawson_fit(iters=2000):
    """Minimax relative error of 1 + f (a + f (b + f c)) against 2^f on
    [0, 1] with a + b + c = 1, by iteratively reweighted least squares."""
    f = np.linspace(0.0, 1.0, 20001)
    y = 2.0 ** f
    A = np.stack([(f ** 2 - f) / y, (f ** 3 - f) / y], 1)
    rhs = (y - 1 - f) / y
    w = np.full_like(f, 1.0 / len(f))
    for _ in range(iters):
        sw = np.sqrt(w)
        coef, *_ = np.linalg.lstsq(A * sw[:, None], rhs * sw, rcond=None)
        err = np.abs(A @ coef - rhs)
        w = w * err
        w /= w.sum()
    b, c = coef
    return 1.0 - b - c, b, c


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fma32(a, b, c):
    # a * b is exact in fp64 for fp32 operands; one rounding to fp32 after
    return f32(a.astype(np.float64) * b + c)


def ex2_fma2_model(x):
    k = constants()
    x = np.fmax(f32(x), np.float32(-127.0))              # fmaxf: NaN -> -127
    j = np.floor(x.astype(np.float64))                    # the add rounded toward -inf
    t = f32(12582912.0 + j)
    f = f32(x.astype(np.float64) - (t.astype(np.float64) - 12582912.0))
    q = fma32(f, np.float32(k["C"]), np.float32(k["B"]))
    q = fma32(q, f, np.float32(k["A"]))
    q = fma32(q, f, np.float32(1.0))
    bits = (q.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_constants_follow_the_stated_fit():
    a, b, c = lawson_fit()
    k = constants()
    assert abs(k["A"] - a) < 1e-6 and abs(k["B"] - b) < 1e-6 and abs(k["C"] - c) < 1e-6
    f = np.linspace(0, 1, 100001)
    p = 1 + f * (a + f * (b + f * c))
    assert np.max(np.abs(p / 2.0 ** f - 1)) < 1.04e-4


def test_relative_error_over_the_softmax_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-126.0, 8.0, 400001), rng.uniform(-30, 8, 200000),
                        np.arange(-126, 9, dtype=np.float64), np.arange(-126, 8) + 0.5])
    x = f32(x)
    got = ex2_fma2_model(x).astype(np.float64)
    ref = 2.0 ** x.astype(np.float64)
    rel = np.abs(got / ref - 1)
    assert rel.max() < 1.1e-4, (x[rel.argmax()], rel.max())


def test_masked_scores_give_exact_zero():
    x = f32([-np.inf, -1e30, -1000.0, -127.0, -127.0 - 2 ** -16, np.nan])
    got = ex2_fma2_model(x)
    assert np.all(got == 0) and not np.any(np.signbit(got))


@pytest.mark.parametrize("x", [-126.999, -126.5, -126.0001])
def test_just_above_the_clamp_stays_tiny_and_non_negative(x):
    got = float(ex2_fma2_model(f32([x]))[0])
    assert 0.0 <= got < 2.0 ** -126
