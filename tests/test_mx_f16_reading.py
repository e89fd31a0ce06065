"""The reading that lets the f16 kernels take OCP MX activations: the
quantise-dequantise (QDQ) of a bf16 row, times the power of two 2^a that puts
the row's largest |x| in [2^14, 2^15), is exactly representable in f16 and
stays below 2^15, for every block whose largest value is within 2^21 (MXFP8)
or 2^35 (MXFP4) of the row's (the smallest code of such a block, times its
scale and 2^a, is still a multiple of f16's subnormal step 2^-24); further
below, a block's smallest values may round.  And the QDQ of a bounded
SwiGLU-OAI intermediate fits f16 as it is.  Checked with the oracle's QDQ
(fp64) and numpy's float16, no GPU."""
import numpy as np
import pytest

import oracle


def _f16_exact(v: np.ndarray) -> bool:
    return bool(np.all(v.astype(np.float16).astype(np.float64) == v))


@pytest.mark.parametrize("fmt", ["mxfp4_dyn", "mxfp8_dyn"])
def test_scaled_qdq_of_bf16_rows_is_exact_f16(fmt):
    rng = np.random.default_rng(7)
    rows, cols = 64, 512
    x = rng.standard_normal((rows, cols))
    # blocks spread over 2^-12 .. 2^6 within a row, some all-zero
    blk = np.exp2(rng.integers(-12, 7, (rows, cols // 32)).astype(np.float64))
    blk[rng.random((rows, cols // 32)) < 0.1] = 0.0
    x = x * np.repeat(blk, 32, axis=1)
    xb = x.astype(np.float32)  # the values a bf16 row holds are exact in fp32
    xb = oracle.bf16_values(oracle.bf16_bits(xb.astype(np.float64))).astype(np.float32)
    q = oracle.qdq_rows(xb, fmt, None)
    for r in range(rows):
        amax = np.abs(xb[r]).max()
        if amax == 0:
            continue
        _, ex = np.frexp(amax)
        a = 15 - int(ex)
        v = q[r] * np.exp2(a)
        assert np.abs(v).max() < 2.0 ** 15
        assert _f16_exact(v), r


@pytest.mark.parametrize("fmt", ["mxfp4_dyn", "mxfp8_dyn"])
def test_qdq_of_bounded_swiglu_intermediate_fits_f16(fmt):
    # |z| <= limit * (limit + |beta|) for the clamped SwiGLU-OAI; with the
    # largest limit and beta the f16 paths take (64) the QDQ stays finite in f16
    # and is exact there (values above f16's subnormal range)
    rng = np.random.default_rng(8)
    bound = 64.0 * (64.0 + 64.0)
    z = (rng.uniform(-1, 1, (32, 256)) * bound).astype(np.float32)
    z[0, :32] = bound  # a block at the bound itself
    q = oracle.qdq_rows(z, fmt, None)
    assert np.abs(q).max() < 65504.0
    assert _f16_exact(q)


def test_the_stated_tail_is_where_exactness_ends():
    # a block 2^-40 below the row's largest value falls under f16's subnormal
    # step after the row's power of two: the tail the reading excludes
    x = np.zeros((1, 64), np.float32)
    x[0, :32] = 3.0
    x[0, 32:] = np.float32(3.0 * 2.0 ** -40) * np.linspace(0.5, 1.0, 32, dtype=np.float32)
    q = oracle.qdq_rows(x, "mxfp8_dyn", None)
    _, ex = np.frexp(3.0)
    v = q[0] * np.exp2(15 - int(ex))
    assert _f16_exact(v[:32]) and not _f16_exact(v[32:])


@pytest.mark.parametrize("fmt,rel", [("mxfp8_dyn", 21), ("mxfp4_dyn", 35)])
def test_exact_up_to_the_stated_distance(fmt, rel):
    # a block whose largest value is 2^-rel of the row's, holding values down
    # to 2^-12 of its own maximum (so its smallest codes occur): still exact
    rng = np.random.default_rng(rel)
    for _ in range(50):
        x = np.zeros((1, 64), np.float32)
        x[0, :32] = np.float32(1.999)
        b = rng.uniform(-1, 1, 32) * np.exp2(rng.uniform(-12, 0, 32))
        b[0] = 1.0
        x[0, 32:] = (b * 1.999 * 2.0 ** -rel).astype(np.float32)
        q = oracle.qdq_rows(x, fmt, None)
        _, ex = np.frexp(np.abs(x).max())
        assert _f16_exact(q[0] * np.exp2(15 - int(ex)))
