"""Shared bits of the parity tests."""
import numpy as np

from oracle.batch import oracle_batch  # noqa: F401

# A finer measure beside the 2e-3 bound: the error in units of the fp16
# spacing at each output row's largest |oracle| value.  The result is rounded
# to fp16 once (at most half a unit per element) and the softmax weights the
# P.V product uses are fp16 (rounding each weight by up to 2^-11 of itself);
# over the seeded random sweep a correct kernel stays within a mean of
# 0.09-0.12 units and a maximum of 1.14, while dropping each sequence's last
# token gives a mean of 4-39 units -- on long contexts, whose outputs are
# ~0.02, that mistake is ~5e-4 and passes the absolute bound.
ROW_ULP_MEAN = 0.25
ROW_ULP_MAX = 3.0


def attention_tolerance():
    """Max |GPU - oracle| allowed on fp16 outputs: the 2e-3 bound stated for
    fp16 inputs with fp32 accumulation."""
    return 2e-3


def row_ulps(got, ref):
    """|got - ref| in fp16 spacings at each row's (last axis) largest |ref|."""
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    unit = np.spacing(scale.astype(np.float16)).astype(np.float64)
    return np.abs(np.asarray(got, dtype=np.float64) - ref) / unit


def assert_matches_oracle(got, ref, what=""):
    """Finite, max |got - ref| <= 2e-3, and in row units a mean of at most
    ROW_ULP_MEAN and a maximum of at most ROW_ULP_MAX."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape, what)
    assert np.isfinite(got).all(), "non-finite output %s" % (what,)
    err = np.abs(got - ref)
    if err.size == 0:
        return
    assert err.max() <= attention_tolerance(), "max abs error %.3g at %s %s" % (
        err.max(), np.unravel_index(err.argmax(), err.shape), what)
    u = row_ulps(got, ref)
    assert u.mean() <= ROW_ULP_MEAN and u.max() <= ROW_ULP_MAX, (
        "row-unit error mean %.3f max %.2f at %s %s" % (
            u.mean(), u.max(), np.unravel_index(u.argmax(), u.shape), what))
