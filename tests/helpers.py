"""Comparison helpers for GPU-vs-oracle parity, with the stated tolerances.

Tolerances (floating point, against the fp64 oracle):
  log p, element-wise relative: 2e-5 for fp32 logits, 1e-5 for bf16 logits;
    exactly 0 where the oracle gives exactly 0 (masked rows, V = 1); never > 0.
    A log p may also differ by 2^-148 absolutely: that of a near-certain
    column is about -(1 - p), which fp32 holds below 2^-126 only as a
    subnormal (2 ulp = 2^-148 of error) and below 2^-149 not at all.
  dlogits, per row ||got - ref||_2 / ||ref||_2: 2e-5 fp32, 4e-3 bf16;
    ignored rows exactly zero.  The dlogits come in the logits' dtype, which
    cannot hold values below half its smallest subnormal (2^-150 fp32,
    2^-134 bf16): each element may also differ from the fp64 value by that
    much (a row whose whole gradient lies below it reads as zero).
  reduced loss, relative: 2e-5.
  row entropy, element-wise relative: 2e-5 for either logit type (the sums
    behind it are fp32 whatever the input type); exactly 0 where the oracle
    gives exactly 0; never negative.
  entropy may also differ by 2^-141 absolutely: it is an fp32 mass (1 - p
    of the reference column) times that mass's mean surprisal, and where the
    mass is below 2^-126 it is a subnormal with an absolute error of up to
    2 ulp = 2^-148, while the surprisal stays under 2^7 nats (-log of a mass
    fp32 can hold, 103.3, plus log V).  A mass below fp32's range reads as 0.
  a DFT-weighted row loss p_y * CE_row may likewise differ by 2^-148 CE_row
    + 2^-149 (p_y subnormal, then the product's rounding); a reduced DFT
    loss by the sum of its rows' floors.
  soft-capped CE (cap_eps): every exponent carries the fp32 error of its
    capped logit, eps = 2.5 ulp(cap) / T; log p and a CE row loss (the
    label's exponent and the log-sum-exp's) may differ by 2 eps more, a DFT
    row loss by 2 eps (|loss| + p_y), a gradient row by 3 eps relative.
  CE gradients near fp32's subnormals: the label element g/T expm1(log p)
    is formed from the fp32 log p (within 2^-148 near 0: the log p floor),
    so a row may move by |g/T| 2^-148; a DFT weight p_y is an fp32 value
    (a subnormal within 2^-150), moving the row by |g/T| 2^-150 sqrt(2); a
    soft-capped element is the plain one times its chain factor, two
    roundings, so one more rounding floor per element.  With label
    smoothing an element is p_j minus its smoothed target, both fp32 values
    of order 1; where p sits on the target the element cancels, and the row
    may move by |g/T| 2^-21 (a few ulps of parts of norm at most 1).
Integer results (item counts, skipped rows) are compared exactly.
"""

import math

import numpy as np
import torch

LOGP_TOL = {torch.float32: 2e-5, torch.bfloat16: 1e-5}
GRAD_TOL = {torch.float32: 2e-5, torch.bfloat16: 4e-3}
LOSS_TOL = 2e-5
ENTROPY_TOL = 2e-5
ZERO_SUM_TOL = {torch.float32: 1e-5, torch.bfloat16: 4e-3}
# half the smallest subnormal of the gradient's dtype: its rounding floor
GRAD_FLOOR = {torch.float32: 2.0 ** -150, torch.bfloat16: 2.0 ** -134}


def cap_eps(cap: float, T: float) -> float:
    """Absolute error, in a soft-capped exponent z / T, of forming z = cap *
    tanh(x / cap) in fp32 at all: tanh within 2 ulp of t (CUDA's bound for
    tanhf) and one rounding of the product, so 2.5 ulp(cap) for |t| < 1,
    divided by T.  0 without a cap."""
    if not cap > 0.0:
        return 0.0
    return 2.5 * 2.0 ** (math.floor(math.log2(cap)) - 23) / T


# a subnormal fp32 mass (2 ulp = 2^-148 of error), alone (a log p near 0) or
# times a surprisal < 2^7 nats (an entropy)
LOGP_FLOOR = 2.0 ** -148
SUBNORMAL_PRODUCT_FLOOR = 2.0 ** -141


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def assert_logp_close(got, ref, dtype, what="logp", tol=None, floor=0.0):
    """Element-wise relative error <= tol, plus LOGP_FLOOR and an extra
    absolute `floor` (scalar or per element) for values that are products of
    a subnormal mass, such as DFT-weighted losses."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isnan(got) == np.isnan(ref)), f"{what}: NaN pattern differs"
    ok = ~np.isnan(ref)
    g, r = got[ok], ref[ok]
    floor = np.broadcast_to(np.asarray(floor, dtype=np.float64), ref.shape)[ok]
    assert np.all(g <= 0.0), f"{what}: positive log p {g.max()}"
    zero = r == 0.0
    assert np.all(g[zero] == 0.0), f"{what}: nonzero where the oracle is exactly 0"
    floor = floor[~zero] + LOGP_FLOOR
    diff = np.abs(g[~zero] - r[~zero])
    rel = diff / np.abs(r[~zero])
    tol = LOGP_TOL[dtype] if tol is None else tol
    worst = rel.max() if rel.size else 0.0
    bad = diff > tol * np.abs(r[~zero]) + floor
    assert not np.any(bad), f"{what}: worst relative error {rel[bad].max():.3e} > {tol:.0e}"
    return worst


def assert_grad_rows_close(got, ref, dtype, what="dlogits", tol=None, extra_floor=None):
    """Per row ||got - ref|| <= tol ||ref|| + the dtype's rounding floor
    (+ `extra_floor[r]`: what fp32 floors of the inputs or of intermediate
    values move the row by, stated by the caller)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    tol = GRAD_TOL[dtype] if tol is None else tol
    worst = 0.0
    for r in range(ref.shape[0]):
        if np.all(np.isnan(ref[r])):
            assert np.all(np.isnan(got[r])), f"{what}: row {r} should be NaN"
            continue
        nr = np.linalg.norm(ref[r])
        if nr == 0.0:
            assert np.all(got[r] == 0.0), f"{what}: row {r} should be exactly zero"
            continue
        diff = np.linalg.norm(got[r] - ref[r])
        e = diff / nr
        worst = max(worst, e)
        floor = GRAD_FLOOR[dtype] * math.sqrt(ref.shape[1])
        if extra_floor is not None:
            floor += float(np.broadcast_to(extra_floor, (ref.shape[0],))[r])
        assert diff <= tol * nr + floor, f"{what}: row {r} relative error {e:.3e} > {tol:.0e}"
    return worst


def assert_zero_sum_rows(got, dtype, rows=None):
    got = np.asarray(got, dtype=np.float64)
    tol = ZERO_SUM_TOL[dtype]
    for r in (range(got.shape[0]) if rows is None else rows):
        row = got[r]
        s_abs = math.fsum(np.abs(row))
        if s_abs == 0.0:
            continue
        assert abs(math.fsum(row)) <= tol * s_abs, f"row {r}: gradient does not sum to zero"


def assert_loss_close(got: float, ref: float, what="loss", floor=0.0):
    """Relative error <= LOSS_TOL (+ an absolute `floor`, for a sum of
    DFT-weighted row losses: the sum of their floors)."""
    if ref == 0.0:
        assert got == 0.0, f"{what}: {got} != 0"
        return
    assert abs(got - ref) <= LOSS_TOL * abs(ref) + floor, f"{what}: {got} vs {ref}"


def assert_entropy_close(got, ref, what="entropy"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isnan(got) == np.isnan(ref)), f"{what}: NaN pattern differs"
    ok = ~np.isnan(ref)
    g, r = got[ok], ref[ok]
    assert np.all(g >= 0.0), f"{what}: negative entropy {g.min()}"
    zero = r == 0.0
    assert np.all(g[zero] == 0.0), f"{what}: nonzero where the oracle is exactly 0"
    diff = np.abs(g[~zero] - r[~zero])
    rel = diff / r[~zero]
    worst = rel.max() if rel.size else 0.0
    bad = diff > ENTROPY_TOL * r[~zero] + SUBNORMAL_PRODUCT_FLOOR
    assert not np.any(bad), (
        f"{what}: worst relative error {rel[bad].max():.3e} > {ENTROPY_TOL:.0e}")
    return worst


def assert_grad_block_close(got, ref, dtype, what="dlogits", tol=None):
    """assert_grad_rows_close for a block of rows at once (vectorized)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    tol = GRAD_TOL[dtype] if tol is None else tol
    nan_rows = np.all(np.isnan(ref), axis=1)
    assert np.all(np.isnan(got[nan_rows])), f"{what}: NaN rows differ"
    ok = ~nan_rows
    nr = np.linalg.norm(ref[ok], axis=1)
    zero = nr == 0.0
    assert np.all(got[ok][zero] == 0.0), f"{what}: a zero row is not exactly zero"
    diff = np.linalg.norm(got[ok][~zero] - ref[ok][~zero], axis=1)
    err = diff / nr[~zero]
    worst = err.max() if err.size else 0.0
    floor = GRAD_FLOOR[dtype] * math.sqrt(ref.shape[1])
    bad = diff > tol * nr[~zero] + floor
    assert not np.any(bad), f"{what}: worst row relative error {err[bad].max():.3e} > {tol:.0e}"
    return worst


def assert_zero_sum_block(got, dtype):
    """assert_zero_sum_rows for a block of rows at once; numpy's pairwise fp64
    sums (error far below the tolerance) instead of exact ones."""
    got = np.asarray(got, dtype=np.float64)
    s = np.abs(np.sum(got, axis=1))
    a = np.sum(np.abs(got), axis=1)
    assert np.all(s <= ZERO_SUM_TOL[dtype] * a), "a gradient row does not sum to zero"
