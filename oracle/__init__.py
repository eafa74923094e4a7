"""fp64 CPU oracle for the row-wise log-softmax / cross-entropy path.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports, links or runs anything here, and nothing here imports the product.

The arithmetic lives in ``ce_oracle.c`` (plain C, fp64, one row at a time);
this module only compiles it with gcc on first use and marshals numpy arrays.
Inputs are taken as exact fp64 copies of the bf16/fp32 logits, and the
temperature as the exact value of its fp32 rounding, so both sides of a parity
check see the same numbers.

Functions and the passages they follow:

* :func:`selective_logsoftmax` -- "perf(rlhf): chunk selective_log_softmax
  instead of looping per token" (ms-swift PR #10337), "PR information":
  gather(log_softmax(logits / T)) at K indices per row with a row mask,
  computed in the collapse-safe form of "Fix softmax collapse in CE, GRPO,
  KL/JSD and softmax" (Liger-Kernel PR #1555), "Details".
* :func:`selective_logsoftmax_backward` -- the gradient of sum_k g_k log p_{t_k}
  (plus g_H H, the row entropy, when given):
  (1/T)(sum_{k: t_k = j} g_k - G p_j), with the gathered columns in the
  -expm1(log p_t) form of the same page's "Summary" (second bullet).
* :func:`entropy` -- -sum_j p_j log p_j per row, the reference column's term
  from its accurate log p (the per-token entropy of the unsloth-zoo #2080
  commit quoted on the same page, "Fix").
* :func:`cross_entropy` -- the same page's "Summary" (loss from the sum that
  excludes the target) with ms-swift PR #10353's "PR information" (analytic
  backward g*softmax - g*onehot, zero weight on ignored labels) and the
  unsloth-zoo #2080 "Fix" section's -expm1(log p_t) target gradient (label
  smoothing included there); the DFT variant weights each row by p_y, held
  constant in the backward (ms-swift PR #10353, "PR information").

* :func:`vocab_slice_partials`, :func:`vocab_slice_combine` -- the same
  log-probs computed from slices of the vocabulary: each slice's max and
  sum over its non-target columns and the target logits it holds, merged
  in slice order (the vocab-parallel bullet of the same page's "Summary").

Pins: closed forms, 120-digit brute force, invariants and the pages' collapse
thresholds, in ``tests/test_oracle_pins.py``; the slice functions against
the full-row log-probs for many slicings and against brute force.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ce_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

REDUCTIONS = {"none": 0, "sum": 1, "mean": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ce_oracle.c into a shared library with gcc (IEEE fp64, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # a test may point this at a deliberately broken copy of the oracle
        # to check that the pins catch planted mistakes
        lib = ctypes.CDLL(os.environ.get("GBCE_ORACLE_LIB") or build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_selective_logsoftmax.restype = i64
        lib.oracle_selective_logsoftmax.argtypes = [
            dp, i64, i64, i64, ip, i64, ctypes.c_double, ctypes.c_void_p, dp]
        lib.oracle_cross_entropy.restype = i64
        lib.oracle_cross_entropy.argtypes = [
            dp, i64, i64, i64, ip, i64, ctypes.c_double, ctypes.c_int, ctypes.c_double,
            ctypes.c_int, ctypes.c_double, ctypes.c_void_p, dp, dp, dp, ip, ctypes.c_void_p, i64]
        lib.oracle_selective_logsoftmax_backward.restype = i64
        lib.oracle_selective_logsoftmax_backward.argtypes = [
            dp, i64, i64, i64, ip, i64, ctypes.c_double, ctypes.c_void_p, dp, ctypes.c_void_p,
            dp, i64]
        lib.oracle_entropy.restype = i64
        lib.oracle_entropy.argtypes = [dp, i64, i64, i64, ip, ctypes.c_double, ctypes.c_void_p, dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _as_rows(x) -> np.ndarray:
    x = np.asarray(x)
    if x.ndim != 2:
        raise ValueError("logits must be 2-D [rows, V]")
    if x.dtype != np.float64:
        x = x.astype(np.float64)  # exact for bf16/fp32 inputs
    if x.strides[1] != 8:
        x = np.ascontiguousarray(x)
    return x


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def exact_temperature(temperature: float) -> float:
    """The fp64 value of the fp32 temperature both sides use."""
    return float(np.float32(temperature))


def selective_logsoftmax(x, index, temperature: float = 1.0, row_mask=None):
    """log p at K gathered indices per row; masked-out rows give 0.

    Returns ``(out[rows, K] float64, n_bad_indices)``.
    """
    lib = _load()
    x = _as_rows(x)
    rows, V = x.shape
    idx = np.ascontiguousarray(np.asarray(index, dtype=np.int64).reshape(rows, -1))
    K = idx.shape[1]
    mask_arr = None
    mask_ptr = None
    if row_mask is not None:
        mask_arr = np.ascontiguousarray(np.asarray(row_mask).reshape(rows).astype(np.uint8))
        mask_ptr = mask_arr.ctypes.data
    out = np.empty((rows, K), dtype=np.float64)
    bad = lib.oracle_selective_logsoftmax(
        _ptr(x, ctypes.c_double), rows, V, x.strides[0] // 8, _ptr(idx, ctypes.c_int64), K,
        exact_temperature(temperature), mask_ptr, _ptr(out, ctypes.c_double))
    return out, int(bad)


def selective_logsoftmax_backward(x, index, grad, temperature: float = 1.0, row_mask=None,
                                  grad_entropy=None):
    """dL/dx for upstream grad[r, k] = dL/d log p_{index[r, k]}; masked rows 0.

    ``grad_entropy`` [rows] (optional) is dL/dH_r for the row entropy H_r
    (:func:`entropy` with reference column index[r, 0]).
    Returns ``(dx[rows, V] float64, n_bad_rows)``.
    """
    lib = _load()
    x = _as_rows(x)
    rows, V = x.shape
    idx = np.ascontiguousarray(np.asarray(index, dtype=np.int64).reshape(rows, -1))
    K = idx.shape[1]
    g = np.ascontiguousarray(np.asarray(grad, dtype=np.float64).reshape(rows, K))
    mask_arr = None
    mask_ptr = None
    if row_mask is not None:
        mask_arr = np.ascontiguousarray(np.asarray(row_mask).reshape(rows).astype(np.uint8))
        mask_ptr = mask_arr.ctypes.data
    gh_arr = None
    gh_ptr = None
    if grad_entropy is not None:
        gh_arr = np.ascontiguousarray(np.asarray(grad_entropy, dtype=np.float64).reshape(rows))
        gh_ptr = gh_arr.ctypes.data
    dx = np.empty((rows, V), dtype=np.float64)
    bad = lib.oracle_selective_logsoftmax_backward(
        _ptr(x, ctypes.c_double), rows, V, x.strides[0] // 8, _ptr(idx, ctypes.c_int64), K,
        exact_temperature(temperature), mask_ptr, _ptr(g, ctypes.c_double), gh_ptr,
        _ptr(dx, ctypes.c_double), V)
    return dx, int(bad)


def entropy(x, ref, temperature: float = 1.0, live=None):
    """-sum_j p_j log p_j per row, column ref[r] entering with its accurate log p.

    Rows with live[r] == 0 give 0.  Returns ``(out[rows] float64, n_bad)``.
    """
    lib = _load()
    x = _as_rows(x)
    rows, V = x.shape
    t = np.ascontiguousarray(np.asarray(ref, dtype=np.int64).reshape(rows))
    live_arr = None
    live_ptr = None
    if live is not None:
        live_arr = np.ascontiguousarray(np.asarray(live).reshape(rows).astype(np.uint8))
        live_ptr = live_arr.ctypes.data
    out = np.empty(rows, dtype=np.float64)
    bad = lib.oracle_entropy(_ptr(x, ctypes.c_double), rows, V, x.strides[0] // 8,
                             _ptr(t, ctypes.c_int64), exact_temperature(temperature), live_ptr,
                             _ptr(out, ctypes.c_double))
    return out, int(bad)


def cross_entropy(x, labels, ignore_index: int = -100, temperature: float = 1.0,
                  reduction: str = "mean", grad_out=None, want_grad: bool = True,
                  label_smoothing: float = 0.0, dft: bool = False, softcap: float = 0.0):
    """Token CE forward (and backward when ``want_grad``).

    ``label_smoothing`` eps puts 1 - eps on the label and eps / V on every
    class; ``dft`` weights each row's loss and gradient by its detached p_y;
    ``softcap`` > 0 caps every logit as softcap * tanh(x / softcap) first.

    ``grad_out`` is the upstream gradient: [rows] for reduction 'none', a
    scalar otherwise (default 1).  Returns a dict with ``logp`` [rows],
    ``loss_rows`` [rows], ``loss`` (float), ``n_items`` (int), ``dlogits``
    [rows, V] or None, and ``n_bad`` (out-of-range labels).
    """
    lib = _load()
    x = _as_rows(x)
    rows, V = x.shape
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.int64).reshape(rows))
    red = REDUCTIONS[reduction]
    g_arr = None
    g_ptr = None
    if want_grad:
        if grad_out is None:
            grad_out = np.ones(rows) if red == 0 else np.ones(1)
        g_arr = np.ascontiguousarray(np.asarray(grad_out, dtype=np.float64).reshape(-1))
        if g_arr.size != (rows if red == 0 else 1):
            raise ValueError("grad_out must have rows entries for 'none', one otherwise")
        g_ptr = g_arr.ctypes.data
    logp = np.empty(rows, dtype=np.float64)
    loss_rows = np.empty(rows, dtype=np.float64)
    loss = np.empty(1, dtype=np.float64)
    n_items = np.empty(1, dtype=np.int64)
    dx = np.empty((rows, V), dtype=np.float64) if want_grad else None
    bad = lib.oracle_cross_entropy(
        _ptr(x, ctypes.c_double), rows, V, x.strides[0] // 8, _ptr(lab, ctypes.c_int64),
        int(ignore_index), exact_temperature(temperature), red, float(label_smoothing),
        int(bool(dft)), float(softcap), g_ptr,
        _ptr(logp, ctypes.c_double), _ptr(loss_rows, ctypes.c_double),
        _ptr(loss, ctypes.c_double), _ptr(n_items, ctypes.c_int64),
        dx.ctypes.data if dx is not None else None, V)
    return {"logp": logp, "loss_rows": loss_rows, "loss": float(loss[0]),
            "n_items": int(n_items[0]), "dlogits": dx, "n_bad": int(bad)}


def vocab_slice_partials(x_slice, index, vocab_offset: int, temperature: float = 1.0,
                         row_mask=None):
    """Statistics of one vocabulary slice, global columns [vocab_offset,
    vocab_offset + n): over its columns that are not gathered targets,
    m = max z_j and s = sum_j exp(z_j - m) (z = x / T), and the logit of
    every target the slice holds (0 for the others).  The vocab-parallel
    form of "Fix softmax collapse in CE, GRPO, KL/JSD and softmax"
    ("Summary", first bullet): every shard keeps the sum without the target.

    Returns ``(m[rows], s[rows], xt[rows, K])`` in fp64; rows with
    row_mask == 0 give (-inf, 0, 0).
    """
    x = _as_rows(x_slice)
    rows, n = x.shape
    idx = np.asarray(index, dtype=np.int64).reshape(rows, -1)
    T = exact_temperature(temperature)
    local = idx - int(vocab_offset)
    owned = (local >= 0) & (local < n)
    z = x / T
    zm = z.copy()
    r_ix = np.repeat(np.arange(rows), idx.shape[1])
    zm[r_ix[owned.ravel()], local[owned]] = -np.inf
    m = zm.max(axis=1) if n else np.full(rows, -np.inf)
    with np.errstate(invalid="ignore"):
        s = np.where(np.isfinite(m), np.exp(zm - m[:, None]).sum(axis=1), 0.0)
    xt = np.zeros(idx.shape, dtype=np.float64)
    xt[owned] = x[r_ix[owned.ravel()], local[owned]]
    if row_mask is not None:
        dead = np.asarray(row_mask).reshape(rows) == 0
        m[dead], s[dead], xt[dead] = -np.inf, 0.0, 0.0
    return m, s, xt


def vocab_slice_combine(parts, offsets, index, temperature: float = 1.0, row_mask=None):
    """log p at the gathered indices from the slices' partials.

    ``parts`` is a list (slice order) of ``(m, s, xt)`` from
    :func:`vocab_slice_partials`; ``offsets`` the slices' first global
    columns plus the vocabulary size at the end.  The (m, s) of all slices
    are merged into the state of every non-target column, each target's
    logit is taken from the slice that holds it, and log p_t follows the
    single-device form: the other targets join t's "others", then
    log p_t = -softplus(log s + (m - x_t) / T).  Masked rows give 0.
    Returns ``(logp[rows, K], xt0[rows])``.
    """
    T = exact_temperature(temperature)
    idx = np.asarray(index, dtype=np.int64)
    rows = idx.shape[0]
    idx = idx.reshape(rows, -1)
    K = idx.shape[1]
    ms = np.stack([p[0] for p in parts])        # [S, rows]
    ss = np.stack([p[1] for p in parts])
    M = ms.max(axis=0)
    with np.errstate(invalid="ignore"):
        S = np.where(np.isfinite(M), np.sum(np.where(np.isfinite(ms), ss * np.exp(ms - M), 0.0),
                                            axis=0), 0.0)
    off = np.asarray(offsets, dtype=np.int64)
    owner = np.searchsorted(off, idx, side="right") - 1   # slice of each target
    xt = np.zeros((rows, K))
    for r in range(rows):
        for k in range(K):
            xt[r, k] = parts[owner[r, k]][2][r, k]
    logp = np.zeros((rows, K))
    for r in range(rows):
        if row_mask is not None and np.asarray(row_mask).reshape(rows)[r] == 0:
            continue
        for k in range(K):
            m, s = M[r], S[r]
            seen = set()
            for j in range(K):
                tj = int(idx[r, j])
                if tj == int(idx[r, k]) or tj in seen:
                    continue
                seen.add(tj)
                zj = xt[r, j] / T
                if zj > m:
                    s = s * np.exp(m - zj) + 1.0
                    m = zj
                else:
                    s = s + np.exp(zj - m)
            a = (np.log(s) if s > 0 else -np.inf) + (m - xt[r, k] / T)
            logp[r, k] = -(max(a, 0.0) + np.log1p(np.exp(-abs(a)))) if np.isfinite(a) else \
                (0.0 if a < 0 else -np.inf)
    return logp, xt[:, 0]
