"""Pins for the fp64 oracle, against things other than itself.

Each test ties the oracle to a fact the pages or the mathematics fix:
closed forms, a 120-digit brute force of the plain definition
log p_t = z_t - log sum_j exp(z_j), a library routine a special case
reduces to, invariants, the pages' printed collapse thresholds and the pages' printed
sparse-supervision workload.  A dropped term, a wrong sign, a missing 1/T, a
wrong index or a wrong reduction scale each fails at least one of them.
"""

import math
from decimal import Context, Decimal

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads
from conftest import read_golden

CTX = Context(prec=120)


def brute_row(row, t, T):
    """Plain definition at 120 digits: (log p_j for all j, log p_t)."""
    Td = Decimal(T)
    z = [CTX.divide(Decimal(float(v)), Td) for v in row]
    s = Decimal(0)
    for zj in z:
        s = CTX.add(s, CTX.exp(zj))
    lse = CTX.ln(s)
    return [CTX.subtract(zj, lse) for zj in z], CTX.subtract(z[t], lse)


def brute_grad_row(row, y, T, g):
    """(g/T) * (softmax(z) - onehot(y)) at 120 digits."""
    logps, _ = brute_row(row, y, T)
    scale = CTX.divide(Decimal(g), Decimal(T))
    out = []
    for j, lp in enumerate(logps):
        p = CTX.exp(lp)
        if j == y:
            p = CTX.subtract(p, Decimal(1))
        out.append(float(CTX.multiply(scale, p)))
    return np.array(out)


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-300))


# --------------------------------------------------------------- closed forms

@pytest.mark.parametrize("V", [1, 2, 7, 4096, 152064])
@pytest.mark.parametrize("T", [1.0, 0.9, 0.7])
def test_uniform_logits_give_minus_log_v(V, T):
    rng = np.random.default_rng(V)
    c = rng.normal()
    x = np.full((3, V), c)
    labels = np.array([0, V - 1, V // 2])
    lp, bad = oracle.selective_logsoftmax(x, labels[:, None], T)
    assert bad == 0
    np.testing.assert_allclose(lp[:, 0], -math.log(V), rtol=1e-14, atol=1e-300)
    g = 0.37
    out = oracle.cross_entropy(x, labels, temperature=T, reduction="sum", grad_out=[g])
    Te = oracle.exact_temperature(T)
    dx = out["dlogits"]
    for r, y in enumerate(labels):
        want = np.full(V, g / (Te * V))
        want[y] = g * (1.0 / V - 1.0) / Te
        np.testing.assert_allclose(dx[r], want, rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(out["loss"], 3 * math.log(V), rtol=1e-14)


@pytest.mark.parametrize("V", [2, 5, 1003, 40001])
@pytest.mark.parametrize("gap", [-3.0, 0.5, 17.0, 20.0, 30.0, 50.0])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_two_level_rows(V, gap, T):
    """Target a, V-1 others b: log p = -log1p((V-1) exp((b-a)/T))."""
    a, b = 1.25 + gap, 1.25
    x = np.full((1, V), b)
    y = V // 3
    x[0, y] = a
    lp, _ = oracle.selective_logsoftmax(x, [[y]], T)
    Te = oracle.exact_temperature(T)
    want = -math.log1p((V - 1) * math.exp((b - a) / Te))
    assert lp[0, 0] == pytest.approx(want, rel=1e-13, abs=0)
    assert lp[0, 0] < 0.0


def test_v2_reduces_to_log_sigmoid():
    rng = np.random.default_rng(7)
    x = rng.normal(scale=6.0, size=(200, 2))
    y = rng.integers(0, 2, size=200)
    for T in (1.0, 0.9, 0.7):
        lp, _ = oracle.selective_logsoftmax(x, y[:, None], T)
        Te = oracle.exact_temperature(T)
        other = x[np.arange(200), 1 - y]
        want = scipy.special.log_expit((x[np.arange(200), y] - other) / Te)
        np.testing.assert_allclose(lp[:, 0], want, rtol=1e-13)


def test_v1_rows_are_certain():
    x = np.array([[3.5], [-2.0]])
    lp, _ = oracle.selective_logsoftmax(x, [[0], [0]], 0.9)
    assert np.all(lp == 0.0)
    out = oracle.cross_entropy(x, [0, 0], reduction="mean")
    assert out["loss"] == 0.0
    assert np.all(out["dlogits"] == 0.0)


# ------------------------------------------------------ brute force, 120 digits

@pytest.mark.parametrize("V", [2, 3, 17, 64])
@pytest.mark.parametrize("T", [1.0, 0.9, 0.7])
def test_brute_force_logp(V, T):
    margins = [0.0, 5.0, 17.0, 20.0, 30.0, 50.0, 80.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    x[0] = np.random.default_rng(V).normal(scale=3.0, size=V)   # an ordinary row
    lp, _ = oracle.selective_logsoftmax(x, y[:, None], T)
    Te = oracle.exact_temperature(T)
    for r in range(len(margins)):
        _, want = brute_row(x[r], y[r], Te)
        assert lp[r, 0] == pytest.approx(float(want), rel=1e-12, abs=0), (r, margins[r])


@pytest.mark.parametrize("V", [2, 9, 64])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_brute_force_gradient(V, T):
    margins = [0.0, 17.0, 30.0, 50.0, 80.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=100 + V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    g = 1.3
    out = oracle.cross_entropy(x, y, temperature=T, reduction="sum", grad_out=[g])
    Te = oracle.exact_temperature(T)
    for r in range(len(margins)):
        want = brute_grad_row(x[r], y[r], Te, g)
        assert rel_err(out["dlogits"][r], want) < 1e-11, (r, margins[r])


def test_brute_force_k_indices_with_duplicates():
    rng = np.random.default_rng(3)
    V = 33
    x = rng.normal(scale=4.0, size=(4, V))
    x[1, 5] = x[1].max() + 30.0
    idx = np.array([[0, 5, 5, 32], [5, 5, 1, 2], [7, 7, 7, 7], [31, 0, 16, 3]])
    lp, _ = oracle.selective_logsoftmax(x, idx, 0.9)
    Te = oracle.exact_temperature(0.9)
    for r in range(4):
        for k in range(4):
            _, want = brute_row(x[r], idx[r, k], Te)
            assert lp[r, k] == pytest.approx(float(want), rel=1e-12, abs=0)
    assert lp[0, 1] == lp[0, 2] and lp[2, 0] == lp[2, 3]


# ----------------------------------------------------------------- invariants

def test_invariants_on_collapse_stress_rows():
    """logp <= 0, zero-sum gradient rows, nonzero target gradient (margins 17-50)."""
    for dtype in (torch.float32, torch.bfloat16):
        w = workloads.collapse_stress(dtype=dtype, rows=48, V=40001, seed=1)
        x = workloads.to_numpy_f64(w.logits)
        lab = w.labels.numpy()
        out = oracle.cross_entropy(x, lab, reduction="mean")
        live = lab != workloads.IGNORE_INDEX
        assert out["n_items"] == int(live.sum())
        assert np.all(out["logp"] <= 0.0)
        dx = out["dlogits"]
        for r in np.nonzero(live)[0]:
            row = dx[r]
            assert abs(math.fsum(row)) <= 1e-12 * math.fsum(np.abs(row))
            assert row[lab[r]] < 0.0
        assert np.all(dx[~live] == 0.0)
        peaked = w.peaked_rows.numpy()
        peaked = peaked[live[peaked]]
        assert np.all(out["logp"][peaked] < 0.0)


def test_probabilities_sum_to_one():
    rng = np.random.default_rng(11)
    V = 50
    x = rng.normal(scale=5.0, size=(6, V))
    x[2, 7] += 40.0
    idx = np.tile(np.arange(V), (6, 1))
    for T in (1.0, 0.7):
        lp, _ = oracle.selective_logsoftmax(x, idx, T)
        s = np.array([math.fsum(np.exp(r)) for r in lp])
        np.testing.assert_allclose(s, 1.0, rtol=1e-14)


def test_permuting_columns_permutes_outputs():
    rng = np.random.default_rng(5)
    V = 257
    x = rng.normal(scale=2.0, size=(5, V))
    y = rng.integers(0, V, size=5)
    perm = rng.permutation(V)
    inv = np.argsort(perm)
    a = oracle.cross_entropy(x, y, temperature=0.9, reduction="sum", grad_out=[1.0])
    b = oracle.cross_entropy(x[:, perm], inv[y], temperature=0.9, reduction="sum",
                             grad_out=[1.0])
    np.testing.assert_allclose(b["logp"], a["logp"], rtol=1e-14)
    np.testing.assert_allclose(b["dlogits"], a["dlogits"][:, perm], rtol=1e-13, atol=1e-300)


def test_finite_difference_gradient():
    """The oracle's dlogits is the derivative of its own reduced loss."""
    rng = np.random.default_rng(21)
    V, rows = 6, 4
    x = rng.normal(scale=2.0, size=(rows, V))
    y = np.array([1, -100, 5, 0])
    x[3, 0] += 8.0
    for red, g in (("mean", [0.7]), ("sum", [1.9]), ("none", [0.3, 5.0, -1.1, 2.0])):
        T = 0.7
        out = oracle.cross_entropy(x, y, temperature=T, reduction=red, grad_out=g)
        h = 1e-6
        num = np.zeros_like(x)
        w = np.asarray(g, dtype=np.float64)
        for r in range(rows):
            for j in range(V):
                xp, xm = x.copy(), x.copy()
                xp[r, j] += h
                xm[r, j] -= h
                fp = oracle.cross_entropy(xp, y, temperature=T, reduction=red, want_grad=False)
                fm = oracle.cross_entropy(xm, y, temperature=T, reduction=red, want_grad=False)
                if red == "none":
                    d = (fp["loss_rows"] - fm["loss_rows"]) @ w / (2 * h)
                else:
                    d = w[0] * (fp["loss"] - fm["loss"]) / (2 * h)
                num[r, j] = d
        np.testing.assert_allclose(out["dlogits"], num, rtol=2e-6, atol=1e-9)


# ------------------------------------------------ library reduction (control)

def test_agrees_with_torch_fp64_on_ordinary_rows():
    """Below the fp64 collapse threshold torch's fp64 log_softmax is exact enough."""
    g = torch.Generator().manual_seed(9)
    rows, V = 24, 3001
    x = torch.randn((rows, V), generator=g, dtype=torch.float64) * 3
    y = torch.randint(0, V, (rows,), generator=g)
    x[torch.arange(8), y[:8]] = x[:8].max(dim=1).values + torch.linspace(1, 8, 8,
                                                                         dtype=torch.float64)
    y[20:] = -100
    for T in (1.0, 0.9):
        Te = oracle.exact_temperature(T)
        out = oracle.cross_entropy(x.numpy(), y.numpy(), temperature=T, reduction="mean")
        xt = x.clone().requires_grad_(True)
        loss = torch.nn.functional.cross_entropy(xt / Te, y, ignore_index=-100)
        loss.backward()
        ref_lp = torch.log_softmax(x / Te, dim=1)
        live = y != -100
        want = ref_lp[torch.arange(rows)[live], y[live]].numpy()
        np.testing.assert_allclose(out["logp"][live.numpy()], want, rtol=1e-11)
        assert out["loss"] == pytest.approx(loss.item(), rel=1e-13, abs=0)
        np.testing.assert_allclose(out["dlogits"], xt.grad.numpy(), rtol=1e-10, atol=1e-18)


# ---------------------------------------------------- the pages' printed values

def test_collapse_thresholds_from_the_pages():
    """The naive forms collapse exactly past the printed thresholds; the oracle does not."""
    gold = read_golden("collapse_thresholds.txt")
    assert round(math.log(2.0 ** 24), 1) == gold["fp32"]
    assert round(math.log(2.0 ** 53), 1) == gold["fp64"]
    for key, dtype in (("fp32", torch.float32), ("fp64", torch.float64)):
        thr = gold[key]
        for margin, collapses in ((thr - 0.3, False), (thr + 0.3, True)):
            # two-column row: the rest's log-sum-exp is exactly the other
            # logit, so the margin over it is `margin`; the naive form's
            # lse - x_y is log(sum exp(x - x_max)) and softmax(x_y) its exp
            row = torch.tensor([[0.0, margin]], dtype=dtype)
            lse_minus_xy = torch.log(torch.exp(row - row.max()).sum()).item()
            p_y = torch.softmax(row, dim=1)[0, 1].item()
            assert (lse_minus_xy == 0.0) == collapses, (key, margin, lse_minus_xy)
            assert (p_y == 1.0) == collapses, (key, margin, p_y)
            lp, _ = oracle.selective_logsoftmax(row.double().numpy(), [[1]], 1.0)
            assert lp[0, 0] < 0.0
            m = float(row.double()[0, 1])  # the margin as the row holds it (fp32: rounded)
            assert lp[0, 0] == pytest.approx(-math.log1p(math.exp(-m)), rel=1e-14, abs=0)


def test_sparse_supervision_workload_matches_page():
    gold = read_golden("sparse_supervision.txt")
    w = workloads.ce_sparse_bf16()
    assert w.rows == gold["rows"] and w.vocab == gold["vocab"]
    out = oracle.cross_entropy(workloads.to_numpy_f64(w.logits), w.labels.numpy(),
                               reduction="none", grad_out=w.grad_out.numpy())
    assert out["n_items"] == gold["supervised"]
    mib = 4 * w.vocab / 2 ** 20
    assert w.rows * mib == gold["fp32_mib_all_rows"]
    assert out["n_items"] * mib == gold["fp32_mib_supervised_rows"]
    live = w.labels.numpy() != workloads.IGNORE_INDEX
    assert np.all(out["dlogits"][~live] == 0.0) and np.all(out["loss_rows"][~live] == 0.0)
    # four contiguous spans per sample
    for s in range(2):
        seg = live[s * 961:(s + 1) * 961].astype(int)
        starts = np.sum(np.diff(np.concatenate([[0], seg])) == 1)
        assert starts == gold["spans_per_sample"]


# ---------------------------------------------------------- selection & errors

def test_reductions_and_item_count():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(10, 40))
    y = np.array([3, -100, 0, 39, -100, 7, 7, 1, -100, 2])
    none = oracle.cross_entropy(x, y, reduction="none", grad_out=np.ones(10))
    s = oracle.cross_entropy(x, y, reduction="sum")
    m = oracle.cross_entropy(x, y, reduction="mean")
    assert s["n_items"] == m["n_items"] == 7
    assert s["loss"] == pytest.approx(math.fsum(none["loss_rows"]), rel=1e-15, abs=0)
    assert m["loss"] == pytest.approx(s["loss"] / 7, rel=1e-15, abs=0)
    np.testing.assert_allclose(m["dlogits"], s["dlogits"] / 7, rtol=1e-15)
    np.testing.assert_allclose(none["dlogits"], s["dlogits"], rtol=1e-15)


def test_all_ignored_mean_is_zero():
    x = np.random.default_rng(0).normal(size=(5, 9))
    out = oracle.cross_entropy(x, np.full(5, -100), reduction="mean")
    assert out["n_items"] == 0 and out["loss"] == 0.0
    assert np.all(out["dlogits"] == 0.0)


def test_masked_rows_are_zero_and_unread():
    x = np.random.default_rng(1).normal(size=(4, 12))
    x[1] = np.nan                     # a masked row is never read
    lp, bad = oracle.selective_logsoftmax(x, [[0], [99], [3], [4]], 1.0,
                                          row_mask=[1, 0, 1, 0])
    assert bad == 0 and lp[1, 0] == 0.0 and lp[3, 0] == 0.0 and np.all(np.isfinite(lp))
    assert lp[0, 0] < 0.0 and lp[2, 0] < 0.0


def test_out_of_range_labels_are_flagged():
    x = np.random.default_rng(1).normal(size=(3, 8))
    out = oracle.cross_entropy(x, [2, 8, -5], reduction="sum")
    assert out["n_bad"] == 2
    assert np.isnan(out["loss_rows"][1]) and np.isnan(out["loss_rows"][2])
    assert np.all(np.isnan(out["dlogits"][1]))
    lp, bad = oracle.selective_logsoftmax(x, [[0], [8], [-1]], 1.0)
    assert bad == 2 and np.isnan(lp[1, 0]) and np.isnan(lp[2, 0])


def test_strided_rows_equal_contiguous():
    x = np.random.default_rng(4).normal(size=(6, 30))
    view = x[:, 3:20]
    lab = np.array([0, 1, 16, 5, 9, 2])
    a = oracle.cross_entropy(view, lab, reduction="sum")
    b = oracle.cross_entropy(np.ascontiguousarray(view), lab, reduction="sum")
    np.testing.assert_array_equal(a["logp"], b["logp"])
    np.testing.assert_array_equal(a["dlogits"], b["dlogits"])


# --------------------------------------------- selective log-softmax backward

def brute_selective_grad(row, idx, g, T):
    """(1/T) (sum_{k: t_k = j} g_k - G p_j) at 120 digits."""
    logps, _ = brute_row(row, 0, T)
    G = Decimal(0)
    for gk in g:
        G = CTX.add(G, Decimal(float(gk)))
    out = []
    for j, lp in enumerate(logps):
        acc = CTX.multiply(CTX.minus(G), CTX.exp(lp))
        for t, gk in zip(idx, g):
            if t == j:
                acc = CTX.add(acc, Decimal(float(gk)))
        out.append(float(CTX.divide(acc, Decimal(T))))
    return np.array(out)


@pytest.mark.parametrize("V", [2, 5, 33])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_selective_backward_brute_force(V, T):
    margins = [0.0, 17.0, 30.0, 50.0, 80.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=200 + V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    rng = np.random.default_rng(V)
    K = 3
    idx = np.stack([y, rng.integers(0, V, size=len(margins)), y], axis=1)  # duplicates of y
    g = rng.normal(size=(len(margins), K))
    dx, bad = oracle.selective_logsoftmax_backward(x, idx, g, T)
    assert bad == 0
    Te = oracle.exact_temperature(T)
    for r in range(len(margins)):
        want = brute_selective_grad(x[r], idx[r], g[r], Te)
        scale = np.max(np.abs(want))
        assert np.max(np.abs(dx[r] - want)) <= 1e-12 * scale, (r, margins[r])
        # the gathered label column keeps its (tiny) exact value
        assert dx[r, y[r]] == pytest.approx(want[y[r]], rel=1e-10, abs=1e-300)


def test_selective_backward_finite_difference():
    rng = np.random.default_rng(31)
    V, rows, K = 7, 3, 2
    x = rng.normal(scale=2.0, size=(rows, V))
    idx = np.array([[1, 4], [2, 2], [6, 0]])
    g = rng.normal(size=(rows, K))
    T = 0.8
    dx, _ = oracle.selective_logsoftmax_backward(x, idx, g, T)
    h = 1e-6
    num = np.zeros_like(x)
    for r in range(rows):
        for j in range(V):
            xp, xm = x.copy(), x.copy()
            xp[r, j] += h
            xm[r, j] -= h
            fp, _ = oracle.selective_logsoftmax(xp, idx, T)
            fm, _ = oracle.selective_logsoftmax(xm, idx, T)
            num[r, j] = np.sum(g * (fp - fm)) / (2 * h)
    np.testing.assert_allclose(dx, num, rtol=2e-6, atol=1e-9)


def test_selective_backward_k1_is_minus_ce_backward():
    """For one gathered index, d(g log p_t)/dx is the CE gradient with upstream -g."""
    w = workloads.collapse_stress(dtype=torch.float32, rows=16, V=3001, seed=5)
    x = workloads.to_numpy_f64(w.logits)
    lab = w.index.numpy()[:, 0]
    g = np.random.default_rng(0).normal(size=16)
    dx, _ = oracle.selective_logsoftmax_backward(x, lab[:, None], g[:, None], 0.9)
    ce = oracle.cross_entropy(x, lab, temperature=0.9, reduction="none", grad_out=-g)
    np.testing.assert_allclose(dx, ce["dlogits"], rtol=1e-12, atol=1e-300)


def test_selective_backward_uniform_rows_and_invariants():
    V, T = 40, 0.9
    x = np.full((3, V), 0.3)
    idx = np.array([[0, 5], [7, 7], [39, 1]])
    g = np.array([[1.0, 2.0], [0.5, 0.25], [-1.0, 3.0]])
    dx, _ = oracle.selective_logsoftmax_backward(x, idx, g, T, row_mask=[1, 1, 0])
    Te = oracle.exact_temperature(T)
    for r in range(2):
        want = np.full(V, -g[r].sum() / (V * Te))
        for t, gk in zip(idx[r], g[r]):
            want[t] += gk / Te
        np.testing.assert_allclose(dx[r], want, rtol=1e-12)
        assert abs(math.fsum(dx[r])) <= 1e-13 * math.fsum(np.abs(dx[r]))
    assert np.all(dx[2] == 0.0)


# --------------------------------------------------------------- row entropy

def brute_entropy(row, T):
    logps, _ = brute_row(row, 0, T)
    h = Decimal(0)
    for lp in logps:
        h = CTX.subtract(h, CTX.multiply(CTX.exp(lp), lp))
    return float(h)


@pytest.mark.parametrize("V", [2, 5, 33])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_entropy_brute_force(V, T):
    margins = [0.0, 5.0, 17.0, 30.0, 50.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=300 + V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    x[0] = np.random.default_rng(V).normal(scale=3.0, size=V)
    h, bad = oracle.entropy(x, y, T)
    assert bad == 0
    Te = oracle.exact_temperature(T)
    for r in range(len(margins)):
        want = brute_entropy(x[r], Te)
        assert h[r] == pytest.approx(want, rel=1e-11, abs=1e-300), (r, margins[r])
        assert h[r] > 0.0          # never collapses to 0 for a finite margin


@pytest.mark.parametrize("V", [5, 33])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_entropy_brute_force_when_another_column_dominates(V, T):
    # the sampled column (the reference passed in) is not the row's dominant
    # one: the dominant column's 1 - p must still not round away
    margins = [17.0, 30.0, 50.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=700 + V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    other = (y + 1 + np.arange(len(margins))) % V
    assert np.all(other != y)
    h, bad = oracle.entropy(x, other, T)
    assert bad == 0
    Te = oracle.exact_temperature(T)
    for r in range(len(margins)):
        want = brute_entropy(x[r], Te)
        assert h[r] == pytest.approx(want, rel=1e-11, abs=1e-300), (r, margins[r])


def test_entropy_closed_forms_and_bounds():
    V = 1000
    x = np.full((2, V), 0.25)
    h, _ = oracle.entropy(x, [3, 999], 0.8)
    np.testing.assert_allclose(h, math.log(V), rtol=1e-14)      # uniform: log V
    # two-level row: target a, V-1 others b
    a, b, T = 4.0, 1.0, 1.0
    x = np.full((1, V), b)
    x[0, 10] = a
    p_t = 1.0 / (1.0 + (V - 1) * math.exp(b - a))
    p_o = (1.0 - p_t) / (V - 1)
    want = -p_t * math.log(p_t) - (V - 1) * p_o * math.log(p_o)
    assert oracle.entropy(x, [10], T)[0][0] == pytest.approx(want, rel=1e-13, abs=0)
    # V = 1: certain, the reference column does not change the value
    assert oracle.entropy(np.array([[2.0]]), [0], 1.0)[0][0] == 0.0
    rng = np.random.default_rng(8)
    x = rng.normal(scale=4, size=(20, 77))
    h1, _ = oracle.entropy(x, rng.integers(0, 77, 20), 0.9)
    h2, _ = oracle.entropy(x, rng.integers(0, 77, 20), 0.9)
    np.testing.assert_allclose(h1, h2, rtol=1e-12)              # any reference column
    assert np.all(h1 >= 0.0) and np.all(h1 <= math.log(77))


def test_entropy_skips_dead_rows_and_flags_bad_references():
    x = np.random.default_rng(1).normal(size=(3, 9))
    h, bad = oracle.entropy(x, [1, 50, 2], 1.0, live=[1, 1, 0])
    assert bad == 1 and np.isnan(h[1]) and h[2] == 0.0 and h[0] > 0.0


def test_entropy_ignores_zero_probability_columns():
    # a column at -inf has p = 0 and adds nothing (0 log 0 = 0), also as the
    # reference column
    rng = np.random.default_rng(21)
    base = rng.normal(scale=2, size=(1, 40))
    x = np.concatenate([base, np.full((1, 3), -np.inf)], axis=1)
    want = oracle.entropy(base, [5], 0.9)[0][0]
    for ref in (5, 40, 42):
        got, bad = oracle.entropy(x, [ref], 0.9)
        assert bad == 0 and got[0] == pytest.approx(want, rel=1e-13, abs=0), ref


# ----------------------------------------------- entropy term of the backward

def brute_entropy_grad(row, T):
    """dH/dx_j = -(1/T) p_j (log p_j + H) at 120 digits, and the size
    max_j p_j (|log p_j| + H) / T of the terms it takes the difference of."""
    logps, _ = brute_row(row, 0, T)
    h = Decimal(0)
    for lp in logps:
        h = CTX.subtract(h, CTX.multiply(CTX.exp(lp), lp))
    Td = Decimal(T)
    grad = [float(-CTX.divide(CTX.multiply(CTX.exp(lp), CTX.add(lp, h)), Td)) for lp in logps]
    size = max(float(CTX.divide(CTX.multiply(CTX.exp(lp), CTX.add(abs(lp), h)), Td))
               for lp in logps)
    return np.array(grad), size


@pytest.mark.parametrize("V", [2, 5, 33])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_entropy_backward_brute_force(V, T):
    margins = [0.0, 17.0, 30.0, 50.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=500 + V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    gh = np.array([1.0, -0.5, 2.0, 0.25])
    zero = np.zeros((len(margins), 1))
    dx, bad = oracle.selective_logsoftmax_backward(x, y[:, None], zero, T, grad_entropy=gh)
    assert bad == 0
    Te = oracle.exact_temperature(T)
    for r in range(len(margins)):
        grad, size = brute_entropy_grad(x[r], Te)
        want = gh[r] * grad
        # log p_j + H cancels near a uniform row: the bound scales with the terms
        assert np.max(np.abs(dx[r] - want)) <= 1e-13 * abs(gh[r]) * size, (r, margins[r])
        # the dominant column's tiny entry keeps its relative accuracy
        assert dx[r, y[r]] == pytest.approx(want[y[r]], rel=1e-9, abs=1e-300)


@pytest.mark.parametrize("V", [5, 33])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_entropy_backward_brute_force_dominant_column_not_gathered(V, T):
    # gathered columns other than the dominant one, with and without log-prob
    # upstream: the dominant column's entry still keeps its relative accuracy
    margins = [17.0, 30.0, 50.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=900 + V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    idx = np.stack([(y + 1) % V, (y + 2) % V], axis=1)
    g = np.array([[0.0, 0.0], [0.5, -1.0], [0.0, 0.0]])
    gh = np.array([1.0, -0.75, 0.5])
    dx, bad = oracle.selective_logsoftmax_backward(x, idx, g, T, grad_entropy=gh)
    assert bad == 0
    Te = oracle.exact_temperature(T)
    for r in range(len(margins)):
        grad, size = brute_entropy_grad(x[r], Te)
        want = gh[r] * grad
        logps, _ = brute_row(x[r], 0, Te)
        for k in range(2):
            t = idx[r, k]
            want[t] += g[r, k] / Te
        want -= g[r].sum() / Te * np.array([float(CTX.exp(lp)) for lp in logps])
        d = y[r]
        assert dx[r, d] == pytest.approx(want[d], rel=1e-9, abs=1e-300), (r, margins[r])
        scale = abs(gh[r]) * size + np.abs(g[r]).sum() / Te
        assert np.max(np.abs(dx[r] - want)) <= 1e-13 * scale, (r, margins[r])


def test_entropy_backward_finite_difference_with_logp_terms():
    rng = np.random.default_rng(41)
    V, rows, K = 9, 3, 2
    x = rng.normal(scale=2.0, size=(rows, V))
    idx = np.array([[1, 4], [2, 2], [8, 0]])
    g = rng.normal(size=(rows, K))
    gh = rng.normal(size=rows)
    T = 0.8
    dx, _ = oracle.selective_logsoftmax_backward(x, idx, g, T, grad_entropy=gh)
    h = 1e-6
    num = np.zeros_like(x)
    for r in range(rows):
        for j in range(V):
            xp, xm = x.copy(), x.copy()
            xp[r, j] += h
            xm[r, j] -= h
            fp, _ = oracle.selective_logsoftmax(xp, idx, T)
            fm, _ = oracle.selective_logsoftmax(xm, idx, T)
            hp, _ = oracle.entropy(xp, idx[:, 0], T)
            hm, _ = oracle.entropy(xm, idx[:, 0], T)
            num[r, j] = (np.sum(g[r] * (fp[r] - fm[r])) + gh[r] * (hp[r] - hm[r])) / (2 * h)
    np.testing.assert_allclose(dx, num, rtol=2e-6, atol=1e-9)


def test_entropy_backward_invariants():
    # uniform rows sit at the entropy maximum: zero entropy gradient; rows sum
    # to zero; a column at -inf gets exactly 0
    V = 50
    x = np.full((1, V), 1.5)
    dx, _ = oracle.selective_logsoftmax_backward(x, [[3]], [[0.0]], 0.9, grad_entropy=[2.0])
    assert np.max(np.abs(dx)) <= 1e-15
    rng = np.random.default_rng(3)
    x = rng.normal(scale=3, size=(4, 60))
    x[1, 7] = -np.inf
    dx, _ = oracle.selective_logsoftmax_backward(x, rng.integers(0, 60, (4, 2)),
                                                 rng.normal(size=(4, 2)), 0.7,
                                                 grad_entropy=rng.normal(size=4))
    assert dx[1, 7] == 0.0
    for r in range(4):
        assert abs(math.fsum(dx[r])) <= 1e-14 * math.fsum(np.abs(dx[r]))


# ------------------------------------------- label smoothing and DFT on the CE

def brute_smoothed_loss(row, y, T, eps, dft):
    logps, lpy = brute_row(row, y, T)
    V = len(row)
    mean_nl = CTX.divide(-sum(logps, Decimal(0)), Decimal(V))
    loss = CTX.add(CTX.multiply(Decimal(1) - Decimal(eps), -lpy),
                   CTX.multiply(Decimal(eps), mean_nl))
    if dft:
        loss = CTX.multiply(CTX.exp(lpy), loss)
    return float(loss)


@pytest.mark.parametrize("V", [2, 5, 33])
@pytest.mark.parametrize("eps,dft", [(0.1, False), (0.0, True), (0.25, True)])
def test_smoothed_and_dft_loss_brute_force(V, eps, dft):
    margins = [0.0, 17.0, 30.0, 50.0]
    w = workloads.peaked_rows_tiny(V, margins, seed=700 + V)
    x = w.logits.numpy()
    y = w.labels.numpy()
    for T in (1.0, 0.7):
        out = oracle.cross_entropy(x, y, temperature=T, reduction="none", want_grad=False,
                                   label_smoothing=eps, dft=dft)
        Te = oracle.exact_temperature(T)
        for r in range(len(margins)):
            want = brute_smoothed_loss(x[r], y[r], Te, eps, dft)
            assert out["loss_rows"][r] == pytest.approx(want, rel=1e-12, abs=1e-300), (r, T)


def test_smoothed_ce_matches_torch_fp64():
    rng = np.random.default_rng(12)
    x = rng.normal(scale=2.5, size=(40, 300))
    y = rng.integers(0, 300, 40)
    y[[3, 17]] = -100
    g = 0.37
    for eps in (0.05, 0.3):
        for red in ("mean", "sum", "none"):
            out = oracle.cross_entropy(x, y, temperature=0.8, reduction=red, label_smoothing=eps,
                                       grad_out=np.full(40, g) if red == "none" else [g])
            xt = torch.tensor(x, requires_grad=True)
            Te = oracle.exact_temperature(0.8)
            ref = torch.nn.functional.cross_entropy(xt / Te, torch.tensor(y), ignore_index=-100,
                                                    reduction=red, label_smoothing=eps)
            (ref * g).sum().backward()
            if red == "none":
                np.testing.assert_allclose(out["loss_rows"], ref.detach().numpy(), rtol=1e-13)
            else:
                assert out["loss"] == pytest.approx(float(ref.detach()), rel=1e-13, abs=0)
            np.testing.assert_allclose(out["dlogits"], xt.grad.numpy(), rtol=1e-11, atol=1e-17)


def test_smoothing_and_dft_closed_forms():
    V = 64
    x = np.full((2, V), -0.4)
    # uniform row: every -log p_j is log V, so any eps gives log V; DFT scales by 1/V
    for eps in (0.0, 0.2, 1.0):
        out = oracle.cross_entropy(x, [1, 60], reduction="none", label_smoothing=eps)
        np.testing.assert_allclose(out["loss_rows"], math.log(V), rtol=1e-14)
        d = oracle.cross_entropy(x, [1, 60], reduction="none", label_smoothing=eps, dft=True)
        np.testing.assert_allclose(d["loss_rows"], math.log(V) / V, rtol=1e-14)
        # and a uniform row's smoothed gradient: (1 - eps)(1/V - 1) at y,
        # 1/V - eps/V = (1 - eps)/V at every other column
        np.testing.assert_allclose(out["dlogits"][0, 1], (1 - eps) * (1.0 / V - 1.0),
                                   rtol=1e-12, atol=1e-16)
        others = np.delete(out["dlogits"][0], 1)
        np.testing.assert_allclose(others, (1 - eps) / V, rtol=1e-12, atol=1e-16)


def test_smoothed_gradient_finite_difference_and_dft_relation():
    rng = np.random.default_rng(77)
    V, rows = 11, 3
    x = rng.normal(scale=2.0, size=(rows, V))
    y = np.array([2, 9, 0])
    eps, T, h = 0.15, 0.9, 1e-6
    out = oracle.cross_entropy(x, y, temperature=T, reduction="sum", label_smoothing=eps)
    num = np.zeros_like(x)
    for r in range(rows):
        for j in range(V):
            xp, xm = x.copy(), x.copy()
            xp[r, j] += h
            xm[r, j] -= h
            fp = oracle.cross_entropy(xp, y, temperature=T, reduction="sum", want_grad=False,
                                      label_smoothing=eps)["loss"]
            fm = oracle.cross_entropy(xm, y, temperature=T, reduction="sum", want_grad=False,
                                      label_smoothing=eps)["loss"]
            num[r, j] = (fp - fm) / (2 * h)
    np.testing.assert_allclose(out["dlogits"], num, rtol=2e-6, atol=1e-9)
    # DFT: the weight p_y is held constant, so the gradient is p_y times the plain one
    d = oracle.cross_entropy(x, y, temperature=T, reduction="sum", label_smoothing=eps, dft=True)
    py = np.exp(out["logp"])
    np.testing.assert_allclose(d["dlogits"], py[:, None] * out["dlogits"], rtol=1e-14)
    np.testing.assert_allclose(d["loss_rows"], py * out["loss_rows"], rtol=1e-14)
    for r in range(rows):
        assert abs(math.fsum(d["dlogits"][r])) <= 1e-14 * math.fsum(np.abs(d["dlogits"][r]))


# -------------------------------------------------- logit soft-capping on the CE

@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_softcapped_ce_matches_torch_fp64(eps):
    rng = np.random.default_rng(33)
    x = rng.normal(scale=20.0, size=(24, 200))      # many logits past the cap's knee
    y = rng.integers(0, 200, 24)
    y[5] = -100
    cap, T = 30.0, 0.8
    out = oracle.cross_entropy(x, y, temperature=T, reduction="sum", label_smoothing=eps,
                               softcap=cap, grad_out=[0.5])
    xt = torch.tensor(x, requires_grad=True)
    Te = oracle.exact_temperature(T)
    z = cap * torch.tanh(xt / cap)
    ref = torch.nn.functional.cross_entropy(z / Te, torch.tensor(y), ignore_index=-100,
                                            reduction="sum", label_smoothing=eps)
    (0.5 * ref).backward()
    assert out["loss"] == pytest.approx(float(ref.detach()), rel=1e-13, abs=0)
    np.testing.assert_allclose(out["dlogits"], xt.grad.numpy(), rtol=1e-10, atol=1e-16)


def test_softcap_limits_closed_form_and_finite_differences():
    rng = np.random.default_rng(4)
    x = rng.normal(scale=3.0, size=(5, 50))
    y = rng.integers(0, 50, 5)
    plain = oracle.cross_entropy(x, y, reduction="none")
    huge = oracle.cross_entropy(x, y, reduction="none", softcap=1e7)
    np.testing.assert_allclose(huge["loss_rows"], plain["loss_rows"], rtol=1e-10)
    np.testing.assert_allclose(huge["dlogits"], plain["dlogits"], rtol=1e-8, atol=1e-18)
    # V = 2: log p_y = -softplus((z_o - z_y) / T), z = cap tanh(x / cap)
    x2 = np.array([[41.0, -7.5]])
    cap, T = 25.0, 0.9
    zo, zy = cap * math.tanh(-7.5 / cap), cap * math.tanh(41.0 / cap)
    Te = oracle.exact_temperature(T)
    a = (zo - zy) / Te
    want = max(a, 0.0) + math.log1p(math.exp(-abs(a)))
    got = oracle.cross_entropy(x2, [0], temperature=T, reduction="none", softcap=cap)
    assert got["loss_rows"][0] == pytest.approx(want, rel=1e-13, abs=0)
    # finite differences through the cap
    x3 = rng.normal(scale=15.0, size=(2, 9))
    y3 = np.array([4, 0])
    d = oracle.cross_entropy(x3, y3, reduction="sum", softcap=cap)["dlogits"]
    h = 1e-6
    for r in range(2):
        for j in range(9):
            xp, xm = x3.copy(), x3.copy()
            xp[r, j] += h
            xm[r, j] -= h
            fp = oracle.cross_entropy(xp, y3, reduction="sum", softcap=cap, want_grad=False)
            fm = oracle.cross_entropy(xm, y3, reduction="sum", softcap=cap, want_grad=False)
            # abs: one ulp of a loss of order 10 over 2h is about 1e-9
            assert d[r, j] == pytest.approx((fp["loss"] - fm["loss"]) / (2 * h),
                                            rel=2e-6, abs=5e-9)


def test_softcap_chain_factor_far_past_the_knee():
    # d/dx [cap tanh(x / cap)] = 4 w / (1 + w)^2, w = e^{-2|u|}, u = x / cap:
    # about 1.7e-17 at u = 20 and 3.5e-26 at u = -30, where 1 - tanh^2(u)
    # is 0 in fp64; the plain softmax gradient (p - onehot) / T carries it
    cap, T = 2.0, 0.5
    x = np.array([[40.0, -60.0, 0.3, -1.7]])   # u = 20, -30, 0.15, -0.85
    out = oracle.cross_entropy(x, [2], temperature=T, reduction="sum", softcap=cap)
    Te = oracle.exact_temperature(T)
    z = np.array([cap * math.tanh(v / cap) for v in x[0]]) / Te
    e = np.exp(z - z.max())
    dz = (e / e.sum() - np.array([0.0, 0.0, 1.0, 0.0])) / Te
    for j, v in enumerate(x[0]):
        w = math.exp(-2.0 * abs(v / cap))
        want = dz[j] * 4.0 * w / (1.0 + w) ** 2
        assert want != 0.0
        assert abs(out["dlogits"][0, j] - want) <= 1e-12 * abs(want)


# ----------------------------------------------- vocabulary-slice partials

@pytest.mark.parametrize("cuts", [[0, 33], [0, 16, 33], [0, 1, 5, 20, 33], [0, 32, 33]])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_vocab_slices_reproduce_the_full_row(cuts, T):
    # slicing the vocabulary anywhere (slices of one column, targets at the
    # edges, duplicates, a masked row, collapse margins) and merging the
    # slices' partials gives the full-row log-probs
    rng = np.random.default_rng(len(cuts) + int(T * 10))
    V = 33
    w = workloads.peaked_rows_tiny(V, [0.0, 17.0, 30.0, 50.0], seed=41)
    x = w.logits.numpy()
    y = w.labels.numpy()
    idx = np.stack([y, rng.integers(0, V, 4), np.full(4, V - 1), y], axis=1)
    mask = np.array([1, 1, 0, 1], dtype=np.uint8)
    full, _ = oracle.selective_logsoftmax(x, idx, T, mask)
    parts = [oracle.vocab_slice_partials(x[:, a:b], idx, a, T, mask)
             for a, b in zip(cuts[:-1], cuts[1:])]
    got, xt0 = oracle.vocab_slice_combine(parts, cuts, idx, T, mask)
    np.testing.assert_allclose(got, full, rtol=1e-13, atol=0.0)
    np.testing.assert_array_equal(xt0[mask == 1], x[np.arange(4), idx[:, 0]][mask == 1])


def test_vocab_slices_brute_force_on_confident_rows():
    V, T = 9, 0.9
    w = workloads.peaked_rows_tiny(V, [17.0, 50.0], seed=43)
    x = w.logits.numpy()
    y = w.labels.numpy()
    idx = y[:, None]
    parts = [oracle.vocab_slice_partials(x[:, a:b], idx, a, T) for a, b in ((0, 4), (4, 9))]
    got, _ = oracle.vocab_slice_combine(parts, [0, 4, 9], idx, T)
    Te = oracle.exact_temperature(T)
    for r in range(2):
        _, want = brute_row(x[r], y[r], Te)
        assert got[r, 0] == pytest.approx(float(want), rel=1e-12, abs=0), r
        assert got[r, 0] < 0.0
