"""A seeded sweep of mixed configurations, every output against the fp64 oracle.

Each case draws its own row count (1 row up to several waves), vocabulary
(1 column up to 70001, aligned and ragged), dtype, temperature, logit
scale, padded row stride, K, ignored labels, masked rows, label smoothing,
DFT, soft-cap and reduction.  It runs the token CE (forward, backward,
fused) and the selective log-softmax with its entropy and backward, all
through the C ABI.  The fixed-shape tests cover each feature alone; this
sweep covers their combinations and the shapes between them.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (GRAD_FLOOR, GRAD_TOL, LOGP_FLOOR, assert_entropy_close,
                     assert_grad_rows_close, assert_logp_close, assert_loss_close, cap_eps,
                     to_f64)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import cross_entropy_gb300 as gbce

DEV = "cuda:0"


def make_configs(seed, n, extreme=False, temps=None):
    """n seeded configurations; `extreme` widens the temperature (0.1 .. 4),
    the logit scale (up to 50) and the soft-cap (1 .. 200); `temps`
    replaces the temperatures drawn from."""
    rng = np.random.default_rng(seed)
    if temps is None:
        temps = [0.1, 0.25, 0.5, 1.0, 4.0] if extreme else [0.5, 0.9, 1.0, 1.7]
    scales = [1.0, 20.0, 50.0] if extreme else [1.0, 4.0, 20.0]
    caps = [0.0, 0.0, 1.0, 30.0, 200.0] if extreme else [0.0, 0.0, 30.0, 5.0]
    out = []
    for i in range(n):
        rows = int(rng.choice([1, 2, 3, 7, 64, 129, 300, 457, 700]))
        V = int(rng.choice([1, 2, 7, 8, 9, 1000, 4096, 4099, 8191, 24001, 32768, 50001, 70001]))
        while rows * V > 6_000_000:
            V //= 2
        out.append(dict(
            seed=int(seed * 1000 + i), rows=rows, V=max(V, 1),
            dtype=str(rng.choice(["f32", "bf16"])),
            T=float(rng.choice(temps)),
            scale=float(rng.choice(scales)),
            pad=int(rng.choice([0, 0, 13])),
            K=int(rng.choice([1, 2, 4, 5, 16])),
            eps=float(rng.choice([0.0, 0.0, 0.1])),
            dft=bool(rng.random() < 0.25),
            cap=float(rng.choice(caps)),
            red=str(rng.choice(["none", "sum", "mean"])),
            p_ignore=float(rng.choice([0.0, 0.1, 0.9])),
            p_mask=float(rng.choice([0.0, 0.2])),
        ))
    return out


CONFIGS = make_configs(2024, 36) + make_configs(106, 60) + make_configs(7, 24, extreme=True) + [
    c for s in (14, 17, 19, 20, 22, 26, 30, 39) for c in make_configs(s, 60, extreme=True)] + (
    make_configs(60, 40, extreme=True, temps=[0.02, 0.05]))


def _id(c):
    return (f"{c['rows']}x{c['V']}-{c['dtype']}-T{c['T']}-s{c['scale']:g}-K{c['K']}-{c['red']}"
            f"{'-ls' if c['eps'] else ''}{'-dft' if c['dft'] else ''}"
            f"{'-cap%g' % c['cap'] if c['cap'] else ''}{'-pad' if c['pad'] else ''}")


def assert_sum_of_parts_close(got, parts, dtype, what, input_floor=None):
    """A gradient that is the sum of separately exact parts (the log-probs'
    upstream and the entropy's), per row: ||got - sum|| <= tol * sum_i
    ||part_i|| (+ the dtype's rounding floor, + `input_floor[r]`, what the
    fp32 floors of the backward's saved inputs move the row by).  Where the
    parts nearly cancel, no fp32 evaluation keeps a relative bound on the
    sum itself: its rounding is relative to the parts."""
    ref = sum(parts)
    tol = GRAD_TOL[dtype]
    floor = GRAD_FLOOR[dtype] * math.sqrt(ref.shape[1])
    for r in range(ref.shape[0]):
        if np.all(np.isnan(ref[r])):
            assert np.all(np.isnan(got[r])), f"{what}: row {r} should be NaN"
            continue
        scale = sum(np.linalg.norm(p[r]) for p in parts)
        if scale == 0.0:
            assert np.all(got[r] == 0.0), f"{what}: row {r} should be exactly zero"
            continue
        diff = np.linalg.norm(got[r] - ref[r])
        extra = 0.0 if input_floor is None else input_floor[r]
        assert diff <= tol * scale + floor + extra, (
            f"{what}: row {r} error {diff / scale:.3e} of its parts > {tol:.0e}")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()
    gbce.load_library()


@pytest.mark.parametrize("c", CONFIGS, ids=[_id(c) for c in CONFIGS])
def test_random_config_matches_oracle(c):
    rows, V, K, T = c["rows"], c["V"], c["K"], c["T"]
    dtype = torch.float32 if c["dtype"] == "f32" else torch.bfloat16
    gen = torch.Generator().manual_seed(c["seed"])
    big = (torch.randn((rows, V + c["pad"]), generator=gen) * c["scale"]).to(dtype)
    x_cpu = big[:, :V]
    lab = torch.randint(0, V, (rows,), generator=gen)
    lab[torch.rand(rows, generator=gen) < c["p_ignore"]] = -100
    idx = torch.randint(0, V, (rows, K), generator=gen)
    idx[:, 0] = torch.where(lab >= 0, lab, idx[:, 0])
    mask = (torch.rand(rows, generator=gen) >= c["p_mask"]).to(torch.uint8)
    g_rows = torch.randn(rows, generator=gen)
    g = g_rows if c["red"] == "none" else torch.tensor([0.75])
    gK = torch.randn((rows, K), generator=gen)
    gH = torch.randn(rows, generator=gen) * 0.1

    x = big.to(DEV)[:, :V]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(temperature=T, reduction=c["red"], label_smoothing=c["eps"], dft=c["dft"],
              softcap=c["cap"], dev_status=status)
    lab_d, g_d = lab.to(DEV), g.to(DEV)
    fwd = gbce.ce_fwd(x, lab_d, **kw)
    fused = gbce.ce_fwd_bwd_fused(x, lab_d, g_d, **kw)
    bwd = gbce.ce_bwd(x, lab_d, g_d, fwd.logp, fwd.n_items, **kw)
    lp, ent = gbce.selective_logsoftmax(x, idx.to(DEV), T, mask.to(DEV), with_entropy=True,
                                        dev_status=status)
    dsel = gbce.selective_logsoftmax_bwd(x, idx.to(DEV), gK.to(DEV), lp, T, mask.to(DEV),
                                         grad_entropy=gH.to(DEV), saved_entropy=ent,
                                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    x64 = workloads.to_numpy_f64(x_cpu)
    ref = oracle.cross_entropy(x64, lab.numpy(), temperature=T, reduction=c["red"],
                               grad_out=g.double().numpy(), label_smoothing=c["eps"],
                               dft=c["dft"], softcap=c["cap"])
    assert int(fwd.n_items.item()) == ref["n_items"] == int(fused.n_items.item())
    # soft-capped: the fp32 error of the capped logits themselves (cap_eps)
    eps = cap_eps(c["cap"], T)
    assert_logp_close(to_f64(fwd.logp), ref["logp"], dtype, "ce_fwd log p", floor=2 * eps)
    assert_logp_close(to_f64(fused.logp), ref["logp"], dtype, "fused log p", floor=2 * eps)
    py = np.exp(ref["logp"])
    row_floor = np.full(rows, 2 * eps)
    if c["dft"]:  # p_y (its CE), p_y an fp32 value that may be subnormal
        ce = np.divide(ref["loss_rows"], py, out=np.zeros(rows), where=py > 0)
        row_floor = 2.0 ** -148 * ce + 2.0 ** -149 + 2 * eps * (np.abs(ref["loss_rows"]) + py)
    row_floor = row_floor + LOGP_FLOOR  # a row loss near 0 is a log p near 0
    row_floor = np.where(ref["logp"] == 0.0, 0.0, row_floor)  # ignored rows stay exact
    if c["red"] == "none":
        assert_logp_close(-to_f64(fwd.loss), -ref["loss_rows"], dtype, "ce_fwd rows",
                          floor=row_floor)
        assert_logp_close(-to_f64(fused.loss), -ref["loss_rows"], dtype, "fused rows",
                          floor=row_floor)
    else:
        assert_loss_close(float(fwd.loss.item()), ref["loss"], "ce_fwd loss",
                          floor=row_floor.sum())
        assert_loss_close(float(fused.loss.item()), ref["loss"], "fused loss",
                          floor=row_floor.sum())
    gtol = GRAD_TOL[dtype] + 3 * eps
    # the fp32 floors near the subnormals (helpers): the label element from
    # the fp32 log p, a subnormal DFT weight, the capped element's 2nd rounding
    n_live = max(int(ref["n_items"]), 1)
    g_row = {"none": np.abs(g_rows.double().numpy()), "sum": np.full(rows, 0.75),
             "mean": np.full(rows, 0.75 / n_live)}[c["red"]] / T
    g_floor = g_row * (2.0 ** -148 + (2.0 ** -150 * math.sqrt(2) if c["dft"] else 0.0))
    if c["eps"]:
        # label smoothing: an element is p_j minus its smoothed target, both
        # of order 1 in fp32 (expm1(log p) + eps (1 - 1/V) at the label): where
        # p sits on the target the difference cancels to a few fp32 ulps of
        # the parts, whose norms are at most 1 each
        g_floor = g_floor + g_row * 2.0 ** -21
    if c["cap"]:
        g_floor = g_floor + GRAD_FLOOR[dtype] * math.sqrt(V)
    assert_grad_rows_close(to_f64(fused.dlogits), ref["dlogits"], dtype, "fused dlogits", tol=gtol,
                           extra_floor=g_floor)
    assert_grad_rows_close(to_f64(bwd), ref["dlogits"], dtype, "ce_bwd dlogits", tol=gtol,
                           extra_floor=g_floor)

    ref_lp, _ = oracle.selective_logsoftmax(x64, idx.numpy(), T, mask.numpy())
    ref_h, _ = oracle.entropy(x64, idx[:, 0].numpy(), T, live=mask.numpy())
    # the backward's two parts: through the log-probs, through the entropy
    ref_dl, _ = oracle.selective_logsoftmax_backward(x64, idx.numpy(), gK.double().numpy(), T,
                                                     mask.numpy())
    ref_dh, _ = oracle.selective_logsoftmax_backward(x64, idx.numpy(), np.zeros((rows, K)), T,
                                                     mask.numpy(),
                                                     grad_entropy=gH.double().numpy())
    assert_logp_close(to_f64(lp), ref_lp, dtype, "selective log p")
    assert_entropy_close(to_f64(ent), ref_h, "entropy")
    # the backward takes the forward's fp32 log p and entropy, each within
    # 2^-148 of exact near 0 (the log p / entropy floors); the row moves by
    # at most (|sum_k g_k| + |g_H|) / T times twice that.  A gathered
    # column's element (g_t (1 - p) - g_o p) / T is formed from the fp32
    # log p and cancels where its two terms meet: a few fp32 ulps of its
    # parts, 2^-22 sum_k |g_k| / T
    g_abs = np.abs(gK.double().numpy()).sum(axis=1)
    in_floor = (g_abs + np.abs(gH.double().numpy())) / T * 2.0 ** -147 + g_abs / T * 2.0 ** -22
    assert_sum_of_parts_close(to_f64(dsel), [ref_dl, ref_dh], dtype, "selective backward",
                              input_floor=in_floor)
