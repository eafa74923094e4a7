"""GPU parity of the token CE with label smoothing and DFT weighting
(ce_fwd, ce_bwd, ce_fwd_bwd_fused) against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (assert_grad_block_close, assert_grad_rows_close, assert_logp_close,
                     assert_loss_close, assert_zero_sum_rows, to_f64)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import cross_entropy_gb300 as gbce

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()
    gbce.load_library()


def check_rows_loss(got_rows, ref_rows, dtype, what):
    # row losses are >= 0: compare them as (negated) log-probs, same bound
    assert_logp_close(-to_f64(got_rows), -np.asarray(ref_rows), dtype, what)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("eps,dft", [(0.1, False), (0.0, True), (0.2, True)])
@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_fwd_bwd_and_fused_match_oracle(dtype, eps, dft, reduction):
    w = workloads.collapse_stress(dtype=dtype, rows=640, V=32003, seed=90)
    x, lab = w.logits.to(DEV), w.labels.to(DEV)
    T = 0.9
    g = (torch.randn(640, generator=torch.Generator().manual_seed(1)) if reduction == "none"
         else torch.tensor([0.75]))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(temperature=T, reduction=reduction, label_smoothing=eps, dft=dft)
    fwd = gbce.ce_fwd(x, lab, dev_status=status, **kw)
    d_sep = gbce.ce_bwd(x, lab, g.to(DEV), fwd.logp, fwd.n_items, dev_status=status, **kw)
    fused = gbce.ce_fwd_bwd_fused(x, lab, g.to(DEV), dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits), w.labels.numpy(),
                               temperature=T, reduction=reduction, grad_out=g.double().numpy(),
                               label_smoothing=eps, dft=dft)
    assert int(fwd.n_items.item()) == ref["n_items"] == int(fused.n_items.item())
    if reduction == "none":
        check_rows_loss(fwd.loss, ref["loss_rows"], dtype, "ce_fwd rows")
        check_rows_loss(fused.loss, ref["loss_rows"], dtype, "fused rows")
    else:
        assert_loss_close(float(fwd.loss.item()), ref["loss"], "ce_fwd")
        assert_loss_close(float(fused.loss.item()), ref["loss"], "fused")
    sel = np.arange(0, 640, 4)
    st = torch.as_tensor(sel, device=DEV)
    for d, name in ((d_sep, "ce_bwd"), (fused.dlogits, "fused")):
        got = to_f64(d[st])
        assert_grad_rows_close(got, ref["dlogits"][sel], dtype, name)
        assert_zero_sum_rows(got, dtype)
    # confident rows keep a nonzero label gradient (negative for g > 0, eps small)
    pk = w.peaked_rows.numpy()
    pk = pk[w.labels.numpy()[pk] >= 0][:20]
    col = w.labels.numpy()[pk]
    gl = to_f64(fused.dlogits[torch.as_tensor(pk, device=DEV)])[np.arange(len(pk)), col]
    want = ref["dlogits"][pk, col]
    assert np.all(np.sign(gl) == np.sign(want)) and np.all(gl != 0.0)


@pytest.mark.parametrize("rows", [2, 100])
def test_split_path_with_smoothing(rows):
    V = 152064
    w = workloads.collapse_stress(dtype=torch.bfloat16, rows=rows, V=V, seed=rows + 3)
    x, lab = w.logits.to(DEV), w.labels.to(DEV)
    fused = gbce.ce_fwd_bwd_fused(x, lab, torch.ones(1, device=DEV), temperature=0.8,
                                  reduction="sum", label_smoothing=0.05, dft=True)
    fwd = gbce.ce_fwd(x, lab, temperature=0.8, reduction="none", label_smoothing=0.05, dft=True)
    torch.cuda.synchronize()
    ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits), w.labels.numpy(),
                               temperature=0.8, reduction="sum", label_smoothing=0.05, dft=True)
    assert_loss_close(float(fused.loss.item()), ref["loss"], "fused sum")
    check_rows_loss(fwd.loss, ref["loss_rows"], torch.bfloat16, "ce_fwd rows")
    sel = np.arange(0, rows, max(1, rows // 20))
    assert_grad_rows_close(to_f64(fused.dlogits[torch.as_tensor(sel, device=DEV)]),
                           ref["dlogits"][sel], torch.bfloat16)


def test_minus_infinity_logit_gives_infinite_smoothed_loss():
    x = torch.randn((2, 4099), device=DEV)
    x[0, 17] = float("-inf")
    lab = torch.tensor([3, 5], device=DEV)
    fwd = gbce.ce_fwd(x, lab, reduction="none", label_smoothing=0.1)
    plain = gbce.ce_fwd(x, lab, reduction="none")
    torch.cuda.synchronize()
    assert torch.isinf(fwd.loss[0]) and torch.isfinite(fwd.loss[1])
    assert torch.isfinite(plain.loss).all()


def test_full_size_grpo_smoothed_dft_fused():
    w = workloads.grpo_bf16(device=DEV)
    out = gbce.ce_fwd_bwd_fused(w.logits, w.labels, torch.ones(1, device=DEV), temperature=0.9,
                                reduction="mean", label_smoothing=0.1, dft=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(9)
    sel = np.sort(np.concatenate([rng.choice(w.rows, 16, replace=False),
                                  w.peaked_rows.cpu().numpy()[:8]]))
    st = torch.as_tensor(sel, device=DEV)
    ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits[st]), w.labels[st].cpu().numpy(),
                               temperature=0.9, reduction="none", label_smoothing=0.1, dft=True,
                               grad_out=np.full(len(sel), 1.0 / w.rows))
    assert_grad_rows_close(to_f64(out.dlogits[st]), ref["dlogits"], torch.bfloat16)
    # the mean over all rows: each sampled row's loss also checked through ce_fwd
    rows_loss = gbce.ce_fwd(w.logits, w.labels, temperature=0.9, reduction="none",
                            label_smoothing=0.1, dft=True).loss
    check_rows_loss(rows_loss[st], ref["loss_rows"], torch.bfloat16, "rows")
    assert_loss_close(float(out.loss.item()), float(rows_loss.double().mean().item()), "mean")


# ------------------------------------------------------ logit soft-capping

def cap_tolerances(dtype, cap, T):
    """The standard bounds: soft-capping gets no extra margin."""
    from helpers import GRAD_TOL, LOGP_TOL
    return LOGP_TOL[dtype], GRAD_TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("eps,dft,scale", [(0.0, False, 1.0), (0.1, True, 1.0), (0.0, False, 12.0)])
def test_softcap_fwd_bwd_fused_match_oracle(dtype, eps, dft, scale):
    # scale 12 pushes most logits past the cap's knee (|x| / cap ~ 0.4 .. 2)
    rows, V, cap, T = 560, 24001, 30.0, 0.9
    w = workloads.collapse_stress(dtype=torch.float32, rows=rows, V=V, seed=70)
    x_cpu = (w.logits * scale).to(dtype)
    x, lab = x_cpu.to(DEV), w.labels.to(DEV)
    g = torch.tensor([0.5])
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(temperature=T, reduction="sum", label_smoothing=eps, dft=dft, softcap=cap)
    fwd = gbce.ce_fwd(x, lab, dev_status=status, **kw)
    rows_fwd = gbce.ce_fwd(x, lab, dev_status=status, **dict(kw, reduction="none"))
    d_sep = gbce.ce_bwd(x, lab, g.to(DEV), fwd.logp, fwd.n_items, dev_status=status, **kw)
    fused = gbce.ce_fwd_bwd_fused(x, lab, g.to(DEV), dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.cross_entropy(workloads.to_numpy_f64(x_cpu), w.labels.numpy(), temperature=T,
                               reduction="sum", grad_out=[0.5], label_smoothing=eps, dft=dft,
                               softcap=cap)
    lp_tol, g_tol = cap_tolerances(dtype, cap, T)
    live = w.labels.numpy() != -100
    assert_logp_close(to_f64(fwd.logp), ref["logp"], dtype, "capped log p", tol=lp_tol)
    assert_logp_close(-to_f64(rows_fwd.loss), -ref["loss_rows"], dtype, "capped rows", tol=lp_tol)
    assert abs(float(fused.loss.item()) - ref["loss"]) <= lp_tol * abs(ref["loss"])
    sel = np.arange(0, rows, 4)
    st = torch.as_tensor(sel, device=DEV)
    for d, name in ((d_sep, "ce_bwd"), (fused.dlogits, "fused")):
        got = to_f64(d[st])
        assert_grad_rows_close(got, ref["dlogits"][sel], dtype, name, tol=g_tol)
    assert np.all(to_f64(fused.dlogits)[~live] == 0.0)


def test_softcap_split_path_and_saturated_logits():
    # few rows take the split statistics + merge; logits up to 1e4 saturate
    V, cap = 152064, 50.0
    gen = torch.Generator().manual_seed(8)
    x_cpu = torch.randn((3, V), generator=gen) * 40.0
    x_cpu[0, 17] = 1e4
    x_cpu[1, 5] = -1e4
    lab = torch.tensor([17, 5, 100])
    x = x_cpu.to(DEV)
    out = gbce.ce_fwd_bwd_fused(x, lab.to(DEV), torch.ones(3, device=DEV), reduction="none",
                                softcap=cap)
    torch.cuda.synchronize()
    ref = oracle.cross_entropy(x_cpu.double().numpy(), lab.numpy(), reduction="none",
                               grad_out=np.ones(3), softcap=cap)
    lp_tol, g_tol = cap_tolerances(torch.float32, cap, 1.0)
    assert_logp_close(-to_f64(out.loss), -ref["loss_rows"], torch.float32, "rows", tol=lp_tol)
    assert_grad_rows_close(to_f64(out.dlogits), ref["dlogits"], torch.float32, tol=g_tol)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,V", [(300, 2), (300, 7), (300, 4099), (3, 70001)])
@pytest.mark.parametrize("cap", [1.0, 3.0])
def test_softcap_chain_factor_far_past_the_knee(dtype, rows, V, cap):
    # logits of 25 cap standard deviations: most lie far past the cap's knee,
    # where the chain factor 1 - tanh^2(x / cap) is tiny and a rounded tanh
    # would leave none of its digits.  Every gradient element against the
    # oracle: the head and tail elements, the label's vector, the
    # lane-by-lane vectors (3 rows: the split path).  Per element: the
    # gradient tolerance relative to the element, plus the dtype's rounding
    # floor (one ulp of its smallest normal magnitude range).
    T = 0.5
    gen = torch.Generator().manual_seed(V + int(cap))
    x_cpu = (torch.randn((rows, V), generator=gen) * (25.0 * cap)).to(dtype)
    lab = torch.randint(0, V, (rows,), generator=gen)
    g = torch.randn(rows, generator=gen)
    x, lab_d, g_d = x_cpu.to(DEV), lab.to(DEV), g.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(temperature=T, reduction="none", softcap=cap, dev_status=status)
    fused = gbce.ce_fwd_bwd_fused(x, lab_d, g_d, **kw)
    fwd = gbce.ce_fwd(x, lab_d, **kw)
    bwd = gbce.ce_bwd(x, lab_d, g_d, fwd.logp, fwd.n_items, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.cross_entropy(workloads.to_numpy_f64(x_cpu), lab.numpy(), temperature=T,
                               reduction="none", grad_out=g.double().numpy(), softcap=cap)
    from helpers import GRAD_TOL
    tol = GRAD_TOL[dtype]
    floor = 2.0 ** -148 if dtype == torch.float32 else 2.0 ** -133
    r = ref["dlogits"]
    far = np.abs(workloads.to_numpy_f64(x_cpu)) > 9.0 * cap
    assert far.mean() > 0.5 and np.all(r[far] != 0.0)
    for d, name in ((fused.dlogits, "fused"), (bwd, "ce_bwd")):
        err = np.abs(to_f64(d) - r)
        bad = err > tol * np.abs(r) + floor
        assert not np.any(bad), (f"{name}: {int(bad.sum())} elements off, worst relative "
                                 f"{(err[bad] / np.abs(r[bad])).max():.3e}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows", [3, 400])
def test_softcap_rows_opening_with_minus_infinity(dtype, rows):
    # a vocabulary mask over each row's first 8192 columns: every thread's
    # first vectors are all -inf, which the cap maps to -cap (finite), so the
    # capped sweep must take them into its max and sum like any other value
    # (3 rows: the split path; 400 rows: one CTA per row and the persistent
    # fused kernel)
    V, cap, T = 32000, 30.0, 0.9
    gen = torch.Generator().manual_seed(rows)
    x_cpu = torch.randn((rows, V), generator=gen) * 3.0
    x_cpu[:, :8192] = float("-inf")
    lab = torch.randint(8192, V, (rows,), generator=gen)
    x_cpu = x_cpu.to(dtype)
    x, lab_d = x_cpu.to(DEV), lab.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fwd = gbce.ce_fwd(x, lab_d, temperature=T, reduction="none", softcap=cap, dev_status=status)
    smooth = gbce.ce_fwd(x, lab_d, temperature=T, reduction="none", softcap=cap,
                         label_smoothing=0.1, dev_status=status)
    fused = gbce.ce_fwd_bwd_fused(x, lab_d, torch.ones(1, device=DEV), temperature=T,
                                  reduction="sum", softcap=cap, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    x64 = workloads.to_numpy_f64(x_cpu)
    ref = oracle.cross_entropy(x64, lab.numpy(), temperature=T, reduction="sum", softcap=cap,
                               grad_out=[1.0])
    ref_s = oracle.cross_entropy(x64, lab.numpy(), temperature=T, reduction="none",
                                 softcap=cap, label_smoothing=0.1)
    check_rows_loss(fwd.loss, ref["loss_rows"], dtype, "capped rows")
    check_rows_loss(smooth.loss, ref_s["loss_rows"], dtype, "capped smoothed rows")
    assert_loss_close(float(fused.loss.item()), ref["loss"], "capped fused sum")
    assert_grad_rows_close(to_f64(fused.dlogits), ref["dlogits"], dtype, "capped fused")


def test_full_size_grpo_softcap_fused_every_row():
    # the benchmark's rows with a soft-cap of 30: the persistent fused kernel
    # with the cap, every row's log p and gradient against the oracle
    w = workloads.grpo_bf16(device=DEV)
    out = gbce.ce_fwd_bwd_fused(w.logits, w.labels, torch.ones(1, device=DEV), temperature=0.9,
                                reduction="mean", softcap=30.0)
    torch.cuda.synchronize()
    lab = w.labels.cpu().numpy()
    total = 0.0
    for r0 in range(0, w.rows, 512):
        r1 = min(w.rows, r0 + 512)
        ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits[r0:r1]), lab[r0:r1],
                                   temperature=0.9, reduction="none", softcap=30.0,
                                   grad_out=np.full(r1 - r0, 1.0 / w.rows))
        assert_logp_close(to_f64(out.logp[r0:r1]), ref["logp"], torch.bfloat16, "capped log p")
        got = to_f64(out.dlogits[r0:r1])
        # (no zero-sum check: the chain factor 1 - tanh^2 differs per column)
        assert_grad_block_close(got, ref["dlogits"], torch.bfloat16, "capped fused")
        total += float(np.sum(ref["loss_rows"]))
        del got, ref
    assert_loss_close(float(out.loss.item()), total / w.rows, "capped mean")
