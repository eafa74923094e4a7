"""Special values in the logits, through the C ABI against the fp64 oracle.

A NaN logit makes its own row's outputs NaN and touches no other row.
Rows holding -inf logits (a vocabulary mask) give the oracle's finite
values, and so does a row whose every column but the label is -inf (log p
0, entropy 0, gradient exactly 0).  The sizes take the persistent fused
kernel (more rows than SMs), the row kernels' next-wave L2 prefetch (more
rows than resident CTAs, rows longer than one ring) and, for 3 rows, the
split path.  Rows led by one column far above their target (hundreds of
nats) check that every gradient keeps its bound there too.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (assert_entropy_close, assert_grad_rows_close, assert_logp_close, to_f64)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import cross_entropy_gb300 as gbce

DEV = "cuda:0"
V = 48000


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()
    gbce.load_library()


def special_rows(rows, dtype, seed):
    """~N(0, 2^2) logits with NaN, -inf and all-but-label -inf rows planted."""
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, V), generator=gen) * 2.0
    lab = torch.randint(4096, V - 1, (rows,), generator=gen)
    second = torch.randint(4096, V - 1, (rows,), generator=gen)
    if rows <= 3:
        nan_rows = {0: [100]}
        mask_rows = [1]
        lone_row = 2
    else:
        nan_rows = {5: [100], 300: [V - 1], rows - 1: [0, 777]}
        mask_rows = [7, 301, rows - 2]
        lone_row = 9
    for r, cols in nan_rows.items():
        for col in cols:
            x[r, col] = float("nan")
    for r in mask_rows:
        x[r, :4096] = float("-inf")          # every thread's first vectors
        x[r, 4096 + 13::97] = float("-inf")  # and scattered columns
        for t in (lab[r], second[r]):
            if not torch.isfinite(x[r, t]):
                x[r, t] = 0.5
    x[lone_row, :] = float("-inf")
    x[lone_row, lab[lone_row]] = 1.0
    second[lone_row] = lab[lone_row]
    return x.to(dtype), lab, torch.stack([lab, second], dim=1), sorted(nan_rows)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows", [3, 600])
def test_special_values_match_the_oracle(dtype, rows):
    x_cpu, lab, idx, nan_rows = special_rows(rows, dtype, seed=rows + 7)
    x, lab_d, idx_d = x_cpu.to(DEV), lab.to(DEV), idx.to(DEV)
    T = 0.9
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fwd = gbce.ce_fwd(x, lab_d, temperature=T, reduction="none", dev_status=status)
    fused = gbce.ce_fwd_bwd_fused(x, lab_d, torch.ones(rows, device=DEV), temperature=T,
                                  reduction="none", dev_status=status)
    mean = gbce.ce_fwd_bwd_fused(x, lab_d, torch.ones(1, device=DEV), temperature=T,
                                 reduction="mean", dev_status=status)
    capped = gbce.ce_fwd(x, lab_d, temperature=T, reduction="none", softcap=30.0,
                         dev_status=status)
    lp, ent = gbce.selective_logsoftmax(x, idx_d, T, with_entropy=True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    x64 = workloads.to_numpy_f64(x_cpu)
    ref = oracle.cross_entropy(x64, lab.numpy(), temperature=T, reduction="none",
                               grad_out=np.ones(rows))
    ref_cap = oracle.cross_entropy(x64, lab.numpy(), temperature=T, reduction="none",
                                   softcap=30.0, want_grad=False)
    ref_lp, _ = oracle.selective_logsoftmax(x64, idx.numpy(), T)
    ref_h, _ = oracle.entropy(x64, idx[:, 0].numpy(), T)

    # the NaN rows are NaN in every output, and only they are
    assert np.all(np.isnan(ref["loss_rows"][nan_rows]))
    assert_logp_close(-to_f64(fwd.loss), -ref["loss_rows"], dtype, "ce_fwd rows")
    assert_logp_close(to_f64(fused.logp), ref["logp"], dtype, "fused log p")
    assert_grad_rows_close(to_f64(fused.dlogits), ref["dlogits"], dtype, "fused dlogits")
    assert_logp_close(-to_f64(capped.loss), -ref_cap["loss_rows"], dtype, "capped rows")
    assert_logp_close(to_f64(lp), ref_lp, dtype, "selective log p")
    assert_entropy_close(to_f64(ent), ref_h, "entropy")
    assert np.isnan(float(mean.loss.item()))
    # a NaN stays in its row: every other row of the mean call's gradient is
    # finite (the NaN loss reaches them only through the mean's 1/n)
    live = np.setdiff1d(np.arange(rows), nan_rows)
    d = to_f64(mean.dlogits[torch.as_tensor(live, device=DEV)])
    assert np.all(np.isfinite(d))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows", [3, 600])
def test_rows_dominated_far_above_their_target(dtype, rows):
    # One column leads each row by 60..400 logit units at T = 0.5 (120..800
    # nats); the label and the gathered indices lie elsewhere.  The gathered
    # log p is then far below 0, and the dominant column's gradient must
    # still meet the gradient bound (in ce_bwd and the selective backward,
    # which only get the saved log p, and in the fused calls).
    Vd, T = 4099, 0.5
    gen = torch.Generator().manual_seed(rows + 11)
    x_cpu = torch.randn((rows, Vd), generator=gen) * 2.0
    dom = torch.randint(0, Vd, (rows,), generator=gen)
    lab = (dom + torch.randint(1, Vd, (rows,), generator=gen)) % Vd
    margin = 60.0 + 340.0 * torch.rand(rows, generator=gen)
    x_cpu[torch.arange(rows), dom] += margin
    x_cpu = x_cpu.to(dtype)
    idx = torch.stack([lab, (lab + 7) % Vd], dim=1)
    idx[:, 1] = torch.where(idx[:, 1] == dom, (lab + 8) % Vd, idx[:, 1])
    g = torch.randn(rows, generator=gen)
    gK = torch.randn((rows, 2), generator=gen)
    gH = torch.full((rows,), 0.05)
    x, lab_d, idx_d = x_cpu.to(DEV), lab.to(DEV), idx.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fwd = gbce.ce_fwd(x, lab_d, temperature=T, reduction="none", dev_status=status)
    fused = gbce.ce_fwd_bwd_fused(x, lab_d, g.to(DEV), temperature=T, reduction="none",
                                  dev_status=status)
    bwd = gbce.ce_bwd(x, lab_d, g.to(DEV), fwd.logp, fwd.n_items, temperature=T,
                      reduction="none", dev_status=status)
    capped = gbce.ce_fwd_bwd_fused(x, lab_d, g.to(DEV), temperature=T, reduction="none",
                                   softcap=150.0, dev_status=status)
    lp, ent = gbce.selective_logsoftmax(x, idx_d, T, with_entropy=True, dev_status=status)
    dsel = gbce.selective_logsoftmax_bwd(x, idx_d, gK.to(DEV), lp, T, dev_status=status)
    dent = gbce.selective_logsoftmax_bwd(x, idx_d, gK.to(DEV), lp, T, grad_entropy=gH.to(DEV),
                                         saved_entropy=ent, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    x64 = workloads.to_numpy_f64(x_cpu)
    ref = oracle.cross_entropy(x64, lab.numpy(), temperature=T, reduction="none",
                               grad_out=g.double().numpy())
    ref_cap = oracle.cross_entropy(x64, lab.numpy(), temperature=T, reduction="none",
                                   grad_out=g.double().numpy(), softcap=150.0)
    assert np.all(ref["logp"] < -100.0)
    assert_logp_close(to_f64(fwd.logp), ref["logp"], dtype, "ce_fwd log p")
    assert_grad_rows_close(to_f64(fused.dlogits), ref["dlogits"], dtype, "fused dlogits")
    assert_grad_rows_close(to_f64(bwd), ref["dlogits"], dtype, "ce_bwd dlogits")
    assert_grad_rows_close(to_f64(capped.dlogits), ref_cap["dlogits"], dtype, "capped dlogits")
    ref_d, _ = oracle.selective_logsoftmax_backward(x64, idx.numpy(), gK.double().numpy(), T)
    ref_de, _ = oracle.selective_logsoftmax_backward(x64, idx.numpy(), gK.double().numpy(), T,
                                                     grad_entropy=gH.double().numpy())
    assert_grad_rows_close(to_f64(dsel), ref_d, dtype, "selective backward")
    assert_grad_rows_close(to_f64(dent), ref_de, dtype, "selective backward + entropy")
