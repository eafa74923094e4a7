"""GPU parity: the CUDA library through its C ABI against the fp64 oracle.

Inputs are the seeded workloads; the oracle sees exact fp64 copies of the
same bf16/fp32 logits.  Tolerances are in tests/helpers.py.
"""

import hashlib
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden
from helpers import (assert_grad_block_close, assert_grad_rows_close, assert_logp_close,
                     assert_loss_close, assert_zero_sum_block, assert_zero_sum_rows, to_f64)

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


def new_status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def run_gpu(w: workloads.Workload, T, red, g):
    """Every entry point on one workload, on the GPU."""
    x = w.logits.to(DEV)
    lab = w.labels.to(DEV)
    status = new_status()
    res = {}
    res["logp_sel"] = gbce.selective_logsoftmax(
        x, w.index.to(DEV), T, None if w.row_mask is None else w.row_mask.to(DEV),
        dev_status=status)
    fwd = gbce.ce_fwd(x, lab, temperature=T, reduction=red, want_lse=True, dev_status=status)
    res["fwd"] = fwd
    res["bwd"] = gbce.ce_bwd(x, lab, g.to(DEV), fwd.logp, fwd.n_items, temperature=T,
                             reduction=red, dev_status=status)
    res["fused"] = gbce.ce_fwd_bwd_fused(x, lab, g.to(DEV), temperature=T, reduction=red,
                                         want_lse=True, dev_status=status)
    torch.cuda.synchronize()
    res["status"] = int(status.item())
    return res


def upstream_rows(w, red, g, sel):
    """Each selected row's upstream gradient (the mean's 1/n_items folded in)."""
    n_full = int((w.labels.cpu().numpy() != workloads.IGNORE_INDEX).sum())
    g_np = g.cpu().double().numpy()
    if red == "none":
        return g_np[sel], n_full
    if red == "sum":
        return np.full(len(sel), g_np[0]), n_full
    return np.full(len(sel), g_np[0] / n_full if n_full else 0.0), n_full


def run_all(w: workloads.Workload, temperature=None, reduction=None, grad_out=None,
            rows_sel=None):
    """Every entry point on one workload; oracle on `rows_sel` (default all rows)."""
    T = w.temperature if temperature is None else temperature
    red = w.reduction if reduction is None else reduction
    g = w.grad_out if grad_out is None else grad_out
    res = run_gpu(w, T, red, g)

    sel = np.arange(w.rows) if rows_sel is None else np.asarray(rows_sel)
    x64 = workloads.to_numpy_f64(w.logits[torch.as_tensor(sel)])
    lab_np = w.labels.cpu().numpy()
    mask_np = None if w.row_mask is None else w.row_mask.cpu().numpy()[sel]
    ref_lp, _ = oracle.selective_logsoftmax(x64, w.index.cpu().numpy()[sel], T, mask_np)
    g_rows, n_full = upstream_rows(w, red, g, sel)
    ref = oracle.cross_entropy(x64, lab_np[sel], temperature=T, reduction="none",
                               grad_out=g_rows)
    ref["n_full"] = n_full
    return res, ref, sel


def check_all(w, res, ref, sel, reduction=None, check_scalar_vs_oracle=True, T=None):
    dt = w.logits.dtype
    red = w.reduction if reduction is None else reduction
    T = w.temperature if T is None else T
    assert res["status"] == 0
    assert_logp_close(to_f64(res["logp_sel"])[sel], ref_logp_sel(w, sel, T), dt, "selective")
    fwd, fused = res["fwd"], res["fused"]
    assert int(fwd.n_items.item()) == ref["n_full"] == int(fused.n_items.item())
    for name, lp in (("ce_fwd logp", fwd.logp), ("fused logp", fused.logp)):
        assert_logp_close(to_f64(lp)[sel], ref["logp"], dt, name)
    live = w.labels.cpu().numpy()[sel] != workloads.IGNORE_INDEX
    lse = to_f64(fwd.lse)[sel]
    assert np.all(lse[~live] == 0.0)
    lse_ref = workloads.to_numpy_f64(w.logits[torch.as_tensor(sel)])[
        np.arange(len(sel)), np.where(live, w.labels.cpu().numpy()[sel], 0)] / \
        oracle.exact_temperature(T) - ref["logp"]
    np.testing.assert_allclose(lse[live], lse_ref[live], rtol=2e-6, atol=2e-6)
    # per-row losses and the reduced loss
    if red == "none":
        assert_logp_close(-to_f64(fwd.loss)[sel], -ref["loss_rows"], dt, "loss rows")
        assert_logp_close(-to_f64(fused.loss)[sel], -ref["loss_rows"], dt, "fused loss rows")
    else:
        lp_all = to_f64(fwd.logp)
        total = -np.sum(lp_all)
        want = total if red == "sum" else (total / ref["n_full"] if ref["n_full"] else 0.0)
        assert_loss_close(float(fwd.loss.item()), want, "ce_fwd loss vs its rows")
        assert_loss_close(float(fused.loss.item()), want, "fused loss vs its rows")
        if check_scalar_vs_oracle and len(sel) == w.rows:
            s = float(np.sum(ref["loss_rows"]))
            want_o = s if red == "sum" else (s / ref["n_full"] if ref["n_full"] else 0.0)
            assert_loss_close(float(fused.loss.item()), want_o, "fused loss vs oracle")
    for name, d in (("ce_bwd", res["bwd"]), ("fused", fused.dlogits)):
        got = to_f64(d[torch.as_tensor(sel, device=d.device)])
        assert_grad_rows_close(got, ref["dlogits"], dt, name)
        assert_zero_sum_rows(got, dt)


def ref_logp_sel(w, sel, T):
    mask = None if w.row_mask is None else w.row_mask.cpu().numpy()[sel]
    out, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(w.logits[torch.as_tensor(sel)]),
                                         w.index.cpu().numpy()[sel], T, mask)
    return out


# ------------------------------------------------------------ the workloads

def test_ce_small_fp32_64x4096():
    w = workloads.ce_small_fp32()
    res, ref, sel = run_all(w)
    check_all(w, res, ref, sel)
    # the 20-margin rows keep a nonzero, negative target gradient
    d = to_f64(res["fused"].dlogits)
    lab = w.labels.numpy()
    for r in w.peaked_rows.numpy():
        assert d[r, lab[r]] < 0.0


def test_ce_sparse_bf16_1922x4096():
    w = workloads.ce_sparse_bf16()
    res, ref, sel = run_all(w)
    check_all(w, res, ref, sel, reduction="none")
    live = w.labels.numpy() != workloads.IGNORE_INDEX
    fused = res["fused"]
    assert int(fused.n_items.item()) == 256
    d = fused.dlogits
    assert torch.all(d[torch.as_tensor(~live, device=DEV)] == 0)
    # upstream weight 1/256 with reduction none == mean with upstream 1
    mean = gbce.ce_fwd_bwd_fused(w.logits.to(DEV), w.labels.to(DEV), torch.ones(1),
                                 reduction="mean")
    assert torch.equal(mean.dlogits, d)
    assert_loss_close(float(mean.loss.item()), float(fused.loss.double().sum().item()) / 256)


@pytest.mark.parametrize("T", [1.0, 0.9])
def test_logp_bf16_1024x32768(T):
    w = workloads.logp_bf16()
    x = w.logits.to(DEV)
    status = new_status()
    got = gbce.selective_logsoftmax(x, w.index.to(DEV), T, w.row_mask.to(DEV),
                                    dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(w.logits), w.index.numpy(), T,
                                         w.row_mask.numpy())
    g = to_f64(got)
    assert_logp_close(g, ref, torch.bfloat16)
    masked = w.row_mask.numpy() == 0
    assert masked.sum() == 154 and np.all(g[masked] == 0.0)


def sample_rows(w, n_plain=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(w.rows, size=n_plain, replace=False).tolist())
    if w.peaked_rows is not None:
        pk = w.peaked_rows.cpu().numpy()
        rows |= set(rng.choice(pk, size=min(24, len(pk)), replace=False).tolist())
    rows |= {0, w.rows - 1}
    return np.array(sorted(rows))


def check_every_row(w, res, T, red, g, block=512):
    """Every row of a full-size run against the oracle, in row blocks (host
    memory stays bounded): both log-probs, the lse, both gradients and
    their zero sums; then the reduced loss against the oracle's own."""
    dt = w.logits.dtype
    assert res["status"] == 0
    fwd, fused = res["fwd"], res["fused"]
    lab_np = w.labels.cpu().numpy()
    mask_np = None if w.row_mask is None else w.row_mask.cpu().numpy()
    g_all, n_full = upstream_rows(w, red, g, np.arange(w.rows))
    assert int(fwd.n_items.item()) == n_full == int(fused.n_items.item())
    loss_rows = np.empty(w.rows)
    Te = oracle.exact_temperature(T)
    worst = {"logp": 0.0, "grad": 0.0}
    for r0 in range(0, w.rows, block):
        r1 = min(w.rows, r0 + block)
        x64 = workloads.to_numpy_f64(w.logits[r0:r1])
        ref_sel, _ = oracle.selective_logsoftmax(
            x64, w.index[r0:r1].cpu().numpy(), T, None if mask_np is None else mask_np[r0:r1])
        assert_logp_close(to_f64(res["logp_sel"][r0:r1]), ref_sel, dt, "selective")
        ref = oracle.cross_entropy(x64, lab_np[r0:r1], temperature=T, reduction="none",
                                   grad_out=g_all[r0:r1])
        for name, lp in (("ce_fwd logp", fwd.logp), ("fused logp", fused.logp)):
            worst["logp"] = max(worst["logp"],
                                assert_logp_close(to_f64(lp[r0:r1]), ref["logp"], dt, name))
        live = lab_np[r0:r1] != workloads.IGNORE_INDEX
        lse = to_f64(fwd.lse[r0:r1])
        assert np.all(lse[~live] == 0.0)
        xy = x64[np.arange(r1 - r0), np.where(live, lab_np[r0:r1], 0)]
        np.testing.assert_allclose(lse[live], (xy / Te - ref["logp"])[live], rtol=2e-6,
                                   atol=2e-6)
        loss_rows[r0:r1] = ref["loss_rows"]
        for name, d in (("ce_bwd", res["bwd"]), ("fused", fused.dlogits)):
            got = to_f64(d[r0:r1])
            worst["grad"] = max(worst["grad"],
                                assert_grad_block_close(got, ref["dlogits"], dt, name))
            assert_zero_sum_block(got, dt)
            del got
        del x64, ref
    total = math.fsum(loss_rows)
    want = total if red == "sum" else (total / n_full if n_full else 0.0)
    assert_loss_close(float(fwd.loss.item()), want, "ce_fwd loss vs oracle")
    assert_loss_close(float(fused.loss.item()), want, "fused loss vs oracle")
    return worst


def test_grpo_bf16_8192x152064_k4_full_size():
    """Full size, launch configuration of the benchmark; every row against the oracle."""
    w = workloads.grpo_bf16(device=DEV)
    res = run_gpu(w, w.temperature, w.reduction, w.grad_out)
    check_every_row(w, res, w.temperature, w.reduction, w.grad_out)
    # invariants on every row
    lp = res["logp_sel"]
    assert bool(torch.all(lp <= 0)) and bool(torch.all(torch.isfinite(lp)))
    fused = res["fused"]
    assert int(fused.n_items.item()) == w.rows
    d = fused.dlogits
    lab = w.labels.to(DEV)
    tgt = d.gather(1, lab[:, None])[:, 0].float()
    assert bool(torch.all(tgt < 0)), "every row keeps a negative target gradient"
    rowsum = d.double().sum(dim=1)
    rowabs = d.double().abs().sum(dim=1)
    assert bool(torch.all(rowsum.abs() <= 4e-3 * rowabs))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_collapse_stress_2048x151936_full_size(dtype):
    w = workloads.collapse_stress(dtype=dtype, device=DEV)
    res = run_gpu(w, w.temperature, w.reduction, w.grad_out)
    worst = check_every_row(w, res, w.temperature, w.reduction, w.grad_out)
    # at least as accurate as the collapse fix's own reported accuracy on the
    # same margins and vocabulary (tests/golden/accuracy_bars.txt)
    bars = read_golden("accuracy_bars.txt")
    grad_bar = bars["grad_fp32_worst_row_rel" if dtype == torch.float32
                    else "grad_bf16_worst_row_rel"]
    assert worst["grad"] <= grad_bar, (worst, grad_bar)
    assert worst["logp"] <= bars["logp_collapsed_rel"], worst
    fused = res["fused"]
    live = (w.labels != workloads.IGNORE_INDEX)
    assert int(fused.n_items.item()) == int(live.sum().item()) == 2048 - 205
    # logp <= 0 and nonzero on every confident row; target gradient nonzero
    lp = fused.logp
    assert bool(torch.all(lp <= 0))
    pk = w.peaked_rows
    assert bool(torch.all(lp[pk] < 0)), "a confident row collapsed to log p = 0"
    tgt = fused.dlogits[pk, w.labels[pk]].float()
    assert bool(torch.all(tgt < 0)), "a confident row lost its target gradient"
    d = fused.dlogits.double()
    tol = 1e-5 if dtype == torch.float32 else 4e-3
    rows_live = live.nonzero()[:, 0]
    assert bool(torch.all(d[rows_live].sum(1).abs() <= tol * d[rows_live].abs().sum(1)))
    assert bool(torch.all(d[~live] == 0))


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [1, 2, 7, 1003, 4099, 40001])
def test_odd_vocab_sizes(dtype, V):
    rows = 37
    w = workloads.collapse_stress(dtype=dtype, rows=rows, V=max(V, 4), seed=V)
    if V < 4:
        x = torch.randn((rows, V), generator=torch.Generator().manual_seed(V)).to(dtype)
        lab = torch.randint(0, V, (rows,), generator=torch.Generator().manual_seed(V + 1))
        lab[::5] = workloads.IGNORE_INDEX
        w.logits, w.labels = x, lab
        w.index = torch.where(lab < 0, 0, lab)[:, None]
        w.row_mask = (lab >= 0).to(torch.uint8)
    res, ref, sel = run_all(w, temperature=0.7)
    check_all(w, res, ref, sel, T=0.7)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_strided_misaligned_rows_and_unaligned_dlogits(dtype):
    g = torch.Generator().manual_seed(5)
    rows, V = 29, 5000
    big = torch.randn((rows, V + 13), generator=g).mul(3).to(dtype)
    x_cpu = big[:, 3:3 + V]            # row starts 6 or 12 bytes past 16-byte boundaries
    lab = torch.randint(0, V, (rows,), generator=g)
    lab[4] = workloads.IGNORE_INDEX
    x = big.to(DEV)[:, 3:3 + V]
    assert x.stride(0) == V + 13
    ref = oracle.cross_entropy(workloads.to_numpy_f64(x_cpu), lab.numpy(), temperature=0.9,
                               reduction="sum", grad_out=[0.5])
    # dlogits with a different 16-byte phase than the logits (scalar-store path)
    dbig = torch.empty((rows, V + 1), dtype=dtype, device=DEV)
    d = dbig[:, 1:]
    out = gbce.ce_fwd_bwd_fused(x, lab.to(DEV), torch.tensor([0.5]), temperature=0.9,
                                reduction="sum", dlogits=d)
    d2 = gbce.ce_bwd(x, lab.to(DEV), torch.tensor([0.5]), out.logp, out.n_items,
                     temperature=0.9, reduction="sum")
    torch.cuda.synchronize()
    assert_logp_close(to_f64(out.logp), ref["logp"], dtype)
    assert_grad_rows_close(to_f64(d), ref["dlogits"], dtype, "fused, unaligned dlogits")
    assert_grad_rows_close(to_f64(d2), ref["dlogits"], dtype, "ce_bwd")
    assert_loss_close(float(out.loss.item()), ref["loss"])


@pytest.mark.parametrize("rows", [1, 3, 64, 100, 200])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_few_rows_split_vocab(rows, dtype):
    """Few rows with a large vocabulary split it: each row's slices run as one
    cluster of CTAs that swap their partials through distributed shared memory
    (8 slices at 1 and 3 rows, 7 at 64, 4 at 100, 2 at 200 on 152 SMs)."""
    w = workloads.collapse_stress(dtype=dtype, rows=rows, V=152064, seed=rows)
    res, ref, sel = run_all(w, temperature=0.9)
    check_all(w, res, ref, sel, T=0.9)


def test_topk_duplicates_and_k16():
    g = torch.Generator().manual_seed(8)
    rows, V = 40, 9000
    x_cpu = torch.randn((rows, V), generator=g).mul(2).to(torch.bfloat16)
    idx = torch.randint(0, V, (rows, 16), generator=g)
    idx[:, 5] = idx[:, 2]                # duplicates
    idx[3, :] = 17                       # all the same column
    x_cpu[7, idx[7, 0]] = 60.0           # a confident gathered column
    mask = torch.ones(rows, dtype=torch.uint8)
    mask[11] = 0
    for K in (16, 4, 1):
        got = gbce.selective_logsoftmax(x_cpu.to(DEV), idx[:, :K].to(DEV), 0.9, mask.to(DEV))
        ref, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(x_cpu), idx[:, :K].numpy(),
                                             0.9, mask.numpy())
        g64 = to_f64(got)
        assert_logp_close(g64, ref, torch.bfloat16, f"K={K}")
        if K == 16:
            assert np.all(g64[:, 5] == g64[:, 2])
            assert np.all(g64[3] == g64[3, 0])


def test_all_ignored_and_mean_is_zero():
    x = torch.randn((9, 300), device=DEV)
    lab = torch.full((9,), -100, device=DEV)
    out = gbce.ce_fwd_bwd_fused(x, lab, torch.ones(1), reduction="mean")
    fwd = gbce.ce_fwd(x, lab, reduction="mean")
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and fwd.loss.item() == 0.0
    assert int(out.n_items.item()) == 0
    assert bool(torch.all(out.dlogits == 0))


def test_empty_batch():
    x = torch.empty((0, 128), device=DEV)
    lab = torch.empty((0,), dtype=torch.int64, device=DEV)
    out = gbce.ce_fwd_bwd_fused(x, lab, torch.ones(1), reduction="mean")
    lp = gbce.selective_logsoftmax(x, lab[:, None], 1.0)
    torch.cuda.synchronize()
    assert out.loss.item() == 0.0 and int(out.n_items.item()) == 0 and lp.numel() == 0


def test_bad_labels_and_indices_are_reported_not_trapped():
    x = torch.randn((6, 500), device=DEV)
    lab = torch.tensor([1, 500, -3, -100, 2, 499], device=DEV)
    status = new_status()
    out = gbce.ce_fwd_bwd_fused(x, lab, torch.ones(1), reduction="sum", dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gbce.DEV_BAD_LABEL
    lp = out.logp.cpu()
    assert torch.isnan(lp[1]) and torch.isnan(lp[2]) and lp[3] == 0
    assert torch.isfinite(lp[[0, 4, 5]]).all()
    assert torch.isnan(out.dlogits[1]).all() and (out.dlogits[3] == 0).all()
    status.zero_()
    idx = torch.tensor([[0, 3], [600, 1], [2, -1], [4, 4], [5, 6], [7, 8]], device=DEV)
    got = gbce.selective_logsoftmax(x, idx, 1.0, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gbce.DEV_BAD_INDEX
    g = got.cpu()
    assert torch.isnan(g[1, 0]) and torch.isnan(g[2, 1]) and torch.isfinite(g[1, 1])
    # the context is still usable
    assert float(torch.ones(1, device=DEV).sum().item()) == 1.0


def test_repeatable_bytes_and_inputs_untouched():
    w = workloads.collapse_stress(dtype=torch.bfloat16, rows=600, V=32000, seed=4)
    x = w.logits.to(DEV)
    lab = w.labels.to(DEV)
    h0 = hashlib.sha256(x.view(torch.int16).cpu().numpy().tobytes()).hexdigest()
    a = gbce.ce_fwd_bwd_fused(x, lab, torch.ones(1), temperature=0.9)
    b = gbce.ce_fwd_bwd_fused(x, lab, torch.ones(1), temperature=0.9)
    fwd = gbce.ce_fwd(x, lab, temperature=0.9)
    d1 = gbce.ce_bwd(x, lab, torch.ones(1), fwd.logp, fwd.n_items, temperature=0.9)
    d2 = gbce.ce_bwd(x, lab, torch.ones(1), fwd.logp, fwd.n_items, temperature=0.9)
    torch.cuda.synchronize()
    assert torch.equal(a.dlogits, b.dlogits) and torch.equal(a.loss, b.loss)
    assert torch.equal(d1, d2)
    # ce_fwd and the fused call run different kernels (each deterministic)
    assert_loss_close(float(fwd.loss.item()), float(a.loss.item()))
    h1 = hashlib.sha256(x.view(torch.int16).cpu().numpy().tobytes()).hexdigest()
    assert h0 == h1, "logits were modified"


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_back_to_back_calls_see_the_kernel_written_inputs(reduction):
    # Each call's logits and labels are written by a kernel just before it on
    # the same stream, and its outputs are read by kernels right after it,
    # alternating two input sets with different ignored rows and one shared
    # workspace.  The fused call's persistent kernel and loss reduction start
    # early, as programmatic dependents of the kernel before them: each must
    # still see the writes before it and finish before the reads after it.
    rows, V, T = 600, 24001, 0.9
    sets = []
    for seed in (11, 12):
        w = workloads.collapse_stress(dtype=torch.bfloat16, rows=rows, V=V, seed=seed)
        lab = w.labels.clone()
        lab[torch.arange(seed, rows, 7)] = -100
        g = torch.randn(rows) if reduction == "none" else torch.tensor([0.75])
        ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits), lab.numpy(), temperature=T,
                                   reduction=reduction, grad_out=g.double().numpy())
        sets.append((w.logits.to(DEV), lab.to(DEV), g.to(DEV), ref))
    x = torch.empty((rows, V), dtype=torch.bfloat16, device=DEV)
    lab_d = torch.empty(rows, dtype=torch.int64, device=DEV)
    ws = gbce.new_workspace(rows, V, 1, device=torch.device(DEV))
    got = []
    for i in range(6):
        src, lab_src, g, _ = sets[i % 2]
        torch.mul(src, 1.0, out=x)
        torch.add(lab_src, 0, out=lab_d)
        out = gbce.ce_fwd_bwd_fused(x, lab_d, g, temperature=T, reduction=reduction,
                                    workspace=ws)
        got.append((out.loss * 1.0, out.n_items * 1, out.dlogits * 1.0, out.logp * 1.0))
    torch.cuda.synchronize()
    for i, (loss, n, d, lp) in enumerate(got):
        ref = sets[i % 2][3]
        assert int(n.item()) == ref["n_items"], f"call {i}: n_items"
        if reduction == "none":
            assert_logp_close(-to_f64(loss), -ref["loss_rows"], torch.bfloat16, f"call {i} rows")
        else:
            assert_loss_close(float(loss.item()), ref["loss"], f"call {i} loss")
        assert_logp_close(to_f64(lp), ref["logp"], torch.bfloat16, f"call {i} log p")
        sel = np.arange(0, rows, 25)
        assert_grad_rows_close(to_f64(d[torch.as_tensor(sel, device=DEV)]), ref["dlogits"][sel],
                               torch.bfloat16, f"call {i} dlogits")


def test_three_d_logits_flatten():
    x = torch.randn((2, 5, 700), device=DEV, dtype=torch.bfloat16)
    idx = torch.randint(0, 700, (2, 5), device=DEV)
    got = gbce.selective_logsoftmax(x, idx, 1.0)
    assert got.shape == (2, 5)
    ref, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(x.reshape(10, 700)),
                                         idx.reshape(10, 1).cpu().numpy(), 1.0)
    assert_logp_close(to_f64(got).reshape(10, 1), ref, torch.bfloat16)


def test_stream_argument_is_honoured():
    s = torch.cuda.Stream()
    w = workloads.ce_small_fp32(device=DEV)
    with torch.cuda.stream(s):
        out = gbce.ce_fwd_bwd_fused(w.logits, w.labels, torch.ones(1, device=DEV))
    s.synchronize()
    ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits), w.labels.cpu().numpy(),
                               reduction="mean")
    assert_loss_close(float(out.loss.item()), ref["loss"])


# ------------------------------------------- persistent fused kernel shapes

@pytest.mark.parametrize("dtype,V", [
    (torch.bfloat16, 40001),     # row 80 KB
    (torch.float32, 100003),     # 400 KB, misaligned rows
    (torch.bfloat16, 262144),    # 512 KB
    (torch.float32, 500000),     # 2 MB: the rows in flight no longer all fit L2
])
def test_fused_persistent_row_sizes(dtype, V):
    w = workloads.collapse_stress(dtype=dtype, rows=520, V=V, seed=V % 97)
    sel = sample_rows(w, n_plain=16, seed=2)
    res, ref, sel = run_all(w, temperature=0.7, rows_sel=sel)
    check_all(w, res, ref, sel, T=0.7)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fused_persistent_strided_rows_and_unaligned_dlogits(dtype):
    g = torch.Generator().manual_seed(17)
    rows, V = 520, 70001
    big = torch.randn((rows, V + 9), generator=g).mul(2).to(dtype)
    x_cpu = big[:, 3:3 + V]
    lab = torch.randint(0, V, (rows,), generator=g)
    lab[::7] = workloads.IGNORE_INDEX
    x_cpu[5, lab[5]] = 80.0
    x = big.to(DEV)[:, 3:3 + V]
    dbig = torch.empty((rows, V + 1), dtype=dtype, device=DEV)
    d = dbig[:, 1:]
    out = gbce.ce_fwd_bwd_fused(x, lab.to(DEV), torch.tensor([0.25]), temperature=0.9,
                                reduction="sum", dlogits=d)
    torch.cuda.synchronize()
    sel = np.array([0, 1, 5, 7, 100, 257, 300, 519])
    ref = oracle.cross_entropy(workloads.to_numpy_f64(x_cpu[sel]), lab.numpy()[sel],
                               temperature=0.9, reduction="none", grad_out=np.full(8, 0.25))
    assert_logp_close(to_f64(out.logp)[sel], ref["logp"], dtype)
    assert_grad_rows_close(to_f64(d[torch.as_tensor(sel, device=DEV)]), ref["dlogits"], dtype)
    total = -np.sum(to_f64(out.logp))
    assert_loss_close(float(out.loss.item()), total)


def test_persistent_stats_many_rows_k16_and_masks():
    g = torch.Generator().manual_seed(23)
    rows, V = 700, 50001
    x_cpu = torch.randn((rows, V), generator=g).mul(3).to(torch.bfloat16)
    idx = torch.randint(0, V, (rows, 16), generator=g)
    idx[:, 9] = idx[:, 1]
    mask = (torch.rand(rows, generator=g) > 0.2).to(torch.uint8)
    got = gbce.selective_logsoftmax(x_cpu.to(DEV), idx.to(DEV), 0.8, mask.to(DEV))
    sel = np.arange(0, rows, 23)
    ref, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(x_cpu[sel]), idx.numpy()[sel],
                                         0.8, mask.numpy()[sel])
    assert_logp_close(to_f64(got)[sel], ref, torch.bfloat16)
    assert np.all(to_f64(got)[mask.numpy() == 0] == 0.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,K,pad", [(4099, 1, 0), (32768, 4, 0), (1000, 16, 13), (32000, 4, 5)])
def test_many_short_rows_every_row(dtype, V, K, pad):
    # several waves of short rows, every row against the oracle: row strides
    # that leave rows off 16-byte boundaries (scalar head and tail), ragged
    # vocabularies, duplicated indices, masked rows, and a few out-of-range
    # indices (NaN for just those, reported).
    rows, T = 1300, 0.7
    g = torch.Generator().manual_seed(V + K)
    big = (torch.randn((rows, V + pad), generator=g) * 3.0).to(dtype)
    x_cpu = big[:, :V]
    idx = torch.randint(0, V, (rows, K), generator=g)
    if K > 1:
        idx[:, K - 1] = idx[:, 0]
    idx[5, 0] = V
    idx[rows - 2, K - 1] = -3
    mask = (torch.rand(rows, generator=g) >= 0.2).to(torch.uint8)
    mask[5] = 1
    mask[rows - 2] = 1
    status = new_status()
    got = gbce.selective_logsoftmax(big.to(DEV)[:, :V], idx.to(DEV), T, mask.to(DEV),
                                    dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gbce.DEV_BAD_INDEX
    ref, n_bad = oracle.selective_logsoftmax(workloads.to_numpy_f64(x_cpu), idx.numpy(), T,
                                             mask.numpy())
    assert n_bad == 2
    assert_logp_close(to_f64(got), ref, dtype)
    assert np.all(to_f64(got)[mask.numpy() == 0] == 0.0)


# ---------------------------------------------------------- size extremes

def test_huge_vocab_few_rows_split_path():
    # 2 rows of 2^25 + 3 columns: the split path at 64 slices of ~524K
    # columns, an odd tail, one confident row
    V = (1 << 25) + 3
    w = workloads.collapse_stress(dtype=torch.bfloat16, rows=2, V=V, seed=101)
    w.labels[:] = torch.tensor([7, V - 1])
    workloads.set_target_margin(w.logits, torch.tensor([1]), torch.tensor([V - 1]),
                                torch.tensor([30.0]))
    w.index = w.labels[:, None].clone()
    w.row_mask = None
    res, ref, sel = run_all(w, temperature=0.9, reduction="sum", grad_out=torch.ones(1))
    check_all(w, res, ref, sel, reduction="sum", T=0.9)


def test_million_column_rows_persistent_path():
    # 520 rows of 1,000,003 fp32 columns (4 MB a row): the persistent fused
    # kernel's rows no longer all fit L2 at once; K = 16 gathered indices
    V, rows = 1_000_003, 520
    g = torch.Generator().manual_seed(5)
    w = workloads.collapse_stress(dtype=torch.float32, rows=rows, V=V, seed=55)
    idx = torch.randint(0, V, (rows, 16), generator=g)
    idx[:, 0] = torch.where(w.labels >= 0, w.labels, idx[:, 0])
    w.index = idx
    sel = np.concatenate([np.arange(0, rows, 53), w.peaked_rows.numpy()[:6]])
    res, ref, sel = run_all(w, temperature=1.0, reduction="mean", grad_out=torch.ones(1),
                            rows_sel=np.sort(sel))
    check_all(w, res, ref, sel, reduction="mean", check_scalar_vs_oracle=False, T=1.0)


def test_binding_refuses_bad_output_buffers_before_any_launch():
    x = torch.randn((6, 300), device=DEV)
    lab = torch.zeros(6, dtype=torch.int64, device=DEV)
    idx = torch.zeros((6, 2), dtype=torch.int64, device=DEV)
    before = gbce.kernel_launches()
    bad_calls = [
        lambda: gbce.selective_logsoftmax(x, idx, out=torch.empty((5, 2), device=DEV)),
        lambda: gbce.selective_logsoftmax(x, idx, out=torch.empty((6, 2), dtype=torch.float64,
                                                                  device=DEV)),
        lambda: gbce.selective_logsoftmax(x, idx, entropy_out=torch.empty(5, device=DEV)),
        lambda: gbce.ce_fwd_bwd_fused(x, lab, dlogits=torch.empty((5, 300), device=DEV)),
        lambda: gbce.ce_fwd_bwd_fused(x, lab, dlogits=torch.empty((6, 300), dtype=torch.bfloat16,
                                                                  device=DEV)),
        lambda: gbce.ce_bwd(x, lab, torch.ones(1), torch.zeros(6), torch.tensor(6),
                            dlogits=torch.empty((6, 299), device=DEV)),
        lambda: gbce.selective_logsoftmax_bwd(x, idx, torch.ones((6, 2)), torch.zeros((6, 2)),
                                              dlogits=torch.empty((6, 300), device=DEV)[:, :299]),
        lambda: gbce.ce_fwd(x, lab, dev_status=torch.zeros(1, dtype=torch.int64, device=DEV)),
        lambda: gbce.ce_fwd(x, lab, workspace=torch.empty(1 << 16, dtype=torch.uint8)),
    ]
    for call in bad_calls:
        with pytest.raises(ValueError):
            call()
    torch.cuda.synchronize()
    assert gbce.kernel_launches() == before
