"""GPU parity of the vocabulary-slice path (vocab_slice_stats, _combine,
_grad) against the fp64 oracle, through the C ABI.  Every slice lives on one
GPU here; across devices only the gather of the partials changes (covered on
CPU with gloo ranks in test_multirank_cpu.py)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (assert_grad_block_close, assert_grad_rows_close, assert_logp_close,
                     assert_zero_sum_block, to_f64)

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


def run_slices(x, idx, cuts, T, mask=None, g=None, ignore_index=-100):
    """Stats per slice, combine, gradient per slice (concatenated)."""
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    V = x.shape[1]
    parts = [gbce.vocab_slice_stats(x[:, a:b], idx, a, V, T, mask, ignore_index=ignore_index,
                                    dev_status=status)
             for a, b in zip(cuts[:-1], cuts[1:])]
    logp, xt0, state = gbce.vocab_slice_combine(torch.stack(parts), cuts, idx, T, mask,
                                                ignore_index=ignore_index, dev_status=status)
    d = None
    if g is not None:
        d = torch.cat([gbce.vocab_slice_grad(x[:, a:b], idx, a, V, g, logp, xt0, T, mask,
                                             row_state=state, ignore_index=ignore_index,
                                             dev_status=status)
                       for a, b in zip(cuts[:-1], cuts[1:])], dim=1)
    torch.cuda.synchronize()
    return logp, xt0, d, int(status.item())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [1, 4])
def test_slices_match_the_oracle(dtype, K):
    # ragged, misaligned slice boundaries; confident rows at margins 17..50;
    # duplicate indices; masked rows
    rows, V, T = 600, 24001, 0.9
    w = workloads.collapse_stress(dtype=dtype, rows=rows, V=V, seed=60 + K)
    gen = torch.Generator().manual_seed(K)
    idx = torch.randint(0, V, (rows, K), generator=gen)
    idx[:, 0] = torch.where(w.labels >= 0, w.labels, idx[:, 0])
    if K > 1:
        idx[::5, 2] = idx[::5, 0]
    mask = (torch.rand(rows, generator=gen) > 0.1).to(torch.uint8)
    g = torch.randn((rows, K), generator=gen)
    cuts = [0, 7001, 7003, 15000, V]
    x = w.logits.to(DEV)
    logp, xt0, d, status = run_slices(x, idx.to(DEV), cuts, T, mask.to(DEV), g.to(DEV))
    assert status == 0
    ref, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(w.logits), idx.numpy(), T,
                                         mask.numpy())
    assert_logp_close(to_f64(logp), ref, dtype, "sliced log p")
    live = mask.numpy() == 1
    np.testing.assert_array_equal(to_f64(xt0)[live],
                                  workloads.to_numpy_f64(w.logits)[np.arange(rows), idx[:, 0]][live])
    # the same log-probs as the single-device call, within the same bound
    whole = gbce.selective_logsoftmax(x, idx.to(DEV), T, mask.to(DEV))
    assert_logp_close(to_f64(logp), to_f64(whole).astype(np.float64), dtype, "vs whole row")
    ref_d, _ = oracle.selective_logsoftmax_backward(workloads.to_numpy_f64(w.logits),
                                                    idx.numpy(), g.double().numpy(), T,
                                                    mask.numpy())
    got = to_f64(d)
    assert_grad_block_close(got, ref_d, dtype, "sliced gradient")
    assert_zero_sum_block(got, dtype)
    assert np.all(got[~live] == 0.0)


def test_token_ce_over_slices_few_rows_and_ignored_labels():
    # the CE case: k = 1, index = labels, ignore_index -100; loss = -log p and
    # the gradient with grad_logp = -upstream; 3 rows of 152064 columns, so
    # each slice's statistics split again over a cluster of CTAs
    rows, V, T = 3, 152064, 1.0
    w = workloads.collapse_stress(dtype=torch.bfloat16, rows=rows, V=V, seed=5)
    lab = torch.tensor([17, -100, V - 1])
    workloads.set_target_margin(w.logits, torch.tensor([2]), torch.tensor([V - 1]),
                                torch.tensor([30.0]))
    x = w.logits.to(DEV)
    up = torch.tensor([0.5, 1.0, -2.0])
    cuts = [0, 76032, V]
    logp, _, d, status = run_slices(x, lab.to(DEV), cuts, T, g=(-up).to(DEV))
    assert status == 0
    ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits), lab.numpy(), temperature=T,
                               reduction="none", grad_out=up.double().numpy())
    assert_logp_close(to_f64(logp)[:, 0], ref["logp"], torch.bfloat16, "sliced CE log p")
    assert to_f64(logp)[1, 0] == 0.0 and np.all(to_f64(d)[1] == 0.0)
    assert_grad_block_close(to_f64(d), ref["dlogits"], torch.bfloat16, "sliced CE gradient")


def test_bad_index_is_reported_by_the_combine():
    x = torch.randn((4, 300), device=DEV)
    idx = torch.tensor([[1], [300], [5], [-7]], device=DEV)
    logp, _, d, status = run_slices(x, idx, [0, 150, 300], 1.0,
                                    g=torch.ones((4, 1), device=DEV))
    assert status & gbce.DEV_BAD_INDEX
    lp = logp.cpu()
    assert torch.isnan(lp[1, 0]) and torch.isnan(lp[3, 0]) and torch.isfinite(lp[[0, 2], 0]).all()
    assert torch.isnan(d[1]).all() and torch.isfinite(d[[0, 2]]).all()


def test_slice_arguments_are_checked_on_the_host():
    x = torch.randn((2, 10), device=DEV)
    idx = torch.zeros((2, 1), dtype=torch.int64, device=DEV)
    with pytest.raises(gbce.GbceError):
        gbce.vocab_slice_stats(x, idx, 95, 100)          # slice past the vocabulary
    parts = torch.zeros((2, 2, 3), device=DEV)
    with pytest.raises(gbce.GbceError):
        gbce.vocab_slice_combine(parts, [0, 10, 10], idx)  # offsets not increasing
    with pytest.raises(gbce.GbceError):
        gbce.vocab_slice_combine(parts, [5, 10, 20], idx)  # not starting at 0


def test_slices_of_rows_dominated_far_above_their_first_index():
    # a column outside the gathered set leads each row by 60..400 units at
    # T = 0.5 (hundreds of nats): the combine's row state keeps the slice
    # gradient within the fp32 bound
    rows, V, T = 300, 9001, 0.5
    gen = torch.Generator().manual_seed(77)
    x_cpu = torch.randn((rows, V), generator=gen) * 2.0
    dom = torch.randint(0, V, (rows,), generator=gen)
    idx = ((dom + torch.randint(1, V, (rows,), generator=gen)) % V)[:, None]
    x_cpu[torch.arange(rows), dom] += 60.0 + 340.0 * torch.rand(rows, generator=gen)
    g = torch.randn((rows, 1), generator=gen)
    cuts = [0, 3000, 6001, V]
    logp, _, d, status = run_slices(x_cpu.to(DEV), idx.to(DEV), cuts, T, g=g.to(DEV))
    assert status == 0
    x64 = x_cpu.double().numpy()
    ref, _ = oracle.selective_logsoftmax(x64, idx.numpy(), T)
    assert np.all(ref < -100.0)
    assert_logp_close(to_f64(logp), ref, torch.float32, "sliced log p")
    ref_d, _ = oracle.selective_logsoftmax_backward(x64, idx.numpy(), g.double().numpy(), T)
    assert_grad_block_close(to_f64(d), ref_d, torch.float32, "sliced gradient")


def slice_config(seed):
    """A seeded vocabulary-slice case: rows, vocabulary, K, dtype,
    temperature, logit scale and 1..5 slices with random boundaries."""
    rng = np.random.default_rng(seed)
    rows = int(rng.choice([1, 3, 64, 300, 700]))
    V = int(rng.choice([2, 9, 1000, 4099, 24001, 50001]))
    K = int(rng.choice([1, 2, 4, 16]))
    dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    T = float(rng.choice([0.1, 0.25, 0.5, 1.0, 4.0]))
    scale = float(rng.choice([1.0, 20.0, 50.0]))
    nsl = int(rng.integers(1, min(V, 5) + 1))
    cuts = sorted(set([0, V] + [int(c) for c in rng.integers(1, V, size=nsl - 1)]))
    return rows, V, K, dtype, T, scale, cuts


@pytest.mark.parametrize("seed", range(48))
def test_seeded_slicings_match_the_oracle(seed):
    # random slicings of random rows (extreme temperatures and scales): the
    # combined log p and the per-slice gradients against the oracle.  The
    # gradient takes the combine's fp32 log p, so a row may also move by
    # 2^-147 sum|g| / T (the log p floor) and, where a gathered column's two
    # terms cancel, by a few fp32 ulps of them, 2^-22 sum|g| / T.
    rows, V, K, dtype, T, scale, cuts = slice_config(seed)
    gen = torch.Generator().manual_seed(seed)
    x_cpu = (torch.randn((rows, V), generator=gen) * scale).to(dtype)
    idx = torch.randint(0, V, (rows, K), generator=gen)
    mask = (torch.rand(rows, generator=gen) > 0.15).to(torch.uint8)
    g = torch.randn((rows, K), generator=gen)
    logp, xt0, d, status = run_slices(x_cpu.to(DEV), idx.to(DEV), cuts, T, mask.to(DEV),
                                      g.to(DEV))
    assert status == 0
    x64 = workloads.to_numpy_f64(x_cpu)
    ref, _ = oracle.selective_logsoftmax(x64, idx.numpy(), T, mask.numpy())
    assert_logp_close(to_f64(logp), ref, dtype, "sliced log p")
    ref_d, _ = oracle.selective_logsoftmax_backward(x64, idx.numpy(), g.double().numpy(), T,
                                                    mask.numpy())
    ga = np.abs(g.double().numpy()).sum(axis=1) / T
    assert_grad_rows_close(to_f64(d), ref_d, dtype, "sliced dlogits",
                           extra_floor=ga * (2.0 ** -147 + 2.0 ** -22))
