"""GPU parity of selective_logsoftmax_bwd (the GRPO-style gradient through the
gathered log-probs) against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (assert_grad_block_close, assert_grad_rows_close, assert_zero_sum_block,
                     assert_zero_sum_rows, to_f64)

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


def run_case(x_cpu, idx, g, T, mask=None, rows_sel=None, dlogits=None, x_dev=None):
    """GPU forward + backward on x; oracle backward on rows_sel."""
    x = x_cpu.to(DEV) if x_dev is None else x_dev
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    m_dev = None if mask is None else mask.to(DEV)
    lp = gbce.selective_logsoftmax(x, idx.to(DEV), T, m_dev, dev_status=status)
    d = gbce.selective_logsoftmax_bwd(x, idx.to(DEV), g.to(DEV), lp, T, m_dev,
                                      dlogits=dlogits, dev_status=status)
    torch.cuda.synchronize()
    sel = np.arange(x_cpu.shape[0]) if rows_sel is None else np.asarray(rows_sel)
    st = torch.as_tensor(sel)
    ref, bad = oracle.selective_logsoftmax_backward(
        workloads.to_numpy_f64(x_cpu[st]), idx.numpy()[sel], g.double().numpy()[sel], T,
        None if mask is None else mask.numpy()[sel])
    got = to_f64(d[st.to(DEV)])
    return got, ref, int(status.item()), bad


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [1, 4])
def test_matches_oracle_with_masks_and_duplicates(dtype, K):
    gen = torch.Generator().manual_seed(40 + K)
    rows, V = 600, 32003
    w = workloads.collapse_stress(dtype=dtype, rows=rows, V=V, seed=K)
    idx = torch.randint(0, V, (rows, K), generator=gen)
    idx[:, 0] = torch.where(w.labels >= 0, w.labels, idx[:, 0])   # confident rows' label first
    if K > 1:
        idx[::3, 2] = idx[::3, 0]                                  # duplicates
    mask = (torch.rand(rows, generator=gen) > 0.1).to(torch.uint8)
    g = torch.randn((rows, K), generator=gen)
    sel = np.arange(0, rows, 7)
    got, ref, status, bad = run_case(w.logits, idx, g, 0.9, mask, rows_sel=sel)
    assert status == 0 and bad == 0
    assert_grad_rows_close(got, ref, dtype, "selective_logsoftmax_bwd")
    assert_zero_sum_rows(got, dtype)
    assert np.all(got[mask.numpy()[sel] == 0] == 0.0)


def test_confident_rows_keep_their_target_gradient():
    w = workloads.collapse_stress(dtype=torch.float32, rows=520, V=151936, seed=9)
    idx = torch.where(w.labels >= 0, w.labels, 0)[:, None]
    g = torch.full((520, 1), -1.0)              # e.g. a positive advantage
    pk = w.peaked_rows.numpy()
    sel = pk[w.labels.numpy()[pk] >= 0][:40]
    got, ref, status, _ = run_case(w.logits, idx, g, 1.0, rows_sel=sel)
    assert status == 0
    assert_grad_rows_close(got, ref, torch.float32)
    cols = idx.numpy()[sel, 0]
    # d(-log p_t)/dx_t = -(1 - p_t) / T: tiny but never rounded to zero
    assert np.all(got[np.arange(len(sel)), cols] < 0.0)
    assert_zero_sum_rows(got, torch.float32)


def test_upstream_sums_that_cancel():
    # K = 16 on three columns: indices 8..15 repeat 0..7 with each upstream
    # negated to within 1e-4, so every column's summed upstream (and every
    # gradient element) is a sum of O(1) terms that cancels to ~1e-4.  In
    # fp32 such a sum keeps only the terms' rounding (~1e-7, about 1e-3 of
    # these rows); the kernel's sums of at most K upstream values are exact
    # enough to meet the row bound.
    rows, V, K, T = 256, 3, 16, 0.8
    gen = torch.Generator().manual_seed(92)
    x_cpu = torch.randn((rows, V), generator=gen) * 2.0
    idx = torch.randint(0, V, (rows, K), generator=gen)
    idx[:, 8:] = idx[:, :8]
    g = torch.randn((rows, K), generator=gen)
    g[:, 8:] = -g[:, :8] + 1e-4 * torch.randn((rows, 8), generator=gen)
    x = x_cpu.to(DEV)
    lp = gbce.selective_logsoftmax(x, idx.to(DEV), T)
    d = gbce.selective_logsoftmax_bwd(x, idx.to(DEV), g.to(DEV), lp, T)
    torch.cuda.synchronize()
    ref, _ = oracle.selective_logsoftmax_backward(workloads.to_numpy_f64(x_cpu), idx.numpy(),
                                                  g.double().numpy(), T)
    assert_grad_rows_close(to_f64(d), ref, torch.float32, "cancelling upstream")


def test_small_upstream_beside_a_large_one():
    # K = 2 with upstream gradients a thousand times apart, on rows confident
    # in their first index: each gathered column's gradient holds the other
    # index's small upstream (times its p), which a difference G - g_t of the
    # fp32 sums would carry only to the large upstream's rounding.  Every
    # gathered element against the oracle, element by element.
    rows, V, T = 512, 4099, 1.0
    gen = torch.Generator().manual_seed(91)
    x_cpu = torch.randn((rows, V), generator=gen) * 2.0
    idx = torch.randint(0, V, (rows, 2), generator=gen)
    x_cpu[torch.arange(rows), idx[:, 0]] += 30.0  # confident in index 0
    g = torch.stack([torch.full((rows,), -1.5), 1e-3 + torch.rand(rows, generator=gen) * 2e-3], dim=1)
    x = x_cpu.to(DEV)
    lp = gbce.selective_logsoftmax(x, idx.to(DEV), T)
    d = gbce.selective_logsoftmax_bwd(x, idx.to(DEV), g.to(DEV), lp, T)
    torch.cuda.synchronize()
    ref, _ = oracle.selective_logsoftmax_backward(workloads.to_numpy_f64(x_cpu), idx.numpy(),
                                                  g.double().numpy(), T)
    got = to_f64(d)
    r = np.arange(rows)
    for k in range(2):
        want = ref[r, idx[:, k].numpy()]
        have = got[r, idx[:, k].numpy()]
        rel = np.abs(have - want) / np.abs(want)
        assert rel.max() <= 2e-5, f"index {k}: worst relative error {rel.max():.3e}"
    assert_grad_rows_close(got, ref, torch.float32, "small upstream")


@pytest.mark.parametrize("rows", [1, 3])
def test_few_rows_split_path(rows):
    w = workloads.collapse_stress(dtype=torch.bfloat16, rows=rows, V=152064, seed=rows)
    idx = torch.randint(0, 152064, (rows, 4), generator=torch.Generator().manual_seed(3))
    g = torch.randn((rows, 4), generator=torch.Generator().manual_seed(4))
    got, ref, status, _ = run_case(w.logits, idx, g, 0.9)
    assert status == 0
    assert_grad_rows_close(got, ref, torch.bfloat16)


def test_strided_rows_unaligned_dlogits():
    gen = torch.Generator().manual_seed(12)
    rows, V = 530, 9001
    big = torch.randn((rows, V + 5), generator=gen).mul(3)
    x_cpu = big[:, 2:2 + V]
    idx = torch.randint(0, V, (rows, 4), generator=gen)
    g = torch.randn((rows, 4), generator=gen)
    dbig = torch.empty((rows, V + 3), device=DEV)
    d = dbig[:, 3:]
    got, ref, status, _ = run_case(x_cpu, idx, g, 0.7, rows_sel=np.arange(0, rows, 11),
                                   dlogits=d, x_dev=big.to(DEV)[:, 2:2 + V])
    assert status == 0
    assert_grad_rows_close(got, ref, torch.float32)


def test_full_size_grpo_k4():
    w = workloads.grpo_bf16(device=DEV)
    g = torch.randn((w.rows, 4), device=DEV, generator=torch.Generator(device=DEV).manual_seed(1))
    lp = gbce.selective_logsoftmax(w.logits, w.index, 0.9)
    d = gbce.selective_logsoftmax_bwd(w.logits, w.index, g, lp, 0.9)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    sel = np.sort(np.concatenate([rng.choice(w.rows, 20, replace=False),
                                  w.peaked_rows.cpu().numpy()[:12]]))
    st = torch.as_tensor(sel, device=DEV)
    ref, _ = oracle.selective_logsoftmax_backward(workloads.to_numpy_f64(w.logits[st]),
                                                  w.index[st].cpu().numpy(),
                                                  g[st].double().cpu().numpy(), 0.9)
    assert_grad_rows_close(to_f64(d[st]), ref, torch.bfloat16)
    rs = d.double().sum(1).abs()
    ra = d.double().abs().sum(1)
    assert bool(torch.all(rs <= 4e-3 * ra))


def test_bad_index_gives_nan_row_and_status():
    x = torch.randn((4, 300), device=DEV)
    idx = torch.tensor([[1, 2], [300, 3], [4, -1], [5, 5]], device=DEV)
    g = torch.ones((4, 2), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp = gbce.selective_logsoftmax(x, idx.clamp(0, 299), 1.0)
    d = gbce.selective_logsoftmax_bwd(x, idx, g, lp, 1.0, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gbce.DEV_BAD_INDEX
    assert torch.isnan(d[1]).all() and torch.isnan(d[2]).all()
    assert torch.isfinite(d[0]).all() and torch.isfinite(d[3]).all()


# ------------------------------------------------ with the row entropy's term

def run_ent_case(x_cpu, idx, g, gh, T, mask=None, rows_sel=None):
    """GPU forward (log p + entropy) and backward with dL/dH; oracle backward."""
    x = x_cpu.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    m_dev = None if mask is None else mask.to(DEV)
    lp, h = gbce.selective_logsoftmax(x, idx.to(DEV), T, m_dev, with_entropy=True,
                                      dev_status=status)
    d = gbce.selective_logsoftmax_bwd(x, idx.to(DEV), g.to(DEV), lp, T, m_dev,
                                      grad_entropy=gh.to(DEV), saved_entropy=h,
                                      dev_status=status)
    torch.cuda.synchronize()
    sel = np.arange(x_cpu.shape[0]) if rows_sel is None else np.asarray(rows_sel)
    st = torch.as_tensor(sel)
    ref, bad = oracle.selective_logsoftmax_backward(
        workloads.to_numpy_f64(x_cpu[st]), idx.numpy()[sel], g.double().numpy()[sel], T,
        None if mask is None else mask.numpy()[sel], grad_entropy=gh.double().numpy()[sel])
    return to_f64(d[st.to(DEV)]), ref, int(status.item()), bad


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [1, 4])
def test_entropy_term_matches_oracle(dtype, K):
    gen = torch.Generator().manual_seed(60 + K)
    rows, V = 560, 24001
    w = workloads.collapse_stress(dtype=dtype, rows=rows, V=V, seed=30 + K)
    idx = torch.randint(0, V, (rows, K), generator=gen)
    idx[:, 0] = torch.where(w.labels >= 0, w.labels, idx[:, 0])
    if K > 1:
        idx[::4, 1] = idx[::4, 0]
    mask = (torch.rand(rows, generator=gen) > 0.1).to(torch.uint8)
    g = torch.randn((rows, K), generator=gen)
    gh = torch.randn(rows, generator=gen)
    sel = np.arange(0, rows, 5)
    got, ref, status, bad = run_ent_case(w.logits, idx, g, gh, 0.9, mask, rows_sel=sel)
    assert status == 0 and bad == 0
    assert_grad_rows_close(got, ref, dtype, "selective_logsoftmax_bwd + entropy")
    assert_zero_sum_rows(got, dtype)
    assert np.all(got[mask.numpy()[sel] == 0] == 0.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [1, 4])
def test_entropy_term_rows_confident_in_another_column(dtype, K):
    # the dominant column (margins 17..50) outside the gathered set, or (K = 4,
    # even rows) gathered at index 1..3; rows 1 and 2 mod 4 have only the
    # entropy's upstream, where that column's entry is most of the gradient
    rows, V = 560, 24001
    w = workloads.dominated_elsewhere(dtype, rows=rows, V=V, K=K, seed=90 + K)
    gen = torch.Generator().manual_seed(91 + K)
    g = torch.randn((rows, K), generator=gen)
    g[(torch.arange(rows) % 4 == 1) | (torch.arange(rows) % 4 == 2)] = 0.0
    gh = torch.randn(rows, generator=gen)
    got, ref, status, bad = run_ent_case(w.logits, w.index, g, gh, 0.9)
    assert status == 0 and bad == 0
    assert_grad_rows_close(got, ref, dtype, "selective_logsoftmax_bwd + entropy")
    assert_zero_sum_rows(got, dtype)
    d = w.labels.numpy()
    at_d = got[np.arange(rows), d]
    want = ref[np.arange(rows), d]
    assert np.all(np.sign(at_d) == np.sign(want)) and np.all(at_d != 0.0)


def test_entropy_only_gradient_of_confident_rows():
    # g = 0: the gradient of the entropy alone; a confident row's dominant
    # column has d H / d x_t = -(p_t / T)(log p_t + H) < 0, tiny but not 0
    rows, V = 520, 151936
    w = workloads.collapse_stress(dtype=torch.float32, rows=rows, V=V, seed=13)
    idx = torch.where(w.labels >= 0, w.labels, 0)[:, None]
    g = torch.zeros((rows, 1))
    gh = torch.ones(rows)
    pk = w.peaked_rows.numpy()
    sel = pk[w.labels.numpy()[pk] >= 0][:32]
    got, ref, status, _ = run_ent_case(w.logits, idx, g, gh, 1.0, rows_sel=sel)
    assert status == 0
    assert_grad_rows_close(got, ref, torch.float32)
    cols = idx.numpy()[sel, 0]
    assert np.all(got[np.arange(len(sel)), cols] < 0.0)
    assert_zero_sum_rows(got, torch.float32)


def test_entropy_term_with_minus_infinity_and_split_path():
    gen = torch.Generator().manual_seed(70)
    for rows, V in ((3, 152064), (530, 7003)):
        x = torch.randn((rows, V), generator=gen).mul(2.0)
        x[:, ::97] = float("-inf")
        idx = torch.randint(0, V, (rows, 2), generator=gen)
        idx[:, 0] = (idx[:, 0] // 97) * 97 + 1           # a finite reference column
        g = torch.randn((rows, 2), generator=gen)
        gh = torch.randn(rows, generator=gen)
        sel = np.arange(0, rows, max(1, rows // 40))
        got, ref, status, _ = run_ent_case(x, idx, g, gh, 0.8, rows_sel=sel)
        assert status == 0
        assert_grad_rows_close(got, ref, torch.float32)
        assert np.all(got[:, ::97] == 0.0)


def test_full_size_grpo_k4_with_entropy():
    w = workloads.grpo_bf16(device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(2)
    g = torch.randn((w.rows, 4), device=DEV, generator=gen)
    gh = torch.randn(w.rows, device=DEV, generator=gen)
    lp, h = gbce.selective_logsoftmax(w.logits, w.index, 0.9, with_entropy=True)
    d = gbce.selective_logsoftmax_bwd(w.logits, w.index, g, lp, 0.9, grad_entropy=gh,
                                      saved_entropy=h)
    torch.cuda.synchronize()
    # every row against the oracle, in row blocks
    for r0 in range(0, w.rows, 512):
        r1 = min(w.rows, r0 + 512)
        ref, _ = oracle.selective_logsoftmax_backward(
            workloads.to_numpy_f64(w.logits[r0:r1]), w.index[r0:r1].cpu().numpy(),
            g[r0:r1].double().cpu().numpy(), 0.9,
            grad_entropy=gh[r0:r1].double().cpu().numpy())
        got = to_f64(d[r0:r1])
        assert_grad_block_close(got, ref, torch.bfloat16)
        assert_zero_sum_block(got, torch.bfloat16)
        del got, ref
