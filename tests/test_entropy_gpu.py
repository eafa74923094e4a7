"""GPU parity of the row entropy that selective_logsoftmax computes in the
same sweep as the log-probs, against the fp64 oracle, through the C ABI."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_entropy_close, assert_logp_close

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


def gpu_logp_entropy(x, idx, T, mask=None):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp, h = gbce.selective_logsoftmax(x, idx, T, mask, with_entropy=True, dev_status=status)
    torch.cuda.synchronize()
    return lp, h, int(status.item())


def oracle_entropy(x_cpu, idx_cpu, T, mask=None, rows_sel=None):
    sel = np.arange(x_cpu.shape[0]) if rows_sel is None else np.asarray(rows_sel)
    st = torch.as_tensor(sel)
    h, bad = oracle.entropy(workloads.to_numpy_f64(x_cpu[st]), idx_cpu.numpy()[sel, 0], T,
                            None if mask is None else mask.numpy()[sel])
    return h, bad


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,T", [(1, 1.0), (4, 0.9)])
def test_matches_oracle_on_confident_rows(dtype, K, T):
    rows, V = 700, 32003
    w = workloads.collapse_stress(dtype=dtype, rows=rows, V=V, seed=20 + K)
    gen = torch.Generator().manual_seed(K)
    idx = torch.randint(0, V, (rows, K), generator=gen)
    idx[:, 0] = torch.where(w.labels >= 0, w.labels, idx[:, 0])   # the confident column first
    if K > 1:
        idx[::5, 3] = idx[::5, 0]                                  # duplicates
    lp, h, status = gpu_logp_entropy(w.logits.to(DEV), idx.to(DEV), T, w.row_mask.to(DEV))
    assert status == 0
    ref, bad = oracle_entropy(w.logits, idx, T, w.row_mask)
    assert bad == 0
    assert_entropy_close(h.cpu().numpy(), ref)
    assert np.all(h.cpu().numpy() <= math.log(V) * (1 + 1e-6))
    # the confident rows keep their tiny positive entropy
    pk = w.peaked_rows.numpy()
    live = pk[w.row_mask.numpy()[pk] != 0]
    assert np.all(h.cpu().numpy()[live] > 0.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,T", [(1, 1.0), (1, 0.7), (4, 0.9)])
def test_rows_confident_in_another_column(dtype, K, T):
    # the dominant column (margins 17/20/30/50) is never the first index:
    # outside the gathered set, or (K = 4, every other row) at index 1..3
    w = workloads.dominated_elsewhere(dtype, rows=600, V=32003, K=K, seed=80 + K)
    lp, h, status = gpu_logp_entropy(w.logits.to(DEV), w.index.to(DEV), T)
    assert status == 0
    ref, bad = oracle_entropy(w.logits, w.index, T)
    assert bad == 0
    assert_entropy_close(h.cpu().numpy(), ref)
    assert np.all(h.cpu().numpy() > 0.0)
    ref_lp, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(w.logits), w.index.numpy(), T)
    assert_logp_close(lp.cpu().numpy(), ref_lp, dtype)


@pytest.mark.parametrize("rows", [3, 100])
def test_rows_confident_in_another_column_split_path(rows):
    # few rows: the slices of a row form a cluster, and its first CTA redoes
    # the entropy around the dominant column over the whole row
    w = workloads.dominated_elsewhere(torch.bfloat16, rows=rows, V=152064, K=2, seed=rows)
    lp, h, status = gpu_logp_entropy(w.logits.to(DEV), w.index.to(DEV), 0.9)
    assert status == 0
    ref, _ = oracle_entropy(w.logits, w.index, 0.9)
    assert_entropy_close(h.cpu().numpy(), ref)
    ref_lp, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(w.logits), w.index.numpy(),
                                            0.9)
    assert_logp_close(lp.cpu().numpy(), ref_lp, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_log_probs_are_unchanged_by_the_entropy(dtype):
    w = workloads.collapse_stress(dtype=dtype, rows=600, V=40001, seed=5)
    x = w.logits.to(DEV)
    idx = torch.randint(0, 40001, (600, 4), generator=torch.Generator().manual_seed(6)).to(DEV)
    plain = gbce.selective_logsoftmax(x, idx, 0.9, w.row_mask.to(DEV))
    lp, _, status = gpu_logp_entropy(x, idx, 0.9, w.row_mask.to(DEV))
    assert status == 0
    assert torch.equal(plain, lp)


@pytest.mark.parametrize("rows", [1, 3, 200])
def test_few_rows_split_path(rows):
    V = 152064
    w = workloads.collapse_stress(dtype=torch.bfloat16, rows=rows, V=V, seed=rows)
    idx = torch.where(w.labels >= 0, w.labels, 0)[:, None].repeat(1, 2)
    idx[:, 1] = torch.randint(0, V, (rows,), generator=torch.Generator().manual_seed(2))
    lp, h, status = gpu_logp_entropy(w.logits.to(DEV), idx.to(DEV), 0.7)
    assert status == 0
    sel = np.arange(0, rows, max(1, rows // 25))
    ref, _ = oracle_entropy(w.logits, idx, 0.7, rows_sel=sel)
    assert_entropy_close(h.cpu().numpy()[sel], ref)
    ref_lp, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(w.logits[torch.as_tensor(sel)]),
                                            idx.numpy()[sel], 0.7)
    assert_logp_close(lp.cpu().numpy()[sel], ref_lp, torch.bfloat16)


def test_zero_probability_columns_and_ragged_rows():
    # -inf logits (p = 0, 0 log 0 = 0), also at the reference column; a row
    # stride that leaves a scalar head and tail; V = 1 and V = 2 rows
    gen = torch.Generator().manual_seed(31)
    rows, V = 520, 5003
    big = torch.randn((rows, V + 3), generator=gen).mul(2.5)
    x_cpu = big[:, 1:1 + V].clone()
    cols = torch.randint(0, V, (rows, 40), generator=gen)
    x_cpu.scatter_(1, cols, float("-inf"))
    big[:, 1:1 + V] = x_cpu
    idx = torch.randint(0, V, (rows, 1), generator=gen)
    idx[::4, 0] = cols[::4, 0]                    # reference column at -inf
    _, h, status = gpu_logp_entropy(big.to(DEV)[:, 1:1 + V], idx.to(DEV), 0.9)
    assert status == 0
    ref, _ = oracle_entropy(x_cpu, idx, 0.9)
    assert_entropy_close(h.cpu().numpy(), ref)
    for v in (1, 2):
        x = torch.randn((3, v), generator=gen)
        i = torch.zeros((3, 1), dtype=torch.int64)
        _, h, status = gpu_logp_entropy(x.to(DEV), i.to(DEV), 1.0)
        ref, _ = oracle_entropy(x, i, 1.0)
        assert status == 0
        assert_entropy_close(h.cpu().numpy(), ref)


def test_bad_reference_index_gives_nan():
    x = torch.randn((4, 300), device=DEV)
    idx = torch.tensor([[1, 2], [300, 3], [4, -1], [5, 5]], device=DEV)
    lp, h, status = gpu_logp_entropy(x, idx, 1.0)
    assert status == gbce.DEV_BAD_INDEX
    assert torch.isnan(h[1]) and torch.isfinite(h[[0, 2, 3]]).all()
    ref, _ = oracle.entropy(x.double().cpu().numpy(), [1, 4, 4, 5], 1.0)
    assert_entropy_close(h[[0, 2, 3]].cpu().numpy(), ref[[0, 2, 3]])


def test_full_size_grpo_k4():
    # every row against the oracle, in row blocks
    w = workloads.grpo_bf16(device=DEV)
    lp, h, status = gpu_logp_entropy(w.logits, w.index, 0.9)
    assert status == 0
    for r0 in range(0, w.rows, 1024):
        r1 = min(w.rows, r0 + 1024)
        ref, _ = oracle.entropy(workloads.to_numpy_f64(w.logits[r0:r1]),
                                w.index[r0:r1, 0].cpu().numpy(), 0.9)
        assert_entropy_close(h[r0:r1].cpu().numpy(), ref)
    hv = h.cpu().numpy()
    assert np.all(hv > 0.0) and np.all(hv <= math.log(w.vocab) * (1 + 1e-6))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_padded_vocabulary_at_minus_infinity(dtype):
    # a vocabulary padded to a multiple of 128 with -inf logits, as some
    # models' heads are: the padding must add exactly nothing
    rows, V, real = 600, 32128, 32003
    gen = torch.Generator().manual_seed(77)
    x = torch.randn((rows, V), generator=gen).mul(2.0)
    x[:, real:] = float("-inf")
    x = x.to(dtype)
    idx = torch.randint(0, real, (rows, 4), generator=gen)
    lp, h, status = gpu_logp_entropy(x.to(DEV), idx.to(DEV), 0.9)
    assert status == 0
    ref, _ = oracle_entropy(x, idx, 0.9)
    assert_entropy_close(h.cpu().numpy(), ref)
    ref_cut, _ = oracle_entropy(x[:, :real].contiguous(), idx, 0.9)
    np.testing.assert_allclose(ref, ref_cut, rtol=1e-13)
    ref_lp, _ = oracle.selective_logsoftmax(workloads.to_numpy_f64(x), idx.numpy(), 0.9)
    assert_logp_close(lp.cpu().numpy(), ref_lp, dtype)
