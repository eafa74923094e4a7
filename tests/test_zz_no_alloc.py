"""ce_fwd_bwd_fused_noalloc: the fused cross-entropy call for callers that
cannot give the library a workspace (a C program or plugin with no device
allocator of its own, which must not call cudaMalloc on its hot path).

Its scratch is a fixed array inside the library, shared by every call.  These
tests call it through the C ABI several times in a row, with different
problems so that each call runs over what the previous one left in the array,
and compare each result with the workspace-taking ce_fwd_bwd_fused on the
same inputs and with the fp64 oracle.  The file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_grad_rows_close, assert_logp_close, assert_loss_close, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SCRATCH_BYTES = 1 << 20


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()
    import cross_entropy_gb300 as gbce

    return gbce.load_library()


def _noalloc(lib, x, lab, grad, T, red):
    """One call of the new entry point through ctypes; returns its outputs."""
    rows, V = x.shape
    loss = torch.full((rows,) if red == 0 else (1,), float("nan"), device=DEV)
    logp = torch.full((rows,), float("nan"), device=DEV)
    lse = torch.full((rows,), float("nan"), device=DEV)
    n = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    d = torch.full_like(x, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    dtype = 1 if x.dtype == torch.bfloat16 else 0
    st = lib.ce_fwd_bwd_fused_noalloc(
        x.data_ptr(), dtype, rows, V, x.stride(0), lab.data_ptr(), -100, ctypes.c_float(T), red,
        grad.data_ptr(), loss.data_ptr(), logp.data_ptr(), lse.data_ptr(), n.data_ptr(),
        d.data_ptr(), d.stride(0), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.gbce_status_string(st)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return loss, logp, lse, n, d


def _reference(x, lab, grad, T, red):
    import cross_entropy_gb300 as gbce

    names = {0: "none", 1: "sum", 2: "mean"}
    return gbce.ce_fwd_bwd_fused(x, lab, grad, temperature=T, reduction=names[red],
                                 want_lse=True)


def _compare(got, ref, dtype):
    loss, logp, lse, n, d = got
    assert int(n.item()) == int(ref.n_items.item())
    assert_logp_close(to_f64(logp), to_f64(ref.logp), dtype, "noalloc logp")
    np.testing.assert_allclose(to_f64(lse), to_f64(ref.lse), rtol=2e-6, atol=2e-6)
    if loss.numel() == 1:
        assert_loss_close(float(loss.item()), float(ref.loss.item()), "noalloc loss")
    else:
        assert_logp_close(-to_f64(loss), -to_f64(ref.loss), dtype, "noalloc loss rows")
    assert_grad_rows_close(to_f64(d), to_f64(ref.dlogits), dtype, "noalloc dlogits")


def _against_oracle(got, w, grad, T, red, dtype):
    """The no-allocation call's outputs against the fp64 oracle."""
    loss, logp, _, n, d = got
    names = {0: "none", 1: "sum", 2: "mean"}
    ref = oracle.cross_entropy(workloads.to_numpy_f64(w.logits), w.labels.numpy(), temperature=T,
                               reduction=names[red], grad_out=grad.double().cpu().numpy())
    assert int(n.item()) == ref["n_items"]
    assert_logp_close(to_f64(logp), ref["logp"], dtype, "noalloc logp vs oracle")
    if red == 0:
        assert_logp_close(-to_f64(loss), -ref["loss_rows"], dtype, "noalloc rows vs oracle")
    else:
        assert_loss_close(float(loss.item()), ref["loss"], "noalloc loss vs oracle")
    assert_grad_rows_close(to_f64(d), ref["dlogits"], dtype, "noalloc dlogits vs oracle")


def test_calls_in_a_row_match_the_workspace_entry_point_and_the_oracle(lib):
    # call 1: many rows, mean, bf16 -> the persistent kernel's row ticket, the
    # per-row losses and the item count in scratch
    w1 = workloads.collapse_stress(dtype=torch.bfloat16, rows=700, V=32000, seed=11)
    x1, l1 = w1.logits.to(DEV), w1.labels.to(DEV)
    g1 = torch.ones(1, device=DEV)
    got1 = _noalloc(lib, x1, l1, g1, 0.9, 2)
    _compare(got1, _reference(x1, l1, g1, 0.9, 2), torch.bfloat16)
    _against_oracle(got1, w1, g1, 0.9, 2, torch.bfloat16)
    # call 2: few rows, large vocabulary, fp32, sum -> a vocabulary split,
    # over what the first call left in the scratch
    w2 = workloads.collapse_stress(dtype=torch.float32, rows=3, V=152064, seed=12)
    x2, l2 = w2.logits.to(DEV), w2.labels.to(DEV)
    g2 = torch.tensor([0.5], device=DEV)
    got2 = _noalloc(lib, x2, l2, g2, 1.0, 1)
    _compare(got2, _reference(x2, l2, g2, 1.0, 1), torch.float32)
    _against_oracle(got2, w2, g2, 1.0, 1, torch.float32)
    # call 3: reduction none with a per-row upstream gradient
    w3 = workloads.collapse_stress(dtype=torch.bfloat16, rows=300, V=4099, seed=13)
    x3, l3 = w3.logits.to(DEV), w3.labels.to(DEV)
    g3 = torch.randn(300, generator=torch.Generator().manual_seed(3)).to(DEV)
    got3 = _noalloc(lib, x3, l3, g3, 0.7, 0)
    _compare(got3, _reference(x3, l3, g3, 0.7, 0), torch.bfloat16)
    _against_oracle(got3, w3, g3, 0.7, 0, torch.bfloat16)
    # and the first problem again, now over the other calls' leftovers
    again = _noalloc(lib, x1, l1, g1, 0.9, 2)
    _compare(again, _reference(x1, l1, g1, 0.9, 2), torch.bfloat16)


def test_oversized_problem_is_refused_before_any_gpu_work(lib):
    rows, V = 200_000, 8
    assert lib.gbce_workspace_size(rows, V, 1) > SCRATCH_BYTES
    fake = 0x10000
    st = lib.ce_fwd_bwd_fused_noalloc(fake, 0, rows, V, V, fake, -100, ctypes.c_float(1.0), 2,
                                      fake, fake, None, None, None, fake * 4096, V, None, None)
    assert st == 4  # GBCE_EWORKSPACE
