"""Row-wise log-softmax and token cross-entropy on one GB300 (sm_103a).

Thin Python binding of ``libgbce.so`` (see ``include/gbce.h``).  The functions
here only check and marshal arguments -- data pointers, strides, the current
CUDA stream -- and allocate outputs with PyTorch; every step of the
computation runs in the library's CUDA kernels.  There is no CPU or PyTorch
fallback: if the library is missing or a tensor is not on a CUDA device,
the call raises.

Functions (same names as the C ABI):

* :func:`selective_logsoftmax` -- log p at K gathered indices per row, with
  temperature and row mask ("perf(rlhf): chunk selective_log_softmax instead
  of looping per token", "PR information"), and optionally each row's softmax
  entropy from the same sweep; :func:`selective_logsoftmax_bwd` its gradient
  (the one a GRPO-style loss sends back), optionally with the entropy's.
* :func:`ce_fwd`, :func:`ce_bwd`, :func:`ce_fwd_bwd_fused` -- token
  cross-entropy in the collapse-safe form of "Fix softmax collapse in CE,
  GRPO, KL/JSD and softmax" ("Summary"), with the analytic backward
  g*softmax - g*onehot of ms-swift PR #10353 ("PR information"), optional
  label smoothing, DFT row weights and logit soft-capping.
* :func:`ce_fwd_bwd_fused_noalloc` -- the fused call without a workspace.
* :func:`vocab_slice_stats`, :func:`vocab_slice_combine`,
  :func:`vocab_slice_grad` -- the selective log-softmax (and token CE) over
  a vocabulary split into slices, e.g. one per device of a vocab-parallel
  head ("Fix softmax collapse ...", "Summary", first bullet), with
  :func:`gather_slice_partials` moving the per-slice statistics between
  ranks through torch.distributed.

Caller-supplied output, scratch and status tensors are checked for device,
dtype and size before any GPU work: the kernels write through their data
pointers.
"""

from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# GBCE_LIBRARY may name another build of the same library (e.g. one built
# with a different kernel option) to load instead of the in-tree one.
LIB_PATH = os.environ.get("GBCE_LIBRARY") or os.path.join(_HERE, "_build", "libgbce.so")

GBCE_F32, GBCE_BF16 = 0, 1
REDUCTIONS = {"none": 0, "sum": 1, "mean": 2}
MAX_K = 16
DEV_BAD_LABEL, DEV_BAD_INDEX, DEV_TIMEOUT = 1, 2, 4

# The C entry points and their argument types, in header order.
_vp, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_i32 = ctypes.c_int
_SIGNATURES = {
    "gbce_workspace_size": (_sz, [_i64, _i64, _i64]),
    "gbce_status_string": (ctypes.c_char_p, [_i32]),
    "gbce_kernel_launches": (ctypes.c_uint64, []),
    "selective_logsoftmax": (_i32, [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _f32, _vp, _vp,
                                    _vp, _vp, _sz, _vp, _vp]),
    "selective_logsoftmax_bwd": (_i32, [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _f32, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _i64, _vp, _vp]),
    "ce_fwd": (_i32, [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _f32, _i32, _vp, _vp, _vp, _vp,
                      _vp, _vp, _sz, _vp, _vp]),
    "ce_bwd": (_i32, [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _f32, _i32, _vp, _vp, _vp, _vp,
                      _vp, _i64, _vp, _vp]),
    "ce_fwd_bwd_fused": (_i32, [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _f32, _i32, _vp, _vp,
                                _vp, _vp, _vp, _vp, _vp, _i64, _vp, _sz, _vp, _vp]),
    "ce_fwd_bwd_fused_noalloc": (_i32, [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _f32, _i32,
                                        _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp]),
    "vocab_slice_stats": (_i32, [_vp, _i32, _i64, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _vp,
                                 _f32, _vp, _vp, _vp]),
    "vocab_slice_combine": (_i32, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _vp, _f32, _vp, _vp,
                                   _vp, _vp, _vp]),
    "vocab_slice_grad": (_i32, [_vp, _i32, _i64, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _vp,
                                _f32, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp]),
}
MAX_SLICES = 64

_lib = None


class GbceError(RuntimeError):
    """A libgbce call returned a non-OK status."""


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libgbce.so (built by ``cross_entropy_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libgbce.so not found at {path}: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        msg = load_library().gbce_status_string(status).decode()
        raise GbceError(f"{what}: {msg}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GBCE_F32
    if t.dtype == torch.bfloat16:
        return GBCE_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _rows_view(logits: torch.Tensor) -> torch.Tensor:
    """[..., V] with unit column stride -> 2-D [rows, V] view (no copy)."""
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor (no CPU path exists)")
    if logits.dim() < 2:
        raise ValueError("logits must have shape [rows, vocab] or [..., vocab]")
    if logits.stride(-1) != 1:
        raise ValueError("logits must have unit stride along the vocabulary")
    if logits.dim() > 2:
        try:
            logits = logits.view(-1, logits.shape[-1])
        except RuntimeError as exc:
            raise ValueError("leading dimensions of logits must flatten without a copy") from exc
    return logits


def _stream_ptr(stream, device=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _check_buffer(t: Optional[torch.Tensor], name: str, dtype, numel: int, device) -> None:
    """A caller-supplied output or scratch tensor: the kernels write exactly
    `numel` elements of `dtype` through its data pointer, so anything else is
    refused here, before any GPU work."""
    if t is None:
        return
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous() or t.numel() != numel:
        raise ValueError(f"{name} must be a contiguous tensor of {numel} elements, "
                         f"got shape {tuple(t.shape)}")


def _check_dlogits(d: torch.Tensor, x: torch.Tensor) -> None:
    if d.device != x.device or d.dtype != x.dtype or tuple(d.shape) != tuple(x.shape):
        raise ValueError(f"dlogits must be a {x.dtype} tensor of shape {tuple(x.shape)} on "
                         f"{x.device} (rows x vocab, unit vocab stride)")


def _check_status(st: Optional[torch.Tensor], device) -> None:
    if st is not None and (st.device != device or st.dtype != torch.int32 or st.numel() < 1):
        raise ValueError("dev_status must be an int32 tensor of at least 1 element on "
                         "the logits' device")


def _dev_int64(x, device) -> torch.Tensor:
    t = torch.as_tensor(x, dtype=torch.int64, device=device)
    return t.contiguous()


def kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(load_library().gbce_kernel_launches())


def workspace_size(rows: int, vocab: int, k: int = 1) -> int:
    return int(load_library().gbce_workspace_size(int(rows), int(vocab), int(k)))


def new_workspace(rows: int, vocab: int, k: int = 1, device=None) -> torch.Tensor:
    """A byte tensor large enough for any call on a [rows, vocab] problem."""
    n = max(workspace_size(rows, vocab, k), 16)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _workspace(ws, rows, vocab, k, device):
    if ws is None:
        ws = new_workspace(rows, vocab, k, device)
    elif ws.device != device or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    return ws, int(ws.data_ptr()), int(ws.numel() * ws.element_size())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def selective_logsoftmax(logits: torch.Tensor, index, temperature: float = 1.0,
                         row_mask: Optional[torch.Tensor] = None, *,
                         out: Optional[torch.Tensor] = None,
                         with_entropy: bool = False,
                         entropy_out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         dev_status: Optional[torch.Tensor] = None, stream=None):
    """log p_{index[r, k]} of each row at temperature T, fp32, shape index.shape.

    ``index`` is [..., K] (or [...] for K = 1) int64; masked-out rows
    (``row_mask == 0``) are not read and give 0.  With ``with_entropy`` (or an
    ``entropy_out`` [...] fp32 buffer) the same sweep also gives each row's
    softmax entropy, and the call returns ``(logp, entropy)``.
    """
    lib = load_library()
    lead_shape = logits.shape[:-1]
    x = _rows_view(logits)
    rows, V = x.shape
    idx = _dev_int64(index, x.device)
    squeeze = idx.dim() == len(lead_shape)
    K = 1 if squeeze else idx.shape[-1]
    idx = idx.reshape(rows, K)
    mask = None
    if row_mask is not None:
        mask = row_mask.to(device=x.device, dtype=torch.uint8).reshape(rows).contiguous()
    if out is None:
        out = torch.empty((rows, K), dtype=torch.float32, device=x.device)
    _check_buffer(out, "out", torch.float32, rows * K, x.device)
    _check_status(dev_status, x.device)
    ent = entropy_out
    if ent is None and with_entropy:
        ent = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check_buffer(ent, "entropy_out", torch.float32, rows, x.device)
    ws, ws_ptr, ws_bytes = _workspace(workspace, rows, V, K, x.device)
    with torch.cuda.device(x.device):  # the library launches on the current device
        st = lib.selective_logsoftmax(x.data_ptr(), _dtype_code(x), rows, V, x.stride(0),
                                      idx.data_ptr(), K, float(temperature), _ptr(mask),
                                      out.data_ptr(), _ptr(ent), ws_ptr, ws_bytes, _ptr(dev_status),
                                      _stream_ptr(stream, x.device))
    _check(st, "selective_logsoftmax")
    res = out.view(*lead_shape, K)
    res = res.squeeze(-1) if squeeze else res
    if ent is None:
        return res
    return res, ent.view(lead_shape)


def selective_logsoftmax_bwd(logits: torch.Tensor, index, grad_logp, saved_logp,
                             temperature: float = 1.0, row_mask: Optional[torch.Tensor] = None,
                             *, grad_entropy=None, saved_entropy: Optional[torch.Tensor] = None,
                             dlogits: Optional[torch.Tensor] = None,
                             dev_status: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """dL/dlogits for upstream grad_logp = dL/d selective_logsoftmax(...).

    ``index``, ``grad_logp`` and ``saved_logp`` have the forward's output
    shape ([..., K], or [...] for K = 1); masked-out rows get zero.  With
    ``grad_entropy`` = dL/d entropy ([...], one per row) the gradient of the
    forward's entropy output is added; ``saved_entropy`` is that output.
    """
    lib = load_library()
    lead_shape = logits.shape[:-1]
    x = _rows_view(logits)
    rows, V = x.shape
    idx = _dev_int64(index, x.device)
    K = 1 if idx.dim() == len(lead_shape) else idx.shape[-1]
    idx = idx.reshape(rows, K)
    g = torch.as_tensor(grad_logp, dtype=torch.float32, device=x.device).reshape(rows, K)
    g = g.contiguous()
    lp = saved_logp.to(device=x.device, dtype=torch.float32).reshape(rows, K).contiguous()
    mask = None
    if row_mask is not None:
        mask = row_mask.to(device=x.device, dtype=torch.uint8).reshape(rows).contiguous()
    gh = hs = None
    if (grad_entropy is None) != (saved_entropy is None):
        raise ValueError("grad_entropy and saved_entropy go together")
    if grad_entropy is not None:
        gh = torch.as_tensor(grad_entropy, dtype=torch.float32,
                             device=x.device).reshape(rows).contiguous()
        hs = saved_entropy.to(device=x.device, dtype=torch.float32).reshape(rows).contiguous()
    if dlogits is None:
        dlogits = torch.empty_like(logits)
    d = _rows_view(dlogits)
    _check_dlogits(d, x)
    _check_status(dev_status, x.device)
    with torch.cuda.device(x.device):  # the library launches on the current device
        st = lib.selective_logsoftmax_bwd(x.data_ptr(), _dtype_code(x), rows, V, x.stride(0),
                                          idx.data_ptr(), K, float(temperature), _ptr(mask),
                                          g.data_ptr(), lp.data_ptr(), _ptr(gh), _ptr(hs),
                                          d.data_ptr(), d.stride(0), _ptr(dev_status),
                                          _stream_ptr(stream, x.device))
    _check(st, "selective_logsoftmax_bwd")
    return dlogits


class CeOptions(ctypes.Structure):
    """gbce_ce_options: label smoothing eps and the DFT row weight."""

    _fields_ = [("label_smoothing", ctypes.c_float), ("dft", ctypes.c_int32),
                ("softcap", ctypes.c_float)]


def _ce_options(label_smoothing: float, dft: bool, softcap: float = 0.0):
    """A CeOptions to pass by reference, or None for plain CE."""
    if label_smoothing == 0.0 and not dft and softcap == 0.0:
        return None
    return ctypes.byref(CeOptions(float(label_smoothing), 1 if dft else 0, float(softcap)))


class CeForward(NamedTuple):
    loss: torch.Tensor              # [rows] for 'none', [] otherwise
    logp: Optional[torch.Tensor]    # [rows] log p of the label (0 for ignored rows)
    lse: Optional[torch.Tensor]     # [rows] logsumexp of logits / T
    n_items: torch.Tensor           # [] int64


class CeFused(NamedTuple):
    loss: torch.Tensor
    dlogits: torch.Tensor
    logp: Optional[torch.Tensor]
    lse: Optional[torch.Tensor]
    n_items: torch.Tensor


def ce_fwd(logits: torch.Tensor, labels, ignore_index: int = -100, temperature: float = 1.0,
           reduction: str = "mean", *, label_smoothing: float = 0.0, dft: bool = False,
           softcap: float = 0.0,
           want_lse: bool = False, workspace: Optional[torch.Tensor] = None,
           dev_status: Optional[torch.Tensor] = None, stream=None) -> CeForward:
    """Cross-entropy forward; returns loss, saved log p (for ce_bwd), lse, n_items.

    ``label_smoothing`` eps, ``dft`` (rows weighted by their detached p_y) and
    ``softcap`` (logits capped as softcap * tanh(x / softcap)) change the loss;
    ce_bwd must be given the same three.
    """
    lib = load_library()
    x = _rows_view(logits)
    rows, V = x.shape
    lab = _dev_int64(labels, x.device).reshape(rows)
    red = REDUCTIONS[reduction]
    loss = torch.empty((rows,) if red == 0 else (1,), dtype=torch.float32, device=x.device)
    logp = torch.empty(rows, dtype=torch.float32, device=x.device)
    lse = torch.empty(rows, dtype=torch.float32, device=x.device) if want_lse else None
    n_items = torch.empty(1, dtype=torch.int64, device=x.device)
    ws, ws_ptr, ws_bytes = _workspace(workspace, rows, V, 1, x.device)
    _check_status(dev_status, x.device)
    with torch.cuda.device(x.device):  # the library launches on the current device
        st = lib.ce_fwd(x.data_ptr(), _dtype_code(x), rows, V, x.stride(0), lab.data_ptr(),
                        int(ignore_index), float(temperature), red,
                        _ce_options(label_smoothing, dft, softcap), loss.data_ptr(),
                        logp.data_ptr(),
                        _ptr(lse), n_items.data_ptr(), ws_ptr, ws_bytes, _ptr(dev_status),
                        _stream_ptr(stream, x.device))
    _check(st, "ce_fwd")
    return CeForward(loss if red == 0 else loss[0], logp, lse, n_items[0])


def ce_bwd(logits: torch.Tensor, labels, grad_out, saved_logp: torch.Tensor, n_items=None,
           ignore_index: int = -100, temperature: float = 1.0, reduction: str = "mean", *,
           label_smoothing: float = 0.0, dft: bool = False, softcap: float = 0.0,
           dlogits: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
           stream=None) -> torch.Tensor:
    """dlogits = g * (softmax - onehot) / T from ce_fwd's saved log p (smoothed /
    DFT-weighted with the same options as the forward)."""
    lib = load_library()
    x = _rows_view(logits)
    rows, V = x.shape
    lab = _dev_int64(labels, x.device).reshape(rows)
    red = REDUCTIONS[reduction]
    g = torch.as_tensor(grad_out, dtype=torch.float32, device=x.device).reshape(-1).contiguous()
    if g.numel() != (rows if red == 0 else 1):
        raise ValueError("grad_out must have one entry per row for 'none', one otherwise")
    n = None if n_items is None else _dev_int64(n_items, x.device).reshape(1)
    if dlogits is None:
        dlogits = torch.empty((rows, V), dtype=x.dtype, device=x.device)
    d = _rows_view(dlogits)
    _check_dlogits(d, x)
    _check_status(dev_status, x.device)
    lp = saved_logp.to(device=x.device, dtype=torch.float32).reshape(rows).contiguous()
    with torch.cuda.device(x.device):  # the library launches on the current device
        st = lib.ce_bwd(x.data_ptr(), _dtype_code(x), rows, V, x.stride(0), lab.data_ptr(),
                        int(ignore_index), float(temperature), red,
                        _ce_options(label_smoothing, dft, softcap), g.data_ptr(), lp.data_ptr(),
                        _ptr(n), d.data_ptr(), d.stride(0), _ptr(dev_status),
                        _stream_ptr(stream, x.device))
    _check(st, "ce_bwd")
    return dlogits


def ce_fwd_bwd_fused(logits: torch.Tensor, labels, grad_out=None, ignore_index: int = -100,
                     temperature: float = 1.0, reduction: str = "mean", *,
                     label_smoothing: float = 0.0, dft: bool = False, softcap: float = 0.0,
                     dlogits: Optional[torch.Tensor] = None, want_logp: bool = True,
                     want_lse: bool = False, workspace: Optional[torch.Tensor] = None,
                     dev_status: Optional[torch.Tensor] = None, stream=None) -> CeFused:
    """Cross-entropy loss and dlogits in one call (upstream gradient known up front)."""
    lib = load_library()
    x = _rows_view(logits)
    rows, V = x.shape
    lab = _dev_int64(labels, x.device).reshape(rows)
    red = REDUCTIONS[reduction]
    if grad_out is None:
        grad_out = torch.ones(rows if red == 0 else 1)
    g = torch.as_tensor(grad_out, dtype=torch.float32, device=x.device).reshape(-1).contiguous()
    if g.numel() != (rows if red == 0 else 1):
        raise ValueError("grad_out must have one entry per row for 'none', one otherwise")
    loss = torch.empty((rows,) if red == 0 else (1,), dtype=torch.float32, device=x.device)
    logp = torch.empty(rows, dtype=torch.float32, device=x.device) if want_logp else None
    lse = torch.empty(rows, dtype=torch.float32, device=x.device) if want_lse else None
    n_items = torch.empty(1, dtype=torch.int64, device=x.device)
    if dlogits is None:
        dlogits = torch.empty((rows, V), dtype=x.dtype, device=x.device)
    d = _rows_view(dlogits)
    _check_dlogits(d, x)
    _check_status(dev_status, x.device)
    ws, ws_ptr, ws_bytes = _workspace(workspace, rows, V, 1, x.device)
    with torch.cuda.device(x.device):  # the library launches on the current device
        st = lib.ce_fwd_bwd_fused(x.data_ptr(), _dtype_code(x), rows, V, x.stride(0),
                                  lab.data_ptr(),
                                  int(ignore_index), float(temperature), red,
                                  _ce_options(label_smoothing, dft, softcap), g.data_ptr(),
                                  loss.data_ptr(), _ptr(logp), _ptr(lse), n_items.data_ptr(),
                                  d.data_ptr(), d.stride(0), ws_ptr, ws_bytes, _ptr(dev_status),
                                  _stream_ptr(stream, x.device))
    _check(st, "ce_fwd_bwd_fused")
    return CeFused(loss if red == 0 else loss[0], dlogits, logp, lse, n_items[0])


def ce_fwd_bwd_fused_noalloc(logits: torch.Tensor, labels, grad_out=None,
                             ignore_index: int = -100, temperature: float = 1.0,
                             reduction: str = "mean", *, dlogits: Optional[torch.Tensor] = None,
                             dev_status: Optional[torch.Tensor] = None, stream=None) -> CeFused:
    """ce_fwd_bwd_fused with the library's built-in scratch instead of a workspace.

    For callers that cannot supply scratch memory (see include/gbce.h).  The
    outputs allocated here are the caller's, as with every other call; the
    library itself allocates nothing.  Calls whose GPU work overlaps share the
    built-in scratch and race.
    """
    lib = load_library()
    x = _rows_view(logits)
    rows, V = x.shape
    lab = _dev_int64(labels, x.device).reshape(rows)
    red = REDUCTIONS[reduction]
    if grad_out is None:
        grad_out = torch.ones(rows if red == 0 else 1)
    g = torch.as_tensor(grad_out, dtype=torch.float32, device=x.device).reshape(-1).contiguous()
    if g.numel() != (rows if red == 0 else 1):
        raise ValueError("grad_out must have one entry per row for 'none', one otherwise")
    loss = torch.empty((rows,) if red == 0 else (1,), dtype=torch.float32, device=x.device)
    logp = torch.empty(rows, dtype=torch.float32, device=x.device)
    n_items = torch.empty(1, dtype=torch.int64, device=x.device)
    if dlogits is None:
        dlogits = torch.empty((rows, V), dtype=x.dtype, device=x.device)
    d = _rows_view(dlogits)
    _check_dlogits(d, x)
    _check_status(dev_status, x.device)
    with torch.cuda.device(x.device):  # the library launches on the current device
        st = lib.ce_fwd_bwd_fused_noalloc(x.data_ptr(), _dtype_code(x), rows, V, x.stride(0),
                                          lab.data_ptr(), int(ignore_index), float(temperature),
                                          red,
                                          g.data_ptr(), loss.data_ptr(), logp.data_ptr(), None,
                                          n_items.data_ptr(), d.data_ptr(), d.stride(0),
                                          _ptr(dev_status), _stream_ptr(stream, x.device))
    _check(st, "ce_fwd_bwd_fused_noalloc")
    return CeFused(loss if red == 0 else loss[0], dlogits, logp, None, n_items[0])


# ------------------------------------------------ vocabulary-parallel path

def _slice_index(index, lead_shape, rows, device):
    idx = _dev_int64(index, device)
    K = 1 if idx.dim() == len(lead_shape) else idx.shape[-1]
    return idx.reshape(rows, K).contiguous(), K


def vocab_slice_stats(logits_slice: torch.Tensor, index, vocab_offset: int, vocab: int,
                      temperature: float = 1.0, row_mask: Optional[torch.Tensor] = None, *,
                      ignore_index: int = -100, out: Optional[torch.Tensor] = None,
                      dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Partials [rows, 2 + K] fp32 of one vocabulary slice: the max and the
    sum over its non-target columns and the logits of the targets it holds.

    ``logits_slice`` [..., n] holds global columns [vocab_offset, vocab_offset
    + n) of a ``vocab``-column vocabulary; ``index`` [..., K] (or [...]) holds
    global columns.  Rows with ``row_mask == 0`` or whose first index equals
    ``ignore_index`` are skipped.
    """
    lib = load_library()
    lead_shape = logits_slice.shape[:-1]
    x = _rows_view(logits_slice)
    rows, n = x.shape
    idx, K = _slice_index(index, lead_shape, rows, x.device)
    mask = None
    if row_mask is not None:
        mask = row_mask.to(device=x.device, dtype=torch.uint8).reshape(rows).contiguous()
    if out is None:
        out = torch.empty((rows, 2 + K), dtype=torch.float32, device=x.device)
    _check_buffer(out, "out", torch.float32, rows * (2 + K), x.device)
    _check_status(dev_status, x.device)
    with torch.cuda.device(x.device):
        st = lib.vocab_slice_stats(x.data_ptr(), _dtype_code(x), rows, n, x.stride(0),
                                   int(vocab_offset), int(vocab), idx.data_ptr(), K,
                                   int(ignore_index), _ptr(mask), float(temperature),
                                   out.data_ptr(), _ptr(dev_status),
                                   _stream_ptr(stream, x.device))
    _check(st, "vocab_slice_stats")
    return out


def gather_slice_partials(partials: torch.Tensor, group=None) -> torch.Tensor:
    """All ranks' partials stacked in rank order, [world, rows, 2 + K]: the one
    exchange of the vocab-parallel path (rank i holds slice i).  With no
    initialised process group, the local partials as a single slice."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return partials.unsqueeze(0)
    world = dist.get_world_size(group)
    parts = [torch.empty_like(partials) for _ in range(world)]
    dist.all_gather(parts, partials.contiguous(), group=group)
    return torch.stack(parts)


def vocab_slice_combine(partials: torch.Tensor, slice_offsets, index, temperature: float = 1.0,
                        row_mask: Optional[torch.Tensor] = None, *, ignore_index: int = -100,
                        dev_status: Optional[torch.Tensor] = None, stream=None):
    """From all slices' partials stacked in slice order, [slices, rows, 2 + K]:
    ``(logp [rows, K], target_logit [rows], row_state [rows, 2])`` -- the
    log-probs, the logit of index[:, 0] and each row's whole (max, sum),
    the last two for :func:`vocab_slice_grad`.  ``slice_offsets`` are the
    slices' first global columns followed by the vocabulary size."""
    lib = load_library()
    if not partials.is_cuda or partials.dtype != torch.float32 or partials.dim() != 3:
        raise ValueError("partials must be a float32 CUDA tensor [slices, rows, 2 + K]")
    slices, rows, width = partials.shape
    K = width - 2
    offs = [int(o) for o in slice_offsets]
    if len(offs) != slices + 1:
        raise ValueError("slice_offsets needs one entry per slice plus the vocabulary size")
    idx = _dev_int64(index, partials.device).reshape(rows, -1).contiguous()
    if idx.shape[1] != K:
        raise ValueError("index must have K columns, as the partials")
    mask = None
    if row_mask is not None:
        mask = row_mask.to(device=partials.device, dtype=torch.uint8).reshape(rows).contiguous()
    part = partials.contiguous()
    logp = torch.empty((rows, K), dtype=torch.float32, device=partials.device)
    xt0 = torch.empty(rows, dtype=torch.float32, device=partials.device)
    state = torch.empty((rows, 2), dtype=torch.float32, device=partials.device)
    host_offs = (ctypes.c_int64 * len(offs))(*offs)
    _check_status(dev_status, partials.device)
    with torch.cuda.device(partials.device):
        st = lib.vocab_slice_combine(part.data_ptr(), slices, ctypes.cast(host_offs, _vp), rows,
                                     idx.data_ptr(), K, int(ignore_index), _ptr(mask),
                                     float(temperature), logp.data_ptr(), xt0.data_ptr(),
                                     state.data_ptr(), _ptr(dev_status),
                                     _stream_ptr(stream, partials.device))
    _check(st, "vocab_slice_combine")
    return logp, xt0, state


def vocab_slice_grad(logits_slice: torch.Tensor, index, vocab_offset: int, vocab: int,
                     grad_logp, logp: torch.Tensor, target_logit: torch.Tensor,
                     temperature: float = 1.0, row_mask: Optional[torch.Tensor] = None, *,
                     row_state: Optional[torch.Tensor] = None, ignore_index: int = -100,
                     dlogits: Optional[torch.Tensor] = None,
                     dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """dL/d logits_slice for upstream grad_logp = dL/d logp, from the combined
    log-probs, target logit and (optional, for rows whose first index lies far
    below the row's max) row state of :func:`vocab_slice_combine`."""
    lib = load_library()
    lead_shape = logits_slice.shape[:-1]
    x = _rows_view(logits_slice)
    rows, n = x.shape
    idx, K = _slice_index(index, lead_shape, rows, x.device)
    g = torch.as_tensor(grad_logp, dtype=torch.float32, device=x.device).reshape(rows, K)
    g = g.contiguous()
    lp = logp.to(device=x.device, dtype=torch.float32).reshape(rows, K).contiguous()
    xt = target_logit.to(device=x.device, dtype=torch.float32).reshape(rows).contiguous()
    rs = None
    if row_state is not None:
        rs = row_state.to(device=x.device, dtype=torch.float32).reshape(rows, 2).contiguous()
    mask = None
    if row_mask is not None:
        mask = row_mask.to(device=x.device, dtype=torch.uint8).reshape(rows).contiguous()
    if dlogits is None:
        dlogits = torch.empty_like(logits_slice)
    d = _rows_view(dlogits)
    _check_dlogits(d, x)
    _check_status(dev_status, x.device)
    with torch.cuda.device(x.device):
        st = lib.vocab_slice_grad(x.data_ptr(), _dtype_code(x), rows, n, x.stride(0),
                                  int(vocab_offset), int(vocab), idx.data_ptr(), K,
                                  int(ignore_index), _ptr(mask), float(temperature),
                                  g.data_ptr(), lp.data_ptr(), xt.data_ptr(), _ptr(rs),
                                  d.data_ptr(), d.stride(0), _ptr(dev_status),
                                  _stream_ptr(stream, x.device))
    _check(st, "vocab_slice_grad")
    return dlogits

