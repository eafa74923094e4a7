"""The C-ABI boundary on the CPU: the library loads, exports every entry point
include/gbce.h declares, and rejects bad arguments on the host (these checks
return before any CUDA call, so they need no GPU)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbce.h")


@pytest.fixture(scope="module")
def lib():
    from cross_entropy_gb300 import build

    path = build.build()
    import cross_entropy_gb300 as gbce

    return gbce.load_library(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


def test_header_declares_the_four_calls_and_helpers():
    names = declared_functions()
    for n in ("selective_logsoftmax", "ce_fwd", "ce_bwd", "ce_fwd_bwd_fused",
              "gbce_workspace_size", "gbce_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from cross_entropy_gb300 import build

    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in declared_functions():
        assert n in exported, f"{n} declared in gbce.h but not exported"
        assert hasattr(lib, n)


def test_binding_names_match_the_abi():
    import cross_entropy_gb300 as gbce

    for n in ("selective_logsoftmax", "ce_fwd", "ce_bwd", "ce_fwd_bwd_fused"):
        assert callable(getattr(gbce, n))
    assert set(gbce._SIGNATURES) == set(declared_functions())


def test_status_strings(lib):
    for code in range(5):
        assert lib.gbce_status_string(code).decode().startswith("GBCE_")


def test_workspace_size_is_pure(lib):
    assert lib.gbce_workspace_size(0, 100, 1) == 0
    a = lib.gbce_workspace_size(8192, 152064, 4)
    assert a == lib.gbce_workspace_size(8192, 152064, 1) and a >= 8192 * 8
    few = lib.gbce_workspace_size(2, 152064, 1)   # split path needs partials
    assert few >= 2 * 18 * 8


FAKE = 0x10000  # never dereferenced: every case fails host validation first


def _logp(lib, **kw):
    a = dict(logits=FAKE, dtype=1, rows=4, vocab=100, stride=100, index=FAKE, k=1, T=1.0,
             mask=None, out=FAKE, entropy=None, ws=FAKE, ws_bytes=1 << 20, status=None,
             stream=None)
    a.update(kw)
    return lib.selective_logsoftmax(a["logits"], a["dtype"], a["rows"], a["vocab"], a["stride"],
                                    a["index"], a["k"], a["T"], a["mask"], a["out"],
                                    a["entropy"], a["ws"], a["ws_bytes"], a["status"],
                                    a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), 2),
    (dict(logits=FAKE + 1), 2),            # bf16 pointer not 2-byte aligned
    (dict(vocab=0), 1),
    (dict(stride=99), 1),
    (dict(rows=-1), 1),
    (dict(T=0.0), 1),
    (dict(T=float("nan")), 1),
    (dict(T=float("inf")), 1),
    (dict(k=0), 1),
    (dict(k=17), 1),
    (dict(logits=None), 1),
    (dict(index=None), 1),
    (dict(out=None), 1),
    (dict(ws=None), 4),
    (dict(ws_bytes=16), 4),
    (dict(ws=FAKE + 8), 4),
    (dict(entropy=FAKE, ws=None), 4),
])
def test_selective_logsoftmax_host_checks(lib, kw, code):
    assert _logp(lib, **kw) == code


def _bwd(lib, **kw):
    a = dict(logits=FAKE, dtype=0, rows=4, vocab=100, stride=100, labels=FAKE, ignore=-100,
             T=1.0, red=2, opt=None, grad=FAKE, logp=FAKE, n=FAKE, d=FAKE * 16, dstride=100)
    a.update(kw)
    return lib.ce_bwd(a["logits"], a["dtype"], a["rows"], a["vocab"], a["stride"], a["labels"],
                      a["ignore"], a["T"], a["red"], a["opt"], a["grad"], a["logp"], a["n"],
                      a["d"], a["dstride"], None, None)


def _opts(eps, dft=0, cap=0.0):
    import ctypes

    import cross_entropy_gb300 as gbce

    return ctypes.byref(gbce.CeOptions(eps, dft, cap))


@pytest.mark.parametrize("kw,code", [
    (dict(d=FAKE + 400), 1),               # dlogits overlaps logits
    (dict(d=FAKE), 1),                     # dlogits aliases logits
    (dict(dstride=50), 1),
    (dict(n=None), 1),                     # mean needs n_items
    (dict(grad=None), 1),
    (dict(logp=None), 1),
    (dict(red=5), 1),
    (dict(d=FAKE * 16 + 2), 2),            # fp32 dlogits misaligned
])
def test_ce_bwd_host_checks(lib, kw, code):
    assert _bwd(lib, **kw) == code


@pytest.mark.parametrize("eps", [-0.1, 1.5, float("nan"), float("inf")])
def test_ce_options_out_of_range_are_refused(lib, eps):
    assert _bwd(lib, opt=_opts(eps)) == 1
    args = [FAKE, 1, 4, 100, 100, FAKE, -100, 1.0, 2, _opts(eps, 1), FAKE, FAKE, None, None,
            None, FAKE * 16, 100, FAKE * 64, 1 << 20, None, None]
    assert lib.ce_fwd_bwd_fused(*args) == 1
    assert lib.ce_fwd(FAKE, 1, 4, 100, 100, FAKE, -100, 1.0, 2, _opts(eps), FAKE, None, None,
                      None, FAKE * 64, 1 << 20, None, None) == 1


def test_fused_host_checks(lib):
    args = [FAKE, 1, 4, 100, 100, FAKE, -100, 1.0, 2, None, FAKE, FAKE, None, None, None,
            FAKE * 16, 100, FAKE * 64, 1 << 20, None, None]
    a = list(args)
    a[15] = FAKE          # dlogits == logits
    assert lib.ce_fwd_bwd_fused(*a) == 1
    a = list(args)
    a[10] = None          # no upstream gradient
    assert lib.ce_fwd_bwd_fused(*a) == 1
    a = list(args)
    a[18] = 8             # workspace too small
    assert lib.ce_fwd_bwd_fused(*a) == 4


def test_binding_refuses_cpu_tensors():
    import torch

    import cross_entropy_gb300 as gbce

    with pytest.raises(ValueError, match="CUDA"):
        gbce.selective_logsoftmax(torch.zeros(2, 8), torch.zeros(2, 1, dtype=torch.int64))
    with pytest.raises(ValueError, match="CUDA"):
        gbce.ce_fwd_bwd_fused(torch.zeros(2, 8), torch.zeros(2, dtype=torch.int64))


def test_missing_library_fails_loudly(tmp_path):
    import cross_entropy_gb300 as gbce

    with pytest.raises(RuntimeError, match="not found"):
        gbce.load_library(str(tmp_path / "libgbce.so"))


def test_selective_backward_entropy_pointers_go_together(lib):
    def call(gh, hs):
        return lib.selective_logsoftmax_bwd(FAKE, 0, 4, 100, 100, FAKE, 1, 1.0, None, FAKE, FAKE,
                                            gh, hs, FAKE * 16, 100, None, None)
    assert call(FAKE, None) == 1
    assert call(None, FAKE) == 1


@pytest.mark.parametrize("cap", [-1.0, float("nan"), float("inf")])
def test_softcap_out_of_range_is_refused(lib, cap):
    assert _bwd(lib, opt=_opts(0.0, 0, cap)) == 1
