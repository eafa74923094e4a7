"""Seeded synthetic inputs for the row-wise log-softmax / cross-entropy path.

Both sides of every parity check (the CUDA library and the fp64 oracle) and
the benchmark draw their inputs from here, so this module holds input
construction only: random draws, row selection and the "target leads the
others by a margin" structure.  It computes no log-softmax, loss or gradient.

The shapes and distributions stand in for the pages' workloads:

* packed RL log-probs, 8192 rows = 8 sequences x 1024 completion tokens at
  vocab 152064 ("perf(rlhf): chunk selective_log_softmax instead of looping
  per token", "Experiment results" and the follow-up comment);
* sparse supervised SFT rows, two 1024-token samples cropped to 1922 rows of
  which 256 are supervised in four assistant spans each, vocab 4096 (ms-swift
  PR #10353, "Experiment results");
* confident rows whose target leads the other logits by 17/20/30/50 at
  vocab 151936 ("Fix softmax collapse in CE, GRPO, KL/JSD and softmax", the
  unsloth-zoo #2080 "Accuracy" section).

No dataset or trained weights are involved; logits are Gaussian.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

IGNORE_INDEX = -100


@dataclass
class Workload:
    """One seeded input set.  Tensors live on ``device``."""

    name: str
    logits: torch.Tensor                 # [rows, V] bf16 or fp32
    labels: torch.Tensor                 # [rows] int64, IGNORE_INDEX = skip
    index: torch.Tensor                  # [rows, K] int64 gather indices
    row_mask: Optional[torch.Tensor]     # [rows] uint8 or None (all live)
    temperature: float
    reduction: str                       # CE reduction
    grad_out: torch.Tensor               # [rows] for 'none', [1] otherwise
    extra_temperatures: tuple = ()
    peaked_rows: Optional[torch.Tensor] = None
    margins: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.logits.shape[0]

    @property
    def vocab(self) -> int:
        return self.logits.shape[1]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(rows: int, V: int, std: float, dtype, g, device, block_rows: int = 1024):
    """N(0, std^2) logits drawn in fp32 in fixed row blocks, then rounded."""
    out = torch.empty((rows, V), dtype=dtype, device=device)
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        blk = torch.randn((r1 - r0, V), generator=g, device=device, dtype=torch.float32)
        out[r0:r1] = (blk * std).to(dtype)
    return out


def set_target_margin(logits: torch.Tensor, rows: torch.Tensor, targets: torch.Tensor,
                      margins: torch.Tensor) -> None:
    """x[r, t] = max_{j != t} x[r, j] + margin, set in fp32, rounded to the dtype."""
    if rows.numel() == 0:
        return
    sub = logits[rows].float()
    ar = torch.arange(rows.numel(), device=logits.device)
    sub[ar, targets] = float("-inf")
    top = sub.max(dim=1).values
    logits[rows, targets] = (top + margins.float()).to(logits.dtype)


def _index_from_labels(labels: torch.Tensor) -> torch.Tensor:
    return torch.where(labels == IGNORE_INDEX, torch.zeros_like(labels), labels).unsqueeze(1)


def ce_small_fp32(device="cpu", seed: int = 0) -> Workload:
    """64 x 4096 fp32 ~N(0,3^2); 6 rows ignored; 8 rows with the target 20 above the rest."""
    rows, V = 64, 4096
    g = _gen(seed, device)
    logits = _normal(rows, V, 3.0, torch.float32, g, device)
    labels = torch.randint(0, V, (rows,), generator=g, device=device)
    perm = torch.randperm(rows, generator=g, device=device)
    ignored, peaked = perm[:6], perm[6:14]
    margins = torch.full((8,), 20.0, device=device)
    set_target_margin(logits, peaked, labels[peaked], margins)
    labels[ignored] = IGNORE_INDEX
    mask = (labels != IGNORE_INDEX).to(torch.uint8)
    return Workload("ce_small_fp32_64x4096", logits, labels, _index_from_labels(labels), mask,
                    1.0, "mean", torch.ones(1, device=device), peaked_rows=peaked,
                    margins=margins)


def _span_labels(samples, per_sample, spans, span_len, V, g, device):
    """Labels that are IGNORE_INDEX except in `spans` non-overlapping runs of
    `span_len` rows per sample, at seeded offsets."""
    rows = samples * per_sample
    labels = torch.full((rows,), IGNORE_INDEX, dtype=torch.int64, device=device)
    free = per_sample - spans * span_len
    for s in range(samples):
        # non-overlapping spans: sorted distinct offsets in the free room,
        # the k-th shifted past the k spans before it
        offs = torch.randperm(free + 1, generator=g, device=device)[:spans].sort().values
        for k in range(spans):
            start = s * per_sample + int(offs[k]) + k * span_len
            labels[start:start + span_len] = torch.randint(
                0, V, (span_len,), generator=g, device=device)
    return labels


def sft_sparse_bf16(device="cpu", seed: int = 0, samples: int = 8, per_sample: int = 1024,
                    spans: int = 4, span_len: int = 64, V: int = 152064) -> Workload:
    """8192 x 152064 bf16 ~N(0,2.5^2): 8 samples of 1024 rows, four 64-row
    supervised spans each (2048 supervised rows, 25%), mean over them.

    The sparse-supervision structure of ms-swift PR #10353 at the packed
    workload's size and vocabulary.
    """
    rows = samples * per_sample
    g = _gen(seed, device)
    logits = _normal(rows, V, 2.5, torch.bfloat16, g, device)
    labels = _span_labels(samples, per_sample, spans, span_len, V, g, device)
    mask = (labels != IGNORE_INDEX).to(torch.uint8)
    return Workload(f"sft_sparse_bf16_{rows}x{V}", logits, labels, _index_from_labels(labels),
                    mask, 1.0, "mean", torch.ones(1, device=device),
                    meta={"supervised": samples * spans * span_len})


def ce_sparse_bf16(device="cpu", seed: int = 0) -> Workload:
    """1922 x 4096 bf16 ~N(0,2^2): two 961-row samples, four 32-row supervised spans each."""
    samples, per_sample, spans, span_len, V = 2, 961, 4, 32, 4096
    rows = samples * per_sample
    g = _gen(seed, device)
    logits = _normal(rows, V, 2.0, torch.bfloat16, g, device)
    labels = _span_labels(samples, per_sample, spans, span_len, V, g, device)
    n_sup = samples * spans * span_len
    grad = torch.full((rows,), 1.0 / n_sup, device=device)
    mask = (labels != IGNORE_INDEX).to(torch.uint8)
    return Workload("ce_sparse_bf16_1922x4096", logits, labels, _index_from_labels(labels), mask,
                    1.0, "none", grad, meta={"supervised": n_sup})


def logp_bf16(device="cpu", seed: int = 0) -> Workload:
    """1024 x 32768 bf16 ~N(0,2^2); one index per row; 154 rows (15%) masked out."""
    rows, V = 1024, 32768
    g = _gen(seed, device)
    logits = _normal(rows, V, 2.0, torch.bfloat16, g, device)
    index = torch.randint(0, V, (rows, 1), generator=g, device=device)
    perm = torch.randperm(rows, generator=g, device=device)
    mask = torch.ones(rows, dtype=torch.uint8, device=device)
    mask[perm[:154]] = 0
    labels = index[:, 0].clone()
    return Workload("logp_bf16_1024x32768", logits, labels, index, mask, 1.0, "mean",
                    torch.ones(1, device=device), extra_temperatures=(0.9,))


def grpo_bf16(device="cpu", seed: int = 0, rows: int = 8192, V: int = 152064,
              K: int = 4) -> Workload:
    """8192 x 152064 bf16 ~N(0,2.5^2) packed log-probs, K=4 indices, T=0.9.

    5% of rows (410 of 8192) have their label logit 8..12 above the rest.
    Column 0 of the index is the label; CE uses it with no ignored rows.
    """
    g = _gen(seed, device)
    logits = _normal(rows, V, 2.5, torch.bfloat16, g, device)
    index = torch.randint(0, V, (rows, K), generator=g, device=device)
    labels = index[:, 0].clone()
    n_peak = (rows * 5 + 50) // 100
    perm = torch.randperm(rows, generator=g, device=device)
    peaked = perm[:n_peak]
    margins = 8.0 + 4.0 * torch.rand((n_peak,), generator=g, device=device)
    set_target_margin(logits, peaked, labels[peaked], margins)
    return Workload(f"grpo_bf16_{rows}x{V}_k{K}", logits, labels, index, None, 0.9, "mean",
                    torch.ones(1, device=device), extra_temperatures=(1.0,),
                    peaked_rows=peaked, margins=margins)


def collapse_stress(dtype=torch.float32, device="cpu", seed: int = 0, rows: int = 2048,
                    V: int = 151936) -> Workload:
    """2048 x 151936 ~N(0,1) in fp32 or bf16; 205 rows ignored; 1024 confident rows.

    The confident rows' label logits lead the other logits by 17, 20, 30 and
    50 in turn (256 rows each at full size), chosen among the non-ignored rows.
    """
    g = _gen(seed, device)
    logits = _normal(rows, V, 1.0, dtype, g, device)
    labels = torch.randint(0, V, (rows,), generator=g, device=device)
    perm = torch.randperm(rows, generator=g, device=device)
    n_ign = (rows * 10 + 50) // 100          # round(10% of rows): 205 of 2048
    n_peak = rows // 2
    ignored, peaked = perm[:n_ign], perm[n_ign:n_ign + n_peak]
    levels = torch.tensor([17.0, 20.0, 30.0, 50.0], device=device)
    margins = levels[torch.arange(n_peak, device=device) % 4]
    set_target_margin(logits, peaked, labels[peaked], margins)
    labels[ignored] = IGNORE_INDEX
    mask = (labels != IGNORE_INDEX).to(torch.uint8)
    tag = "fp32" if dtype == torch.float32 else "bf16"
    return Workload(f"collapse_{tag}_{rows}x{V}", logits, labels, _index_from_labels(labels),
                    mask, 1.0, "mean", torch.ones(1, device=device), peaked_rows=peaked,
                    margins=margins)


def peaked_rows_tiny(V: int, margins, dtype=torch.float64, temperature: float = 1.0,
                     seed: int = 0, device="cpu") -> Workload:
    """One row per margin, N(0,1) others, target at a seeded column, for small-V checks."""
    g = _gen(seed, device)
    m = torch.as_tensor(margins, dtype=torch.float64)
    rows = m.numel()
    logits = torch.randn((rows, V), generator=g, device=device, dtype=torch.float64).to(dtype)
    labels = torch.randint(0, V, (rows,), generator=g, device=device)
    set_target_margin(logits, torch.arange(rows, device=device), labels, m.to(device))
    return Workload(f"peaked_{rows}x{V}", logits, labels, labels.unsqueeze(1), None, temperature,
                    "sum", torch.ones(1, device=device), peaked_rows=torch.arange(rows),
                    margins=m)


def dominated_elsewhere(dtype, rows: int, V: int, K: int, seed: int = 0,
                        device="cpu") -> Workload:
    """Confident rows whose dominant column is not the first gathered index.

    N(0,1) logits; every row gets one column d with x_d = max_{j != d} x_j +
    margin, margins cycling 17/20/30/50 (the collapse margins).  The first
    gathered index is never d.  With K > 1, every other row gathers d at an
    index k > 0; the other rows leave d out of the gathered set (a sampled
    token that is not the row's argmax).
    """
    g = _gen(seed, "cpu")
    logits = torch.randn((rows, V), generator=g).to(dtype)
    d = torch.randint(0, V, (rows,), generator=g)
    margins = torch.tensor([17.0, 20.0, 30.0, 50.0]).repeat((rows + 3) // 4)[:rows]
    set_target_margin(logits, torch.arange(rows), d, margins)
    index = torch.randint(0, V, (rows, K), generator=g)
    index = torch.where(index == d[:, None], (index + 1) % V, index)
    if K > 1:
        k = 1 + torch.arange(rows) % (K - 1)
        even = torch.arange(rows) % 2 == 0
        index[even, k[even]] = d[even]
    return Workload(f"dominated_elsewhere_{rows}x{V}_k{K}", logits.to(device), d.to(device),
                    index.to(device), None, 1.0, "sum", torch.ones(1, device=device),
                    peaked_rows=torch.arange(rows), margins=margins)


def to_numpy_f64(t: torch.Tensor):
    """Exact fp64 copy of bf16/fp32/fp64 logits for the oracle."""
    return t.detach().to("cpu").to(torch.float64).numpy()
