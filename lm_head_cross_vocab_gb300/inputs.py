"""Seeded synthetic workloads for the fused LM-head + CE + KL distillation loss.

This module only draws random inputs; it computes none of the loss arithmetic.
Both the CUDA library's tests/benchmark and the CPU oracle consume the tensors
it returns (the oracle receives exact fp64 upcasts of the same bytes).

Workload recipes (shapes, distributions, masks) follow the five synthetic
configurations of this project:

1. tiny tied fp32       N=64,    D=64,            V=512,    forward KL, T=2
2. separate-teacher bf16 N=4096, D_s=2048, D_t=4096, V=32000, Jeffreys, T=2, w_tce=0.5
3. large-vocab scoring   N=8192, student logits,  D_t=4096, V=248320, forward KL, T=1
4. sparse top-K          N=32768, D=4096,         V=151936, K=100, sequence chunk 2048
5. logit pairs           N=16384, V=128256,       forward/reverse/skew-JS(beta=0.1), T=2

"N(0, s)" means standard deviation s.  Ignore masks are seeded Bernoulli
draws.  Top-K teachers hold K distinct random column ids per token (in random
order) and probabilities softmax(N(0,2) draws) * M with M ~ U(0.85, 0.99),
not renormalised (the Full-Chunked-KL-Loss README, "Methods").
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

SEED_BASE = 1000


@dataclasses.dataclass(frozen=True)
class Workload:
    """Static description of one synthetic configuration."""

    cfg: int
    name: str
    n_tokens: int
    vocab: int
    d_student: int          # 0 when the student arrives as logits
    d_teacher: int          # 0 when the teacher arrives as logits / top-K
    dtype: str              # "bf16" | "fp32"
    student: str            # "hidden" | "logits"
    teacher: str            # "tied" | "separate" | "logits" | "topk"
    variant: str            # "forward" | "reverse" | "jeffreys" | "skew_js"
    t_student: float
    t_teacher: float
    w_student_ce: float
    w_teacher_ce: float
    w_kl: float
    beta: float
    ignore_index: int
    ignore_frac: float
    topk: int = 0
    vocab_chunk: int = 0
    seq_chunk: int = 0
    backward: bool = True
    student_logit_std: float = 0.0
    teacher_noise_std: float = 0.0

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    1: Workload(1, "tiny_tied_fp32", 64, 512, 64, 64, "fp32", "hidden", "tied", "forward",
                2.0, 2.0, 1.0, 1.0, 1.0, 0.5, -100, 0.10, vocab_chunk=128),
    2: Workload(2, "separate_teacher_bf16", 4096, 32000, 2048, 4096, "bf16", "hidden", "separate",
                "jeffreys", 2.0, 2.0, 1.0, 0.5, 1.0, 0.5, -100, 0.05),
    3: Workload(3, "large_vocab_scoring", 8192, 248320, 0, 4096, "bf16", "logits", "separate",
                "forward", 1.0, 1.0, 1.0, 0.0, 1.0, 0.5, -1, 0.03, vocab_chunk=16384,
                backward=False, student_logit_std=3.0),
    4: Workload(4, "sparse_topk", 32768, 151936, 4096, 0, "bf16", "hidden", "topk", "forward",
                1.0, 1.0, 0.0, 0.0, 1.0, 0.5, -100, 0.0, topk=100, seq_chunk=2048),
    5: Workload(5, "logit_pair", 16384, 128256, 0, 0, "bf16", "logits", "logits", "forward",
                2.0, 2.0, 0.0, 0.0, 1.0, 0.1, -100, 0.08,
                student_logit_std=4.0, teacher_noise_std=1.0),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def _normal(shape, std, dtype, g, device):
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_labels(n, vocab, ignore_index, ignore_frac, g, device):
    labels = torch.randint(0, vocab, (n,), generator=g, device=device, dtype=torch.int64)
    if ignore_frac > 0:
        drop = torch.rand(n, generator=g, device=device) < ignore_frac
        labels[drop] = ignore_index
    return labels


def make_topk(n, vocab, k, g, device, mass_lo=0.85, mass_hi=0.99):
    """K distinct random column ids per row (unsorted) and non-renormalised probabilities."""
    idx = torch.randint(0, vocab, (n, k), generator=g, device=device, dtype=torch.int64)
    for _ in range(64):
        s, _ = torch.sort(idx, dim=1)
        dup_rows = (s[:, 1:] == s[:, :-1]).any(dim=1)
        if not bool(dup_rows.any()):
            break
        rows = dup_rows.nonzero().flatten()
        idx[rows] = torch.randint(0, vocab, (rows.numel(), k), generator=g, device=device,
                                  dtype=torch.int64)
    else:  # pragma: no cover - astronomically unlikely for K << V
        raise RuntimeError("could not draw distinct top-K ids")
    raw = torch.randn(n, k, generator=g, device=device, dtype=torch.float32) * 2.0
    mass = mass_lo + (mass_hi - mass_lo) * torch.rand(n, 1, generator=g, device=device)
    p = torch.softmax(raw, dim=1) * mass
    return idx.to(torch.int32), p.contiguous()


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw every input tensor of workload ``w`` on ``device``.

    Returns a dict with keys among h_s, w_s, logits_s, h_t, w_t, logits_t,
    labels, topk_idx, topk_p (absent keys are unused by the workload).
    """
    seed = SEED_BASE + w.cfg if seed is None else seed
    g = _gen(device, seed)
    dt = _torch_dtype(w.dtype)
    out = {}
    n, v = w.n_tokens, w.vocab
    if w.student == "hidden":
        out["h_s"] = _normal((n, w.d_student), 1.0, dt, g, device)
        out["w_s"] = _normal((v, w.d_student), 0.02, dt, g, device)
    else:
        out["logits_s"] = _normal((n, v), w.student_logit_std, dt, g, device)
    if w.teacher == "tied":
        out["h_t"] = _normal((n, w.d_student), 1.0, dt, g, device)
    elif w.teacher == "separate":
        out["h_t"] = _normal((n, w.d_teacher), 1.0, dt, g, device)
        out["w_t"] = _normal((v, w.d_teacher), 0.02, dt, g, device)
    elif w.teacher == "logits":
        if w.student == "logits" and w.teacher_noise_std > 0:
            zt = out["logits_s"].float()
            zt.add_(torch.randn(n, v, generator=g, device=device) * w.teacher_noise_std)
            out["logits_t"] = zt.to(dt)
            del zt
        else:
            out["logits_t"] = _normal((n, v), max(w.student_logit_std, 1.0), dt, g, device)
    if w.teacher == "topk":
        out["topk_idx"], out["topk_p"] = make_topk(n, v, w.topk, g, device)
    if w.ignore_frac > 0 or w.w_student_ce > 0 or w.w_teacher_ce > 0:
        out["labels"] = make_labels(n, v, w.ignore_index, w.ignore_frac, g, device)
    return out
