"""Benchmark of the fused LM-head + CE + KL distillation loss (forward + backward).

One step = the whole hot path through the C ABI on one batch of synthetic
input: kd_fwd (label check, fused tcgen05 projection + online-softmax CE/KL,
split combine, loss reduction) and kd_bwd (recomputed logits -> closed-form
gradient chunks -> dH and dW on tcgen05).  Default workload: the separate-
teacher bf16 configuration (4096 tokens, D_s = 2048, D_t = 4096, V = 32000,
Jeffreys KL, T = 2, teacher CE weight 0.5, 5 % ignored labels).

    python bench.py [--gpus N --steps K --warmup W] [--config C] [--impl reference]

Multi-GPU (torchrun): every rank runs its own batch (data parallel, weak
scaling); no collective is on the data path.  `--impl reference` times the
fp64 CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from lm_head_cross_vocab_gb300 import inputs as I  # noqa: E402

L2_BYTES = 129 * 2 ** 20
NOMINAL_BF16_TFLOPS = 2250.0  # dense (no 2:4 sparsity), GB300


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def flops_per_step(w: I.Workload):
    """Algorithmic FLOPs: projections forward, recompute + dH + dW backward."""
    n, v = w.n_tokens, w.vocab
    proj_s = 2 * n * v * w.d_student if w.student == "hidden" else 0
    proj_t = 2 * n * v * (w.d_teacher if w.teacher == "separate"
                          else w.d_student if w.teacher == "tied" else 0)
    fwd = proj_s + proj_t
    bwd = (fwd + 2 * proj_s) if w.backward else 0
    return fwd, bwd


def bytes_per_step(w: I.Workload):
    """Algorithmic HBM bytes of the logits-streaming path (bf16 logits)."""
    n, v = w.n_tokens, w.vocab
    fwd = 2 * n * v * (1 + (w.teacher == "logits"))
    bwd = 2 * n * v * (2 + (w.teacher == "logits")) if w.backward else 0
    return fwd, bwd


# library sources behind each measured family: the projection and the mixing
# kernels stand alone; the loss path is everything else in csrc/
SOURCE_GROUPS = {"project": ("kd_project.cu",), "mix": ("kd_mix.cu",)}


def kernel_sources_hash(group: str = "loss") -> str:
    """Hash of the library sources a kernel family depends on (its kernels,
    the shared headers and the launch planning)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lm_head_cross_vocab_gb300", "csrc")
    own = {f for g in SOURCE_GROUPS.values() for f in g}
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh", ".h")):
            continue
        if f.endswith(".cu") and (f not in SOURCE_GROUPS[group] if group in SOURCE_GROUPS
                                  else f in own):
            continue
        h.update(f.encode())
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(group: str = "loss") -> dict:
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum from
    one ncu capture, profiles/traffic.json), keyed "workload:kernel family";
    empty once the sources of that group differ from the ones captured."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    g = d.get("groups", {}).get(group, {})
    if g.get("sources_sha256_16") != kernel_sources_hash(group):
        return {}
    return g.get("bytes_per_launch", {})


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU)

def oracle_step(w: I.Workload, cpu: dict, rows: np.ndarray):
    """fwd + bwd of the oracle on the sampled token rows (row-local work)."""
    from oracle import kd_oracle as O
    sub = {k: (v[rows] if k in ("h_s", "h_t", "logits_s", "logits_t", "labels", "topk_idx",
                                "topk_p") else v) for k, v in cpu.items()}
    lab = sub["labels"].numpy() if "labels" in sub else None
    if w.student == "hidden":
        z_s = O.project(sub["h_s"], sub["w_s"])
    else:
        z_s = O.as_f64(sub["logits_s"])
    z_t = None
    if w.teacher == "separate":
        z_t = O.project(sub["h_t"], sub["w_t"])
    elif w.teacher == "tied":
        z_t = O.project(sub["h_t"], sub["w_s"])
    elif w.teacher == "logits":
        z_t = O.as_f64(sub["logits_t"])
    kw = dict(variant=w.variant, t_student=w.t_student, t_teacher=w.t_teacher, beta=w.beta,
              w_student_ce=w.w_student_ce, w_teacher_ce=w.w_teacher_ce, w_kl=w.w_kl,
              ignore_index=w.ignore_index)
    topk = {}
    if w.teacher == "topk":
        topk = dict(topk_idx=sub["topk_idx"].numpy(), topk_p=sub["topk_p"].numpy())
    out = O.forward(z_s, z_t, lab, **topk, **kw)
    if w.backward:
        g_s, g_t = O.grad_logits(z_s, z_t, lab, **topk, **kw)
        if w.student == "hidden":
            O.hidden_grads(sub["h_s"], sub["w_s"], g_s, sub.get("h_t"), g_t,
                           tied=w.teacher == "tied")
    return out["loss"]


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def time_oracle(w: I.Workload, rows_per_step: int, steps: int, warmup: int, seed: int):
    cpu = I.make_inputs(w, "cpu")
    rng = np.random.default_rng(seed)
    for _ in range(warmup):
        oracle_step(w, cpu, np.sort(rng.choice(w.n_tokens, rows_per_step, replace=False)))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(w, cpu, np.sort(rng.choice(w.n_tokens, rows_per_step, replace=False)))
    dt = time.perf_counter() - t0
    return rows_per_step * steps / dt, dt


def run_reference(args, w: I.Workload, rank: int):
    if rank != 0:
        return
    rows = args.ref_rows
    value, dt = time_oracle(w, rows, args.steps, args.warmup, 7)
    line = {
        "impl": "reference", "metric": "fused linear+CE+KD fwd+bwd tokens/s", "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.n_tokens, "vocab": w.vocab,
                   "d_student": w.d_student, "d_teacher": w.d_teacher},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(),
                         "kind": "oracle",
                         "sample": f"{rows} seeded random tokens of the workload per step "
                                   f"(fp64 numpy oracle, fwd+bwd)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def smi_index(local: int) -> int:
    """nvidia-smi index of this process's GPU (the first CUDA_VISIBLE_DEVICES
    entry when it is numeric, else the local rank)."""
    first = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    return int(first) if first.isdigit() else local


def time_cpu_oracle(fn, seconds):
    """Tokens/s of fn(rows) (the CPU oracle on a seeded sample of `rows` token
    rows), the sample grown from 8 rows until one call takes about `seconds`;
    returns (rate, rows, elapsed)."""
    rows = 8
    while True:
        t0 = time.perf_counter()
        fn(rows)
        dt = time.perf_counter() - t0
        if dt >= seconds or rows >= 4096:
            return rows / dt, rows, dt
        rows = min(4096, rows * 4, max(rows * 2, int(rows * seconds / max(dt, 1e-3))))


def run_diag_gemm(args, rank):
    """The tensor-core GEMM core on its own (kd_diag_gemm_bf16: C = A B^T, bf16
    operands stored K-major, fp32 C) against torch.matmul (cuBLAS) on the same
    bf16 operands: a check of the mainloop shared by the fused kernels."""
    from lm_head_cross_vocab_gb300 import kd
    lib = kd.load_library()
    dev = torch.device("cuda", 0)
    out = []
    for (m, n, k) in ((8192, 8192, 8192), (4096, 6400, 6144), (16384, 8192, 4096)):
        g = torch.Generator(device=dev).manual_seed(m + n + k)
        a = torch.randn(m, k, generator=g, device=dev).to(torch.bfloat16)
        b = torch.randn(n, k, generator=g, device=dev).to(torch.bfloat16)
        c = torch.empty(m, n, device=dev, dtype=torch.float32)
        st = torch.cuda.current_stream(dev).cuda_stream

        def ours():
            r = lib.kd_diag_gemm_bf16(a.data_ptr(), b.data_ptr(), c.data_ptr(), m, n, k, 0, st)
            assert r == kd.KD_OK, r

        def cublas():
            torch.matmul(a, b.t())

        res = {"m": m, "n": n, "k": k}
        for name, fn in (("kd_diag_gemm_bf16", ours), ("torch_matmul", cublas)):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            for _ in range(args.steps):
                fn()
            s1.record()
            torch.cuda.synchronize()
            res[name + "_tflops"] = 2 * m * n * k / (s0.elapsed_time(s1) / args.steps) / 1e9
        out.append(res)
    if rank == 0:
        print(json.dumps({"metric": "tensor-core GEMM TFLOP/s (diagnostic)", "unit": "TFLOP/s",
                          "dtype": "bf16", "data": "synthetic", "steps": args.steps,
                          "warmup": args.warmup, "shapes": out}), flush=True)


def _projection_map(v_t, v_s):
    """The synthetic cross-tokenizer token map of the projection legs: 80 % of
    the student ids reached by one teacher token, 3 % by two, the other teacher
    tokens unmatched (seeded)."""
    rng = np.random.default_rng(1006)
    tmap = np.full(v_t, -1, dtype=np.int32)
    src = rng.permutation(v_t)
    one = rng.permutation(v_s)[: int(0.8 * v_s)]
    tmap[src[: one.size]] = one
    two = rng.choice(one, int(0.03 * v_s), replace=False)
    tmap[src[one.size: one.size + two.size]] = two
    return tmap


def run_project_loss(args, rank):
    """Cross-tokenizer distillation with the projected teacher inside the loss
    (KD_TEACHER_PROJECTED): bf16 teacher logits ~N(0,4) over 151936 ids, the
    projection map of --project, bf16 student logits ~N(0,4) over 128256 ids,
    8 % ignored labels, forward KL, T = 2, w_sce = 0.  One step = kd_fwd +
    kd_bwd (d z_s); no projected tensor is stored.  The same step through the
    unfused composition (kd_project_teacher_logits, then a logits teacher at
    T = 1) is timed beside it."""
    from lm_head_cross_vocab_gb300 import kd
    kd.load_library()
    n = args.tokens or 16384
    v_t, v_s, T = 151936, 128256, 2.0
    dev = torch.device("cuda", 0)
    tmap_d = torch.from_numpy(_projection_map(v_t, v_s)).to(dev)
    g = torch.Generator(device=dev).manual_seed(1008)
    z_t = (torch.randn(n, v_t, generator=g, device=dev) * 4.0).to(torch.bfloat16)
    z_s = (torch.randn(n, v_s, generator=g, device=dev) * 4.0).to(torch.bfloat16)
    labels = torch.randint(0, v_s, (n,), generator=g, device=dev)
    labels[torch.rand(n, generator=g, device=dev) < 0.08] = -100
    t = {"logits_s": z_s, "logits_t": z_t, "labels": labels, "token_map": tmap_d}
    common = dict(n_tokens=n, vocab=v_s, dtype="bf16", student="logits", variant="forward",
                  t_student=T, w_student_ce=0.0, w_teacher_ce=0.0, w_kl=1.0, ignore_index=-100)
    prob = kd.Problem(teacher="projected", t_teacher=T, vocab_teacher=v_t, **common)
    prob_u = kd.Problem(teacher="logits", t_teacher=1.0, **common)
    ws_f, ws_b, ws_p = kd.Workspace(), kd.Workspace(), kd.Workspace()
    fo = bo = fu = bu = None
    zp = None

    def fused():
        nonlocal fo, bo
        fo = kd.forward(prob, t, ws_f, check=False, out=fo)
        bo = kd.backward(prob, t, fo["stats"], want=("logits_s",), workspace=ws_b, check=False,
                         out=bo)

    def unfused():
        nonlocal fu, bu, zp
        zp = kd.project_teacher_logits(tmap_d, z_t, v_s, temperature=T, workspace=ws_p,
                                       check=False)
        tu = {"logits_s": z_s, "logits_t": zp, "labels": labels}
        fu = kd.forward(prob_u, tu, ws_f, check=False, out=fu)
        bu = kd.backward(prob_u, tu, fu["stats"], want=("logits_s",), workspace=ws_b,
                         check=False, out=bu)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / steps

    launches0 = kd.kd_launch_count()
    with ClockSampler(smi_index(0)) as clk:
        ms = timed(fused, args.steps)
    launches = kd.kd_launch_count() - launches0
    kd.check_status(fo["dev_status"])
    ms_u = timed(unfused, max(3, args.steps // 2))
    zp = None
    peak_gib = torch.cuda.max_memory_allocated(dev) / 2 ** 30
    nbytes = n * (4 * v_t + 6 * v_s)  # fwd: z_t, z_s; bwd: z_t, z_s, d z_s (bf16)
    peaks, peak_src = load_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "cross-vocab fused linear+KD fwd+bwd tokens/s (projected teacher)",
            "value": n / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "cross_vocab_projected_teacher", "tokens": n,
                       "v_teacher": v_t, "v_student": v_s, "temperature": T,
                       "variant": "forward", "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "kernel": "k_proj_loss (fwd + bwd, + inverse map)",
                         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src} copy",
                         "bytes_per_step": nbytes, "traffic": None},
            "sections": {"unfused_project_then_logits_teacher": {
                "ms_per_step": ms_u, "tokens_per_s": n / (ms_u / 1e3),
                "note": "kd_project_teacher_logits -> kd_fwd / kd_bwd, projected logits stored"}},
            "peak_hbm_gib": peak_gib, "clocks": clk.summary(), "gpu_launches": launches}),
            flush=True)


def run_projection(args, rank):
    """Cross-vocabulary token-map projection (kd_project_teacher_logits) on a
    synthetic cross-tokenizer case: bf16 teacher logits ~N(0,4) over a
    151936-id vocabulary projected at T = 2 onto a 128256-id student vocabulary
    through a seeded exact-map-like token map (80 % of the student ids reached
    by one teacher token, 3 % by two, the other teacher tokens unmatched)."""
    from lm_head_cross_vocab_gb300 import kd
    kd.load_library()
    n = args.tokens or 16384
    v_t, v_s = 151936, 128256
    dev = torch.device("cuda", 0)
    tmap = _projection_map(v_t, v_s)
    tmap_d = torch.from_numpy(tmap).to(dev)
    g = torch.Generator(device=dev).manual_seed(1006)
    z = (torch.randn(n, v_t, generator=g, device=dev) * 4.0).to(torch.bfloat16)
    out = torch.empty(n, v_s, device=dev, dtype=torch.bfloat16)
    ws = kd.Workspace()
    for _ in range(args.warmup):
        kd.project_teacher_logits(tmap_d, z, v_s, temperature=2.0, workspace=ws, check=False)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = kd.kd_launch_count()
    with ClockSampler(smi_index(0)) as clk:
        s.record()
        for _ in range(args.steps):
            out = kd.project_teacher_logits(tmap_d, z, v_s, temperature=2.0, workspace=ws,
                                            check=False)
        e.record()
        torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.steps
    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import kd_oracle as O
        gc = torch.Generator().manual_seed(1007)

        def oracle(rows):
            O.project_teacher_logits((torch.randn(rows, v_t, generator=gc) * 4.0).to(
                torch.bfloat16), tmap, v_s, temperature=2.0)
        v_cpu, rows, dt = time_cpu_oracle(oracle, min(args.cpu_seconds, 6.0))
        cpu_base = {"value": v_cpu, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                    "sample": f"{rows} seeded token rows of the same map, fp64 numpy oracle "
                              f"({dt:.1f} s)"}
    nbytes = n * v_t * 2 + n * v_s * 2  # teacher logits read once, projected logits written
    peaks, peak_src = load_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "token-map projection tokens/s", "value": n / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "cross_vocab_projection", "tokens": n, "v_teacher": v_t,
                       "v_student": v_s, "temperature": 2.0,
                       "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "kernel": "k_project_exchange (+ inverse map, exchange lists)",
                         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src} copy",
                         "bytes_per_launch": nbytes,
                         "traffic": None if args.tokens else
                         load_traffic("project").get("cross_vocab_projection:k_project")},
            "cpu_baseline": cpu_base, "clocks": clk.summary(),
            "gpu_launches": kd.kd_launch_count() - launches0}), flush=True)


def run_mix(args, rank):
    """Multi-teacher mixing (kd_mix_teacher_logits): two bf16 teachers' cached
    logits ~N(0, 2^2) and ~N(0, 3^2) over a 151936-id vocabulary, weights
    0.6 / 0.4, mixed into one bf16 log-distribution per token."""
    from lm_head_cross_vocab_gb300 import kd
    kd.load_library()
    n = args.tokens or 16384
    v = 151936
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(2718)
    zs = [(torch.randn(n, v, generator=g, device=dev) * s).to(torch.bfloat16) for s in (2.0, 3.0)]
    w = [0.6, 0.4]
    for _ in range(args.warmup):
        kd.mix_teacher_logits(zs, w, args.mix, check=False)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = kd.kd_launch_count()
    with ClockSampler(smi_index(0)) as clk:
        s.record()
        for _ in range(args.steps):
            out = kd.mix_teacher_logits(zs, w, args.mix, check=False)
        e.record()
        torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.steps
    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import kd_oracle as O
        gc = torch.Generator().manual_seed(2719)

        def oracle(rows):
            O.mix_teacher_logits([(torch.randn(rows, v, generator=gc) * sd).to(torch.bfloat16)
                                  for sd in (2.0, 3.0)], w, args.mix)
        v_cpu, rows, dt = time_cpu_oracle(oracle, min(args.cpu_seconds, 6.0))
        cpu_base = {"value": v_cpu, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                    "sample": f"{rows} seeded token rows of two teachers, fp64 numpy oracle "
                              f"({dt:.1f} s)"}
    nbytes = 2 * n * v * 2 + n * v * 2  # both teachers read once, the mixture written once
    peaks, peak_src = load_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "multi-teacher mixing tokens/s", "value": n / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"mix_2_teachers_{args.mix}", "tokens": n, "vocab": v,
                       "teachers": 2, "weights": w, "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "kernel": "k_mix_cluster", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "peak_source": f"{peak_src} copy", "bytes_per_launch": nbytes,
                         "traffic": None if args.tokens else
                         load_traffic("mix").get(f"mix_2_teachers_{args.mix}:k_mix")},
            "cpu_baseline": cpu_base, "clocks": clk.summary(),
            "gpu_launches": kd.kd_launch_count() - launches0}), flush=True)
    del out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload at this many tokens (small cases for profiler captures)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--cpu-rows", type=int, default=0, help="oracle sample size (0: sized by time)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--project", action="store_true",
                    help="time the cross-vocabulary token-map projection instead of the loss")
    ap.add_argument("--diag-gemm", action="store_true",
                    help="time the tensor-core GEMM core against torch.matmul (diagnostic)")
    ap.add_argument("--project-loss", action="store_true",
                    help="time cross-vocabulary distillation with the projected teacher inside "
                         "the loss (fwd + bwd)")
    ap.add_argument("--mix", choices=["arithmetic", "geometric"],
                    help="time multi-teacher mixing (this mode) instead of the loss")
    ap.add_argument("--variant", choices=["forward", "reverse", "jeffreys", "skew_js",
                                          "skew_forward", "skew_reverse"],
                    help="run the workload with this KL variant")
    ap.add_argument("--forward-only", action="store_true",
                    help="forward-only scoring: kd_fwd with no saved statistics, no backward")
    ap.add_argument("--no-serialised", action="store_true",
                    help="skip the extra pass that times the gradient producer with the "
                         "backward GEMMs serialised")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from lm_head_cross_vocab_gb300 import dist as D
    rank, world, local = D.world_from_env()
    w = I.WORKLOADS[args.config]
    if args.tokens > 0:
        w = w.scaled(n_tokens=args.tokens)
    if args.variant:
        w = w.scaled(variant=args.variant)
    if args.forward_only:
        w = w.scaled(backward=False)

    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if args.project:
        run_projection(args, rank)
        return
    if args.project_loss:
        run_project_loss(args, rank)
        return
    if args.diag_gemm:
        run_diag_gemm(args, rank)
        return
    if args.mix:
        run_mix(args, rank)
        return

    from lm_head_cross_vocab_gb300 import kd
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    kd.load_library()
    if not kd.kd_device_supported(local):
        raise SystemExit("bench needs an sm_103 GPU")

    # inputs resident in HBM; each rank owns its own batch (weak scaling)
    t = I.make_inputs(w, dev, seed=I.SEED_BASE + w.cfg + 7919 * rank)
    prob = kd.problem_for(w, vocab_chunk=0, seq_chunk=0)
    ws_f, ws_b = kd.Workspace(), kd.Workspace()
    fwd_out = None
    bwd_out = None
    want = ("h_s", "w_s") if w.student == "hidden" else ("logits_s",)

    save_stats = w.backward  # forward-only scoring keeps no statistics

    def step():
        nonlocal fwd_out, bwd_out
        fwd_out = kd.forward(prob, t, ws_f, check=False, out=fwd_out, save_stats=save_stats)
        if w.backward:
            bwd_out = kd.backward(prob, t, fwd_out["stats"], want=want, workspace=ws_b,
                                  check=False, out=bwd_out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    kd.check_status(fwd_out["dev_status"])

    # per-section events (fused forward launch; backward recompute + dH/dW)
    # and, on the tensor-core path, one event pair per gradient-producer and
    # per backward GEMM launch
    n = args.steps
    plan = kd.kd_plan_info(prob.to_c())
    n_chunks = 0
    if w.backward and plan["path"] == 2 and w.student == "hidden":
        n_chunks = -(-w.n_tokens // plan["chunk_rows"]) * -(-w.vocab // plan["chunk_cols"])

    def new_events(k):
        return [torch.cuda.Event(enable_timing=True) for _ in range(k)]

    evs = [new_events(4) for _ in range(n)]
    lev = [(new_events(n_chunks), new_events(n_chunks), new_events(2 * n_chunks),
            new_events(2 * n_chunks)) for _ in range(n)]
    for e4 in evs + [e for grp in lev for e in grp]:
        for e in e4:
            e.record()  # materialise the handles
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_index = smi_index(local)
    launches0 = kd.kd_launch_count()
    with ClockSampler(gpu_index) as clk:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        start.record()
        for i in range(n):
            kd.kd_set_profile_events(*evs[i]) if w.backward else \
                kd.kd_set_profile_events(evs[i][0], evs[i][1])
            if n_chunks:
                kd.kd_set_profile_launch_events(0, lev[i][0], lev[i][1])
                kd.kd_set_profile_launch_events(1, lev[i][2], lev[i][3])
            step()
        stop.record()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    kd.kd_set_profile_events()
    kd.kd_set_profile_launch_events(0)
    kd.kd_set_profile_launch_events(1)
    launches = kd.kd_launch_count() - launches0
    ms = D.max_over_ranks(start.elapsed_time(stop), dev)
    ms_step = ms / n
    tokens = w.n_tokens * world
    value = tokens / (ms_step / 1e3)
    fwd_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][1]) for i in range(n))
    bwd_ms = statistics.mean(evs[i][2].elapsed_time(evs[i][3]) for i in range(n)) \
        if w.backward else 0.0
    # per-step device time (first forward event to the last event of the step)
    step_ms = [evs[i][0].elapsed_time(evs[i][3] if w.backward else evs[i][1]) for i in range(n)]
    step_ms_median = statistics.median(step_ms)

    peaks, peak_src = load_peaks()
    # a timed region under a second runs at the burst clock: the burst peak
    # applies; longer regions settle under the power cap (sustained peak)
    burst = ms < 1000.0
    f_fwd, f_bwd = flops_per_step(w)
    # kernel families of one step: device time per step, launches per step and
    # algorithmic work per step (FLOPs on the tensor-core path, HBM bytes on
    # the streaming path).  The roofline is reported for the largest family
    # on the caller's stream; the backward GEMMs run on a second stream,
    # concurrently with the next gradient chunk, so their event times include
    # waiting for SMs the producer holds (reported, never chosen).
    fams = {}
    side_stream = {"backward_gemm"}
    if f_fwd > 0:
        unit, scale = "TFLOP/s", 1e12
        peak = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
        bound = "tensor"
        psrc = (f"{peak_src} cuBLAS bf16 {'burst' if burst else 'sustained'} "
                f"(timed region {ms:.0f} ms {'<' if burst else '>='} 1 s)")
        fams["fused_forward"] = ("k_tc<EPI_FWD>: fused projections + online CE/KL", fwd_ms, 1, f_fwd)
        if n_chunks:
            def launch_ms(k0, k1, cnt):
                return statistics.mean(sum(lev[i][k0][j].elapsed_time(lev[i][k1][j])
                                           for j in range(cnt)) for i in range(n))
            fams["gradient_producer"] = ("k_tc<EPI_GRAD>: recomputed projections -> G chunk",
                                         launch_ms(0, 1, n_chunks), n_chunks, f_fwd)
            fams["backward_gemm"] = ("k_tc<EPI_GEMM>: dH = G W, dW = G^T H",
                                     launch_ms(2, 3, 2 * n_chunks), 2 * n_chunks, f_bwd - f_fwd)
    else:
        unit, scale, peak = "GB/s", 1e9, peaks["hbm_gbs"]
        bound, psrc = "hbm", f"{peak_src} copy bandwidth"
        b_fwd, b_bwd = bytes_per_step(w)
        fams["stream_forward"] = ("k_fwd: streamed logits -> online CE/KL", fwd_ms, 1, b_fwd)
        if w.backward:
            fams["stream_backward"] = ("k_bwd: streamed logits -> d z_s", bwd_ms, 1, b_bwd)
    dom = max((f for f in fams if f not in side_stream), key=lambda k: fams[k][1])
    name, k_ms, k_n, k_work = fams[dom]
    per_launch_ms = k_ms / k_n
    achieved = (k_work / k_n) / (per_launch_ms / 1e3) / scale
    # (captured at the workload's own size and variant only)
    traffic = (load_traffic().get(f"{w.name}:{dom}")
               if not args.tokens and not args.variant else None)
    step_work = (f_fwd + f_bwd) if bound == "tensor" else sum(bytes_per_step(w))
    step_achieved = step_work / (ms_step / 1e3) / scale
    roofline = {"bound": bound, "kernel": name, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "peak_source": psrc, "traffic": traffic,
                ("flops_per_launch" if bound == "tensor" else "bytes_per_launch"): k_work / k_n,
                "launch_ms": per_launch_ms, "launches_per_step": k_n,
                "step_achieved": step_achieved, "step_frac": step_achieved / peak}
    if bound == "tensor":
        roofline["step_frac_nominal"] = step_achieved / NOMINAL_BF16_TFLOPS
        roofline["nominal_peak_source"] = "dense bf16 tensor peak, 2250 TFLOP/s (GB300 nominal)"
    if dom == "gradient_producer":
        roofline["launch_note"] = ("live launch time: the backward GEMMs of the previous "
                                   "gradient chunk share the SMs on a second stream")
    sections = {f: {"ms_per_step": v[1], "launches": v[2],
                    "achieved": v[3] / (v[1] / 1e3) / scale if v[1] else None, "unit": unit,
                    **({"overlapped": True} if f in side_stream else {})}
                for f, v in fams.items()}
    if f_fwd > 0:
        sections["step_tflops"] = (f_fwd + f_bwd) / (ms_step / 1e3) / 1e12
    # the gradient producer again with the backward GEMMs on the caller's
    # stream (one stream): its launches then hold the GPU alone
    if n_chunks and not args.no_serialised:
        old_env = os.environ.get("KD_BWD_STREAMS")
        os.environ["KD_BWD_STREAMS"] = "1"
        try:
            for _ in range(2):
                step()
            ns = min(n, 10)
            torch.cuda.synchronize()
            for i in range(ns):
                kd.kd_set_profile_launch_events(0, lev[i][0], lev[i][1])
                step()
            torch.cuda.synchronize()
            kd.kd_set_profile_launch_events(0)
            ser_ms = statistics.mean(sum(lev[i][0][j].elapsed_time(lev[i][1][j])
                                         for j in range(n_chunks)) for i in range(ns)) / n_chunks
        finally:
            if old_env is None:
                os.environ.pop("KD_BWD_STREAMS", None)
            else:
                os.environ["KD_BWD_STREAMS"] = old_env
        ser = (f_fwd / n_chunks) / (ser_ms / 1e3) / 1e12
        sections["gradient_producer_serialised"] = {
            "launch_ms": ser_ms, "achieved": ser, "unit": "TFLOP/s", "frac": ser / peak,
            "note": "KD_BWD_STREAMS=1, outside the timed region"}
        if dom == "gradient_producer":
            roofline["launch_ms_serialised"] = ser_ms
            roofline["frac_serialised"] = ser / peak

    # end to end through the C ABI with host buffers: every step uploads all of
    # its inputs (hidden states, head weights, labels) from pinned host memory
    # and downloads its results (loss, gradients).  Copies run on their own
    # stream and overlap the neighbouring steps' compute: two device sets of
    # inputs and outputs, step i+1's inputs uploading and step i's results
    # downloading while step i computes.
    e2e = None
    if not args.no_e2e:
        host = {k: v.cpu().pin_memory() for k, v in t.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        sets = [{"t": t, "fo": fwd_out, "bo": bwd_out},
                {"t": {k: torch.empty_like(v) for k, v in t.items()}, "fo": None, "bo": None}]

        def results(st):
            return [st["fo"]["loss"]] + ([st["bo"][k] for k in st["bo"] if k.startswith("d_")]
                                         if w.backward else [])

        def step_on(st):
            st["fo"] = kd.forward(prob, st["t"], ws_f, check=False, out=st["fo"],
                                  save_stats=save_stats)
            if w.backward:
                st["bo"] = kd.backward(prob, st["t"], st["fo"]["stats"], want=want,
                                       workspace=ws_b, check=False, out=st["bo"])

        for st in sets:  # allocate both output sets
            step_on(st)
        torch.cuda.synchronize()
        res_host = [torch.empty_like(r, device="cpu").pin_memory() for r in results(sets[0])]
        d2h = sum(r.numel() * r.element_size() for r in results(sets[0]))
        comp, copy = torch.cuda.current_stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        up, done, down = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def upload(i):
            with torch.cuda.stream(copy):
                for k, v in host.items():
                    sets[i % 2]["t"][k].copy_(v, non_blocking=True)
                up[i % 2].record(copy)

        def run(nsteps, start=None):
            if start is not None:
                copy.wait_event(start)  # the first upload is inside the timed region
            upload(0)
            for i in range(nsteps):
                sb = i % 2
                comp.wait_event(up[sb])
                if i >= 2:
                    comp.wait_event(down[sb])  # step i-2's results are read
                step_on(sets[sb])
                done[sb].record(comp)
                with torch.cuda.stream(copy):
                    if i + 1 < nsteps:  # set 1-sb is free once step i-1 is done
                        if i >= 1:
                            copy.wait_event(done[1 - sb])
                        upload(i + 1)
                    copy.wait_event(done[sb])
                    for r_h, r_d in zip(res_host, results(sets[sb])):
                        r_h.copy_(r_d, non_blocking=True)
                    down[sb].record(copy)
            comp.wait_event(down[(nsteps - 1) % 2])

        run(args.warmup)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ne = max(3, n)  # the same number of timed steps as the device-resident value
        s2.record(comp)
        run(ne, s2)
        e2.record(comp)
        torch.cuda.synchronize()
        ms_e = D.max_over_ranks(s2.elapsed_time(e2), dev)
        e2e = {"value": tokens / (ms_e / ne / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e / ne, "steps": ne,
               "copies": "own stream, overlapping neighbouring steps"}

    peak_gib = torch.cuda.max_memory_allocated(dev) / 2 ** 30
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # a probe sizes the sample to about --cpu-seconds of oracle work
        probe = min(64, w.n_tokens)
        v_probe, _ = time_oracle(w, probe, 1, 0, 13)
        rows = int(min(w.n_tokens, max(probe, args.cpu_seconds * v_probe)))
        if args.cpu_rows > 0:
            rows = min(args.cpu_rows, w.n_tokens)
        v_cpu, dt = time_oracle(w, rows, 1, 0, 11)
        cpu_base = {"value": v_cpu, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                    "sample": f"{rows} seeded random tokens of the {w.name} workload, fwd+bwd, "
                              f"fp64 numpy oracle ({dt:.1f} s)"}

    in_bytes = sum(v.numel() * v.element_size() for v in t.values())
    if rank == 0:
        metric = ("fused linear+CE+KD fwd+bwd tokens/s" if w.backward else
                  "fused linear+CE+KD forward-only scoring tokens/s")
        line = {
            "metric": metric, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": n, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_median": step_ms_median,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "tokens_per_gpu": w.n_tokens, "vocab": w.vocab,
                       "d_student": w.d_student, "d_teacher": w.d_teacher,
                       "variant": w.variant, "teacher": w.teacher,
                       "parallelism": f"dp{world}",
                       "l2": "inputs larger than L2" if in_bytes > L2_BYTES else "L2 not flushed"},
            "roofline": roofline, "sections": sections,
            "peak_hbm_gib": peak_gib, "cpu_baseline": cpu_base, "e2e": e2e,
            "clocks": clk.summary(), "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
