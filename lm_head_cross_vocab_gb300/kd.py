"""Thin Python binding of the ``kd.h`` C ABI (argument marshalling only).

Every step of the loss runs inside ``libkdgb.so``; this module only turns
PyTorch tensors into device pointers, allocates outputs / workspace with the
PyTorch caching allocator and passes the current CUDA stream.  There is no
fallback: if the library is missing or the device is not an sm_103 GPU the
calls raise.

Low-level names mirror the ABI one to one: ``kd_workspace_size``, ``kd_fwd``,
``kd_bwd``, ``kd_status_string``, ``kd_device_supported``, ``kd_abi_version``,
``kd_diag_gemm_bf16``.  ``forward`` / ``backward`` are conveniences that build
the structs from keyword arguments and tensors.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkdgb.so")

# ---------------------------------------------------------------- enums
KD_OK, KD_ERR_INVALID_ARG, KD_ERR_UNSUPPORTED, KD_ERR_WORKSPACE = 0, 1, 2, 3
KD_ERR_BAD_LABEL, KD_ERR_BAD_TOPK, KD_ERR_TIMEOUT, KD_ERR_CUDA, KD_ERR_NO_DEVICE = 4, 5, 6, 7, 8
KD_DEV_BAD_LABEL, KD_DEV_BAD_TOPK, KD_DEV_TIMEOUT, KD_DEV_BAD_MAP = 0x1, 0x2, 0x4, 0x8
KD_DEV_MAP_UNSUPPORTED = 0x10
KD_BF16, KD_FP32 = 0, 1
KD_STUDENT_HIDDEN, KD_STUDENT_LOGITS = 0, 1
KD_TEACHER_NONE, KD_TEACHER_TIED, KD_TEACHER_SEPARATE, KD_TEACHER_LOGITS, KD_TEACHER_TOPK = range(5)
KD_TEACHER_PROJECTED = 5
KD_KL_FORWARD, KD_KL_REVERSE, KD_KL_JEFFREYS, KD_KL_SKEW_JS = range(4)
KD_KL_SKEW_FORWARD, KD_KL_SKEW_REVERSE = 4, 5
KD_REDUCE_MEAN, KD_REDUCE_SUM = 0, 1
KD_STATS_PER_TOKEN = 8
KD_STATIC_SCRATCH_BYTES = 32 << 20
KD_ABI_VERSION = 5  # the kd.h this binding follows

DTYPES = {"bf16": KD_BF16, "fp32": KD_FP32}
STUDENTS = {"hidden": KD_STUDENT_HIDDEN, "logits": KD_STUDENT_LOGITS}
TEACHERS = {"none": KD_TEACHER_NONE, "tied": KD_TEACHER_TIED, "separate": KD_TEACHER_SEPARATE,
            "logits": KD_TEACHER_LOGITS, "topk": KD_TEACHER_TOPK,
            "projected": KD_TEACHER_PROJECTED}
VARIANTS = {"forward": KD_KL_FORWARD, "reverse": KD_KL_REVERSE, "jeffreys": KD_KL_JEFFREYS,
            "skew_js": KD_KL_SKEW_JS, "skew_forward": KD_KL_SKEW_FORWARD,
            "skew_reverse": KD_KL_SKEW_REVERSE}
REDUCTIONS = {"mean": KD_REDUCE_MEAN, "sum": KD_REDUCE_SUM}


class kd_problem(ctypes.Structure):
    _fields_ = [
        ("n_tokens", ctypes.c_int64), ("vocab", ctypes.c_int64), ("d_student", ctypes.c_int64),
        ("d_teacher", ctypes.c_int64), ("topk", ctypes.c_int64),
        ("dtype", ctypes.c_int32), ("student", ctypes.c_int32), ("teacher", ctypes.c_int32),
        ("variant", ctypes.c_int32), ("reduction", ctypes.c_int32),
        ("t_student", ctypes.c_float), ("t_teacher", ctypes.c_float),
        ("w_student_ce", ctypes.c_float), ("w_teacher_ce", ctypes.c_float),
        ("w_kl", ctypes.c_float), ("beta", ctypes.c_float),
        ("ignore_index", ctypes.c_int64), ("num_batch_labels", ctypes.c_int64),
        ("assume_valid_labels", ctypes.c_int32), ("teacher_grads", ctypes.c_int32),
        ("vocab_chunk", ctypes.c_int64), ("seq_chunk", ctypes.c_int64),
        ("vocab_teacher", ctypes.c_int64),
    ]


class kd_inputs(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("h_s", "w_s", "logits_s", "h_t", "w_t", "logits_t", "labels", "topk_idx",
                 "topk_p", "token_map")]


class KDError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {kd_status_string(status)} (status {status})")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libkdgb.so (built by ``lm_head_cross_vocab_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I, vp = ctypes.POINTER(kd_problem), ctypes.POINTER(kd_inputs), ctypes.c_void_p
    sz = ctypes.POINTER(ctypes.c_size_t)
    lib.kd_workspace_size.argtypes = [P, sz, sz]
    lib.kd_fwd.argtypes = [P, I, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.kd_bwd.argtypes = [P, I, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, ctypes.c_size_t,
                           vp]
    lib.kd_status_string.argtypes = [ctypes.c_int]
    lib.kd_status_string.restype = ctypes.c_char_p
    lib.kd_device_supported.argtypes = [ctypes.c_int]
    lib.kd_diag_gemm_bf16.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64, ctypes.c_int, vp]
    lib.kd_set_profile_events.argtypes = [vp, vp, vp, vp]
    lib.kd_set_profile_launch_events.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int]
    lib.kd_plan_info.argtypes = [P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
    lib.kd_fwd_static_scratch.argtypes = [P, I, vp, vp, vp, vp, vp, vp, vp]
    lib.kd_project_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64, sz]
    lib.kd_project_teacher_logits.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp,
                                              ctypes.c_int64, ctypes.c_int32, ctypes.c_float, vp,
                                              ctypes.c_int32, vp, vp, ctypes.c_size_t, vp]
    lib.kd_mix_teacher_logits.argtypes = [vp, ctypes.c_int32, vp, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int32, ctypes.c_int32, vp, ctypes.c_int32, vp,
                                          vp]
    lib.kd_bwd_grads.argtypes = [P, I, vp, vp, ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp]
    lib.kd_launch_count.restype = ctypes.c_uint64
    for f in ("kd_workspace_size", "kd_fwd", "kd_bwd", "kd_device_supported", "kd_abi_version",
              "kd_diag_gemm_bf16", "kd_set_profile_events", "kd_set_profile_launch_events",
              "kd_fwd_static_scratch", "kd_project_workspace_size", "kd_project_teacher_logits",
              "kd_plan_info", "kd_mix_teacher_logits", "kd_bwd_grads"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


# ---------------------------------------------------------------- raw ABI

def kd_status_string(status: int) -> str:
    return load_library().kd_status_string(int(status)).decode()


def kd_device_supported(device: int = 0) -> bool:
    return bool(load_library().kd_device_supported(int(device)))


def kd_abi_version() -> int:
    return int(load_library().kd_abi_version())


def kd_workspace_size(problem: kd_problem):
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = load_library().kd_workspace_size(ctypes.byref(problem), ctypes.byref(f), ctypes.byref(b))
    if st != KD_OK:
        raise KDError(st, "kd_workspace_size")
    return int(f.value), int(b.value)


def kd_fwd(problem, inputs, ce_s, ce_t, kl, stats, loss, dev_status, workspace, ws_bytes, stream):
    return int(load_library().kd_fwd(ctypes.byref(problem), ctypes.byref(inputs), ce_s, ce_t, kl,
                                     stats, loss, dev_status, workspace, ws_bytes, stream))


def kd_fwd_static_scratch(problem, inputs, ce_s, ce_t, kl, stats, loss, dev_status, stream):
    return int(load_library().kd_fwd_static_scratch(ctypes.byref(problem), ctypes.byref(inputs),
                                                    ce_s, ce_t, kl, stats, loss, dev_status,
                                                    stream))


def kd_bwd(problem, inputs, stats, d_loss, grad_scale, d_h_s, d_w_s, d_logits_s, dev_status,
           workspace, ws_bytes, stream):
    return int(load_library().kd_bwd(ctypes.byref(problem), ctypes.byref(inputs), stats, d_loss,
                                     ctypes.c_float(grad_scale), d_h_s, d_w_s, d_logits_s,
                                     dev_status, workspace, ws_bytes, stream))


def kd_diag_gemm_bf16(a: torch.Tensor, b: torch.Tensor, a_kmajor: bool = True,
                      b_kmajor: bool = True) -> torch.Tensor:
    """C = A B^T on the library's tcgen05 GEMM core (diagnostic).  `a` is A
    [M, K] (a_kmajor) or A^T stored [K, M]; `b` is B [N, K] or B^T stored [K, N]."""
    assert a.dtype == torch.bfloat16 and b.dtype == torch.bfloat16 and a.is_contiguous() \
        and b.is_contiguous()
    m, ka = (a.shape[0], a.shape[1]) if a_kmajor else (a.shape[1], a.shape[0])
    n, kb = (b.shape[0], b.shape[1]) if b_kmajor else (b.shape[1], b.shape[0])
    assert ka == kb
    c = torch.empty(m, n, device=a.device, dtype=torch.float32)
    layout = (0 if a_kmajor else 1) | (0 if b_kmajor else 2)
    st = load_library().kd_diag_gemm_bf16(a.data_ptr(), b.data_ptr(), c.data_ptr(), m, n, ka,
                                          layout, _stream(a.device))
    if st != KD_OK:
        raise KDError(st, "kd_diag_gemm_bf16")
    return c


def kd_set_profile_events(fwd_start=None, fwd_stop=None, bwd_start=None, bwd_stop=None):
    """Record torch.cuda.Event objects around the fused forward / backward sections."""
    h = [None if e is None else e.cuda_event for e in (fwd_start, fwd_stop, bwd_start, bwd_stop)]
    st = load_library().kd_set_profile_events(*h)
    if st != KD_OK:
        raise KDError(st, "kd_set_profile_events")


_launch_event_arrays = {}  # kind -> (starts, stops, events): kept alive while set


def kd_set_profile_launch_events(kind: int, starts=(), stops=()):
    """Record torch.cuda.Event pairs around each gradient-producer launch (kind
    0) or backward GEMM launch (kind 1) of later kd_bwd calls; () stops."""
    starts, stops = list(starts), list(stops)
    assert len(starts) == len(stops)
    n = len(starts)
    arr_s = (ctypes.c_void_p * max(n, 1))(*[e.cuda_event for e in starts])
    arr_t = (ctypes.c_void_p * max(n, 1))(*[e.cuda_event for e in stops])
    st = load_library().kd_set_profile_launch_events(kind, ctypes.addressof(arr_s),
                                                     ctypes.addressof(arr_t), n)
    if st != KD_OK:
        raise KDError(st, "kd_set_profile_launch_events")
    if n:
        _launch_event_arrays[kind] = (arr_s, arr_t, starts + stops)
    else:
        _launch_event_arrays.pop(kind, None)


def kd_plan_info(problem: kd_problem) -> dict:
    path, splits = ctypes.c_int32(0), ctypes.c_int32(0)
    rows, cols = ctypes.c_int64(0), ctypes.c_int64(0)
    st = load_library().kd_plan_info(ctypes.byref(problem), ctypes.byref(path), ctypes.byref(splits),
                                     ctypes.byref(rows), ctypes.byref(cols))
    if st != KD_OK:
        raise KDError(st, "kd_plan_info")
    return {"path": path.value, "vocab_splits": splits.value, "chunk_rows": rows.value,
            "chunk_cols": cols.value}


def kd_launch_count() -> int:
    return int(load_library().kd_launch_count())


# ---------------------------------------------------------------- helpers

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


@dataclasses.dataclass
class Problem:
    """Keyword form of ``kd_problem`` (orda-kernel style parameter names)."""

    n_tokens: int
    vocab: int
    d_student: int = 0
    d_teacher: int = 0
    topk: int = 0
    dtype: str = "bf16"
    student: str = "hidden"
    teacher: str = "tied"
    variant: str = "forward"
    reduction: str = "mean"
    t_student: float = 1.0
    t_teacher: Optional[float] = None
    w_student_ce: float = 1.0
    w_teacher_ce: float = 0.0
    w_kl: float = 1.0
    beta: float = 0.5
    ignore_index: int = -100
    num_batch_labels: int = 0
    assume_valid_labels: bool = False
    vocab_chunk: int = 0
    seq_chunk: int = 0
    teacher_grads: bool = False  # the backward may be asked for d_h_t / d_w_t
    vocab_teacher: int = 0       # V_t of a "projected" teacher (token map over V_t ids)

    def to_c(self) -> kd_problem:
        p = kd_problem()
        p.n_tokens, p.vocab = self.n_tokens, self.vocab
        p.d_student, p.d_teacher, p.topk = self.d_student, self.d_teacher, self.topk
        p.dtype, p.student = DTYPES[self.dtype], STUDENTS[self.student]
        p.teacher, p.variant = TEACHERS[self.teacher], VARIANTS[self.variant]
        p.reduction = REDUCTIONS[self.reduction]
        p.t_student = self.t_student
        p.t_teacher = self.t_student if self.t_teacher is None else self.t_teacher
        p.w_student_ce, p.w_teacher_ce, p.w_kl = self.w_student_ce, self.w_teacher_ce, self.w_kl
        p.beta, p.ignore_index = self.beta, self.ignore_index
        p.num_batch_labels = self.num_batch_labels
        p.assume_valid_labels = int(self.assume_valid_labels)
        p.teacher_grads = int(self.teacher_grads)
        p.vocab_chunk, p.seq_chunk = self.vocab_chunk, self.seq_chunk
        p.vocab_teacher = self.vocab_teacher
        return p


class kd_grads(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("d_h_s", "d_w_s", "d_logits_s", "d_h_t", "d_w_t")]


def make_inputs(t: dict) -> kd_inputs:
    i = kd_inputs()
    for k in ("h_s", "w_s", "logits_s", "h_t", "w_t", "logits_t", "labels", "topk_idx", "topk_p",
              "token_map"):
        v = t.get(k)
        if v is not None:
            assert v.is_cuda and v.is_contiguous(), f"{k} must be a contiguous CUDA tensor"
        setattr(i, k, _ptr(v))
    return i


def _device_of(t: dict):
    for v in t.values():
        if v is not None:
            return v.device
    return torch.device("cuda")


class Workspace:
    """Reusable device workspace (PyTorch allocation, 256-byte aligned)."""

    def __init__(self):
        self.buf = None

    def get(self, nbytes: int, device):
        if self.buf is None or self.buf.numel() < nbytes + 256 or self.buf.device != device:
            self.buf = None
            self.buf = torch.empty(max(nbytes, 1) + 256, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        return (base + 255) // 256 * 256, nbytes


def check_status(dev_status: torch.Tensor, assume_valid: bool = False):
    s = int(dev_status.item())
    if s & KD_DEV_TIMEOUT:
        raise KDError(KD_ERR_TIMEOUT, "device")
    if s & KD_DEV_MAP_UNSUPPORTED:
        raise KDError(KD_ERR_UNSUPPORTED, "token map too skewed for the fused projected teacher")
    if s & KD_DEV_BAD_MAP:
        raise KDError(KD_ERR_INVALID_ARG, "token map entry outside [-1, V_student)")
    if not assume_valid:
        if s & KD_DEV_BAD_LABEL:
            raise KDError(KD_ERR_BAD_LABEL, "device")
        if s & KD_DEV_BAD_TOPK:
            raise KDError(KD_ERR_BAD_TOPK, "device")


def forward(problem: Problem, tensors: dict, workspace: Optional[Workspace] = None,
            check: bool = True, out: Optional[dict] = None, save_stats: bool = True):
    """Run kd_fwd; returns dict(ce_s, ce_t, kl, stats, loss, dev_status).

    save_stats=False is forward-only scoring (flash_kd API doc: only the
    forward pass exists, scoring runs without gradients): no per-token
    statistics are kept for a backward, and ``stats`` is None."""
    dev = _device_of(tensors)
    n = problem.n_tokens
    if out is None:
        out = {
            "ce_s": torch.empty(n, device=dev, dtype=torch.float32),
            "ce_t": torch.empty(n, device=dev, dtype=torch.float32),
            "kl": torch.empty(n, device=dev, dtype=torch.float32),
            "stats": (torch.empty(n, KD_STATS_PER_TOKEN, device=dev, dtype=torch.float32)
                      if save_stats else None),
            "loss": torch.empty((), device=dev, dtype=torch.float32),
            "dev_status": torch.zeros((), device=dev, dtype=torch.int32),
        }
    cp = problem.to_c()
    fb, _ = kd_workspace_size(cp)
    ws = workspace or Workspace()
    wptr, wbytes = ws.get(fb, dev)
    st = kd_fwd(cp, make_inputs(tensors), _ptr(out["ce_s"]), _ptr(out["ce_t"]), _ptr(out["kl"]),
                _ptr(out["stats"]), _ptr(out["loss"]), _ptr(out["dev_status"]), wptr, wbytes,
                _stream(dev))
    if st != KD_OK:
        raise KDError(st, "kd_fwd")
    if check:
        check_status(out["dev_status"], problem.assume_valid_labels)
    return out


def backward(problem: Problem, tensors: dict, stats: torch.Tensor, *, d_loss=None,
             grad_scale: float = 1.0, want=("h_s", "w_s", "logits_s"),
             workspace: Optional[Workspace] = None, check: bool = True,
             out: Optional[dict] = None):
    """Run kd_bwd; returns dict of the requested gradients (+ dev_status)."""
    dev = _device_of(tensors)
    if out is None:
        out = {"dev_status": torch.zeros((), device=dev, dtype=torch.int32)}
        for k in want:
            src = tensors.get(k)
            if src is not None:
                out["d_" + k] = torch.empty_like(src)
    cp = problem.to_c()
    _, bb = kd_workspace_size(cp)
    ws = workspace or Workspace()
    wptr, wbytes = ws.get(bb, dev)
    if out.get("d_h_t") is None and out.get("d_w_t") is None:
        st = kd_bwd(cp, make_inputs(tensors), _ptr(stats), _ptr(d_loss), grad_scale,
                    _ptr(out.get("d_h_s")), _ptr(out.get("d_w_s")), _ptr(out.get("d_logits_s")),
                    _ptr(out["dev_status"]), wptr, wbytes, _stream(dev))
        name = "kd_bwd"
    else:
        g = kd_grads(*[_ptr(out.get(k)) for k in ("d_h_s", "d_w_s", "d_logits_s", "d_h_t",
                                                   "d_w_t")])
        st = load_library().kd_bwd_grads(ctypes.byref(cp), ctypes.byref(make_inputs(tensors)),
                                         _ptr(stats), _ptr(d_loss), ctypes.c_float(grad_scale),
                                         ctypes.byref(g), _ptr(out["dev_status"]), wptr, wbytes,
                                         _stream(dev))
        name = "kd_bwd_grads"
    if st != KD_OK:
        raise KDError(st, name)
    if check:
        check_status(out["dev_status"], problem.assume_valid_labels)
    return out


def problem_for(w, **overrides) -> Problem:
    """Problem matching a synthetic workload description (inputs.Workload)."""
    kw = dict(n_tokens=w.n_tokens, vocab=w.vocab, d_student=w.d_student, d_teacher=w.d_teacher,
              topk=w.topk, dtype=w.dtype, student=w.student, teacher=w.teacher,
              variant=w.variant, t_student=w.t_student, t_teacher=w.t_teacher,
              w_student_ce=w.w_student_ce, w_teacher_ce=w.w_teacher_ce, w_kl=w.w_kl, beta=w.beta,
              ignore_index=w.ignore_index, vocab_chunk=w.vocab_chunk, seq_chunk=w.seq_chunk)
    kw.update(overrides)
    return Problem(**kw)


# ---------------------------------------------------------------- cross-vocabulary

def build_exact_token_map(student_vocab, teacher_vocab) -> torch.Tensor:
    """Token map for kd_project_teacher_logits: entry j is the student id of the
    teacher token string teacher_vocab[j], or -1 when the student vocabulary has
    no identical string (orda-kernel README, "Cross-vocabulary distillation":
    build_exact_token_map).  Vocabularies are sequences of token strings indexed
    by id; a string listed twice in the student vocabulary maps to its first id.
    Host-side preparation of a constant input (int32 CPU tensor)."""
    first = {}
    for i, tok in enumerate(student_vocab):
        first.setdefault(tok, i)
    return torch.tensor([first.get(tok, -1) for tok in teacher_vocab], dtype=torch.int32)


def project_teacher_logits(token_map: torch.Tensor, logits_t: torch.Tensor, v_student: int,
                           temperature: float = 1.0, out_dtype=None,
                           workspace: Optional[Workspace] = None, check: bool = True):
    """kd_project_teacher_logits: teacher logits [N, V_t] -> student-vocabulary
    logits [N, V_s] (tempered; unmatched ids at the dtype's most negative value)."""
    dev = logits_t.device
    dtype = logits_t.dtype if out_dtype is None else out_dtype
    tm = token_map.to(device=dev, dtype=torch.int32).contiguous()
    zt = logits_t.contiguous()
    n, vt = zt.shape
    assert tm.numel() == vt
    out = torch.empty(n, v_student, device=dev, dtype=dtype)
    dev_status = torch.zeros(1, device=dev, dtype=torch.int32)
    nbytes = ctypes.c_size_t(0)
    lib = load_library()
    st = lib.kd_project_workspace_size(vt, v_student, ctypes.byref(nbytes))
    if st != KD_OK:
        raise KDError(st, "kd_project_workspace_size")
    ws = workspace or Workspace()
    wptr, wbytes = ws.get(nbytes.value, dev)
    dt = {torch.bfloat16: KD_BF16, torch.float32: KD_FP32}
    st = lib.kd_project_teacher_logits(tm.data_ptr(), vt, v_student, zt.data_ptr(), n,
                                       dt[zt.dtype], float(temperature), out.data_ptr(),
                                       dt[dtype], dev_status.data_ptr(), wptr, wbytes,
                                       _stream(dev))
    if st != KD_OK:
        raise KDError(st, "kd_project_teacher_logits")
    if check and int(dev_status.item()) & KD_DEV_BAD_MAP:
        raise KDError(KD_ERR_INVALID_ARG, "token map entry outside [-1, V_student)")
    return out


KD_MIX_ARITHMETIC, KD_MIX_GEOMETRIC = 0, 1
KD_MIX_MAX_TEACHERS = 8
MIX_MODES = {"arithmetic": KD_MIX_ARITHMETIC, "geometric": KD_MIX_GEOMETRIC}


def mix_teacher_logits(logits, weights=None, mode: str = "arithmetic", out_dtype=None,
                       check: bool = True):
    """kd_mix_teacher_logits: K teacher logit tensors [N, V] (same device, dtype
    and shape) -> the mixture's log-probabilities [N, V] (probability average
    or product of experts; weights normalised, uniform when None)."""
    zs = [z.contiguous() for z in logits]
    if not zs or len(zs) > KD_MIX_MAX_TEACHERS:
        raise ValueError(f"1..{KD_MIX_MAX_TEACHERS} teachers")
    z0 = zs[0]
    if any(z.shape != z0.shape or z.dtype != z0.dtype or z.device != z0.device for z in zs):
        raise ValueError("teachers must share shape, dtype and device")
    n, v = z0.shape
    dev = z0.device
    dtype = z0.dtype if out_dtype is None else out_dtype
    out = torch.empty(n, v, device=dev, dtype=dtype)
    ptrs = (ctypes.c_void_p * len(zs))(*[z.data_ptr() for z in zs])
    w = None
    if weights is not None:
        w = (ctypes.c_float * len(zs))(*[float(x) for x in weights])
        if len(weights) != len(zs):
            raise ValueError("one weight per teacher")
    dev_status = torch.zeros(1, device=dev, dtype=torch.int32)
    dt = {torch.bfloat16: KD_BF16, torch.float32: KD_FP32}
    st = load_library().kd_mix_teacher_logits(ptrs, len(zs), w, n, v, dt[z0.dtype],
                                              MIX_MODES[mode], out.data_ptr(), dt[dtype],
                                              dev_status.data_ptr(), _stream(dev))
    if st != KD_OK:
        raise KDError(st, "kd_mix_teacher_logits")
    if check and int(dev_status.item()) & KD_DEV_TIMEOUT:
        raise KDError(KD_ERR_TIMEOUT, "a bounded wait timed out")
    return out
