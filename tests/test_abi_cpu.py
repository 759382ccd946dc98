"""CPU-side checks of the C ABI: the library loads, exports every symbol that
include/kd.h declares, the ctypes structs match the C layout, and host-side
validation / planning behave (no kernel is launched on this machine)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kd.h")


@pytest.fixture(scope="session")
def kd():
    from lm_head_cross_vocab_gb300 import build, kd as K
    build.build()
    K.load_library()
    return K


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:kd_status|const char\*|int)\s+(kd_\w+)\s*\(", src,
                                 flags=re.M)))


def test_header_declares_the_api():
    names = _declared_functions()
    for f in ("kd_workspace_size", "kd_fwd", "kd_bwd", "kd_status_string", "kd_device_supported",
              "kd_abi_version", "kd_diag_gemm_bf16"):
        assert f in names


def test_library_exports_every_declared_symbol(kd):
    lib = kd.load_library()
    out = subprocess.run(["nm", "-D", "--defined-only", kd.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (kd_\w+)", out))
    for f in _declared_functions():
        assert f in exported, f
        assert hasattr(lib, f)


def test_abi_version_and_status_strings(kd):
    assert kd.kd_abi_version() == kd.KD_ABI_VERSION == 5
    for code in range(9):
        s = kd.kd_status_string(code)
        assert s and s != "unknown status"
    assert kd.kd_status_string(99) == "unknown status"


def test_ctypes_struct_layout_matches_c(kd, tmp_path):
    """Compile a tiny C probe of sizeof/offsetof against kd.h and compare."""
    fields = [f for f, _ in kd.kd_problem._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "kd.h"', "int main(void){",
            'printf("%zu\\n", sizeof(kd_problem));',
            'printf("%zu\\n", sizeof(kd_inputs));']
    prog += [f'printf("%zu\\n", offsetof(kd_problem, {f}));' for f in fields]
    prog += ["return 0;}"]
    c = tmp_path / "probe.c"
    c.write_text("\n".join(prog))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(c), "-o",
                    str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(kd.kd_problem)
    assert vals[1] == ctypes.sizeof(kd.kd_inputs)
    for f, off in zip(fields, vals[2:]):
        assert getattr(kd.kd_problem, f).offset == off, f


def _prob(kd, **kw):
    base = dict(n_tokens=64, vocab=512, d_student=64, dtype="fp32", teacher="tied",
                t_student=2.0, w_teacher_ce=1.0)
    base.update(kw)
    return kd.Problem(**base).to_c()


@pytest.mark.parametrize("bad", [
    dict(n_tokens=-1), dict(vocab=0), dict(t_student=0.0), dict(t_student=float("nan")),
    dict(w_kl=-1.0), dict(w_student_ce=float("inf")), dict(variant="skew_js", beta=1.0),
    dict(variant="skew_js", beta=0.0), dict(student="logits", teacher="tied"),
    dict(d_student=0), dict(teacher="separate", d_teacher=0),
    dict(teacher="topk", topk=0, w_teacher_ce=0.0),
    dict(teacher="topk", topk=2000, w_teacher_ce=0.0),
    dict(teacher="none", w_teacher_ce=1.0), dict(teacher="tied", d_teacher=32),
])
def test_invalid_problems_are_rejected_synchronously(kd, bad):
    p = _prob(kd, **bad)
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = kd.load_library().kd_workspace_size(ctypes.byref(p), ctypes.byref(f), ctypes.byref(b))
    assert st == kd.KD_ERR_INVALID_ARG


def test_unsupported_combinations(kd):
    lib = kd.load_library()
    f = ctypes.c_size_t(0)
    # bf16 tensor-core path needs 16-byte row pitches (D multiple of 8)
    p = _prob(kd, dtype="bf16", d_student=60)
    assert lib.kd_workspace_size(ctypes.byref(p), ctypes.byref(f), None) == kd.KD_ERR_UNSUPPORTED
    # top-K teachers carry no logits for a teacher CE
    p = _prob(kd, teacher="topk", topk=4, w_teacher_ce=1.0)
    assert lib.kd_workspace_size(ctypes.byref(p), ctypes.byref(f), None) == kd.KD_ERR_UNSUPPORTED


def test_projected_teacher_argument_rules(kd):
    """KD_TEACHER_PROJECTED (orda-kernel README, "Cross-vocabulary distillation"):
    the teacher vocabulary size is required, the student must arrive as logits,
    and the token map and teacher logits are required inputs."""
    lib = kd.load_library()
    f, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    base = dict(student="logits", teacher="projected", d_student=0, vocab=5000)
    p = _prob(kd, **base, vocab_teacher=7000)
    assert lib.kd_workspace_size(ctypes.byref(p), ctypes.byref(f), ctypes.byref(b)) == kd.KD_OK
    assert f.value > 0 and b.value > 0
    p = _prob(kd, **base, vocab_teacher=0)
    assert lib.kd_workspace_size(ctypes.byref(p), ctypes.byref(f), None) == kd.KD_ERR_INVALID_ARG
    p = _prob(kd, teacher="projected", vocab_teacher=7000)  # hidden student
    assert lib.kd_workspace_size(ctypes.byref(p), ctypes.byref(f), None) == kd.KD_ERR_UNSUPPORTED
    # a teacher row that would need more than 8 CTAs of the fused kernel
    p = _prob(kd, **base, vocab_teacher=1 << 22)
    assert lib.kd_workspace_size(ctypes.byref(p), ctypes.byref(f), None) == kd.KD_ERR_UNSUPPORTED
    fake = 1 << 20
    p = _prob(kd, **base, vocab_teacher=7000)
    ins = kd.kd_inputs(logits_s=fake, logits_t=fake, labels=fake)  # no token map
    st = lib.kd_fwd(ctypes.byref(p), ctypes.byref(ins), None, None, None, None, None, None, None,
                    0, None)
    assert st == kd.KD_ERR_INVALID_ARG


def test_null_inputs_and_workspace_errors(kd):
    lib = kd.load_library()
    p = _prob(kd)
    ins = kd.kd_inputs()  # all NULL
    st = lib.kd_fwd(ctypes.byref(p), ctypes.byref(ins), None, None, None, None, None, None, None,
                    0, None)
    assert st == kd.KD_ERR_INVALID_ARG
    # well-formed pointers (never dereferenced on the host) but no workspace
    fake = 1 << 20
    ins = kd.kd_inputs(h_s=fake, w_s=fake, h_t=fake, labels=fake)
    st = lib.kd_fwd(ctypes.byref(p), ctypes.byref(ins), None, None, None, None, None, None, None,
                    0, None)
    assert st == kd.KD_ERR_WORKSPACE
    # CE weights without labels
    ins = kd.kd_inputs(h_s=fake, w_s=fake, h_t=fake)
    st = lib.kd_fwd(ctypes.byref(p), ctypes.byref(ins), None, None, None, None, None, None, None,
                    0, None)
    assert st == kd.KD_ERR_INVALID_ARG


def test_backward_argument_rules(kd):
    lib = kd.load_library()
    fake = 1 << 20
    p = _prob(kd)
    ins = kd.kd_inputs(h_s=fake, w_s=fake, h_t=fake, labels=fake)
    # d_logits_s makes no sense for a hidden-state student
    st = lib.kd_bwd(ctypes.byref(p), ctypes.byref(ins), fake, None, ctypes.c_float(1.0), None,
                    None, fake, None, fake, 1 << 30, None)
    assert st == kd.KD_ERR_INVALID_ARG
    st = lib.kd_bwd(ctypes.byref(p), ctypes.byref(ins), fake, None, ctypes.c_float(float("nan")),
                    fake, None, None, None, fake, 1 << 30, None)
    assert st == kd.KD_ERR_INVALID_ARG


def test_no_scratch_buffer_spans_tokens_by_vocab(kd):
    """The backward's gradient chunk is at most a quarter of the (tokens x vocab)
    matrix for every workload (its two bf16 buffers together at most half a bf16
    logits matrix), and the forward never holds logits at all."""
    from lm_head_cross_vocab_gb300 import inputs as I
    for cfg in (1, 2, 3, 4, 5):
        w = I.WORKLOADS[cfg]
        p = kd.problem_for(w, vocab_chunk=0, seq_chunk=0).to_c()
        info = kd.kd_plan_info(p)
        fb, bb = kd.kd_workspace_size(p)
        full = w.n_tokens * w.vocab
        if info["path"] != 0:  # streaming path keeps no chunk
            assert info["chunk_rows"] * info["chunk_cols"] <= max(full // 4, 128 * 256), (cfg, info)
        assert fb < full * 2, (cfg, fb)


def test_device_query_without_gpu(kd):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    assert kd.kd_device_supported(0) is False


def test_mix_argument_rules(kd):
    """kd_mix_teacher_logits rejects bad arguments synchronously (before any
    device work); well-formed calls reach the device check."""
    lib = kd.load_library()
    fake = 1 << 20
    ptrs = (ctypes.c_void_p * 9)(*([fake] * 9))

    def call(k=2, weights=(1.0, 1.0), n=4, v=10, din=kd.KD_BF16, mode=kd.KD_MIX_ARITHMETIC,
             dout=kd.KD_FP32, out=fake):
        w = None if weights is None else (ctypes.c_float * len(weights))(*weights)
        return lib.kd_mix_teacher_logits(ptrs, k, w, n, v, din, mode, out, dout, None, None)

    bad = [dict(k=0), dict(k=9, weights=None), dict(weights=(1.0, -1.0)), dict(weights=(0.0, 0.0)),
           dict(weights=(1.0, float("nan"))), dict(v=0), dict(n=-1), dict(din=7), dict(dout=7),
           dict(mode=2), dict(out=None)]
    for kw in bad:
        assert call(**kw) == kd.KD_ERR_INVALID_ARG, kw
    for kw in (dict(), dict(weights=None), dict(weights=(0.0, 2.0), mode=kd.KD_MIX_GEOMETRIC),
               dict(k=8, weights=None)):
        assert call(**kw) == kd.KD_ERR_NO_DEVICE, kw


def test_teacher_grads_argument_rules(kd):
    """kd_bwd_grads: teacher gradients need a hidden student, a tied / separate
    teacher and teacher_grads = 1; d_w_t only for a separate teacher."""
    lib = kd.load_library()
    fake = 1 << 20
    ins = kd.kd_inputs(h_s=fake, w_s=fake, h_t=fake, w_t=fake, labels=fake)

    def call(teacher="separate", tg=1, **g):
        p = _prob(kd, teacher=teacher, d_teacher=64)
        p.teacher_grads = tg
        grads = kd.kd_grads(**{k: fake for k in g})
        return lib.kd_bwd_grads(ctypes.byref(p), ctypes.byref(ins), fake, None, 1.0,
                                ctypes.byref(grads), None, None, 0, None)

    assert call(tg=0, d_h_t=1) == kd.KD_ERR_INVALID_ARG
    assert call(teacher="tied", d_w_t=1) == kd.KD_ERR_INVALID_ARG
    assert lib.kd_bwd_grads(ctypes.byref(_prob(kd)), ctypes.byref(ins), fake, None, 1.0, None,
                            None, None, 0, None) == kd.KD_ERR_INVALID_ARG
    # well-formed requests get as far as the workspace / device checks
    assert call(d_h_t=1, d_w_t=1) in (kd.KD_ERR_WORKSPACE, kd.KD_ERR_NO_DEVICE)
