"""Teacher gradients on the GPU against the oracle (orda-kernel README,
"Teacher descriptors": a teacher whose teacher_ce_weight is > 0 is trained by
its CE term; the KL variants detach it): d H_t and d W_t of separate teachers
and d H_t of tied ones, on the fp32 SIMT path and the bf16 tensor-core path,
in one vocabulary / token chunk and in several (fp32 accumulators)."""
import numpy as np
import pytest
import torch

from lm_head_cross_vocab_gb300 import inputs as I
from lm_head_cross_vocab_gb300 import kd
from oracle import kd_oracle as O
from tests.parity_util import GRAD_TOL, oracle_kwargs, oracle_logits, rel_l2

pytestmark = pytest.mark.gpu

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kd.load_library()
    assert kd.kd_device_supported(0), "tests need an sm_103 GPU"


def _run(w, **overrides):
    dev = torch.device("cuda:0")
    cpu = I.make_inputs(w, "cpu")
    t = {k: v.to(dev) for k, v in cpu.items()}
    prob = kd.problem_for(w, teacher_grads=True, **overrides)
    fwd = kd.forward(prob, t)
    want = ("h_s", "w_s", "h_t") + (("w_t",) if w.teacher == "separate" else ())
    bwd = kd.backward(prob, t, fwd["stats"], want=want)
    torch.cuda.synchronize()
    lab = cpu["labels"].numpy()
    z_s, z_t = oracle_logits(cpu, w)
    kw = oracle_kwargs(w, prob)
    g_s, g_t = O.grad_logits(z_s, z_t, lab, **kw)
    tied = w.teacher == "tied"
    d_hs, d_ws = O.hidden_grads(cpu["h_s"], cpu["w_s"], g_s, cpu["h_t"], g_t, tied=tied)
    d_ht, d_wt = O.teacher_hidden_grads(cpu["h_t"], cpu["w_s" if tied else "w_t"], g_t)
    got = {k: bwd[k].cpu().double().numpy() for k in bwd if k.startswith("d_")}
    valid = lab != w.ignore_index
    return got, {"d_h_s": d_hs, "d_w_s": d_ws, "d_h_t": d_ht, "d_w_t": d_wt}, valid


def _check(got, ref, valid, dtype):
    for k in got:
        assert rel_l2(got[k], ref[k]) <= GRAD_TOL[dtype], k
    assert np.all(got["d_h_t"][~valid] == 0), "ignored tokens give zero teacher rows"


@pytest.mark.parametrize("variant", ["forward", "jeffreys", "skew_reverse"])
def test_separate_teacher_grads_fp32_multichunk(variant):
    w = W[2].scaled(n_tokens=77, d_student=40, d_teacher=24, vocab=333, dtype="fp32",
                    variant=variant)
    got, ref, valid = _run(w, vocab_chunk=64, seq_chunk=32)
    _check(got, ref, valid, "fp32")


def test_tied_teacher_grads_fp32():
    got, ref, valid = _run(W[1])
    _check(got, ref, valid, "fp32")


@pytest.mark.parametrize("variant", ["forward", "jeffreys", "skew_reverse"])
def test_separate_teacher_grads_bf16(variant):
    w = W[2].scaled(n_tokens=300, d_student=128, d_teacher=256, vocab=1000, variant=variant)
    got, ref, valid = _run(w)
    _check(got, ref, valid, "bf16")


@pytest.mark.parametrize("vchunk,schunk", [(256, 128), (512, 0), (0, 128)])
def test_separate_teacher_grads_bf16_chunked(vchunk, schunk):
    """Several vocabulary chunks (d H_t accumulated in fp32) and / or several
    token chunks (d W_t accumulated in fp32)."""
    w = W[2].scaled(n_tokens=300, d_student=64, d_teacher=128, vocab=1100)
    got, ref, valid = _run(w, vocab_chunk=vchunk, seq_chunk=schunk)
    _check(got, ref, valid, "bf16")


def test_tied_teacher_grads_bf16():
    w = W[1].scaled(n_tokens=257, d_student=64, d_teacher=64, vocab=777, dtype="bf16")
    got, ref, valid = _run(w)
    _check(got, ref, valid, "bf16")


def test_teacher_grads_zero_without_teacher_ce():
    w = W[2].scaled(n_tokens=64, d_student=64, d_teacher=64, vocab=500, w_teacher_ce=0.0)
    got, ref, valid = _run(w)
    assert np.all(got["d_h_t"] == 0) and np.all(got["d_w_t"] == 0)
    assert rel_l2(got["d_h_s"], ref["d_h_s"]) <= GRAD_TOL["bf16"]


def test_teacher_grads_need_the_workspace_flag():
    w = W[2].scaled(n_tokens=64, d_student=64, d_teacher=64, vocab=500)
    dev = torch.device("cuda:0")
    t = {k: v.to(dev) for k, v in I.make_inputs(w, "cpu").items()}
    prob = kd.problem_for(w)  # teacher_grads off
    fwd = kd.forward(prob, t)
    with pytest.raises(kd.KDError):
        kd.backward(prob, t, fwd["stats"], want=("h_s", "h_t"))


@pytest.mark.parametrize("streams", ["1", "2"])
def test_separate_teacher_grads_bf16_stream_schedules(streams, monkeypatch):
    """The teacher GEMMs on the backward's single-stream and two-stream
    schedules (KD_BWD_STREAMS, read on every call), several chunks each way."""
    monkeypatch.setenv("KD_BWD_STREAMS", streams)
    w = W[2].scaled(n_tokens=300, d_student=64, d_teacher=128, vocab=1100)
    got, ref, valid = _run(w, vocab_chunk=256, seq_chunk=128)
    _check(got, ref, valid, "bf16")
