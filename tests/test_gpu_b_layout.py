"""Both operand layouts of the backward GEMMs against the oracle.  dH = G W and
dW = G^T H take W and H either as stored (MN-major B operands) or from a
per-backward transpose (K-major B operands); the plan picks one by problem
shape, and the KD_TC_KMAJOR_B debug override forces each here on small,
ragged problems with several row and vocabulary chunks."""
import pytest

from lm_head_cross_vocab_gb300 import inputs as I
from tests.parity_util import assert_parity, run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["0", "1"], ids=["stored_mn", "transposed_k"])
def b_layout(request, monkeypatch):
    monkeypatch.setenv("KD_TC_KMAJOR_B", request.param)
    return request.param


def test_separate_teacher_chunked(b_layout):
    w = I.WORKLOADS[2].scaled(n_tokens=300, d_student=136, d_teacher=256, vocab=1000)
    assert_parity(run_and_compare(w, vocab_chunk=384, seq_chunk=128), "bf16")


def test_tied_teacher_ce_chunked(b_layout):
    """Tied teacher with teacher CE: dW also gets G_t^T H_t as a second K segment."""
    w = I.WORKLOADS[1].scaled(dtype="bf16", n_tokens=200, d_student=72, d_teacher=72, vocab=900)
    assert_parity(run_and_compare(w, vocab_chunk=256, seq_chunk=128), "bf16")


def test_topk_chunked(b_layout):
    w = I.WORKLOADS[4].scaled(n_tokens=260, d_student=128, vocab=3000, topk=20)
    assert_parity(run_and_compare(w, vocab_chunk=512, seq_chunk=128), "bf16")
