"""The single-CTA tensor-core tiles (KD_TC_PAIR=0 debug override) against the oracle,
so both tile geometries of the tcgen05 kernels stay covered."""
import pytest

from lm_head_cross_vocab_gb300 import inputs as I
from tests.parity_util import assert_parity, run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _single_cta(monkeypatch):
    monkeypatch.setenv("KD_TC_PAIR", "0")


def test_single_cta_separate_teacher():
    w = I.WORKLOADS[2].scaled(n_tokens=300, d_student=128, d_teacher=256, vocab=1000)
    assert_parity(run_and_compare(w), "bf16")


def test_single_cta_topk_chunked():
    w = I.WORKLOADS[4].scaled(n_tokens=260, d_student=128, vocab=3000, topk=20)
    assert_parity(run_and_compare(w, vocab_chunk=512, seq_chunk=128), "bf16")
