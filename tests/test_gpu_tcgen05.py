"""The opt-in tcgen05 form of the bf16 attention tile (MSA_BF16_ATTENTION=tcgen05)
against the oracle: QK^T and P.V on the fifth-generation tensor cores with S and
O in tensor memory. The same checks as the default kernel's: reduced workloads
in both compositions, edge lengths, and never-written cache slots holding NaN."""
import numpy as np
import pytest

from block_sparse_attention_07_gb300 import msa, synth

import parity
from test_gpu_pipeline import REDUCED

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture
def tcgen05(monkeypatch):
    monkeypatch.setenv("MSA_BF16_ATTENTION", "tcgen05")


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", ["b32_32k", "ragged", "spec8", "tiny"])
def test_reduced_workloads(tcgen05, name, fused):
    w = REDUCED[name]
    dw = parity.build(w)
    dw.step_fused() if fused else dw.step_separate()
    assert "bf16_tma_tcgen05" in msa.last_dispatch()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


def test_edge_lengths(tcgen05):
    lens = np.array([1, 5, 127, 128, 129, 255, 1921, 2100], dtype=np.int32)
    w = synth.scaled(W["b32_32k"], batch=len(lens), ctx=None, ctx_range=None)
    dw = parity.build(w, lens=lens)
    dw.step_separate()
    assert "bf16_tma_tcgen05" in msa.last_dispatch()
    parity.verify_workload(dw, w, lens, run_step=False)


def test_two_kv_heads_three_positions(tcgen05):
    w = synth.scaled(W["spec8"], batch=2, ctx=2947, q_len=3, n_heads=32, n_kv_heads=2, n_idx_heads=2)
    dw = parity.build(w)
    dw.step_fused()
    assert "bf16_tma_tcgen05" in msa.last_dispatch()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


def test_unwritten_slots_hold_nan(tcgen05):
    w = REDUCED["spec8"]
    dw = parity.build(w)
    parity.poison_unwritten_slots(dw)
    dw.step_fused()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


def test_default_stays_on_mma_sync():
    w = REDUCED["b32_32k"]
    dw = parity.build(w)
    dw.step_separate()
    assert "bf16_tma_mma" in msa.last_dispatch()
