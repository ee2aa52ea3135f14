"""FP8 K/V attention against the oracle: ragged tails, several positions,
three KV heads, a small top-k, more rows than SMs (CTAs that carry several
rows, copies running ahead across a row boundary), the selection inside the
launch, and bit-identical repeats.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa, synth

import parity

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

CASES = {
    "b3": synth.scaled(W["fp8kv_32k"], batch=3, ctx=2400),
    "q5": synth.scaled(W["spec8"], batch=2, ctx=2693, q_len=5, kv_dtype="fp8"),
    "g3": synth.scaled(W["fp8kv_32k"], batch=2, ctx=2300, n_heads=48, n_kv_heads=3, n_idx_heads=3),
    "top3": synth.scaled(W["fp8kv_32k"], batch=2, ctx=2500, topk=3),
    "rows_over_sms": synth.scaled(W["fp8kv_32k"], batch=48, ctx=1500),
}


def _expect_fp8():
    d = msa.last_dispatch()
    assert "fp8_tma_cvt_f16_mma" in d, d


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", list(CASES))
def test_fp8_matches_oracle(case, fused):
    w = CASES[case]
    dw = parity.build(w)
    dw.step_fused() if fused else dw.step_separate()
    _expect_fp8()
    sample = None if len(dw.which) <= 4 else [0, 17, len(dw.which) - 1]
    parity.verify_workload(dw, w, synth.seq_lens(w), sample=sample, run_step=False)


def test_fp8_edge_lengths():
    """No candidates, one block, block boundaries."""
    lens = np.array([1, 127, 128, 129, 257, 1921, 2049], dtype=np.int32)
    w = synth.scaled(W["fp8kv_32k"], batch=len(lens), ctx=None, ctx_range=None)
    dw = parity.build(w, lens=lens)
    dw.step_separate()
    _expect_fp8()
    parity.verify_workload(dw, w, lens, run_step=False)


def test_fp8_repeats_bitwise():
    """Six identical steps give bit-identical outputs, cache slots past each
    length poisoned with NaN patterns; 8 positions straddle block ends."""
    lens = np.array([8, 9, 130, 136, 1028, 2951], dtype=np.int32)
    w = synth.scaled(W["spec8"], batch=len(lens), ctx=None, ctx_range=None, kv_dtype="fp8")
    dw = parity.build(w, lens=lens)
    parity.poison_unwritten_slots(dw)
    outs = []
    for _ in range(6):
        dw.step_fused()
        torch.cuda.synchronize()
        outs.append(dw.out.clone())
    assert dw.check_flags() == 0
    for k, o in enumerate(outs[1:], 1):
        assert torch.equal(o, outs[0]), f"step {k} differs from step 0"
    parity.verify_workload(dw, w, lens, run_step=False)
