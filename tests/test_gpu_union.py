"""Several query positions with bf16 K/V: the form that streams the union of a
(request, KV head) group's selected blocks once ("MiniMax M3 vLLM サポート：…",
section "EAGLE3 を用いた投機的デコード": all draft positions of a request in
one pass), forced on small cases through MSA_MULTIPOS_ATTENTION=union and
checked against the oracle like the per-position form."""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa, synth

import parity

pytestmark = pytest.mark.gpu

# the tcgen05 form (M = 128 query rows: 8 positions x 16 heads) and the mma.sync form
FORMS = ["union", "union_mma"]

W = synth.WORKLOADS

CASES = {
    "spec8": synth.scaled(W["spec8"], batch=3, ctx=3000),
    "q2": synth.scaled(W["spec8"], batch=3, ctx=2946, q_len=2),
    "q3": synth.scaled(W["spec8"], batch=3, ctx=2947, q_len=3),
    "q7": synth.scaled(W["spec8"], batch=2, ctx=2950, q_len=7),
    "g2": synth.scaled(W["spec8"], batch=2, ctx=2951, n_heads=32, n_kv_heads=2, n_idx_heads=2),
    "fp4idx": synth.scaled(W["spec8"], batch=3, ctx=3000, idx_dtype="nvfp4"),
    "top5": synth.scaled(W["spec8"], batch=2, ctx=2600, topk=5),
}


def _check_union_ran():
    assert "union_of_positions" in msa.last_dispatch(), msa.last_dispatch()


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", list(CASES))
def test_union_matches_oracle(case, fused, form, monkeypatch):
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", form)
    w = CASES[case]
    dw = parity.build(w)
    dw.step_fused() if fused else dw.step_separate()
    _check_union_ran()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


@pytest.mark.parametrize("form", FORMS)
def test_union_edge_lengths(form, monkeypatch):
    """Lengths below, at and just past block boundaries: the 8 positions' local
    blocks differ, some requests have fewer candidates than k - 1, one has
    none."""
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", form)
    lens = np.array([8, 9, 130, 135, 136, 1028, 2948, 2951, 2952], dtype=np.int32)
    w = synth.scaled(W["spec8"], batch=len(lens), ctx=None, ctx_range=None)
    dw = parity.build(w, lens=lens)
    dw.step_separate()
    _check_union_ran()
    parity.verify_workload(dw, w, lens, run_step=False)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("fused", [False, True])
def test_union_unwritten_slots_hold_nan(fused, form, monkeypatch):
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", form)
    w = CASES["spec8"]
    assert (synth.seq_lens(w) % 128 != 0).all()
    dw = parity.build(w)
    parity.poison_unwritten_slots(dw)
    dw.step_fused() if fused else dw.step_separate()
    _check_union_ran()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


@pytest.mark.parametrize("form", FORMS)
def test_union_large_logits(form, monkeypatch):
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", form)
    plain = synth.request

    def scaled_request(w, b, length):
        r = dict(plain(w, b, length))
        r["q"] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(r["q"]) * np.float32(64.0))
        return r

    monkeypatch.setattr(synth, "request", scaled_request)
    w = CASES["spec8"]
    dw = parity.build(w)
    dw.step()
    _check_union_ran()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


@pytest.mark.parametrize("form", FORMS)
def test_union_persistent_groups_and_repeat(form, monkeypatch):
    """More groups than CTAs (each CTA runs several groups in turn, its stages
    and tags carried across them), two steps in a row giving the same output,
    and the per-position form agreeing within the oracle tolerance."""
    w = synth.scaled(W["spec8"], batch=200, ctx=1400)
    dw = parity.build(w)
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", form)
    dw.step_separate()
    _check_union_ran()
    torch.cuda.synchronize()
    first = dw.out.clone()
    dw.step_separate()
    torch.cuda.synchronize()
    assert torch.equal(dw.out, first)
    parity.verify_workload(dw, w, synth.seq_lens(w), sample=[0, 1, 77, 199], run_step=False)
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", "rows")
    dw.attend()
    assert "union_of_positions" not in msa.last_dispatch()
    torch.cuda.synchronize()
    assert dw.check_flags() == 0
    err = (dw.out.float() - first.float()).abs()
    assert err.max().item() <= parity.OUT_MAX_ABS and err.mean().item() <= parity.OUT_MEAN_ABS


@pytest.mark.parametrize("form", FORMS)
def test_union_bad_inputs_are_flagged(form, monkeypatch):
    """A selected block past a position's local block and a bad page id are
    flagged and skipped; the kernel neither traps nor hangs."""
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", form)
    w = CASES["spec8"]
    dw = parity.build(w)
    dw.step_separate()
    assert dw.check_flags() == 0
    sel = dw.selected.clone()
    sel[0, 0, 0, 0] = int(dw.lens[0]) // 128 + 3          # beyond the local block
    dw.selected.copy_(sel)
    dw.block_table_d[1, int(sel[1, 2, 1, 0])] = dw.num_pages + 9
    dw.attend()
    flags = dw.check_flags()
    assert flags & msa.FLAG_BAD_BLOCK and flags & msa.FLAG_BAD_PAGE and not flags & msa.FLAG_TIMEOUT
    assert torch.isfinite(dw.out.float()).all()
