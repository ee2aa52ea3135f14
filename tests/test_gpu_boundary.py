"""Inputs only the device can check: the kernels skip the bad block or token,
raise a flag bit, and neither trap nor hang."""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa, synth

import parity

pytestmark = pytest.mark.gpu


def _small():
    w = synth.scaled(synth.WORKLOADS["b32_32k"], batch=2, ctx=1500)
    return w, parity.build(w)


def test_clean_run_has_no_flags():
    w, dw = _small()
    dw.step()
    assert dw.check_flags() == 0


def test_corrupt_block_table_entry_is_flagged():
    w, dw = _small()
    dw.step()
    assert dw.check_flags() == 0
    dw.block_table_d[0, 3] = dw.num_pages + 7
    dw.block_table_d[1, 0] = -5
    dw.index_score()
    dw.select()
    dw.attend()
    flags = dw.check_flags()
    assert flags & msa.FLAG_BAD_PAGE
    assert torch.isfinite(dw.out.float()).all()
    S = dw.scores.cpu().numpy()
    assert np.isneginf(S[0, 0, :, 3]).all() and np.isneginf(S[1, 0, :, 0]).all()


def test_bad_seq_len_is_flagged():
    w, dw = _small()
    dw.seq_lens_d[1] = dw.dims.max_blocks_per_seq * 128 + 1
    dw.index_score()
    dw.select()
    dw.attend()
    assert dw.check_flags() & msa.FLAG_BAD_SEQLEN
    sel = dw.selected.cpu().numpy()
    assert (sel[1] == -1).all()


def test_selected_block_beyond_local_is_flagged():
    w, dw = _small()
    dw.index_score()
    dw.select()
    torch.cuda.synchronize()
    sel = dw.selected.clone()
    sel[0, 0, 0, -1] = 11          # local block of L=1500 is 11; 11 is legal
    sel[0, 0, 1, -1] = 12          # beyond the local block
    dw.attend(selected=sel)
    assert dw.check_flags() & msa.FLAG_BAD_BLOCK


def test_workspace_too_small_is_rejected_before_launch():
    w, dw = _small()
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(msa.MSAError) as e:
        msa.sparse_gqa_decode(dw.dims, dw.q, dw.cache, dw.block_table_d, dw.seq_lens_d, dw.selected, dw.out,
                              dw.lse, small, dw.flags)
    assert e.value.status == msa.ERR_WORKSPACE


def test_dispatch_record_names_the_variant():
    w, dw = _small()
    dw.index_score()
    assert "index_score fp8_mma_f16" in msa.last_dispatch()
    dw.select()
    assert "select_blocks" in msa.last_dispatch()
    dw.attend()
    assert "sparse_gqa bf16_tma_mma" in msa.last_dispatch()
    w4 = synth.scaled(synth.WORKLOADS["nvfp4_256k"], batch=1, ctx=700)
    dw4 = parity.build(w4)
    dw4.step()
    assert "sparse_gqa nvfp4_regk_f16_mma 8warps" in msa.last_dispatch()
    w5 = synth.scaled(synth.WORKLOADS["b32_32k_fp4idx"], batch=1, ctx=700)
    dw5 = parity.build(w5)
    dw5.index_score()
    assert "index_score nvfp4_group_cols_mma_f16" in msa.last_dispatch()
    w6 = synth.scaled(synth.WORKLOADS["spec8"], batch=1, ctx=700, idx_dtype="nvfp4")
    dw6 = parity.build(w6)
    dw6.index_score()
    assert "index_score nvfp4_mma_f16" in msa.last_dispatch()
    w8 = synth.scaled(synth.WORKLOADS["fp8kv_32k"], batch=1, ctx=700)
    dw8 = parity.build(w8)
    dw8.step()
    assert "sparse_gqa fp8_tma_cvt_f16_mma" in msa.last_dispatch()
    wt = synth.scaled(synth.WORKLOADS["tiny"], batch=1, ctx=700)
    dwt = parity.build(wt)
    dwt.index_score()
    assert "index_score f32_fma" in msa.last_dispatch()


def test_fused_selection_flags_bad_pages_and_lengths():
    """The selection inside the attention launch meets the same invalid inputs:
    a page id outside the cache and a request with an impossible length."""
    w, dw = _small()
    dw.step_fused()
    assert dw.check_flags() == 0
    dw.block_table_d[0, 3] = dw.num_pages + 7
    dw.index_score()
    dw.select_attend()
    assert dw.check_flags() & msa.FLAG_BAD_PAGE
    assert torch.isfinite(dw.out.float()).all()
    dw.flags.zero_()
    dw.block_table_d.copy_(torch.from_numpy(dw.block_table))
    dw.seq_lens_d[1] = 0
    dw.index_score()
    dw.select_attend()
    assert dw.check_flags() & msa.FLAG_BAD_SEQLEN
    assert (dw.selected[1] == -1).all()
    assert torch.isfinite(dw.out.float()).all()


def test_bounded_wait_gives_up_and_reports():
    """A kernel whose barrier wait runs out (nothing completes it; no copy in
    flight) sets MSA_FLAG_TIMEOUT and returns; the context stays usable: a
    decode step afterwards runs clean and matches the one before."""
    w, dw = _small()
    dw.step()
    assert dw.check_flags() == 0
    before = dw.out.clone()
    msa.selftest_bounded_wait(dw.flags)
    assert dw.check_flags() == msa.FLAG_TIMEOUT
    dw.flags.zero_()
    dw.step()
    assert dw.check_flags() == 0
    assert torch.equal(dw.out, before)
