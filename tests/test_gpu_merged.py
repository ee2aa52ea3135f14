"""The step's insert inside the index launch (msa_insert_index_score): with one
query position, each request's new token sits in its local block, which the
scoring never reads. The merged launch must write the same cache bytes and
scores as the two separate calls, and reject a token that is not at its
request's last position."""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa, synth

import parity
from test_gpu_pipeline import REDUCED

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
MERGED = ["b32_32k", "fp8kv_32k", "b32_32k_fp4idx", "nvfp4_256k", "tiny"]


def _cache_tensors(dw):
    c, ic = dw.cache, dw.idx_cache
    return [t for t in (c.k, c.v, c.k_scale, c.v_scale, ic.keys, ic.scale, ic.block_scale) if t is not None]


def _clear_step_slots(dw):
    """Zero the cache rows of the step's new tokens (written at build time)."""
    slots = dw.new_slots.cpu().numpy()
    for t in _cache_tensors(dw):
        for s in slots:
            t[int(s) // 128, :, int(s) % 128] = 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", MERGED)
def test_merged_step_matches_oracle(name):
    w = REDUCED[name]
    dw = parity.build(w)
    assert dw.merges_insert
    _clear_step_slots(dw)
    dw.step()
    torch.cuda.synchronize()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


@pytest.mark.parametrize("name", MERGED)
def test_merged_launch_writes_the_same_bytes(name):
    w = REDUCED[name]
    a, b = parity.build(w), parity.build(w)
    _clear_step_slots(a)
    _clear_step_slots(b)
    a.insert_step_tokens()
    a.index_score()
    b.insert_index_score()
    torch.cuda.synchronize()
    assert "insert+index_score" in msa.last_dispatch()
    assert a.check_flags() == 0 and b.check_flags() == 0
    for x, y in zip(_cache_tensors(a), _cache_tensors(b)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    assert torch.equal(a.scores, b.scores)


def test_token_off_its_last_position_is_flagged_and_skipped():
    w = REDUCED["b32_32k"]
    dw = parity.build(w)
    _clear_step_slots(dw)
    good = dw.new_slots.clone()
    dw.new_slots[1] = good[1] - 1                 # one position early: not the request's last token
    dw.new_slots[2] = -1                          # a padding token: skipped silently
    dw.insert_index_score(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert dw.check_flags() == msa.FLAG_BAD_SLOT
    s1, s0 = int(good[1]), int(good[0])
    assert not dw.cache.k[s1 // 128, :, s1 % 128].any()     # not written
    assert dw.cache.k[s0 // 128, :, s0 % 128].any()         # request 0 written


def test_unsupported_shapes_are_rejected():
    w = REDUCED["spec8"]                          # 8 query positions
    dw = parity.build(w)
    with pytest.raises(msa.MSAError):
        msa.insert_index_score(dw.dims, dw.new_k, dw.new_v, dw.new_idx, dw.new_slots, dw.cache, dw.q_idx,
                               dw.idx_cache, dw.block_table_d, dw.seq_lens_d, dw.scores, dw.flags)
