"""The allocation-free sparse GQA entry point, for callers that cannot allocate
device memory (its scratch is a fixed array inside the library instead of a
caller-provided workspace).

Called through the C ABI and compared with msa_sparse_gqa_decode, which takes
a workspace, on two calls in a row (the second call finds the scratch holding
the first call's partials). This file is collected last so that a run stopping
at its first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa, synth

import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,changes", [("b32_32k", dict(batch=4, ctx=3000)),
                                          ("nvfp4_256k", dict(batch=2, ctx=2600)),
                                          ("spec8", dict(batch=2, ctx=2948))])
def test_noalloc_matches_workspace_entry_point(name, changes):
    w = synth.scaled(synth.WORKLOADS[name], **changes)
    dw = parity.build(w)
    dw.index_score()
    dw.select()
    dw.attend()
    torch.cuda.synchronize()
    ref_out = dw.out.float().cpu().numpy()
    ref_lse = dw.lse.cpu().numpy()
    for call in range(2):
        out = torch.full_like(dw.out, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        msa.sparse_gqa_decode_noalloc(dw.dims, dw.q, dw.cache, dw.block_table_d, dw.seq_lens_d, dw.selected, out,
                                      lse, dw.flags)
        assert msa.read_device_flags(dw.flags) == 0
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(l).all(), f"call {call}"
        err = np.abs(o - ref_out)
        assert err.max() <= parity.OUT_MAX_ABS and err.mean() <= parity.OUT_MEAN_ABS, f"call {call}"
        assert np.abs(l - ref_lse).max() <= parity.LSE_ABS, f"call {call}"


def test_noalloc_split_rows_across_changing_shapes(monkeypatch):
    """NVFP4 K/V rows are split over CTAs and merged through the scratch array
    (the balanced form, forced for the small batch too). A large batch, then a
    small one with other lengths, then the large one again: each call finds
    the previous call's partials and tickets in the array (laid out for
    another shape) and must still match the workspace entry point."""
    monkeypatch.setenv("MSA_NVFP4_SPLIT", "tickets")
    big = parity.build(synth.scaled(synth.WORKLOADS["nvfp4_256k"], batch=64, ctx=3000))
    small = parity.build(synth.scaled(synth.WORKLOADS["nvfp4_256k"], batch=3, ctx=None, ctx_range=(900, 5000),
                                      seed=20261301))
    refs = {}
    for name, dw in (("big", big), ("small", small)):
        dw.index_score()
        dw.select()
        dw.attend()
        torch.cuda.synchronize()
        assert msa.read_device_flags(dw.flags) == 0
        refs[name] = (dw.out.float().cpu().numpy(), dw.lse.cpu().numpy())
    for name, dw in (("big", big), ("small", small), ("big", big)):
        out = torch.full_like(dw.out, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        msa.sparse_gqa_decode_noalloc(dw.dims, dw.q, dw.cache, dw.block_table_d, dw.seq_lens_d, dw.selected, out,
                                      lse, dw.flags)
        assert msa.read_device_flags(dw.flags) == 0
        o, l = out.float().cpu().numpy(), lse.cpu().numpy()
        ro, rl = refs[name]
        assert np.isfinite(o).all() and np.isfinite(l).all(), name
        err = np.abs(o - ro)
        assert err.max() <= parity.OUT_MAX_ABS and err.mean() <= parity.OUT_MEAN_ABS, name
        assert np.abs(l - rl).max() <= parity.LSE_ABS, name


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 64 MiB holds about 8,000 split-K partials of 8,320 bytes
    dims = msa.make_dims(64, 8, max_blocks_per_seq=4, num_pages=8)      # 64 * 8 * 4 * 16 = 32768 partials
    x = torch.zeros(16, dtype=torch.uint8, device="cuda")
    kv = msa.KVCache(msa.BF16, x, x)
    with pytest.raises(msa.MSAError) as e:
        msa.sparse_gqa_decode_noalloc(dims, x, kv, x, x, x, x, None, x)
    assert e.value.status == msa.ERR_WORKSPACE
