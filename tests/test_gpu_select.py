"""The selection on hand-made score rows, against the oracle's selection of the
same fp32 values: random rows, rows of equal scores (order by block id), -inf
scores, short rows, and a row shaped so that the first threshold keeps hundreds
of candidates (the exact-threshold path). Each case runs through the selection
kernel and through the fused select + sparse-GQA launch (one warp per row)."""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa
from oracle import msa as om

pytestmark = pytest.mark.gpu


def _run(scores: np.ndarray, lens, q_len=1, topk=16, fused=False):
    B, Q, I, NB = scores.shape
    s = torch.from_numpy(scores.astype(np.float32)).cuda()
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sel = torch.full((B, Q, I, topk), -7, dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    if not fused:
        dims = msa.make_dims(B, q_len, 16 * I, I, I, 128, 128, NB, NB * B, topk)
        msa.select_blocks(dims, s, sl, sel, flags)
    else:
        # every request maps block n to page n of one zero K/V cache
        G, H, P = I, 16 * I, NB
        dims = msa.make_dims(B, q_len, H, G, I, 128, 128, NB, P, topk)
        cache = msa.KVCache(msa.BF16, *[torch.zeros((P, G, 128, 128), dtype=torch.bfloat16, device="cuda")
                                        for _ in range(2)])
        bt = torch.arange(NB, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous()
        q = torch.zeros((B, Q, H, 128), dtype=torch.bfloat16, device="cuda")
        out, lse = torch.empty_like(q), torch.empty((B, Q, H), dtype=torch.float32, device="cuda")
        ws = torch.empty(msa.sparse_gqa_workspace_size(dims, msa.BF16), dtype=torch.uint8, device="cuda")
        msa.select_sparse_gqa_decode(dims, q, cache, bt, sl, s, sel, out, lse, ws, flags)
        assert "select+sparse_gqa" in msa.last_dispatch()
    assert msa.read_device_flags(flags) == 0
    return sel.cpu().numpy()


def _check(scores, lens, sel, q_len, topk):
    B, Q, I, NB = scores.shape
    for b in range(B):
        for j in range(Q):
            ell = (lens[b] - q_len + j) // 128
            for g in range(I):
                want, _ = om.select_row(scores[b, j, g].astype(np.float32).astype(np.float64), ell, topk)
                assert sel[b, j, g].tolist() == want.tolist(), (b, j, g)


def _adversarial_row(NB, rng):
    ell = NB - 1
    row = rng.uniform(0, 40, NB)
    n = np.arange(NB)
    big = (n % 32) < 14
    row[big] = 100 + 0.001 * n[big]          # lanes 0..13: every element above the threshold
    lane14 = (n % 32) == 14
    row[lane14] = 0.0
    row[14] = 50.0
    return row, ell


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("topk", [16, 5, 1])
def test_select_patterns(topk, fused):
    rng = np.random.default_rng(7)
    NB = 2048
    lens = [NB * 128, 128 * 700 + 5, 37, 128 * 20]
    scores = np.full((4, 1, 4, NB), -np.inf)
    for b, L in enumerate(lens):
        ell = (L - 1) // 128
        scores[b, 0, 0, :ell] = rng.standard_normal(ell)
        scores[b, 0, 1, :ell] = 3.25                                   # all equal: lowest ids win
        scores[b, 0, 2, :ell] = np.round(rng.standard_normal(ell), 1)  # many ties
        row = rng.standard_normal(ell)
        row[rng.random(ell) < 0.3] = -np.inf
        scores[b, 0, 3, :ell] = row
    adv, ell = _adversarial_row(NB, rng)
    scores[0, 0, 2, :ell] = adv[:ell]
    sel = _run(scores, lens, topk=topk, fused=fused)
    _check(scores, lens, sel, 1, topk)


@pytest.mark.parametrize("fused", [False, True])
def test_select_spec_positions(fused):
    rng = np.random.default_rng(8)
    NB, Q = 600, 8
    lens = [128 * 500 + 3, 128 * 300 + 4]           # positions straddle a block boundary
    scores = np.full((2, Q, 4, NB), -np.inf)
    for b, L in enumerate(lens):
        for j in range(Q):
            ell = (L - Q + j) // 128
            scores[b, j, :, :ell] = rng.standard_normal((4, ell))
    sel = _run(scores, lens, q_len=Q, fused=fused)
    _check(scores, lens, sel, Q, 16)


@pytest.mark.parametrize("fused", [False, True])
def test_nan_scores_count_as_minus_inf(fused):
    rng = np.random.default_rng(9)
    NB = 300
    base = rng.standard_normal((1, 1, 4, NB))
    base[0, 0, :, rng.random(NB) < 0.5] = np.nan
    lens = [NB * 128]
    with_nan = _run(base, lens, fused=fused)
    as_inf = _run(np.where(np.isnan(base), -np.inf, base), lens, fused=fused)
    assert np.array_equal(with_nan, as_inf)
