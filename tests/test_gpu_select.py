"""The selection kernel on hand-made score rows, against the oracle's selection of
the same fp32 values: random rows, rows of equal scores (order by block id),
-inf scores, short rows, and a row shaped so that the first threshold keeps
hundreds of candidates (the kernel's exact-threshold path)."""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa
from oracle import msa as om

pytestmark = pytest.mark.gpu


def _run(scores: np.ndarray, lens, q_len=1, topk=16):
    B, Q, I, NB = scores.shape
    dims = msa.make_dims(B, q_len, 16 * I, I, I, 128, 128, NB, NB * B, topk)
    s = torch.from_numpy(scores.astype(np.float32)).cuda()
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sel = torch.empty((B, Q, I, topk), dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.select_blocks(dims, s, sl, sel, flags)
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


@pytest.mark.parametrize("topk", [16, 5, 1])
def test_select_patterns(topk):
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
    sel = _run(scores, lens, topk=topk)
    _check(scores, lens, sel, 1, topk)


def test_select_spec_positions():
    rng = np.random.default_rng(8)
    NB, Q = 600, 8
    lens = [128 * 500 + 3, 128 * 300 + 4]           # positions straddle a block boundary
    scores = np.full((2, Q, 4, NB), -np.inf)
    for b, L in enumerate(lens):
        for j in range(Q):
            ell = (L - Q + j) // 128
            scores[b, j, :, :ell] = rng.standard_normal((4, ell))
    sel = _run(scores, lens, q_len=Q)
    _check(scores, lens, sel, Q, 16)


def test_nan_scores_count_as_minus_inf():
    rng = np.random.default_rng(9)
    NB = 300
    base = rng.standard_normal((1, 1, 4, NB))
    base[0, 0, :, rng.random(NB) < 0.5] = np.nan
    lens = [NB * 128]
    with_nan = _run(base, lens)
    as_inf = _run(np.where(np.isnan(base), -np.inf, base), lens)
    assert np.array_equal(with_nan, as_inf)
