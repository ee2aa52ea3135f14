"""Seeded random decode steps against the oracle.

Each case draws a small workload: the K/V and index-key formats, 1 to 8 query
positions, 1, 2 or 4 KV heads (16 query heads and one index head each), a top-k
from 1 to 16, ragged lengths from a few tokens to a few thousand, the
composition (selection inside the attention launch or not), for NVFP4 K/V the
split form and for bf16 K/V with several positions the union form. The draws
are fixed by the seed, so a failure names a reproducible case.
"""
import numpy as np
import pytest

from block_sparse_attention_07_gb300 import msa, synth

import parity

pytestmark = pytest.mark.gpu

N_CASES = 48


def _draw(k):
    rng = np.random.default_rng([20261203, k])
    kv = ["bf16", "fp8", "nvfp4"][int(rng.integers(3))]
    idx = ["fp8", "nvfp4"][int(rng.integers(2))]
    q_len = int(rng.integers(1, 9))
    g = [1, 2, 4][int(rng.integers(3))]
    topk = int(rng.integers(1, 17))
    batch = int(rng.integers(1, 5))
    lo = max(q_len, int(rng.integers(1, 400)))
    hi = lo + int(rng.integers(0, 3000))
    fused = bool(rng.integers(2))
    split = ["auto", "tickets", "cluster2", "cluster4", "cluster8"][int(rng.integers(5))]
    multipos = ["auto", "union", "union_mma", "rows"][int(rng.integers(4))]
    w = synth.scaled(synth.WORKLOADS["ragged"], name=f"fuzz{k}", batch=batch, q_len=q_len, ctx=None,
                     ctx_range=(lo, hi), idx_dtype=idx, kv_dtype=kv, planted=False, n_heads=16 * g,
                     n_kv_heads=g, n_idx_heads=g, topk=topk, seed=20261300 + k)
    return w, fused, split, multipos


@pytest.mark.parametrize("k", range(N_CASES))
def test_fuzz_case_matches_oracle(k, monkeypatch):
    w, fused, split, multipos = _draw(k)
    for var, val in (("MSA_NVFP4_SPLIT", split), ("MSA_MULTIPOS_ATTENTION", multipos)):
        if val == "auto":
            monkeypatch.delenv(var, raising=False)
        else:
            monkeypatch.setenv(var, val)
    dw = parity.build(w)
    dw.step_fused() if fused else dw.step_separate()
    d = msa.last_dispatch()
    assert "sparse_gqa" in d, d
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)
