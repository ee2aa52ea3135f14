"""Parity of the whole decode step (insert, score, select, attend) against the oracle.

Reduced-size versions of every workload (several tiles, ragged tails) are
checked request by request; the full-size workloads run in the same launch
configuration as the benchmark and are checked on sampled requests.
"""
import numpy as np
import pytest

from block_sparse_attention_07_gb300 import synth

import parity

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

REDUCED = {
    "tiny": W["tiny"],
    "b32_32k": synth.scaled(W["b32_32k"], batch=3, ctx=2000),
    "ragged": synth.scaled(W["ragged"], batch=5, ctx_range=(300, 5000)),
    "spec8": synth.scaled(W["spec8"], batch=3, ctx=3000),
    "nvfp4_256k": synth.scaled(W["nvfp4_256k"], batch=2, ctx=3000),
    "b32_32k_fp4idx": synth.scaled(W["b32_32k_fp4idx"], batch=3, ctx=2300),
    "fp4_256k": synth.scaled(W["fp4_256k"], batch=2, ctx=2900),
    # NVFP4 index keys with 8 query positions (the per-value block-scale path;
    # one position takes the per-group path)
    "spec8_fp4idx": synth.scaled(W["spec8"], batch=3, ctx=3000, idx_dtype="nvfp4"),
    "fp8kv_32k": synth.scaled(W["fp8kv_32k"], batch=3, ctx=2400),
    # FP8 K/V with 8 positions (causal limits inside the local block)
    "spec8_fp8kv": synth.scaled(W["spec8"], batch=2, ctx=2700, kv_dtype="fp8"),
}


@pytest.mark.parametrize("name", list(REDUCED))
def test_reduced_workload(name):
    w = REDUCED[name]
    dw = parity.build(w)
    parity.verify_workload(dw, w, synth.seq_lens(w))


EDGE_LENS = {
    # (workload base, lengths): L < 128 (no candidates), exact multiples +-1,
    # fewer candidates than k-1, long enough for a full top-16.
    "short_and_multiples": ("b32_32k", [1, 5, 127, 128, 129, 255, 256, 257, 1919, 1920, 1921, 2100]),
    "spec_straddle": ("spec8", [8, 9, 130, 135, 136, 1028, 2948, 2951, 2952]),
    "nvfp4_edges": ("nvfp4_256k", [1, 128, 129, 1500, 2049]),
    "tiny_f32_edges": ("tiny", [1, 200, 4095]),
    "fp4idx_edges": ("b32_32k_fp4idx", [1, 129, 257, 2100]),
    "spec_fp4idx_edges": ("spec8", [8, 9, 136, 1028, 2951], {"idx_dtype": "nvfp4"}),
    "fp8kv_edges": ("fp8kv_32k", [1, 127, 128, 129, 1921, 2049]),
}


@pytest.mark.parametrize("case", list(EDGE_LENS))
def test_edge_lengths(case):
    base, lens, *more = EDGE_LENS[case]
    w = synth.scaled(W[base], batch=len(lens), ctx=None, ctx_range=None, **(more[0] if more else {}))
    lens = np.array(lens, dtype=np.int32)
    dw = parity.build(w, lens=lens)
    parity.verify_workload(dw, w, lens)


@pytest.mark.parametrize("topk", [1, 2, 7, 16])
def test_topk_values(topk):
    w = synth.scaled(W["b32_32k"], batch=2, ctx=3100, topk=topk)
    dw = parity.build(w)
    parity.verify_workload(dw, w, synth.seq_lens(w))


@pytest.mark.parametrize("name", list(W))
def test_full_size_sampled(name):
    """Full-size workload, benchmark launch configuration, two sampled requests."""
    w = W[name]
    dw = parity.build(w)
    lens = synth.seq_lens(w)
    dw.step()
    dw.step()          # a second step (the benchmark repeats steps) gives the same result
    sample = [0, len(dw.which) - 1]
    parity.verify_workload(dw, w, lens, sample=sample, run_step=False)


@pytest.mark.parametrize("name", ["b32_32k", "nvfp4_256k", "spec8", "fp8kv_32k"])
def test_fused_select_attend_step(name):
    """The step with selection and attention in one launch (msa_select_sparse_gqa_decode):
    same checks, including the selection it writes back; NVFP4 rows are split over CTAs."""
    w = REDUCED[name]
    dw = parity.build(w)
    dw.step_fused()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


NAN_TAIL = {
    # (workload, selection inside the attention launch); no length is a multiple of 128
    "bf16": (REDUCED["b32_32k"], False),
    "bf16_fused": (REDUCED["b32_32k"], True),
    "fp8kv_fused": (REDUCED["fp8kv_32k"], True),
    "nvfp4": (REDUCED["nvfp4_256k"], False),
    "spec8": (REDUCED["spec8"], True),
    "spec8_fp8kv": (REDUCED["spec8_fp8kv"], False),
    "tiny_f32": (synth.scaled(W["tiny"], ctx=3950), False),
    "fp4idx": (REDUCED["b32_32k_fp4idx"], False),
}


@pytest.mark.parametrize("case", list(NAN_TAIL))
def test_unwritten_slots_hold_nan(case):
    """Outputs stay finite and match the oracle when the never-written slots of
    the local page hold NaN patterns (a cache in reused memory)."""
    w, fused = NAN_TAIL[case]
    assert (synth.seq_lens(w) % 128 != 0).all()
    dw = parity.build(w)
    parity.poison_unwritten_slots(dw)
    dw.step_fused() if fused else dw.step_separate()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


@pytest.mark.parametrize("name,fused", [("b32_32k", True), ("tiny", False), ("b32_32k_fp4idx", False),
                                        ("spec8", True), ("spec8_fp4idx", False)])
def test_scores_scale_exactly_with_index_queries(name, fused):
    """Multiplying every index query by 2^k multiplies every block score by
    exactly 2^k (products, fp32 sums and scale multiplies all commute with a
    power of two) and so leaves every selection unchanged."""
    import torch
    w = REDUCED[name]
    dw = parity.build(w)
    run = dw.step_fused if fused else dw.step_separate
    run()
    torch.cuda.synchronize()
    S0, sel0 = dw.scores.cpu().numpy().copy(), dw.selected.cpu().numpy().copy()
    scale = 1.0
    for k in (5, -3, -4):
        dw.q_idx.mul_(2.0 ** k)
        scale *= 2.0 ** k
        run()
        torch.cuda.synchronize()
        assert dw.check_flags() == 0
        assert np.array_equal(dw.selected.cpu().numpy(), sel0), f"selection changed at 2^{k}"
        S = dw.scores.cpu().numpy()
        assert np.array_equal(S, (S0 * np.float32(scale)).astype(np.float32)), f"scores not scaled exactly at 2^{k}"


QLENS = {
    # query positions between 1 and 8: the index kernel's unused mma columns,
    # per-position causal limits (some straddling a block boundary), and the
    # per-position selections and attention rows
    "q2_bf16": synth.scaled(W["spec8"], batch=3, ctx=2946, q_len=2),
    "q3_bf16": synth.scaled(W["spec8"], batch=3, ctx=2947, q_len=3),
    "q5_fp8kv": synth.scaled(W["spec8"], batch=2, ctx=2693, q_len=5, kv_dtype="fp8"),
    "q7_bf16": synth.scaled(W["spec8"], batch=2, ctx=2950, q_len=7),
    "q3_fp4idx": synth.scaled(W["spec8"], batch=3, ctx=2305, q_len=3, idx_dtype="nvfp4"),
    "q2_nvfp4kv": synth.scaled(W["nvfp4_256k"], batch=2, ctx=3001, q_len=2),
}


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", list(QLENS))
def test_query_lengths(case, fused):
    w = QLENS[case]
    dw = parity.build(w)
    dw.step_fused() if fused else dw.step_separate()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


HEADS = {
    # 1 to 3 KV heads (index heads = KV heads, 16 query heads each): the index
    # kernel's consumer warps, page strides and every row enumeration follow G
    "g1": synth.scaled(W["b32_32k"], batch=3, ctx=2100, n_heads=16, n_kv_heads=1, n_idx_heads=1),
    "g2_spec": synth.scaled(W["spec8"], batch=2, ctx=2951, n_heads=32, n_kv_heads=2, n_idx_heads=2),
    "g3_fp4idx": synth.scaled(W["b32_32k_fp4idx"], batch=2, ctx=2400, n_heads=48, n_kv_heads=3, n_idx_heads=3),
    "g2_nvfp4kv": synth.scaled(W["nvfp4_256k"], batch=2, ctx=2700, n_heads=32, n_kv_heads=2, n_idx_heads=2),
    "g3_fp8kv": synth.scaled(W["fp8kv_32k"], batch=2, ctx=2300, n_heads=48, n_kv_heads=3, n_idx_heads=3),
    "g1_tiny_f32": synth.scaled(W["tiny"], ctx=1500, n_heads=16, n_kv_heads=1, n_idx_heads=1),
}


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", list(HEADS))
def test_head_counts(case, fused):
    w = HEADS[case]
    dw = parity.build(w)
    dw.step_fused() if fused else dw.step_separate()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


@pytest.mark.parametrize("base", ["b32_32k", "b32_32k_fp4idx", "spec8", "nvfp4_256k"])
def test_max_batch(base):
    """The largest batch the API takes (4,096 requests) with short contexts. This
    exercises the index kernel's per-request prefix (16 KB of shared memory at
    this batch), every row enumeration and the selection padding (2 candidates
    for 15 slots). With 8 positions there are 131,072 attention rows and the
    split-K workspace is over 4 GiB. Sampled requests are checked."""
    w = synth.scaled(W[base], batch=4096, ctx=260)
    dw = parity.build(w)
    dw.step()
    parity.verify_workload(dw, w, synth.seq_lens(w), sample=[0, 1, 2047, 4095], run_step=False)


@pytest.mark.parametrize("name", ["b32_32k", "fp8kv_32k", "nvfp4_256k", "spec8"])
def test_large_logits(name, monkeypatch):
    """Attention queries scaled by 2^6 (exact in bf16) on both sides. Logits reach a
    few hundred, the softmax is nearly one-hot, and the running maximum rises by
    more than the rescale slack on most blocks. So the output rescale path runs far
    more often than on unit-scale data."""
    plain = synth.request

    def scaled_request(w, b, length):
        r = dict(plain(w, b, length))
        r["q"] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(r["q"]) * np.float32(64.0))
        return r

    monkeypatch.setattr(synth, "request", scaled_request)
    w = REDUCED[name]
    dw = parity.build(w)
    dw.step()
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


@pytest.mark.parametrize("kv,mode", [("bf16", "rows"), ("fp8", "rows"), ("bf16", "union"), ("bf16", "union_mma")])
def test_repeated_steps_are_bitwise_identical(kv, mode, monkeypatch):
    """The same step six times in a row gives bit-identical outputs (the
    kernels' merges are deterministic and nothing they read changes): 8
    positions, contexts straddling block boundaries and some shorter than a
    block, cache slots past each length poisoned with NaN patterns. This is
    the check that exposed V rows cleared inside a pipeline stage racing with
    the copy that refills it."""
    import torch
    monkeypatch.setenv("MSA_MULTIPOS_ATTENTION", mode)
    lens = np.array([8, 9, 130, 135, 136, 1028, 2948, 2951, 2952], dtype=np.int32)
    w = synth.scaled(W["spec8"], batch=len(lens), ctx=None, ctx_range=None, kv_dtype=kv)
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
