"""The seeded input generator: deterministic, per-request streams, workload recipes (CPU only)."""
import numpy as np

from block_sparse_attention_07_gb300 import synth


def test_workload_shapes_and_lengths():
    w = synth.WORKLOADS["ragged"]
    lens = synth.seq_lens(w)
    assert lens.shape == (64,) and (lens >= 8192).all() and (lens <= 131073).all()
    assert (lens % 128 != 0).all()
    for name in ("tiny", "b32_32k", "spec8", "nvfp4_256k"):
        w = synth.WORKLOADS[name]
        assert (synth.seq_lens(w) == w.ctx).all()


def test_page_table_is_a_permutation():
    w = synth.scaled(synth.WORKLOADS["ragged"], batch=5, ctx_range=(300, 1000))
    lens = synth.seq_lens(w)
    table, P = synth.page_table(w, lens)
    nb = synth.blocks_per_seq(w, lens)
    used = np.concatenate([table[b, : nb[b]] for b in range(w.batch)])
    assert sorted(used.tolist()) == list(range(P))
    for b in range(w.batch):
        assert (table[b, nb[b]:] == -1).all()


def test_request_streams_are_deterministic_and_independent():
    w = synth.scaled(synth.WORKLOADS["b32_32k"], batch=3, ctx=700)
    a = synth.request(w, 1, 700)
    b = synth.request(w, 1, 700)
    c = synth.request(w, 2, 700)
    for k in a:
        assert np.array_equal(a[k], b[k])
        assert not np.array_equal(a[k], c[k])
    assert a["k"].dtype == np.uint16 and a["k"].shape == (700, 4, 128)
    assert a["q"].shape == (1, 64, 128) and a["q_idx"].dtype == np.uint16
    t = synth.request(synth.WORKLOADS["tiny"], 0, 4096)
    assert t["idx_k"].dtype == np.float32 and t["q_idx"].dtype == np.float32


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(bits)
    assert back.tolist()[:4] == [1.0, 1.0, 1.0 + 2 ** -6, -2.5]


def test_block_offsets_make_scores_vary():
    """The planted offset along the unit index query shifts whole blocks."""
    w = synth.scaled(synth.WORKLOADS["ragged"], batch=1, ctx_range=(20000, 20000))
    r = synth.request(w, 0, 20001)
    qi = synth.bf16_bits_to_f32(r["q_idx"]).astype(np.float64)[0]          # [I, D]
    k = synth.bf16_bits_to_f32(r["idx_k"]).astype(np.float64)[:156 * 128]   # [T, I, D]
    mean_dot = np.einsum("tid,id->ti", k, qi).reshape(156, 128, 4).mean(1)  # [n, I]
    sig = np.linalg.norm(qi, axis=1)
    hi = mean_dot > sig                                                        # planted: +2 sigma
    assert 0.03 < hi.mean() < 0.2
