"""Pins for ``oracle.run.run_request``, the entry point every GPU parity test uses.

``run_request`` takes a request's raw inputs, quantises them with the oracle's
own quantisers in token chunks, gathers only the KV rows of the selected
blocks into a token-indexed view, and runs the three stages of
"MiniMax M3 vLLM サポート：…", section "MSA 実行プロセス" (block scoring,
top-k selection with the local block, sparse GQA). These tests build the same
request a second way, the way a serving cache holds it: every token quantised
in one piece, written into a paged cache through a shuffled block table,
gathered back in logical order and decoded whole, and then fed to
``oracle.msa.decode_step`` / ``oracle.msa.sparse_gqa``. None of the chunking,
the block gather or the selection and head overrides of ``run_request`` is on
that second route, so a wrong token-to-row map, a dropped chunk or a misapplied
override fails here. Outputs must agree exactly (same fp64 operations on the
same values).
"""
import numpy as np
import pytest

from block_sparse_attention_07_gb300 import synth
from oracle import formats as F
from oracle import msa as M
from oracle import quant as QT
from oracle import run as R

BS = 128


def _paged(values: np.ndarray, slots: np.ndarray, num_pages: int) -> np.ndarray:
    """Per-token rows [T, X, ...] -> a paged cache [P, X, BS, ...] (slot = page * BS + offset)."""
    T, X = values.shape[:2]
    flat = np.zeros((num_pages * BS, X) + values.shape[2:], dtype=values.dtype)
    flat[slots] = values
    return np.moveaxis(flat.reshape((num_pages, BS, X) + values.shape[2:]), 1, 2)


def _decoded_request(w, req, L, kv_global, idx_global):
    """(q, q_idx, keys, key_scale, K, V) of one request as fp64 arrays, read back
    from paged caches filled with whole-request quantisation."""
    w1 = synth.scaled(w, batch=1)
    table, P = synth.page_table(w1, np.array([L], dtype=np.int32))
    slots = synth.slot_mapping(w1, table, 0, L)
    row = table[0]

    def kv(x):
        f = synth.bf16_bits_to_f32(x)
        if w.kv_dtype == "bf16":
            return M.gather_tokens(_paged(f, slots, P), row, L, BS).astype(np.float64)
        if w.kv_dtype == "fp8":
            codes = M.gather_tokens(_paged(QT.quant_kv_fp8(f, kv_global), slots, P), row, L, BS)
            return F.e4m3_decode(codes) * float(np.float32(kv_global))
        codes, scl = QT.quant_nvfp4(f, kv_global)
        return F.nvfp4_decode(M.gather_tokens(_paged(codes, slots, P), row, L, BS),
                              M.gather_tokens(_paged(scl, slots, P), row, L, BS), kv_global)

    if w.idx_dtype == "f32":
        keys = M.gather_tokens(_paged(req["idx_k"], slots, P), row, L, BS).astype(np.float64)
        kscale = None
        q_idx = req["q_idx"].astype(np.float64)
    else:
        xi = synth.bf16_bits_to_f32(req["idx_k"])
        q_idx = synth.bf16_bits_to_f32(req["q_idx"]).astype(np.float64)
        if w.idx_dtype == "fp8":
            codes, s = QT.quant_index_keys_fp8(xi)
            keys = F.e4m3_decode(M.gather_tokens(_paged(codes, slots, P), row, L, BS))
            kscale = M.gather_tokens(_paged(s[..., None], slots, P), row, L, BS)[..., 0].astype(np.float64)
        else:
            codes, scl = QT.quant_nvfp4(xi, idx_global)
            keys = F.nvfp4_decode(M.gather_tokens(_paged(codes, slots, P), row, L, BS),
                                  M.gather_tokens(_paged(scl, slots, P), row, L, BS), idx_global)
            kscale = None
    q = synth.bf16_bits_to_f32(req["q"]).astype(np.float64)
    return q, q_idx, keys, kscale, kv(req["k"]), kv(req["v"])


def _other_selection(own: np.ndarray, L: int, Q: int, topk: int, seed: int) -> np.ndarray:
    """A valid selection that differs from ``own``: per (position, head) a seeded
    random set of earlier blocks plus the local block, ascending, padded with -1;
    some rows take fewer blocks than they could."""
    rng = np.random.default_rng(seed)
    G = own.shape[1]
    out = np.full(own.shape, -1, dtype=np.int32)
    for j in range(Q):
        ell = (L - Q + j) // BS
        for g in range(G):
            n = min(topk - 1, ell)
            n = int(rng.integers(0, n + 1)) if (j + g) % 3 == 0 else n
            pick = np.sort(rng.choice(ell, size=n, replace=False)) if n else np.zeros(0, dtype=np.int64)
            row = sorted(pick.tolist() + [ell])
            out[j, g, :len(row)] = row
    assert not np.array_equal(out, own)
    return out


CASES = [
    # (base workload, kv, idx, Q, L, topk): every KV and index-key format, a
    # position window straddling a block boundary, and lengths past the
    # oracle's 16,384-token quantisation chunk.
    ("tiny", "bf16", "f32", 1, 900, 4),
    ("b32_32k", "fp8", "fp8", 8, 5 * BS + 3, 3),
    ("b32_32k", "nvfp4", "nvfp4", 2, 1000, 5),
    ("spec8", "bf16", "fp8", 8, 16384 + 300, 16),
    ("nvfp4_256k", "nvfp4", "fp8", 1, 16384 + BS + 1, 16),
    ("b32_32k", "fp8", "nvfp4", 3, 16384 + 2 * BS - 1, 16),
]


@pytest.mark.parametrize("base,kv,idx,Q,L,topk", CASES)
def test_run_request_equals_paged_decode_step(base, kv, idx, Q, L, topk):
    w = synth.scaled(synth.WORKLOADS[base], batch=2, q_len=Q, ctx=L, ctx_range=None, kv_dtype=kv, idx_dtype=idx,
                     topk=topk)
    req = synth.request(w, 1, L)
    kv_g = synth.kv_scale(w)
    idx_g = float(np.float32(synth.NVFP4_IDX_SYNTH_GLOBAL)) if idx == "nvfp4" else 1.0
    q, q_idx, keys, kscale, K, V = _decoded_request(w, req, L, kv_g, idx_g)
    want = M.decode_step(q, q_idx, keys, kscale, K, V, L, topk, w.softmax_scale, BS)

    got = R.run_request(req, L, topk, w.softmax_scale, BS, idx, kv, kv_g, kv_g, idx_global=idx_g)
    assert np.array_equal(got["S"], want["S"])
    assert np.array_equal(got["sel"], want["sel"]) and np.array_equal(got["sel_used"], want["sel"])
    np.testing.assert_array_equal(got["margin"], want["margin"])
    np.testing.assert_allclose(got["out"], want["out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["lse"], want["lse"], rtol=0, atol=1e-12)

    # a selection made elsewhere replaces the oracle's own in the attention stage only
    alt = _other_selection(want["sel"], L, Q, topk, seed=L + Q)
    got2 = R.run_request(req, L, topk, w.softmax_scale, BS, idx, kv, kv_g, kv_g, sel=alt, idx_global=idx_g)
    out2, lse2 = M.sparse_gqa(q, K, V, L, alt, w.softmax_scale, BS)
    assert np.array_equal(got2["sel"], want["sel"]) and np.array_equal(got2["sel_used"], alt)
    np.testing.assert_allclose(got2["out"], out2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got2["lse"], lse2, rtol=0, atol=1e-12)
    assert not np.allclose(out2, want["out"])

    # a head subset: those heads as in the full run (each against its own KV head), the rest NaN
    heads = [0, 15, 16, 47, 63]
    got3 = R.run_request(req, L, topk, w.softmax_scale, BS, idx, kv, kv_g, kv_g, sel=alt, heads=heads,
                         idx_global=idx_g)
    np.testing.assert_allclose(got3["out"][:, heads], out2[:, heads], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got3["lse"][:, heads], lse2[:, heads], rtol=0, atol=1e-12)
    rest = [h for h in range(w.n_heads) if h not in heads]
    assert np.isnan(got3["out"][:, rest]).all() and np.isnan(got3["lse"][:, rest]).all()


def test_paged_route_sees_a_wrong_row_map():
    """The comparison above is sensitive to the token-to-row map: the same request
    with two tokens of a selected block swapped in K gives a different output."""
    w = synth.scaled(synth.WORKLOADS["b32_32k"], batch=2, q_len=1, ctx=700, topk=4)
    req = synth.request(w, 0, 700)
    q, q_idx, keys, kscale, K, V = _decoded_request(w, req, 700, 1.0, 1.0)
    want = M.decode_step(q, q_idx, keys, kscale, K, V, 700, 4, w.softmax_scale, BS)
    blk = int(want["sel"][0, 0, 0])
    K2 = K.copy()
    K2[[blk * BS, blk * BS + 1]] = K2[[blk * BS + 1, blk * BS]]
    V2 = V.copy()
    V2[blk * BS] = V2[blk * BS + 2]
    bad = M.sparse_gqa(q, K2, V2, 700, want["sel"], w.softmax_scale, BS)[0]
    assert np.abs(bad - want["out"]).max() > 1e-6
