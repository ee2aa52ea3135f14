"""Pins for the oracle's three MSA stages (CPU only).

The oracle is checked against things other than itself: hand-worked examples
(golden files), closed forms, brute force (dense attention, a library SDPA),
library re-computations of the scores, and invariants of the method (positive
score scale, page permutation, key cap). Each pin is chosen so that a plausible
mistake (dropped scale, wrong head map, missing causal mask, transposed
operand, wrong tie order) fails at least one test.
"""
import math

import numpy as np
import pytest
import torch

from conftest import load_golden, num
from oracle import formats as F
from oracle import msa as M


def _arr(x):
    return np.array([[num(v) for v in row] for row in x]) if isinstance(x[0], list) else np.array([num(v) for v in x])


def test_hand_example_all_cases():
    g = load_golden("hand_example.json")
    BS = g["block_size"]
    for case in g["cases"]:
        L, Q, k = case["seq_len"], case["q_len"], case["topk"]
        qi = np.tile(np.array(g["index_query"])[None, None, :], (Q, 1, 1))
        keys = np.array(g["index_keys"])[:, None, :]
        q = np.tile(np.array(g["query"])[None, None, :], (Q, 1, 1))
        K = np.array(g["keys"])[:, None, :]
        V = np.array(g["values"])[:, None, :]
        r = M.decode_step(q, qi, keys, None, K, V, L, k, g["softmax_scale"], BS)
        assert np.array_equal(r["S"][:, 0, :], _arr(case["scores"]))
        assert r["sel"][:, 0, :].tolist() == case["sel"]
        np.testing.assert_allclose(r["out"][:, 0, :], np.array(case["out"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(r["lse"][:, 0], np.array(case["lse"]), rtol=0, atol=1e-14)


def test_tie_break_lower_block_id():
    g = load_golden("tie_break.json")
    BS, L = g["block_size"], g["seq_len"]
    qi = np.array(g["index_query"])[None, None, :]
    keys = np.array(g["index_keys"])[:, None, :]
    S = M.index_scores(qi, keys, None, L, BS)
    assert np.array_equal(S[0, 0], _arr(g["scores"]))
    K = np.zeros((L, 1, 2))
    V = np.stack([np.arange(L, dtype=np.float64), np.ones(L)], axis=1)[:, None, :]
    q = np.ones((1, 1, 2))
    for case in g["cases"]:
        sel, _ = M.select_blocks(S, L, case["topk"], BS)
        assert sel[0, 0].tolist() == case["sel"]
        out, lse = M.sparse_gqa(q, K, V, L, sel, g["softmax_scale"], BS)
        np.testing.assert_allclose(out[0, 0], case["out"], atol=1e-14)
        assert lse[0, 0] == pytest.approx(case["lse"], abs=1e-14)


def test_fp8_index_example():
    g = load_golden("fp8_index_example.json")
    keys = F.e4m3_decode(np.array(g["codes"], dtype=np.uint8))[:, None, :]
    s = np.array(g["scales"])[:, None]
    qi = np.array(g["index_query"])[None, None, :]
    S = M.index_scores(qi, keys, s, g["seq_len"], g["block_size"])
    assert np.array_equal(S[0, 0], _arr(g["scores"]))


def _rand_case(rng, L=1000, Q=1, H=8, G=2, I=2, D=16, BS=16):
    q = rng.standard_normal((Q, H, D))
    qi = rng.standard_normal((Q, I, D))
    keys = rng.standard_normal((L, I, D))
    ks = rng.uniform(0.1, 2.0, (L, I))
    K = rng.standard_normal((L, G, D))
    V = rng.standard_normal((L, G, D))
    return q, qi, keys, ks, K, V


def test_sparse_equals_dense_when_k_covers_every_block():
    rng = np.random.default_rng(11)
    for L, Q in ((1000, 1), (1000, 5), (17, 3), (16, 1), (5, 2)):
        q, qi, keys, ks, K, V = _rand_case(rng, L=L, Q=Q)
        BS = 16
        k = (L + BS - 1) // BS + 1
        r = M.decode_step(q, qi, keys, ks, K, V, L, k, 0.25, BS)
        od, ld = M.dense_gqa(q, K, V, L, 0.25)
        np.testing.assert_allclose(r["out"], od, atol=1e-12, rtol=0)
        np.testing.assert_allclose(r["lse"], ld, atol=1e-12, rtol=0)


def test_dense_matches_library_sdpa():
    rng = np.random.default_rng(12)
    L, Q, H, G, D = 300, 4, 8, 2, 16
    q, _, _, _, K, V = _rand_case(rng, L=L, Q=Q, H=H, G=G, D=D)
    od, _ = M.dense_gqa(q, K, V, L, 0.3)
    rep = H // G
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                       # [1, H, Q, D]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(rep, 0)[None]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(rep, 0)[None]
    pos = torch.arange(L - Q, L)[:, None]
    mask = torch.arange(L)[None, :] <= pos                                # [Q, L]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.3)
    np.testing.assert_allclose(od, ref[0].permute(1, 0, 2).numpy(), atol=1e-12)


def test_scores_match_library_recomputation():
    """Scores from torch's float8 decode + torch einsum + torch amax (a separate code path)."""
    rng = np.random.default_rng(13)
    L, Q, I, D, BS = 700, 3, 2, 32, 32
    codes = rng.integers(0, 256, (L, I, D), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38                                  # no NaN codes
    ks = rng.uniform(0.01, 3.0, (L, I)).astype(np.float32)
    qi = rng.standard_normal((Q, I, D))
    S = M.index_scores(qi, F.e4m3_decode(codes), ks, L, BS)
    kt = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    dots = torch.einsum("qid,tid->qit", torch.from_numpy(qi), kt) * torch.from_numpy(ks.astype(np.float64)).T[None]
    pos = torch.arange(L - Q, L)
    for j in range(Q):
        ell = int(pos[j]) // BS
        ref = dots[j, :, : ell * BS].reshape(I, ell, BS).amax(-1).numpy()
        np.testing.assert_allclose(S[j, :, :ell], ref, rtol=1e-13, atol=0)
        assert np.isneginf(S[j, :, ell:]).all()


def test_selection_matches_library_lexsort():
    rng = np.random.default_rng(14)
    for _ in range(50):
        n = int(rng.integers(1, 300))
        s = rng.integers(-5, 5, n).astype(np.float64)                    # many ties
        for k in (1, 2, 16, 400):
            sel, _ = M.select_row(s, n, k)
            order = np.lexsort((np.arange(n), -s))                         # score desc, id asc
            want = sorted(order[: min(k - 1, n)].tolist() + [n])
            want = want + [-1] * (k - len(want))
            assert sel.tolist() == want


def test_selection_invariant_to_positive_score_scale():
    """Multiplying the index query by c > 0 scales every score by c and keeps the top-k."""
    rng = np.random.default_rng(15)
    q, qi, keys, ks, K, V = _rand_case(rng, L=2000, Q=4)
    S1 = M.index_scores(qi, keys, ks, 2000, 16)
    sel1, _ = M.select_blocks(S1, 2000, 16, 16)
    for c in (0.125, 3.0, 1e-3, 1e3):
        S2 = M.index_scores(qi * c, keys, ks, 2000, 16)
        sel2, _ = M.select_blocks(S2, 2000, 16, 16)
        assert np.array_equal(sel1, sel2)


def test_per_token_scale_is_applied():
    """Two identical keys with different scales: the block holding the larger scale wins."""
    BS, L = 4, 13
    keys = np.ones((L, 1, 2))
    ks = np.ones((L, 1))
    ks[5] = 3.0                      # block 1
    S = M.index_scores(np.array([[[1.0, 1.0]]]), keys, ks, L, BS)
    assert S[0, 0, 1] == 6.0 and S[0, 0, 0] == 2.0 and S[0, 0, 2] == 2.0
    sel, _ = M.select_blocks(S, L, 2, BS)
    assert sel[0, 0].tolist() == [1, 3]


def test_gqa_head_map_closed_form():
    """V is constant per KV head, so head h must output h // (H/G) + 1 exactly."""
    rng = np.random.default_rng(16)
    L, Q, H, G, D, BS = 200, 2, 8, 4, 8, 16
    q = rng.standard_normal((Q, H, D))
    K = rng.standard_normal((L, G, D))
    V = np.broadcast_to((np.arange(G) + 1.0)[None, :, None], (L, G, D)).copy()
    sel = np.tile(np.array([0, 3, 12, -1])[None, None, :], (Q, G, 1))
    out, _ = M.sparse_gqa(q, K, V, L, sel, 0.5, BS)
    want = (np.arange(H) // (H // G) + 1.0)[None, :, None]
    np.testing.assert_allclose(out, np.broadcast_to(want, out.shape), atol=1e-13)


def test_causal_mask_inside_local_block_closed_form():
    """Zero keys give uniform weights; V[t] = t, so the output is the mean attended token id."""
    L, Q, BS = 70, 8, 16
    K = np.zeros((L, 1, 4))
    V = np.broadcast_to(np.arange(L, dtype=np.float64)[:, None, None], (L, 1, 4)).copy()
    q = np.ones((Q, 1, 4))
    sel = np.array([[[4]]] * Q)                          # local block only (tokens 64..69)
    out, lse = M.sparse_gqa(q, K, V, L, sel, 1.0, BS)
    for j in range(Q):
        p = L - Q + j
        if p >= 64:
            toks = np.arange(64, p + 1)
            assert out[j, 0, 0] == pytest.approx(toks.mean(), abs=1e-12)
            assert lse[j, 0] == pytest.approx(math.log(toks.size), abs=1e-12)
        else:
            assert lse[j, 0] == -np.inf                 # block 4 lies wholly in the future
    od, _ = M.dense_gqa(q, K, V, L, 1.0)
    for j in range(Q):
        assert od[j, 0, 0] == pytest.approx((L - Q + j) / 2, abs=1e-12)


def test_block_table_permutation_invariance():
    """Scattering a request into shuffled pages and gathering it back gives the same stages."""
    rng = np.random.default_rng(17)
    L, BS, G = 300, 16, 2
    nb = (L + BS - 1) // BS
    tok = rng.standard_normal((nb * BS, G, 8))
    pages = np.zeros((nb + 3, G, BS, 8))
    perm = rng.permutation(nb + 3)[:nb]
    for n in range(nb):
        pages[perm[n]] = np.moveaxis(tok[n * BS:(n + 1) * BS], 0, 1)
    back = M.gather_tokens(pages, perm, L, BS)
    assert np.array_equal(back, tok[:L])


def test_key_cap_2048_and_traffic_fraction():
    """16 blocks of 128 tokens: never more than 2,048 keys, which is 12.5 % of a 16K context."""
    c = load_golden("page_constants.json")
    BS, k = c["block_size"], 16
    rng = np.random.default_rng(18)
    for L in (1, 127, 128, 129, 2048, 2049, 5000, 16384):
        S = rng.standard_normal((1, 1, (L + BS - 1) // BS))
        sel, _ = M.select_blocks(S, L, k, BS)
        t = M.attended_tokens(sel[0, 0], L - 1, L, BS)
        assert t.size <= c["keys_per_query_cap"]
        assert t.size == min(L, c["keys_per_query_cap"]) or L % BS != 0
    assert k * BS / 16384 == c["long_context_traffic_fraction"]


def test_selection_edge_cases():
    # no candidates: only the local block
    sel, m = M.select_row(np.array([]), 0, 16)
    assert sel.tolist() == [0] + [-1] * 15 and m == np.inf
    # fewer candidates than k-1
    sel, m = M.select_row(np.array([1.0, 5.0, 3.0]), 3, 16)
    assert sel.tolist() == [0, 1, 2, 3] + [-1] * 12 and m == np.inf
    # exactly k-1 candidates
    s = np.arange(15, dtype=np.float64)
    sel, m = M.select_row(s, 15, 16)
    assert sel.tolist() == list(range(16)) and m == np.inf
    # margin between last chosen and first unchosen
    s = np.array([4.0, 1.0, 2.0, 3.0])
    sel, m = M.select_row(s, 4, 3)
    assert sel.tolist() == [0, 3, 4] and m == pytest.approx((3.0 - 2.0) / 3.0)


def test_nvfp4_index_keys_exact_when_representable():
    """Keys whose 16-groups have amax 6 and E2M1 values quantise exactly (global 1):
    the scores equal the exact dot-product maxima."""
    from oracle import run as orun
    rng = np.random.default_rng(19)
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    L, I, D, BS = 600, 2, 128, 128
    keys = rng.choice(vals, (L, I, D)) * rng.choice([-1, 1], (L, I, D))
    keys.reshape(L, I, D // 16, 16)[..., 0] = 6.0                 # amax 6 in every group -> block scale 1
    dec, scale = orun.cached_index_keys(keys.astype(np.float32), "nvfp4", 1.0)
    assert scale is None and np.array_equal(dec, keys)
    qi = rng.standard_normal((1, I, D))
    S = M.index_scores(qi, dec, None, L, BS)
    ell = (L - 1) // BS
    want = np.einsum("id,tid->it", qi[0], keys[: ell * BS]).reshape(I, ell, BS).max(-1)
    np.testing.assert_allclose(S[0, :, :ell], want, rtol=1e-13)


def test_fp8_kv_cache_exact_when_representable():
    """K/V values that are E4M3 codes times a power-of-two tensor scale are stored
    exactly, so a request on an FP8 cache equals the same request on a bf16 cache."""
    from oracle import formats as F
    from oracle import run as orun
    from block_sparse_attention_07_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["tiny"], batch=1, ctx=700)
    req = synth.request(w, 0, 700)
    rng = np.random.default_rng(23)
    s = 2.0 ** -5
    for f in ("k", "v"):
        codes = rng.integers(0, 256, req[f].shape).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0                           # no NaN codes
        req[f] = synth.f32_to_bf16_bits((F.e4m3_decode(codes) * s).astype(np.float32))
    a = orun.run_request(req, 700, w.topk, w.softmax_scale, w.block_size, w.idx_dtype, "bf16")
    b = orun.run_request(req, 700, w.topk, w.softmax_scale, w.block_size, w.idx_dtype, "fp8", s, s)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
    assert np.array_equal(orun.cached_kv_rows(req["k"], "fp8", s), orun.to_f32(req["k"]).astype(np.float64))
