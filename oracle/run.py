"""Runs the oracle on one request of a synthetic workload.

TEST INFRASTRUCTURE (see the package docstring).

Takes the raw (pre-cache) inputs of a request exactly as the generator drew
them, fills the caches with the oracle's own quantisers, decodes them to fp64
and runs the three stages. Nothing here comes from the CUDA path.

Large requests are handled in pieces that do not change any result: index keys
are quantised and decoded in token chunks (the quantiser works per token and
head), and only the KV blocks that the selection uses are quantised and
decoded for the attention stage.
"""
from __future__ import annotations

import numpy as np

from . import formats, msa, quant

_CHUNK = 16384


def to_f32(a: np.ndarray) -> np.ndarray:
    """uint16 arrays are bf16 bit patterns; float32 arrays are taken as they are."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(a, dtype=np.float32)


def cached_index_keys(idx_k: np.ndarray, idx_dtype: str, idx_global: float = 1.0):
    """The index cache's content for these tokens, decoded: (keys fp64 [L, I, D], scale fp64 [L, I] or None).

    FP8 keys carry a per-token scale; NVFP4 keys (E2M1 x E4M3 block scale x
    global scale) decode to their value and have no per-token scale.
    """
    L = idx_k.shape[0]
    keys = np.empty(idx_k.shape, dtype=np.float64)
    scale = np.empty(idx_k.shape[:2], dtype=np.float64) if idx_dtype == "fp8" else None
    for t0 in range(0, L, _CHUNK):
        x = to_f32(idx_k[t0:t0 + _CHUNK])
        if idx_dtype == "f32":
            keys[t0:t0 + _CHUNK] = x
        elif idx_dtype == "nvfp4":
            codes, sc = quant.quant_nvfp4(x, idx_global)
            keys[t0:t0 + _CHUNK] = formats.nvfp4_decode(codes, sc, idx_global)
        else:
            codes, s = quant.quant_index_keys_fp8(x)
            keys[t0:t0 + _CHUNK] = formats.e4m3_decode(codes)
            scale[t0:t0 + _CHUNK] = s
    return keys, scale


def cached_kv_rows(x: np.ndarray, kv_dtype: str, global_scale: float) -> np.ndarray:
    """The KV cache's content for these token rows [T, G, D], decoded to fp64."""
    f = to_f32(x)
    if kv_dtype == "bf16":
        return f.astype(np.float64)
    if kv_dtype == "fp8":
        return formats.e4m3_decode(quant.quant_kv_fp8(f, global_scale)) * float(np.float32(global_scale))
    codes, scales = quant.quant_nvfp4(f, global_scale)
    return formats.nvfp4_decode(codes, scales, global_scale)


class _Rows:
    """K or V restricted to a set of token ids; indexable as [t, g] like the full array."""

    def __init__(self, tokens: np.ndarray, rows: np.ndarray, length: int):
        self.pos = np.full(length, -1, dtype=np.int64)
        self.pos[tokens] = np.arange(tokens.size)
        self.rows = rows
        self.shape = (length,) + rows.shape[1:]

    def __getitem__(self, idx):
        t, g = idx
        p = self.pos[t]
        assert (p >= 0).all(), "token outside the decoded blocks"
        return self.rows[p, g]


def run_request(req: dict, seq_len: int, topk: int, softmax_scale: float, block_size: int, idx_dtype: str,
                kv_dtype: str, k_global: float = 1.0, v_global: float = 1.0, sel=None, heads=None,
                idx_global: float = 1.0):
    """All three stages for one request.

    ``sel`` ([Q, G, topk]) replaces the oracle's own selection in the attention
    stage (to check attention on a selection made elsewhere). ``heads``
    restricts the attention stage to some query heads (others are NaN).
    Returns dict(S, sel, margin, out, lse, sel_used).
    """
    keys, kscale = cached_index_keys(req["idx_k"], idx_dtype, idx_global)
    qi = to_f32(req["q_idx"]).astype(np.float64)
    S = msa.index_scores(qi, keys, kscale, seq_len, block_size)
    del keys
    own_sel, margin = msa.select_blocks(S, seq_len, topk, block_size)
    use = own_sel if sel is None else np.asarray(sel)

    blocks = np.unique(use[use >= 0])
    tok = (blocks[:, None] * block_size + np.arange(block_size)[None, :]).reshape(-1)
    tok = tok[tok < seq_len]
    K = _Rows(tok, cached_kv_rows(req["k"][tok], kv_dtype, k_global), seq_len)
    V = _Rows(tok, cached_kv_rows(req["v"][tok], kv_dtype, v_global), seq_len)
    q = to_f32(req["q"]).astype(np.float64)
    Q, H, D = q.shape
    G = K.shape[1]
    if heads is None:
        out, lse = msa.sparse_gqa(q, K, V, seq_len, use, softmax_scale, block_size)
    else:
        out = np.full(q.shape, np.nan)
        lse = np.full((Q, H), np.nan)
        grp = H // G
        for h in heads:
            g = h // grp
            Kg = _Rows(tok, K.rows[:, g:g + 1], seq_len)
            Vg = _Rows(tok, V.rows[:, g:g + 1], seq_len)
            o1, l1 = msa.sparse_gqa(q[:, h:h + 1], Kg, Vg, seq_len, use[:, g:g + 1], softmax_scale, block_size)
            out[:, h], lse[:, h] = o1[:, 0], l1[:, 0]
    return dict(S=S, sel=own_sel, margin=margin, out=out, lse=lse, sel_used=use)
