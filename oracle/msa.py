"""The three MSA decode stages, per request, in fp64.

TEST INFRASTRUCTURE (see the package docstring).

Stages ("MiniMax M3 vLLM サポート：…", section "MSA 実行プロセス"):
  1. Block scoring: a small index head scores every candidate KV block.
  2. Block selection: the top-k blocks, with local_blocks=1 keeping the block
     that holds the query token.
  3. Sparse GQA: online-softmax attention over the selected blocks only.

Notation: L tokens cached for the request (query tokens included), Q query
positions p_j = L - Q + j, local block l_j = p_j // BS, H query heads sharing G
KV heads (query head h reads KV head h // (H / G)), I index heads.

Readings where the pages are silent (each is listed in the design notes):
  * The block score is the maximum over the block's tokens of the index dot
    product s_t * (q_idx . k_t), s_t being the key's per-token scale (1 for fp32
    keys). The positive global score scale is left out: it cannot change the
    order ("vLLM、AMD Instinct MI355X上で…", question 2).
  * Index head g selects the blocks that KV head g attends over (one selection
    per index head; the MI355X page's TP8 shape keeps one KV head and one index
    head per rank).
  * Candidates for position j are the blocks n < l_j (all fully visible). The
    local block l_j is always taken and does not compete. k counts the local
    block: top-(k-1) + local, so 16 blocks are 2,048 keys ("MiniMax-M3.1-Flash
    Day-0 対応", section "MSAの仕組み").
  * Order: higher score first, then lower block id. The selection is returned as
    ascending block ids padded with -1.
  * Inside the local block only tokens t <= p_j are attended (causal).
  * Attention logits are softmax_scale * q . k; no cap, no sink.
"""
from __future__ import annotations

import numpy as np


def query_positions(seq_len: int, q_len: int) -> np.ndarray:
    return seq_len - q_len + np.arange(q_len)


def gather_tokens(pages: np.ndarray, table_row: np.ndarray, n_tokens: int, block_size: int) -> np.ndarray:
    """Paged cache [P, X, BS, ...] -> the request's tokens [n_tokens, X, ...] in logical order."""
    nb = (n_tokens + block_size - 1) // block_size
    blk = pages[np.asarray(table_row[:nb], dtype=np.int64)]          # [nb, X, BS, ...]
    blk = np.moveaxis(blk, 2, 1)                                     # [nb, BS, X, ...]
    return blk.reshape((nb * block_size,) + blk.shape[2:])[:n_tokens]


def index_scores(q_idx, keys, key_scale, seq_len: int, block_size: int) -> np.ndarray:
    """Stage 1. Returns S [Q, I, nb] (nb = ceil(L / BS)); S = -inf where n >= l_j.

    q_idx [Q, I, D]; keys [>= l_max * BS, I, D] decoded index keys; key_scale
    [>= l_max * BS, I] or None.
    """
    q_idx = np.asarray(q_idx, dtype=np.float64)
    Q, I, D = q_idx.shape
    BS = block_size
    pos = query_positions(seq_len, Q)
    ell = pos // BS
    nb = (seq_len + BS - 1) // BS
    S = np.full((Q, I, nb), -np.inf)
    lmax = int(ell.max())
    if lmax == 0:
        return S
    k = np.asarray(keys[: lmax * BS], dtype=np.float64).reshape(lmax, BS, I, D)
    dots = np.einsum("qid,ntid->qint", q_idx, k)                     # [Q, I, n, t]
    if key_scale is not None:
        s = np.asarray(key_scale[: lmax * BS], dtype=np.float64).reshape(lmax, BS, I)
        dots = dots * np.transpose(s, (2, 0, 1))[None]                # s_t * (q . k_t)
    bmax = dots.max(axis=3)                                           # max over the block's tokens
    for j in range(Q):
        S[j, :, : ell[j]] = bmax[j, :, : ell[j]]
    return S


def select_row(scores: np.ndarray, ell: int, topk: int):
    """Stage 2 for one (position, head): returns (ascending ids padded with -1, margin).

    margin = relative gap between the last chosen and the first unchosen
    competing candidate (inf when every candidate was chosen).
    """
    cand = sorted(range(ell), key=lambda n: (-float(scores[n]), n))
    take = min(topk - 1, ell)
    chosen = cand[:take]
    sel = sorted(chosen + [ell])
    sel = np.array(sel + [-1] * (topk - len(sel)), dtype=np.int32)
    if 0 < take < ell:
        a, b = float(scores[cand[take - 1]]), float(scores[cand[take]])
        den = max(abs(a), abs(b))
        margin = 0.0 if den == 0 else (a - b) / den
    else:
        margin = np.inf     # the chosen set does not depend on the scores
    return sel, margin


def select_blocks(S: np.ndarray, seq_len: int, topk: int, block_size: int):
    """Stage 2 for a request: S [Q, I, nb] -> (sel [Q, I, topk] int32, margin [Q, I])."""
    Q, I, _ = S.shape
    ell = query_positions(seq_len, Q) // block_size
    sel = np.empty((Q, I, topk), dtype=np.int32)
    margin = np.empty((Q, I))
    for j in range(Q):
        for g in range(I):
            sel[j, g], margin[j, g] = select_row(S[j, g], int(ell[j]), topk)
    return sel, margin


def attended_tokens(sel_row, pos: int, seq_len: int, block_size: int) -> np.ndarray:
    """Token ids of the selected blocks that the query at ``pos`` may see."""
    toks = [np.arange(b * block_size, (b + 1) * block_size) for b in sel_row if b >= 0]
    if not toks:
        return np.zeros(0, dtype=np.int64)
    t = np.concatenate(toks)
    return t[(t <= pos) & (t < seq_len)]


def _softmax_attend(q, K, V, scale):
    s = scale * (K @ q)
    m = s.max()
    w = np.exp(s - m)
    z = w.sum()
    return (w @ V) / z, m + np.log(z)


def sparse_gqa(q, K, V, seq_len: int, sel, softmax_scale: float, block_size: int):
    """Stage 3. q [Q, H, D]; K, V [L, G, D] decoded; sel [Q, G, topk].

    Returns out [Q, H, D] and lse [Q, H] (natural log of the softmax denominator
    including the max).
    """
    q = np.asarray(q, dtype=np.float64)
    Q, H, D = q.shape
    G = K.shape[1]
    pos = query_positions(seq_len, Q)
    out = np.zeros((Q, H, D))
    lse = np.full((Q, H), -np.inf)
    for j in range(Q):
        for h in range(H):
            g = h // (H // G)
            t = attended_tokens(sel[j, g], int(pos[j]), seq_len, block_size)
            if t.size == 0:
                continue
            out[j, h], lse[j, h] = _softmax_attend(q[j, h], K[t, g], V[t, g], softmax_scale)
    return out, lse


def dense_gqa(q, K, V, seq_len: int, softmax_scale: float):
    """Causal attention of every query position over all tokens t <= p_j (no selection)."""
    q = np.asarray(q, dtype=np.float64)
    Q, H, D = q.shape
    G = K.shape[1]
    pos = query_positions(seq_len, Q)
    out = np.zeros((Q, H, D))
    lse = np.zeros((Q, H))
    for j in range(Q):
        n = int(pos[j]) + 1
        for h in range(H):
            g = h // (H // G)
            logits = softmax_scale * np.einsum("td,d->t", K[:n, g], q[j, h])
            m = np.max(logits)
            e = np.exp(logits - m)
            out[j, h] = np.einsum("t,td->d", e, V[:n, g]) / e.sum()
            lse[j, h] = m + np.log(e.sum())
    return out, lse


def decode_step(q, q_idx, keys, key_scale, K, V, seq_len: int, topk: int, softmax_scale: float,
                block_size: int):
    """All three stages for one request; returns dict(S, sel, margin, out, lse)."""
    S = index_scores(q_idx, keys, key_scale, seq_len, block_size)
    sel, margin = select_blocks(S, seq_len, topk, block_size)
    out, lse = sparse_gqa(q, K, V, seq_len, sel, softmax_scale, block_size)
    return dict(S=S, sel=sel, margin=margin, out=out, lse=lse)
