"""Shared parity checks: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (written here once, used by every GPU test):
  * Block scores: |gpu - oracle| <= SCORE_REL * A, with A = max over the block's
    tokens of s_t * sum_d |q_d k_td|. Each product of a bf16 query and an E4M3
    (or E2M1 x E4M3) key is exact in fp32 and the kernel sums 128 of them in
    fp32 before one multiply by s_t (or the global scale), so the error is
    below (128 + 2) * 2^-24 * A ~ 7.8e-6 * A.
  * Selections: bit-exact, except that where the oracle's last chosen and first
    unchosen competing scores differ by less than NEAR_TIE relative, the GPU may
    swap blocks that lie inside that band.
  * Attention output (bf16): max-abs <= 2e-2 and mean-abs <= 2e-3 against the
    oracle run on the GPU's own selection; lse within 1e-3 absolute (logit
    error ~1e-5, fp32 sums of <= 2,048 terms).
"""
from __future__ import annotations

import numpy as np
import torch

from block_sparse_attention_07_gb300 import synth
from oracle import run as orun

SCORE_REL = 2e-5
NEAR_TIE = 1e-4
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def build(w, which=None, lens=None):
    from block_sparse_attention_07_gb300.workload import DeviceWorkload
    return DeviceWorkload(w, "cuda", which=which, lens=lens)


def idx_global(w):
    return float(np.float32(synth.NVFP4_IDX_SYNTH_GLOBAL)) if w.idx_dtype == "nvfp4" else 1.0


def score_bound(req, w, L):
    """A[j, g, n] = max_t s_t * sum_d |q_jgd k_tgd| over the block's tokens."""
    keys, scale = orun.cached_index_keys(req["idx_k"], w.idx_dtype, idx_global(w))
    qi = np.abs(orun.to_f32(req["q_idx"]).astype(np.float64))
    BS = w.block_size
    nb = (L + BS - 1) // BS
    lmax = (L - 1) // BS
    A = np.zeros((w.q_len, w.n_idx_heads, nb))
    if lmax == 0:
        return A
    k = np.abs(keys[: lmax * BS]).reshape(lmax, BS, w.n_idx_heads, -1)
    d = np.einsum("qid,ntid->qint", qi, k)
    if scale is not None:
        d = d * np.transpose(scale[: lmax * BS].reshape(lmax, BS, -1), (2, 0, 1))[None]
    A[:, :, :lmax] = d.max(axis=3)
    return A


def check_scores(gpu_S, ora_S, A, where=""):
    fin = np.isfinite(ora_S)
    assert np.array_equal(np.isfinite(gpu_S), fin), f"{where}: -inf pattern differs"
    err = np.abs(gpu_S[fin] - ora_S[fin])
    lim = SCORE_REL * A[fin] + 1e-30
    bad = err > lim
    assert not bad.any(), f"{where}: {bad.sum()} scores off, worst {np.max(err / lim):.3g}x the bound"


def check_selection(gpu_sel, ora_S, L, w, gpu_S=None, where=""):
    """GPU selection == oracle selection up to near ties; and == oracle selection of the GPU's own scores."""
    from oracle import msa as om
    Q = w.q_len
    BS = w.block_size
    pos = L - Q + np.arange(Q)
    for j in range(Q):
        ell = int(pos[j]) // BS
        for g in range(w.n_idx_heads):
            gs = gpu_sel[j, g]
            if gpu_S is not None:
                exact, _ = om.select_row(gpu_S[j, g].astype(np.float64), ell, w.topk)
                assert np.array_equal(gs, exact), f"{where}: select kernel != oracle select on GPU scores (j={j} g={g})"
            os_, margin = om.select_row(ora_S[j, g], ell, w.topk)
            if np.array_equal(gs, os_):
                continue
            assert margin < NEAR_TIE, f"{where}: selection differs with margin {margin:.3g} (j={j} g={g})"
            sc = ora_S[j, g]
            take = min(w.topk - 1, ell)
            order = sorted(range(ell), key=lambda n: (-sc[n], n))
            a = sc[order[take - 1]]
            band = {n for n in range(ell) if abs(sc[n] - a) <= NEAR_TIE * max(abs(sc[n]), abs(a))}
            diff = set(gs[gs >= 0].tolist()) ^ set(os_[os_ >= 0].tolist())
            assert diff <= band, f"{where}: blocks {diff - band} outside the near-tie band"


def check_attention(gpu_out, gpu_lse, ora_out, ora_lse, where="", heads=None):
    if heads is not None:
        gpu_out, ora_out = gpu_out[:, heads], ora_out[:, heads]
        gpu_lse, ora_lse = gpu_lse[:, heads], ora_lse[:, heads]
    err = np.abs(gpu_out.astype(np.float64) - ora_out)
    assert np.isfinite(gpu_out).all(), f"{where}: non-finite output"
    assert err.max() <= OUT_MAX_ABS, f"{where}: max-abs {err.max():.3g}"
    assert err.mean() <= OUT_MEAN_ABS, f"{where}: mean-abs {err.mean():.3g}"
    fin = np.isfinite(ora_lse)
    assert np.array_equal(np.isfinite(gpu_lse), fin), f"{where}: lse -inf pattern differs"
    if fin.any():
        le = np.abs(gpu_lse[fin] - ora_lse[fin])
        assert le.max() <= LSE_ABS, f"{where}: lse max-abs {le.max():.3g}"


def kv_globals(w):
    """Per-tensor K/V scales of the workload's cache (1 for bf16)."""
    s = synth.kv_scale(w)
    return s, s


def verify_workload(dw, w, full_lens, sample=None, heads=None, run_step=True):
    """Runs a decode step on the device and checks the sampled requests against the oracle."""
    if run_step:
        dw.step()
    torch.cuda.synchronize()
    flags = dw.check_flags()
    assert flags == 0, f"device flags {flags:#x}"
    S = dw.scores.cpu().numpy()
    sel = dw.selected.cpu().numpy()
    out = dw.out.float().cpu().numpy()
    lse = dw.lse.cpu().numpy()
    kg, vg = kv_globals(w)
    idx = range(len(dw.which)) if sample is None else sample
    for bi in idx:
        b = dw.which[bi]
        L = int(full_lens[b])
        req = synth.request(w, b, L)
        ora = orun.run_request(req, L, w.topk, w.softmax_scale, w.block_size, w.idx_dtype, w.kv_dtype, kg, vg,
                               sel=sel[bi], heads=heads, idx_global=idx_global(w))
        nb = ora["S"].shape[2]
        where = f"{w.name} b={b} L={L}"
        check_scores(S[bi, :, :, :nb], ora["S"], score_bound(req, w, L), where)
        assert np.isneginf(S[bi, :, :, nb:]).all(), f"{where}: scores beyond the request not -inf"
        check_selection(sel[bi], ora["S"], L, w, gpu_S=S[bi, :, :, :nb], where=where)
        check_attention(out[bi], lse[bi], ora["out"], ora["lse"], where, heads=heads)


def poison_unwritten_slots(dw):
    """Fills every cache slot past each request's length (the tail of its last
    page, which no step has written) with NaN bit patterns: bf16 0xFFFF, E4M3
    0xFF, NVFP4 block scales 0x7F (E4M3 NaN), fp32 NaN. The method reads none of
    them: the indexer scores only whole blocks before the local one, and the
    attention gives tokens past the causal limit probability 0."""
    import torch
    c, ic = dw.cache, dw.idx_cache
    for bi, L in enumerate(dw.lens):
        off = int(L) % 128
        if off == 0:
            continue
        page = int(dw.block_table[bi, (int(L) - 1) // 128])
        if c.k.dtype == torch.bfloat16:
            c.k.view(torch.int16)[page, :, off:] = -1
            c.v.view(torch.int16)[page, :, off:] = -1
        else:
            c.k[page, :, off:] = 0xFF
            c.v[page, :, off:] = 0xFF
            if c.k_scale is not None:
                c.k_scale[page, :, off:] = 0x7F
                c.v_scale[page, :, off:] = 0x7F
        if ic.keys.dtype == torch.float32:
            ic.keys[page, :, off:] = float("nan")
        else:
            ic.keys[page, :, off:] = 0xFF
            if ic.scale is not None:
                ic.scale[page, :, off:] = float("nan")
            if ic.block_scale is not None:
                ic.block_scale[page, :, off:] = 0x7F
    torch.cuda.synchronize()
