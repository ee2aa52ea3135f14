"""The step in front of the decode path: per-head RMS normalisation of the query
and key projections, rotary position embedding, and insertion into the caches.

TEST INFRASTRUCTURE (see the package docstring).

"MiniMax-M3.1-Flash Day-0 対応" (aisoku.org), section "最適化と数値": a fused
QKV GEMM + norm + RoPE + KV insert; "MiniMax M3 vLLM サポート：…"
(agentlenshq.com), section "カーネル融合": QKNorm + RoPE + KV insertion fused
to save HBM round trips and launches; "vLLM、AMD Instinct MI355X上で…",
question 3: the fused projection also normalises, rotates and writes the index
query/key, and a layer that reuses another layer's selection skips that
branch. The pages give no formulas; the readings here are this project's:

* RMSNorm of one head's D values x with weight w (fp32, per dim) and eps:
  y_d = x_d / sqrt(mean_d(x^2) + eps) * w_d.
* Rotary embedding at position pos with base theta, rotating over all D dims
  in the half-split layout: for i < D/2, phi_i = pos * theta^(-2i/D),
  (y_i, y_{i+D/2}) = (x_i cos phi_i - x_{i+D/2} sin phi_i,
                      x_i sin phi_i + x_{i+D/2} cos phi_i).
* Applied to the attention query and key heads and the index query and key
  heads (each with its own weight); V passes unchanged.
* The results are rounded to bf16 (as an unfused norm/RoPE operator would
  emit them); the caches store the bf16 key and V through the cache's own
  quantiser (``quant``), exactly as the plain insert does.

Computed in fp64 here.
"""
from __future__ import annotations

import numpy as np

from . import formats


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """[..., D] -> [..., D], fp64."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(w, dtype=np.float64)


def rope_angles(pos: np.ndarray, D: int, theta: float) -> np.ndarray:
    """phi[t, i] = pos_t * theta^(-2i/D), i < D/2, fp64."""
    i = np.arange(D // 2, dtype=np.float64)
    inv = float(theta) ** (-2.0 * i / D)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """x [T, heads, D] at positions pos [T] -> rotated [T, heads, D], fp64."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    phi = rope_angles(pos, D, theta)[:, None, :]          # [T, 1, D/2]
    c, s = np.cos(phi), np.sin(phi)
    a, b = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> the nearest bf16 (ties to even) as uint16 bits, via an fp32 round
    that cannot change the bf16 decision (fp64 -> fp32 keeps 24 bits)."""
    f = np.asarray(x, dtype=np.float64)
    f32 = f.astype(np.float32)
    # A double rounding fp64 -> fp32 -> bf16 can only differ from the direct one
    # when the fp32 value lands exactly on a bf16 tie; resolve those from fp64.
    u = f32.view(np.uint32)
    lsb = (u >> 16) & 1
    tie = (u & 0xFFFF) == 0x8000
    rounded = ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)
    if tie.any():
        down = (u >> 16).astype(np.uint16)
        lo = formats.bf16_to_f64(down)
        up = formats.bf16_to_f64((down + 1).astype(np.uint16))
        exact = np.abs(f - lo) == np.abs(up - f)
        nearer_up = np.abs(up - f) < np.abs(f - lo)
        pick = np.where(exact, rounded, np.where(nearer_up, down + 1, down)).astype(np.uint16)
        rounded = np.where(tie, pick, rounded).astype(np.uint16)
    return rounded


def norm_rope(x: np.ndarray, w: np.ndarray, pos: np.ndarray, eps: float, theta: float) -> np.ndarray:
    """RMSNorm then rotary embedding of x [T, heads, D] (bf16 bits or floats) -> bf16 bits."""
    if x.dtype == np.uint16:
        x = formats.bf16_to_f64(x)
    return to_bf16(rope(rms_norm(x, w, eps), pos, theta))
