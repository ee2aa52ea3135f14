"""Seeded synthetic inputs for the MSA decode path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no scoring, selection, attention or quantisation). Both the
CUDA path (through the tests and the benchmark) and the fp64 oracle are fed from
here, so the two sides always see the same inputs.

Every array of request ``b`` comes from its own numpy PCG64 stream, keyed by
(workload seed, request, field). A test can therefore regenerate the inputs of a
few sampled requests of a full-size workload without generating the rest.

Workloads (sizes and value recipes of the MiniMax-M3 decode shapes: 64 query
heads, 4 KV heads, 4 index heads, head_dim 128, 128-token KV blocks, top-16
blocks including the local one, at most 2,048 keys per query):

* ``tiny``      batch 2, 4,096 tokens each, 1 query token, fp32 index keys.
* ``b32_32k``   batch 32, 32,768 tokens, 1 query token, FP8 index keys, bf16 KV.
* ``ragged``    batch 64, lengths uniform in [8192, 131072] (never a multiple
                of 128), 10 % of blocks planted +2 sigma.
* ``spec8``     batch 32, 65,536 tokens, 8 query positions per request.
* ``nvfp4_256k`` batch 16, 262,144 tokens, NVFP4 KV.
* ``b32_32k_fp4idx`` and ``fp4_256k``: as ``b32_32k`` and ``nvfp4_256k`` with
  NVFP4 index keys.
* ``fp8kv_32k``: as ``b32_32k`` with FP8 E4M3 K/V (one scale per tensor).
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BLOCK = 128
HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    q_len: int
    ctx: int | None            # fixed context length, or None for ragged
    ctx_range: tuple | None    # (lo, hi) for ragged lengths
    idx_dtype: str             # "f32" (fp32 index keys/query), "fp8" or "nvfp4" (bf16 source, quantised cache)
    kv_dtype: str              # "bf16", "fp8" or "nvfp4"
    planted: bool              # ragged recipe: 10 % of blocks offset by +2 sigma
    n_heads: int = 64
    n_kv_heads: int = 4
    n_idx_heads: int = 4
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK
    topk: int = 16
    seed: int = 20261202

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS = {
    "tiny": Workload("tiny", 2, 1, 4096, None, "f32", "bf16", False, seed=20261202),
    "b32_32k": Workload("b32_32k", 32, 1, 32768, None, "fp8", "bf16", False, seed=20261203),
    "ragged": Workload("ragged", 64, 1, None, (8192, 131072), "fp8", "bf16", True, seed=20261204),
    "spec8": Workload("spec8", 32, 8, 65536, None, "fp8", "bf16", False, seed=20261205),
    "nvfp4_256k": Workload("nvfp4_256k", 16, 1, 262144, None, "fp8", "nvfp4", False, seed=20261206),
    # NVFP4 index keys (the indexer format of the NVFP4 checkpoint's serving recipe)
    "b32_32k_fp4idx": Workload("b32_32k_fp4idx", 32, 1, 32768, None, "nvfp4", "bf16", False, seed=20261207),
    "fp4_256k": Workload("fp4_256k", 16, 1, 262144, None, "nvfp4", "nvfp4", False, seed=20261208),
    # FP8 E4M3 K/V with a per-tensor scale (the other published KV format)
    "fp8kv_32k": Workload("fp8kv_32k", 32, 1, 32768, None, "fp8", "fp8", False, seed=20261209),
}

# Field ids of the per-request random streams.
_F_LEN, _F_PERM, _F_Q, _F_QIDX, _F_IDXK, _F_OFF, _F_K, _F_V, _F_PLANT = range(9)

# NVFP4 global scale used by the synthetic recipe: a per-tensor calibration
# constant (amax 6, i.e. six standard deviations of N(0,1) data, over the
# largest E2M1 magnitude times the largest E4M3 magnitude).
NVFP4_SYNTH_GLOBAL = 6.0 / (6.0 * 448.0)
# Index keys carry block offsets on top of N(0,1); their calibration amax is 8.
NVFP4_IDX_SYNTH_GLOBAL = 8.0 / (6.0 * 448.0)
# FP8 K/V per-tensor scale: amax 6 over the largest E4M3 magnitude.
FP8_KV_SYNTH_SCALE = 6.0 / 448.0


# Seed offset between the attention layers of one model (layer l uses seed + l * stride).
LAYER_SEED_STRIDE = 7919


# Synthetic parameters of the norm / rotary step in front of the decode path
# (the pages give none): RMSNorm epsilon and rotary base.
PROLOGUE_EPS = 1e-6
PROLOGUE_THETA = 10000.0


def norm_weights(w: Workload) -> dict:
    """Per-dim fp32 RMSNorm weights of the query, key, index query and index key
    projections: 1 + 0.1 * N(0, 1), seeded per workload."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 99991])))
    return {name: (1.0 + 0.1 * rng.standard_normal(w.head_dim)).astype(np.float32)
            for name in ("q", "k", "idx_q", "idx_k")}


def kv_scale(w: Workload) -> float:
    """The per-tensor K/V scale of the workload's cache format (fp32 value)."""
    s = {"bf16": 1.0, "fp8": FP8_KV_SYNTH_SCALE, "nvfp4": NVFP4_SYNTH_GLOBAL}[w.kv_dtype]
    return float(np.float32(s))


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def _rng(w: Workload, b: int, field: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, b, field])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def seq_lens(w: Workload) -> np.ndarray:
    """Context length of every request (tokens in the cache, query tokens included)."""
    if w.ctx is not None:
        return np.full(w.batch, w.ctx, dtype=np.int32)
    lo, hi = w.ctx_range
    out = np.empty(w.batch, dtype=np.int32)
    for b in range(w.batch):
        n = int(_rng(w, b, _F_LEN).integers(lo, hi + 1))
        if n % w.block_size == 0:
            n += 1
        out[b] = n
    return out


def blocks_per_seq(w: Workload, lens: np.ndarray) -> np.ndarray:
    return (lens.astype(np.int64) + w.block_size - 1) // w.block_size


def page_table(w: Workload, lens: np.ndarray, spare_pages: int = 0):
    """Logical block -> physical page map, pages shuffled by a seeded permutation.

    Returns (block_table [B, max_blocks] int32 padded with -1, num_pages).
    """
    nb = blocks_per_seq(w, lens)
    max_blocks = int(nb.max())
    num_pages = int(nb.sum()) + spare_pages
    perm = _rng(w, 0, _F_PERM).permutation(num_pages).astype(np.int32)
    table = np.full((w.batch, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        table[b, : nb[b]] = perm[off: off + nb[b]]
        off += int(nb[b])
    return table, num_pages


def request(w: Workload, b: int, length: int) -> dict:
    """All inputs of request ``b`` with ``length`` cached tokens.

    Returns host arrays:
      q      [Q, H, D]  uint16 bf16 bits      (attention query)
      q_idx  [Q, I, D]  float32 (f32 index) or uint16 bf16 bits (fp8 index)
      idx_k  [L, I, D]  float32 or uint16 bf16 bits  (index keys before caching)
      k, v   [L, G, D]  uint16 bf16 bits      (keys/values before caching)
    """
    Q, H, G, I, D, BS = w.q_len, w.n_heads, w.n_kv_heads, w.n_idx_heads, w.head_dim, w.block_size
    out = {}
    out["q"] = f32_to_bf16_bits(_rng(w, b, _F_Q).standard_normal((Q, H, D), dtype=np.float32))
    qi = _rng(w, b, _F_QIDX).standard_normal((Q, I, D), dtype=np.float32)
    if w.idx_dtype != "f32":
        qi = bf16_bits_to_f32(f32_to_bf16_bits(qi))
    out["q_idx"] = qi if w.idx_dtype == "f32" else f32_to_bf16_bits(qi)

    # Index keys: N(0,1) plus a per-block offset along the unit mean index query
    # of each index head, so that block scores differ from block to block.
    nblk = (length + BS - 1) // BS
    keys = _rng(w, b, _F_IDXK).standard_normal((nblk * BS, I, D), dtype=np.float32)
    qmean = qi.astype(np.float64).mean(axis=0)                       # [I, D]
    qhat = qmean / np.linalg.norm(qmean, axis=1, keepdims=True)       # [I, D]
    if w.planted:
        # 10 % of blocks get keys += 2 * qhat: a dot-product offset of +2 sigma,
        # sigma = |q_idx| being the std of q.k for k ~ N(0, I).
        plant = _rng(w, b, _F_PLANT).random((nblk, I)) < 0.10
        off = np.where(plant, 2.0, 0.0)
    else:
        off = 0.5 * _rng(w, b, _F_OFF).standard_normal((nblk, I))
    keys = keys.reshape(nblk, BS, I, D)
    keys += (off[:, None, :, None] * qhat[None, None, :, :]).astype(np.float32)
    keys = keys.reshape(nblk * BS, I, D)[:length]
    out["idx_k"] = np.ascontiguousarray(keys) if w.idx_dtype == "f32" else f32_to_bf16_bits(keys)

    out["k"] = f32_to_bf16_bits(_rng(w, b, _F_K).standard_normal((length, G, D), dtype=np.float32))
    out["v"] = f32_to_bf16_bits(_rng(w, b, _F_V).standard_normal((length, G, D), dtype=np.float32))
    return out


def requests(w: Workload, lens: np.ndarray, which=None, workers: int = 8):
    """Yield (b, request dict) for the requested batch indices, generated in parallel, in order."""
    which = list(range(w.batch)) if which is None else list(which)
    with ThreadPoolExecutor(max_workers=max(1, workers)) as ex:
        futs = [ex.submit(request, w, b, int(lens[b])) for b in which[: workers + 1]]
        nxt = len(futs)
        for i, b in enumerate(which):
            r = futs[i].result()
            futs[i] = None
            if nxt < len(which):
                futs.append(ex.submit(request, w, which[nxt], int(lens[which[nxt]])))
                nxt += 1
            yield b, r


def slot_mapping(w: Workload, block_table: np.ndarray, b: int, length: int) -> np.ndarray:
    """Cache slot (page * block_size + offset) of every token of request ``b``."""
    t = np.arange(length, dtype=np.int64)
    return block_table[b, t // w.block_size].astype(np.int64) * w.block_size + t % w.block_size
