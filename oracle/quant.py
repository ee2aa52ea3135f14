"""Cache insertion and quantisation (the step that fills the paged caches).

TEST INFRASTRUCTURE (see the package docstring).

The pages say the KV cache is ordinary paged KV with 128-token blocks
("MiniMax M3 vLLM サポート：…", section "KV キャッシュ統合"), that a separate
keys-only index cache sits beside it ("vLLM、AMD Instinct MI355X上で…",
question 5), that the roadmap adds an FP8 indexer ("MiniMax M3 vLLM サポート：…",
section "技術ロードマップ") and that NVFP4 KV costs 34,560 bytes per token over
60 layers ("MiniMax-M3.1-Flash Day-0 対応", section "何が新しいか"). They give no
quantisation formulas; the readings below are this project's:

* FP8 index keys: one fp32 scale per (token, index head), s = amax / 448 with
  amax the largest |x| over the head's 128 values; codes = E4M3(x / s). If
  amax is 0 the scale and all codes are 0.
* NVFP4 K/V: the per-tensor fp32 global scale g is an input (a calibration
  constant, as a checkpoint would carry). For each 16 consecutive values of a
  (token, KV head) row: sb = E4M3((amax16 / 6) / g); codes = E2M1(x / (sb * g));
  if sb decodes to 0 every code is 0. Nibble order: the low nibble holds the
  even element.
* FP8 K/V ("MiniMax-M3.1-Flash Day-0 対応", section "何が新しいか": 61,440 bytes
  per token over 60 layers, i.e. one byte per K and V value and no per-token
  scale): one fp32 scale per tensor s (an input, like the NVFP4 global);
  code = E4M3(x / s), saturating at +-448.
* NVFP4 index keys: the same rule per (token, index head) row, with the index
  cache's own global scale (the pages name the format but not its rule:
  "MiniMax-M3.1-Flash Day-0 対応", section "何が新しいか" — the NVFP4 cache
  covers the indexer — and section "試し方" — indexer_kv_dtype nvfp4).

These steps are carried out in fp32 with IEEE round-to-nearest operations (one
rounding per operation, in the order written), which is the precision in which
a GPU makes the same integer decisions; the results are therefore exact
functions of the inputs and are compared byte for byte.
"""
from __future__ import annotations

import numpy as np

from .formats import e2m1_encode, e4m3_decode, e4m3_encode, nvfp4_pack

F32 = np.float32


def quant_index_keys_fp8(x: np.ndarray):
    """[T, I, D] fp32 (or bf16-valued) -> (codes [T, I, D] uint8, scale [T, I] fp32)."""
    x = np.asarray(x, dtype=F32)
    amax = np.max(np.abs(x), axis=-1)                     # exact in fp32
    scale = (amax / F32(448.0)).astype(F32)               # one RN division
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (x / scale[..., None]).astype(F32)            # one RN division per value
    codes = e4m3_encode(y)
    codes = np.where(scale[..., None] > 0, codes, np.uint8(0)).astype(np.uint8)
    return codes, scale


def quant_kv_fp8(x: np.ndarray, scale: float) -> np.ndarray:
    """[T, G, D] fp32 (or bf16-valued) -> E4M3 codes [T, G, D] uint8, value = code x scale."""
    x = np.asarray(x, dtype=F32)
    s = F32(scale)
    y = (x / s).astype(F32)                               # one RN division per value
    return e4m3_encode(y)


def quant_nvfp4(x: np.ndarray, global_scale: float):
    """[T, G, D] fp32 -> (packed codes [T, G, D/2] uint8, block scales [T, G, D/16] uint8 E4M3)."""
    x = np.asarray(x, dtype=F32)
    g = F32(global_scale)
    shp = x.shape
    xb = x.reshape(shp[:-1] + (shp[-1] // 16, 16))
    amax = np.max(np.abs(xb), axis=-1)                    # [..., D/16]
    sb_in = ((amax / F32(6.0)).astype(F32) / g).astype(F32)
    sb_code = e4m3_encode(sb_in)
    sb_val = e4m3_decode(sb_code).astype(F32)             # exact in fp32
    denom = (sb_val * g).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (xb / denom[..., None]).astype(F32)
    nib = e2m1_encode(y)
    nib = np.where(denom[..., None] > 0, nib, np.uint8(0)).astype(np.uint8)
    nib = nib.reshape(shp)
    return nvfp4_pack(nib), sb_code


def insert_tokens(cache: np.ndarray, values: np.ndarray, slots: np.ndarray, block_size: int):
    """Write per-token rows into a paged cache laid out [P, X, block_size, ...].

    ``values`` is [T, X, ...]; ``slots[t]`` = page * block_size + offset; a
    negative slot means "skip this token".
    """
    for t, s in enumerate(np.asarray(slots).tolist()):
        if s < 0:
            continue
        page, off = divmod(int(s), block_size)
        cache[page, :, off] = values[t]
