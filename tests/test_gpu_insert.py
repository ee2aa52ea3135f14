"""The insert/quantise kernel against the oracle's quantisers, byte for byte."""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa, synth
from oracle import formats as F
from oracle import quant as Qz

pytestmark = pytest.mark.gpu


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(synth.f32_to_bf16_bits(x).view(np.int16)).view(torch.bfloat16).cuda()


def _insert(k, v, idx, idx_dtype, kv_dtype, g=1.0, P=4, G=4):
    """Inserts T tokens at slots 0..T-1 of fresh caches; returns host copies of the caches."""
    T = k.shape[0]
    dims = msa.make_dims(1, 1, 16 * G, G, G, 128, 128, P, P, 16)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    if kv_dtype == "bf16":
        cache = msa.KVCache(msa.BF16, torch.zeros((P, G, 128, 128), dtype=torch.bfloat16, device="cuda"),
                            torch.zeros((P, G, 128, 128), dtype=torch.bfloat16, device="cuda"))
    elif kv_dtype == "fp8":
        cache = msa.KVCache(msa.FP8_E4M3, torch.zeros((P, G, 128, 128), dtype=torch.uint8, device="cuda"),
                            torch.zeros((P, G, 128, 128), dtype=torch.uint8, device="cuda"), None, None, g, g)
    else:
        cache = msa.KVCache(msa.NVFP4, *[torch.zeros((P, G, 128, n), dtype=torch.uint8, device="cuda")
                                         for n in (64, 64, 8, 8)], g, g)
    if idx_dtype == "fp8":
        ic = msa.IndexCache(msa.FP8_E4M3, torch.zeros((P, G, 128, 128), dtype=torch.uint8, device="cuda"),
                            torch.zeros((P, G, 128), dtype=torch.float32, device="cuda"))
    elif idx_dtype == "nvfp4":
        ic = msa.IndexCache(msa.NVFP4, torch.zeros((P, G, 128, 64), dtype=torch.uint8, device="cuda"), None,
                            torch.zeros((P, G, 128, 8), dtype=torch.uint8, device="cuda"), g)
    else:
        ic = msa.IndexCache(msa.F32, torch.zeros((P, G, 128, 128), dtype=torch.float32, device="cuda"))
    slots = torch.arange(T, dtype=torch.int64, device="cuda")
    if idx.dtype == np.float32:
        idx_t, new_dt = torch.from_numpy(idx).cuda(), msa.F32
    else:   # uint16 bf16 bit patterns
        idx_t, new_dt = torch.from_numpy(idx.view(np.int16)).view(torch.bfloat16).cuda(), msa.BF16
    msa.kv_insert_quant(dims, _bf16(k), _bf16(v), idx_t, new_dt, slots, cache, ic, flags)
    assert msa.read_device_flags(flags) == 0
    # token t lives at page t // 128, offset t % 128: [P, G, BS, ...] -> [T, G, ...]
    tok = lambda a: a.cpu().numpy().transpose(0, 2, 1, *range(3, a.dim())).reshape(P * 128, G, *a.shape[3:])[:T]
    out = {"idx_keys": tok(ic.keys)}
    if ic.block_scale is not None:
        out["idx_block_scale"] = tok(ic.block_scale)
    if ic.scale is not None:
        out["idx_scale"] = ic.scale.cpu().numpy().transpose(0, 2, 1).reshape(P * 128, G)[:T]
    if kv_dtype == "bf16":
        out["k"] = tok(cache.k.view(torch.int16)).view(np.uint16)
        out["v"] = tok(cache.v.view(torch.int16)).view(np.uint16)
    elif kv_dtype == "fp8":
        out.update(k=tok(cache.k), v=tok(cache.v))
    else:
        out.update(k=tok(cache.k), v=tok(cache.v), ks=tok(cache.k_scale), vs=tok(cache.v_scale))
    return out


def test_fp8_index_keys_bit_exact_random_and_midpoints():
    rng = np.random.default_rng(1)
    T, G = 300, 4
    x = (rng.standard_normal((T, G, 128)) * rng.uniform(1e-3, 50, (T, G, 1))).astype(np.float32)
    # token 0 head 0: amax 448 so s = 1 and the values sit on E4M3 midpoints (ties to even)
    vals = F.e4m3_decode(np.arange(0, 0x7E))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x[0, 0, :] = 0
    x[0, 0, 0] = 448
    x[0, 0, 1:128] = np.resize(mids, 127) * np.where(np.arange(127) % 2, -1, 1)
    x[1, 2, :] = 0.0                                  # zero row -> scale 0, codes 0
    x[2, 1, :] = 1e-30                                # tiny values
    k = rng.standard_normal((T, G, 128)).astype(np.float32)
    got = _insert(k, k, x, "fp8", "bf16")
    codes, scale = Qz.quant_index_keys_fp8(x)
    assert np.array_equal(got["idx_scale"].view(np.uint32), scale.view(np.uint32))
    assert np.array_equal(got["idx_keys"], codes)


def test_fp8_index_keys_from_bf16_source():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((260, 4, 128)).astype(np.float32)
    xb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x))
    got = _insert(x, x, synth.f32_to_bf16_bits(x), "fp8", "bf16")
    codes, scale = Qz.quant_index_keys_fp8(xb)
    assert np.array_equal(got["idx_keys"], codes)
    assert np.array_equal(got["idx_scale"].view(np.uint32), scale.view(np.uint32))


def test_bf16_and_f32_copies_exact():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((200, 4, 128)).astype(np.float32)
    v = rng.standard_normal((200, 4, 128)).astype(np.float32)
    idx = rng.standard_normal((200, 4, 128)).astype(np.float32)
    got = _insert(k, v, idx, "f32", "bf16")
    assert np.array_equal(got["k"], synth.f32_to_bf16_bits(k))
    assert np.array_equal(got["v"], synth.f32_to_bf16_bits(v))
    assert np.array_equal(got["idx_keys"], idx)


@pytest.mark.parametrize("g", [1.0, float(np.float32(6.0 / (6 * 448))), 0.37])
def test_nvfp4_bit_exact(g):
    rng = np.random.default_rng(4)
    T, G = 300, 4
    k = rng.standard_normal((T, G, 128)).astype(np.float32)
    v = (rng.standard_normal((T, G, 128)) * 3).astype(np.float32)
    # E2M1 midpoints with a unit block scale (amax 6 and g = 1 give sb = 1): ties to even
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0])
    k[0, 0, :16] = mids
    k[0, 1, :16] = 0.0                                # zero group -> scale 0, codes 0
    k[0, 2, :16] = 1e-20                              # block scale underflows to 0
    k[0, 3, :16] = 1e4                                # block scale saturates at 448
    kb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(k))
    vb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v))
    got = _insert(k, v, k, "f32", "nvfp4", g=g)
    kc, ks = Qz.quant_nvfp4(kb, g)
    vc, vs = Qz.quant_nvfp4(vb, g)
    assert np.array_equal(got["ks"], ks)
    assert np.array_equal(got["k"], kc)
    assert np.array_equal(got["vs"], vs)
    assert np.array_equal(got["v"], vc)


def test_nvfp4_bytes_per_token():
    """576 bytes per token per layer for 4 KV heads x 128 dims (K and V): the pages' 34,560 / 60."""
    got = _insert(np.zeros((1, 4, 128), np.float32), np.zeros((1, 4, 128), np.float32),
                  np.zeros((1, 4, 128), np.float32), "f32", "nvfp4")
    per_token = sum(got[n][0].nbytes for n in ("k", "v", "ks", "vs"))
    assert per_token == 576 and per_token * 60 == 34560


def test_negative_slots_skip_and_bad_slots_flag():
    dims = msa.make_dims(1, 1, 64, 4, 4, 128, 128, 2, 2, 16)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = msa.KVCache(msa.BF16, torch.zeros((2, 4, 128, 128), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((2, 4, 128, 128), dtype=torch.bfloat16, device="cuda"))
    k = torch.ones((3, 4, 128), dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([-1, 5, 10 ** 6], dtype=torch.int64, device="cuda")
    msa.kv_insert_quant(dims, k, k, None, msa.F32, slots, cache, None, flags)
    assert msa.read_device_flags(flags) == msa.FLAG_BAD_SLOT
    c = cache.k.float().cpu()
    assert c[0, :, 5].eq(1).all() and c.sum().item() == 4 * 128


@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_nvfp4_index_keys_bit_exact(src):
    rng = np.random.default_rng(6)
    T, G = 280, 4
    x = (rng.standard_normal((T, G, 128)) * rng.uniform(0.1, 3, (T, G, 1))).astype(np.float32)
    x[0, 0, :16] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0]
    x[1, 1, :] = 0.0
    g = float(np.float32(8.0 / (6 * 448)))
    k = rng.standard_normal((T, G, 128)).astype(np.float32)
    idx = x if src == "f32" else synth.f32_to_bf16_bits(x)
    xv = x if src == "f32" else synth.bf16_bits_to_f32(idx)
    got = _insert(k, k, idx, "nvfp4", "bf16", g=g)
    codes, scales = Qz.quant_nvfp4(xv, g)
    assert np.array_equal(got["idx_block_scale"], scales)
    assert np.array_equal(got["idx_keys"], codes)


def test_fp8_kv_bit_exact():
    """FP8 E4M3 K/V with one scale per tensor: E4M3 midpoints (ties to even), values
    past the saturation point, zeros and random values, byte for byte."""
    rng = np.random.default_rng(31)
    T, G = 290, 4
    s = np.float32(synth.FP8_KV_SYNTH_SCALE)
    k = (rng.standard_normal((T, G, 128)) * rng.uniform(0.01, 4, (T, G, 1))).astype(np.float32)
    v = rng.standard_normal((T, G, 128)).astype(np.float32)
    vals = F.e4m3_decode(np.arange(0, 0x7E))
    mids = ((vals[:-1] + vals[1:]) / 2 * s).astype(np.float32)          # midpoints of x / s
    k[0, 0, :] = np.resize(mids, 128)
    k[1, 1, :8] = [7.0, -7.0, 100.0, -1e4, 6.0, -6.0, 0.0, -0.0]     # saturation and zeros
    v[2, 3, :] = 0.0
    kb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(k))             # the kernel reads bf16
    vb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v))
    idx = np.zeros((T, G, 128), dtype=np.float32)
    got = _insert(k, v, idx, "f32", "fp8", g=float(s))
    assert np.array_equal(got["k"], Qz.quant_kv_fp8(kb, s))
    assert np.array_equal(got["v"], Qz.quant_kv_fp8(vb, s))
