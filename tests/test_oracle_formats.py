"""Pins for the oracle's number formats and quantisers (CPU only).

Each format is checked against its published definition (golden tables), a
library implementation where one exists (torch's float8_e4m3fn), exhaustive
round trips and error bounds that follow from round-to-nearest.
"""
import numpy as np
import pytest
import torch

from conftest import load_golden, num
from oracle import formats as F
from oracle import quant as Qz


def test_e4m3_golden_codes():
    g = load_golden("formats.json")
    for row in g["e4m3"]:
        v = F.e4m3_decode(np.array([row["code"]]))[0]
        want = num(row["value"])
        if np.isnan(want):
            assert np.isnan(v)
        else:
            assert v == want and np.signbit(v) == np.signbit(want), row


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert (F.e4m3_encode(F.e4m3_decode(codes)) == codes).all()


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    # exact midpoints between neighbours exercise ties-to-even
    vals = F.e4m3_decode(np.arange(0, 0x7E))
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([x, mids, -mids]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = F.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (ours == ref).all()


def test_e4m3_rounding_golden():
    for x, want in load_golden("formats.json")["e4m3_rounding"]:
        assert F.e4m3_decode(F.e4m3_encode(np.array([x])))[0] == want, x


def test_e2m1_table_and_rounding():
    g = load_golden("formats.json")
    dec = F.e2m1_decode(np.arange(16))
    want = np.array(g["e2m1"])
    assert (dec == want).all() and (np.signbit(dec) == np.signbit(want)).all()
    for x, w in g["e2m1_rounding"]:
        assert F.e2m1_decode(F.e2m1_encode(np.array([x])))[0] == w, x
    assert (F.e2m1_encode(dec) == np.arange(16)).all()


def test_nvfp4_pack_order():
    nib = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    packed = F.nvfp4_pack(nib)
    assert packed.tolist() == [[0x21, 0x43]]          # low nibble = even element
    assert (F.nvfp4_unpack(packed) == nib).all()


def test_fp8_index_quant_properties():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((300, 4, 128)) * rng.uniform(0.01, 20, (300, 4, 1))).astype(np.float32)
    x[5, 2] = 0.0                                       # all-zero row
    codes, scale = Qz.quant_index_keys_fp8(x)
    assert codes.dtype == np.uint8 and scale.dtype == np.float32
    assert scale[5, 2] == 0 and (codes[5, 2] == 0).all()
    dec = F.e4m3_decode(codes) * scale[..., None]
    # amax maps to 448 (up to one rounding of the scale)
    amax_code = np.max(np.abs(F.e4m3_decode(codes)), axis=-1)
    assert (amax_code[scale > 0] == 448).all()
    # round-to-nearest error bound: half the E4M3 spacing at each value (relative 2^-4 for normals)
    y = x / np.where(scale > 0, scale, 1)[..., None]
    half_ulp = np.where(np.abs(y) >= 2 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2 ** -6))) - 4), 2.0 ** -10)
    err = np.abs(dec / np.where(scale > 0, scale, 1)[..., None] - y)
    assert (err <= half_ulp * (1 + 1e-6) + 1e-7).all()


def test_nvfp4_quant_properties():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((200, 4, 128)).astype(np.float32)
    x[3, 1, 16:32] = 0.0
    g = np.float32(6.0 / (6 * 448))
    packed, sc = Qz.quant_nvfp4(x, g)
    assert packed.shape == (200, 4, 64) and sc.shape == (200, 4, 8)
    dec = F.nvfp4_decode(packed, sc, g)
    assert (dec[3, 1, 16:32] == 0).all()
    # each 16-group: the largest element sits near the top of the E2M1 range
    xb = x.reshape(200, 4, 8, 16).astype(np.float64)
    sbv = F.e4m3_decode(sc) * float(g)
    amax = np.abs(xb).max(-1)
    ok = amax > 0
    r = amax[ok] / sbv[ok]
    assert (r >= 6 / 1.0625 - 1e-6).all() and (r <= 6 / 0.9375 + 1e-6).all()
    # rounding bound: half the E2M1 spacing (0.25 below 2, 0.5 in [2,4), 1 above), plus saturation
    y = xb / np.where(sbv > 0, sbv, 1)[..., None]
    d = dec.reshape(xb.shape) / np.where(sbv > 0, sbv, 1)[..., None]
    a = np.abs(y)
    half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    err = np.where(a > 6, np.abs(np.abs(d) - 6), np.abs(d - y))
    assert (err[ok] <= half[ok] + 1e-6).all()


def test_fp8_kv_quant_matches_torch_and_saturates():
    """E4M3 K/V with one scale per tensor: codes equal torch's float8_e4m3fn cast of
    x / s inside the E4M3 range, and saturate to +-448 beyond it."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((300, 4, 128)) * 2.5).astype(np.float32)
    x[0, 0, :4] = [7.0, -9.0, 6.5, -6.0001]                 # beyond the calibrated amax 6
    s = np.float32(6.0 / 448.0)
    codes = Qz.quant_kv_fp8(x, s)
    assert codes.dtype == np.uint8 and codes.shape == x.shape
    y = x / s
    inr = np.abs(y) <= 448
    ref = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[inr], ref[inr])
    dec = F.e4m3_decode(codes)
    assert (~inr).sum() > 4 and np.array_equal(dec[~inr], np.sign(y[~inr]) * 448.0)


def test_kv_byte_counts_match_pages():
    """576 bytes/token/layer NVFP4 (x60 = 34,560) and 1,024 FP8 (x60 = 61,440)."""
    c = load_golden("page_constants.json")
    G, D = c["n_kv_heads"], 128
    x = np.zeros((1, G, D), dtype=np.float32)
    packed, sc = Qz.quant_nvfp4(x, 1.0)
    per_layer_nvfp4 = 2 * (packed.nbytes + sc.nbytes)          # K and V
    per_layer_fp8 = 2 * Qz.quant_kv_fp8(x, 1.0).nbytes           # K and V
    assert per_layer_nvfp4 * c["layers"] == c["nvfp4_kv_bytes_per_token_all_layers"]
    assert per_layer_fp8 * c["layers"] == c["fp8_kv_bytes_per_token_all_layers"]
    saving = 100 * (1 - per_layer_nvfp4 / per_layer_fp8)
    assert saving == pytest.approx(c["nvfp4_saving_percent"])


def test_insert_tokens_scatter_and_skip():
    cache = np.zeros((3, 1, 4, 2))
    vals = np.arange(10, dtype=np.float64).reshape(5, 1, 2)
    Qz.insert_tokens(cache, vals, np.array([5, -1, 0, 11, 6]), 4)
    assert (cache[1, 0, 1] == vals[0, 0]).all()
    assert (cache[0, 0, 0] == vals[2, 0]).all()
    assert (cache[2, 0, 3] == vals[3, 0]).all()
    assert (cache[1, 0, 2] == vals[4, 0]).all()
    assert np.count_nonzero(cache) == 4 * 2 - 1      # vals[0] holds one zero
