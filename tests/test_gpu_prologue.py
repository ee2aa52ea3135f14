"""The fused QK-norm + RoPE + insert kernel against the oracle (oracle/prologue.py).

bf16 results (queries, index queries, the bf16 key cache) are within one bf16
ulp of the fp64 oracle on the same bf16 inputs, plus the kernel's fp32 error
(a few 1e-6 absolute for unit-scale rows, which matters where the rotation
cancels to a tiny value): a value that close to a bf16 rounding boundary may
round either way (it does for well under 1 % of values). Cache quantisation is
checked byte for byte on the same bf16 values: the index branch is fed the key
branch's rows and weights, so the kernel's rotated index keys equal the keys it
stores in a bf16 cache, and the FP8 / NVFP4 caches must equal the oracle
quantisers applied to those.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import msa, synth
from oracle import formats as F
from oracle import prologue as Pr
from oracle import quant as Qz

pytestmark = pytest.mark.gpu

H, G, I, D, P = 64, 4, 4, 128, 6
# fp32 error of the norm (tree sum of 128 squares, IEEE sqrt and division) and
# the rotation (two products of values <= ~6 by cos/sin rounded to fp32)
FP32_SLACK = 4e-6


def _bf16_dev(x):
    return torch.from_numpy(synth.f32_to_bf16_bits(x).view(np.int16)).view(torch.bfloat16).cuda()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _case(T=70, seed=5):
    rng = np.random.default_rng(seed)
    raw = {n: (rng.standard_normal((T, c, D)) * rng.uniform(0.2, 5, (T, c, 1))).astype(np.float32)
           for n, c in (("q", H), ("k", G), ("v", G))}
    pos = np.concatenate([[0, 1, 127, 128, 4095], rng.integers(0, 262144, T - 6), [262143]]).astype(np.int32)
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    slots[3] = -1                                       # skipped token
    wts = synth.norm_weights(synth.WORKLOADS["b32_32k"])
    return raw, pos, slots, wts


def _run(raw, pos, slots, wts, kv="bf16", idx="fp8", with_idx=True, theta=synth.PROLOGUE_THETA):
    T = raw["q"].shape[0]
    dims = msa.make_dims(1, 1, H, G, I, D, 128, P, P, 16)
    s = float(np.float32(synth.FP8_KV_SYNTH_SCALE))
    g = float(np.float32(synth.NVFP4_SYNTH_GLOBAL))
    if kv == "bf16":
        cache = msa.KVCache(msa.BF16, *[torch.zeros((P, G, 128, D), dtype=torch.bfloat16, device="cuda")
                                        for _ in range(2)])
    elif kv == "fp8":
        cache = msa.KVCache(msa.FP8_E4M3, *[torch.zeros((P, G, 128, D), dtype=torch.uint8, device="cuda")
                                            for _ in range(2)], None, None, s, s)
    else:
        cache = msa.KVCache(msa.NVFP4, *[torch.zeros((P, G, 128, n), dtype=torch.uint8, device="cuda")
                                         for n in (64, 64, 8, 8)], g, g)
    if idx == "fp8":
        ic = msa.IndexCache(msa.FP8_E4M3, torch.zeros((P, I, 128, D), dtype=torch.uint8, device="cuda"),
                            torch.zeros((P, I, 128), dtype=torch.float32, device="cuda"))
    else:
        ic = msa.IndexCache(msa.NVFP4, torch.zeros((P, I, 128, 64), dtype=torch.uint8, device="cuda"), None,
                            torch.zeros((P, I, 128, 8), dtype=torch.uint8, device="cuda"), g)
    w_dev = {n: torch.from_numpy(a).cuda() for n, a in wts.items()}
    # the index branch gets the key branch's rows and weights (see the module docstring)
    nr = msa.make_norm_rope(w_dev["q"], w_dev["k"], w_dev["q"], w_dev["k"], synth.PROLOGUE_EPS, theta)
    q, k, v = _bf16_dev(raw["q"]), _bf16_dev(raw["k"]), _bf16_dev(raw["v"])
    q_out = torch.zeros_like(q)
    iq_out = torch.zeros((T, I, D), dtype=torch.bfloat16, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.qk_norm_rope_insert(dims, q, k, v, q[:, :I].contiguous() if with_idx else None, k if with_idx else None,
                            torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(), nr, q_out,
                            iq_out if with_idx else None, cache, ic if with_idx else None, flags)
    torch.cuda.synchronize()
    tok = lambda a: a.cpu().numpy().transpose(0, 2, 1, *range(3, a.dim())).reshape(P * 128, a.shape[1], *a.shape[3:])
    return dict(q_out=_bits(q_out), iq_out=_bits(iq_out), cache=cache, ic=ic, tok=tok, flags=flags)


def _within_one_ulp(got_bits, want_bits, where):
    g = F.bf16_to_f64(got_bits)
    w = F.bf16_to_f64(want_bits)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(w), 2.0 ** -126))) - 7)
    err = np.abs(g - w)
    lim = ulp * 1.0000001 + FP32_SLACK
    assert (err <= lim).all(), f"{where}: off by more than one bf16 ulp + fp32 error ({(err / lim).max():.3g}x)"
    frac = np.mean(got_bits != want_bits)
    assert frac < 0.01, f"{where}: {frac:.2%} of values differ by one ulp"


def test_norm_rope_outputs_and_bf16_cache():
    raw, pos, slots, wts = _case()
    r = _run(raw, pos, slots, wts)
    assert msa.read_device_flags(r["flags"]) == 0
    eps, th = synth.PROLOGUE_EPS, synth.PROLOGUE_THETA
    bits = {n: synth.f32_to_bf16_bits(a) for n, a in raw.items()}     # what the kernel reads
    want_q = Pr.norm_rope(bits["q"], wts["q"], pos, eps, th)
    _within_one_ulp(r["q_out"], want_q, "q")
    _within_one_ulp(r["iq_out"], want_q[:, :I], "index q")
    want_k = Pr.norm_rope(bits["k"], wts["k"], pos, eps, th)
    kc = r["tok"](r["cache"].k.view(torch.int16)).view(np.uint16)
    vc = r["tok"](r["cache"].v.view(torch.int16)).view(np.uint16)
    live = slots >= 0
    _within_one_ulp(kc[slots[live]], want_k[live], "k cache")
    assert np.array_equal(vc[slots[live]], synth.f32_to_bf16_bits(raw["v"])[live])   # V unchanged
    # the index key equals the stored key (same rows and weights): quantised byte for byte
    kf = synth.bf16_bits_to_f32(kc[slots[live]])
    codes, scale = Qz.quant_index_keys_fp8(kf)
    assert np.array_equal(r["tok"](r["ic"].keys)[slots[live]], codes)
    sc = r["ic"].scale.cpu().numpy().transpose(0, 2, 1).reshape(P * 128, I)
    assert np.array_equal(sc[slots[live]].view(np.uint32), scale.view(np.uint32))
    # the skipped slot left the caches untouched
    assert int(np.count_nonzero(kc.reshape(P * 128, -1).any(1))) == live.sum()


@pytest.mark.parametrize("kv,idx", [("fp8", "nvfp4"), ("nvfp4", "fp8")])
def test_quantised_caches_byte_exact(kv, idx):
    raw, pos, slots, wts = _case(seed=6)
    ref = _run(raw, pos, slots, wts, "bf16", "fp8")
    r = _run(raw, pos, slots, wts, kv, idx)
    assert msa.read_device_flags(r["flags"]) == 0
    live = slots >= 0
    kf = synth.bf16_bits_to_f32(ref["tok"](ref["cache"].k.view(torch.int16)).view(np.uint16)[slots[live]])
    vf = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(raw["v"]))[live]
    c = r["cache"]
    if kv == "fp8":
        s = np.float32(synth.FP8_KV_SYNTH_SCALE)
        assert np.array_equal(r["tok"](c.k)[slots[live]], Qz.quant_kv_fp8(kf, s))
        assert np.array_equal(r["tok"](c.v)[slots[live]], Qz.quant_kv_fp8(vf, s))
    else:
        g = np.float32(synth.NVFP4_SYNTH_GLOBAL)
        for got, gs, x in ((c.k, c.k_scale, kf), (c.v, c.v_scale, vf)):
            codes, scales = Qz.quant_nvfp4(x, g)
            assert np.array_equal(r["tok"](got)[slots[live]], codes)
            assert np.array_equal(r["tok"](gs)[slots[live]], scales)
    if idx == "nvfp4":
        codes, scales = Qz.quant_nvfp4(kf, np.float32(synth.NVFP4_SYNTH_GLOBAL))
        assert np.array_equal(r["tok"](r["ic"].keys)[slots[live]], codes)
        assert np.array_equal(r["tok"](r["ic"].block_scale)[slots[live]], scales)


def test_reusing_layer_skips_the_index_branch():
    raw, pos, slots, wts = _case(seed=7)
    r = _run(raw, pos, slots, wts, with_idx=False)
    assert msa.read_device_flags(r["flags"]) == 0
    assert not r["ic"].keys.any() and not r["ic"].scale.any()
    assert not r["iq_out"].any()
    want = Pr.norm_rope(synth.f32_to_bf16_bits(raw["q"]), wts["q"], pos, synth.PROLOGUE_EPS, synth.PROLOGUE_THETA)
    _within_one_ulp(r["q_out"], want, "q")


def test_bad_slot_is_flagged_and_skipped():
    raw, pos, slots, wts = _case(T=20, seed=8)
    slots[5] = P * 128 + 3
    r = _run(raw, pos, slots, wts)
    assert msa.read_device_flags(r["flags"]) == msa.FLAG_BAD_SLOT
