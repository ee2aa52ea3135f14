"""The C-ABI library builds, loads and exports every symbol include/msa.h
declares; host-side validation rejects bad arguments before any launch. CPU only:
no call here reaches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    from block_sparse_attention_07_gb300 import _build
    _build.build()
    from block_sparse_attention_07_gb300 import msa
    return msa


def test_every_declared_function_is_exported(m):
    with open(os.path.join(ROOT, "include", "msa.h")) as f:
        header = f.read()
    declared = set(re.findall(r"^\s*(?:[\w\*]+\s+)+\**(msa_\w+)\s*\(", header, re.M))
    assert declared == set(m.EXPORTED)
    lib = ctypes.CDLL(m.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(m):
    assert m.lib.msa_abi_version() == 2
    assert m.status_string(m.OK) == "MSA_OK"
    assert m.status_string(m.ERR_WORKSPACE) == "MSA_ERR_WORKSPACE"
    assert m.status_string(99) == "MSA_ERR_UNKNOWN"


def test_dims_validation(m):
    lib = m.lib
    assert lib.msa_select_blocks(None, None, None, None, None, None) == m.ERR_INVALID_ARG
    d = m.make_dims(2, 1, max_blocks_per_seq=4, num_pages=8)
    fake = ctypes.c_void_p(0x10000)
    # shape rules the kernels do not implement
    for field, val in (("head_dim", 64), ("block_size", 64), ("local_blocks", 2), ("topk", 17),
                       ("q_len", 9), ("n_heads", 32)):
        bad = m.make_dims(2, 1, max_blocks_per_seq=4, num_pages=8)
        setattr(bad, field, val)
        assert lib.msa_select_blocks(ctypes.byref(bad), fake, fake, fake, fake, None) == m.ERR_UNSUPPORTED, field
    for field, val in (("batch", 0), ("topk", 0), ("softmax_scale", -1.0)):
        bad = m.make_dims(2, 1, max_blocks_per_seq=4, num_pages=8)
        setattr(bad, field, val)
        assert lib.msa_select_blocks(ctypes.byref(bad), fake, fake, fake, fake, None) == m.ERR_INVALID_ARG, field
    # null output pointer
    assert lib.msa_select_blocks(ctypes.byref(d), fake, fake, None, fake, None) == m.ERR_INVALID_ARG


def test_workspace_size_and_rejection(m):
    d = m.make_dims(3, 2, max_blocks_per_seq=4, num_pages=8)
    need = m.sparse_gqa_workspace_size(d, m.BF16)
    rows = 3 * 2 * 4
    assert need == rows * 16 * (16 * 128 + 32) * 4 + rows * 8      # partials, then one ticket per row
    fake = ctypes.c_void_p(0x10000)
    kv = m._KVCache(m.BF16, fake, fake, None, None, 1.0, 1.0)
    st = m.lib.msa_sparse_gqa_decode(ctypes.byref(d), fake, ctypes.byref(kv), fake, fake, fake, fake, None, fake,
                                     need - 1, fake, None)
    assert st == m.ERR_WORKSPACE
    # misaligned query pointer
    st = m.lib.msa_sparse_gqa_decode(ctypes.byref(d), ctypes.c_void_p(0x10008), ctypes.byref(kv), fake, fake,
                                     fake, fake, None, fake, need, fake, None)
    assert st == m.ERR_INVALID_ARG


def test_dtype_combinations_rejected(m):
    d = m.make_dims(1, 1, max_blocks_per_seq=4, num_pages=8)
    fake = ctypes.c_void_p(0x10000)
    ic = m._IndexCache(m.FP8_E4M3, fake, fake)
    st = m.lib.msa_index_score(ctypes.byref(d), fake, m.F32, ctypes.byref(ic), fake, fake, fake, fake, None)
    assert st == m.ERR_UNSUPPORTED
    ic = m._IndexCache(m.BF16, fake, None, None, 1.0)                # no bf16 index cache
    st = m.lib.msa_index_score(ctypes.byref(d), fake, m.BF16, ctypes.byref(ic), fake, fake, fake, fake, None)
    assert st == m.ERR_UNSUPPORTED
    ic = m._IndexCache(m.NVFP4, fake, None, None, 1.0)               # NVFP4 keys need their block scales
    st = m.lib.msa_index_score(ctypes.byref(d), fake, m.BF16, ctypes.byref(ic), fake, fake, fake, fake, None)
    assert st == m.ERR_INVALID_ARG
    ic = m._IndexCache(m.NVFP4, fake, None, fake, 0.0)               # and a positive global scale
    st = m.lib.msa_index_score(ctypes.byref(d), fake, m.BF16, ctypes.byref(ic), fake, fake, fake, fake, None)
    assert st == m.ERR_INVALID_ARG
    kv = m._KVCache(m.NVFP4, fake, fake, fake, fake, 0.0, 1.0)      # global scale must be > 0
    st = m.lib.msa_kv_insert_quant(ctypes.byref(d), fake, fake, None, m.F32, fake, 4, ctypes.byref(kv), None,
                                   fake, None)
    assert st == m.ERR_INVALID_ARG
    for ks, vs in ((0.0, 1.0), (1.0, -2.0), (float("nan"), 1.0)):    # FP8 K/V: per-tensor scales > 0
        kv = m._KVCache(m.FP8_E4M3, fake, fake, None, None, ks, vs)
        st = m.lib.msa_kv_insert_quant(ctypes.byref(d), fake, fake, None, m.F32, fake, 4, ctypes.byref(kv), None,
                                       fake, None)
        assert st == m.ERR_INVALID_ARG
        need = m.lib.msa_sparse_gqa_workspace_size(ctypes.byref(d), m.FP8_E4M3)
        st = m.lib.msa_sparse_gqa_decode(ctypes.byref(d), fake, ctypes.byref(kv), fake, fake, fake, fake, None,
                                         fake, need, fake, None)
        assert st == m.ERR_INVALID_ARG
    kv = m._KVCache(m.F32, fake, fake, None, None, 1.0, 1.0)         # no fp32 K/V cache
    st = m.lib.msa_kv_insert_quant(ctypes.byref(d), fake, fake, None, m.F32, fake, 4, ctypes.byref(kv), None,
                                   fake, None)
    assert st == m.ERR_UNSUPPORTED


def test_dispatch_record_before_any_launch(m):
    assert isinstance(m.last_dispatch(), str)


def test_empty_inserts_launch_nothing(m):
    """Zero new tokens is a valid call that launches nothing (checked before any
    device pointer is touched, so it runs here without a GPU)."""
    lib = m.lib
    d = m.make_dims(2, 1, max_blocks_per_seq=4, num_pages=8)
    fake = ctypes.c_void_p(0x10000)
    kc = m._KVCache(m.BF16, fake, fake, None, None, 1.0, 1.0)
    assert lib.msa_kv_insert_quant(ctypes.byref(d), None, None, None, m.BF16, None, 0, ctypes.byref(kc), None,
                                   fake, None) == m.OK
    assert m.last_dispatch() == "kv_insert empty"
    assert lib.msa_kv_insert_quant(ctypes.byref(d), None, None, None, m.BF16, None, -1, ctypes.byref(kc), None,
                                   fake, None) == m.ERR_INVALID_ARG


def test_workspace_size_above_4_gib(m):
    """The workspace size is a size_t all the way to Python: the largest shapes
    the API takes need more than 2^32 bytes."""
    d = m.make_dims(4096, 8, max_blocks_per_seq=4, num_pages=8)
    rows = 4096 * 8 * 4
    assert m.sparse_gqa_workspace_size(d, m.BF16) == rows * (16 * (16 * 128 + 32) * 4 + 8)
    assert m.sparse_gqa_workspace_size(d, m.BF16) > 2 ** 32

