"""Thin ctypes binding over libmsa.so (include/msa.h).

Argument marshalling only: every step of the MSA decode path runs in the
library's CUDA kernels. Tensors are torch tensors (used for device memory and
streams); each call passes their data pointers and the current CUDA stream.
Importing this module loads the library and raises if it was not built: there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmsa.so")

F32, BF16, FP8_E4M3, NVFP4 = 0, 1, 2, 3

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_DEVICE_FLAG = range(6)

FLAG_BAD_PAGE, FLAG_BAD_BLOCK, FLAG_BAD_SEQLEN, FLAG_BAD_SLOT, FLAG_TIMEOUT, FLAG_Q_RANGE = (
    0x1, 0x2, 0x4, 0x8, 0x10, 0x20)

# Every function include/msa.h declares.
EXPORTED = ("msa_abi_version", "msa_status_string", "msa_get_last_dispatch", "msa_kv_insert_quant",
            "msa_index_score", "msa_insert_index_score", "msa_select_blocks", "msa_sparse_gqa_workspace_size",
            "msa_sparse_gqa_decode", "msa_sparse_gqa_decode_noalloc", "msa_read_device_flags",
            "msa_qk_norm_rope_insert", "msa_select_sparse_gqa_decode", "msa_selftest_bounded_wait")


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_len", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("n_idx_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("topk", ctypes.c_int32), ("local_blocks", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]


class _KVCache(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("k_global", ctypes.c_float),
                ("v_global", ctypes.c_float)]


class _IndexCache(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("keys", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("block_scale", ctypes.c_void_p), ("global_scale", ctypes.c_float)]


class NormRope(ctypes.Structure):
    """msa_norm_rope_t: device fp32 [D] RMSNorm weights (pointers), eps, rotary base."""
    _fields_ = [("q_weight", ctypes.c_void_p), ("k_weight", ctypes.c_void_p), ("idx_q_weight", ctypes.c_void_p),
                ("idx_k_weight", ctypes.c_void_p), ("eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


class MSAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libmsa.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.msa_abi_version.restype = ctypes.c_int
    lib.msa_status_string.restype = ctypes.c_char_p
    lib.msa_status_string.argtypes = [ctypes.c_int]
    lib.msa_get_last_dispatch.argtypes = [ctypes.c_char_p, sz]
    lib.msa_kv_insert_quant.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, ctypes.c_int, vp, i32,
                                        ctypes.POINTER(_KVCache), ctypes.POINTER(_IndexCache), vp, vp]
    lib.msa_index_score.argtypes = [ctypes.POINTER(Dims), vp, ctypes.c_int, ctypes.POINTER(_IndexCache), vp, vp,
                                    vp, vp, vp]
    lib.msa_insert_index_score.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, vp, ctypes.POINTER(_KVCache), vp,
                                           ctypes.POINTER(_IndexCache), vp, vp, vp, vp, vp]
    lib.msa_select_blocks.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, vp, vp]
    lib.msa_sparse_gqa_workspace_size.restype = sz
    lib.msa_sparse_gqa_workspace_size.argtypes = [ctypes.POINTER(Dims), ctypes.c_int]
    lib.msa_sparse_gqa_decode.argtypes = [ctypes.POINTER(Dims), vp, ctypes.POINTER(_KVCache), vp, vp, vp, vp, vp,
                                          vp, sz, vp, vp]
    lib.msa_select_sparse_gqa_decode.argtypes = [ctypes.POINTER(Dims), vp, ctypes.POINTER(_KVCache), vp, vp, vp,
                                                 vp, vp, vp, vp, sz, vp, vp]
    lib.msa_sparse_gqa_decode_noalloc.argtypes = [ctypes.POINTER(Dims), vp, ctypes.POINTER(_KVCache), vp, vp, vp,
                                                  vp, vp, vp, vp]
    lib.msa_read_device_flags.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.msa_selftest_bounded_wait.argtypes = [vp, vp]
    lib.msa_qk_norm_rope_insert.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, vp, vp, vp, vp, i32,
                                            ctypes.POINTER(NormRope), vp, vp, ctypes.POINTER(_KVCache),
                                            ctypes.POINTER(_IndexCache), vp, vp]
    for name in EXPORTED:       # every other entry point returns msa_status_t
        if name not in ("msa_abi_version", "msa_status_string", "msa_sparse_gqa_workspace_size"):
            getattr(lib, name).restype = ctypes.c_int
    return lib


lib = _load()
LIB_PATH = _LIB_PATH


def status_string(status: int) -> str:
    return lib.msa_status_string(status).decode()


def last_dispatch() -> str:
    buf = ctypes.create_string_buffer(512)
    lib.msa_get_last_dispatch(buf, 512)
    return buf.value.decode()


def _check(status: int, what: str):
    if status != OK:
        raise MSAError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def make_dims(batch, q_len, n_heads=64, n_kv_heads=4, n_idx_heads=4, head_dim=128, block_size=128,
              max_blocks_per_seq=1, num_pages=1, topk=16, local_blocks=1, softmax_scale=None) -> Dims:
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    return Dims(batch, q_len, n_heads, n_kv_heads, n_idx_heads, head_dim, block_size, max_blocks_per_seq,
                num_pages, topk, local_blocks, softmax_scale)


@dataclasses.dataclass
class KVCache:
    """bf16: k, v [P, G, BS, D]. FP8_E4M3: k, v uint8 E4M3 [P, G, BS, D], k_global / v_global the
    per-tensor scales. NVFP4: k, v uint8 [P, G, BS, D/2], k_scale, v_scale uint8 [P, G, BS, D/16]."""
    dtype: int
    k: object
    v: object
    k_scale: object = None
    v_scale: object = None
    k_global: float = 1.0
    v_global: float = 1.0

    def c(self):
        return _KVCache(self.dtype, _ptr(self.k), _ptr(self.v), _ptr(self.k_scale), _ptr(self.v_scale),
                        self.k_global, self.v_global)


@dataclasses.dataclass
class IndexCache:
    """F32: keys f32 [P, I, BS, D]. FP8_E4M3: keys uint8 [P, I, BS, D], scale f32 [P, I, BS].
    NVFP4: keys uint8 [P, I, BS, D/2], block_scale uint8 [P, I, BS, D/16], global_scale (host float)."""
    dtype: int
    keys: object
    scale: object = None
    block_scale: object = None
    global_scale: float = 1.0

    def c(self):
        return _IndexCache(self.dtype, _ptr(self.keys), _ptr(self.scale), _ptr(self.block_scale), self.global_scale)


class Prepared:
    """A library call whose arguments were marshalled once; calling it launches again.

    Holds the ctypes structures the arguments point to. Used on launch-bound
    paths (the same call issued every decode step)."""
    __slots__ = ("fn", "args", "keep", "what")

    def __init__(self, fn, args, keep, what):
        self.fn, self.args, self.keep, self.what = fn, args, keep, what

    def __call__(self):
        st = self.fn(*self.args)
        if st != OK:
            raise MSAError(st, self.what)


def _call(fn, args, keep, what, prepare):
    if prepare:
        return Prepared(fn, args, keep, what)
    _check(fn(*args), what)
    return None


def kv_insert_quant(dims: Dims, k_new, v_new, idx_k_new, idx_new_dtype: int, slot_mapping, cache: KVCache,
                    idx_cache: IndexCache | None, flags, stream=None, prepare=False):
    kc = cache.c()
    ic = idx_cache.c() if idx_cache is not None else None
    args = (ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(idx_k_new), idx_new_dtype, _ptr(slot_mapping),
            int(k_new.shape[0]), ctypes.byref(kc), ctypes.byref(ic) if ic is not None else None, _ptr(flags),
            _stream(stream))
    return _call(lib.msa_kv_insert_quant, args, (dims, kc, ic), "msa_kv_insert_quant", prepare)


def select_sparse_gqa_decode(dims: Dims, q, cache: KVCache, block_table, seq_lens, scores, selected, out, lse,
                             workspace, flags, stream=None, prepare=False):
    """Selection (written to ``selected``) and sparse GQA in one launch."""
    kc = cache.c()
    args = (ctypes.byref(dims), _ptr(q), ctypes.byref(kc), _ptr(block_table), _ptr(seq_lens), _ptr(scores),
            _ptr(selected), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(flags), _stream(stream))
    return _call(lib.msa_select_sparse_gqa_decode, args, (dims, kc), "msa_select_sparse_gqa_decode", prepare)


def make_norm_rope(q_weight, k_weight, idx_q_weight=None, idx_k_weight=None, eps=1e-6, rope_theta=10000.0):
    """msa_norm_rope_t from device fp32 [D] weight tensors (kept alive by the caller)."""
    return NormRope(_ptr(q_weight), _ptr(k_weight), _ptr(idx_q_weight), _ptr(idx_k_weight), eps, rope_theta)


def qk_norm_rope_insert(dims: Dims, q, k, v, idx_q, idx_k, positions, slot_mapping, nr: NormRope, q_out,
                        idx_q_out, cache: KVCache, idx_cache: IndexCache | None, flags, stream=None, prepare=False):
    kc = cache.c()
    ic = idx_cache.c() if idx_cache is not None else None
    args = (ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(idx_q), _ptr(idx_k), _ptr(positions),
            _ptr(slot_mapping), int(q.shape[0]), ctypes.byref(nr), _ptr(q_out), _ptr(idx_q_out), ctypes.byref(kc),
            ctypes.byref(ic) if ic is not None else None, _ptr(flags), _stream(stream))
    return _call(lib.msa_qk_norm_rope_insert, args, (dims, nr, kc, ic), "msa_qk_norm_rope_insert", prepare)


def index_score(dims: Dims, idx_q, q_dtype: int, idx_cache: IndexCache, block_table, seq_lens, scores, flags,
                stream=None, prepare=False):
    ic = idx_cache.c()
    args = (ctypes.byref(dims), _ptr(idx_q), q_dtype, ctypes.byref(ic), _ptr(block_table), _ptr(seq_lens),
            _ptr(scores), _ptr(flags), _stream(stream))
    return _call(lib.msa_index_score, args, (dims, ic), "msa_index_score", prepare)


def insert_index_score(dims: Dims, k_new, v_new, idx_k_new, slot_mapping, cache: KVCache, idx_q,
                       idx_cache: IndexCache, block_table, seq_lens, scores, flags, stream=None, prepare=False):
    """msa_insert_index_score: the step's new tokens (one per request, at its last position)
    inserted and every block scored, in one launch; one query position only."""
    kc, ic = cache.c(), idx_cache.c()
    args = (ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(idx_k_new), _ptr(slot_mapping), ctypes.byref(kc),
            _ptr(idx_q), ctypes.byref(ic), _ptr(block_table), _ptr(seq_lens), _ptr(scores), _ptr(flags),
            _stream(stream))
    return _call(lib.msa_insert_index_score, args, (dims, kc, ic), "msa_insert_index_score", prepare)


def select_blocks(dims: Dims, scores, seq_lens, selected, flags, stream=None, prepare=False):
    args = (ctypes.byref(dims), _ptr(scores), _ptr(seq_lens), _ptr(selected), _ptr(flags), _stream(stream))
    return _call(lib.msa_select_blocks, args, (dims,), "msa_select_blocks", prepare)


def sparse_gqa_workspace_size(dims: Dims, kv_dtype: int) -> int:
    return int(lib.msa_sparse_gqa_workspace_size(ctypes.byref(dims), kv_dtype))


def sparse_gqa_decode(dims: Dims, q, cache: KVCache, block_table, seq_lens, selected, out, lse, workspace, flags,
                      stream=None, prepare=False):
    kc = cache.c()
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (ctypes.byref(dims), _ptr(q), ctypes.byref(kc), _ptr(block_table), _ptr(seq_lens), _ptr(selected),
            _ptr(out), _ptr(lse), _ptr(workspace), nbytes, _ptr(flags), _stream(stream))
    return _call(lib.msa_sparse_gqa_decode, args, (dims, kc), "msa_sparse_gqa_decode", prepare)


def sparse_gqa_decode_noalloc(dims: Dims, q, cache: KVCache, block_table, seq_lens, selected, out, lse, flags,
                              stream=None):
    """msa_sparse_gqa_decode without a workspace argument, for callers that cannot allocate
    device memory; its scratch is a fixed 64 MiB array inside the library (see include/msa.h)."""
    kc = cache.c()
    st = lib.msa_sparse_gqa_decode_noalloc(ctypes.byref(dims), _ptr(q), ctypes.byref(kc), _ptr(block_table),
                                           _ptr(seq_lens), _ptr(selected), _ptr(out), _ptr(lse), _ptr(flags),
                                           _stream(stream))
    _check(st, "msa_sparse_gqa_decode_noalloc")


def selftest_bounded_wait(flags, stream=None):
    """msa_selftest_bounded_wait: a kernel whose barrier wait runs out (about 2 s)
    and reports MSA_FLAG_TIMEOUT in ``flags``."""
    _check(lib.msa_selftest_bounded_wait(_ptr(flags), _stream(stream)), "msa_selftest_bounded_wait")


def read_device_flags(flags, stream=None) -> int:
    """Synchronises the stream and returns the flag word (0 = no kernel-reported problem)."""
    host = ctypes.c_uint32(0)
    st = lib.msa_read_device_flags(_ptr(flags), ctypes.byref(host), _stream(stream))
    if st not in (OK, ERR_DEVICE_FLAG):
        _check(st, "msa_read_device_flags")
    return int(host.value)


def decode_step(dims: Dims, q, idx_q, q_idx_dtype: int, idx_cache: IndexCache, cache: KVCache, block_table,
                seq_lens, scores, selected, out, lse, workspace, flags, stream=None):
    """The three MSA stages back to back on one stream: score, select, sparse GQA."""
    index_score(dims, idx_q, q_idx_dtype, idx_cache, block_table, seq_lens, scores, flags, stream)
    select_blocks(dims, scores, seq_lens, selected, flags, stream)
    sparse_gqa_decode(dims, q, cache, block_table, seq_lens, selected, out, lse, workspace, flags, stream)
