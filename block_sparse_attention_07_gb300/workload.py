"""Device-resident MSA decode workloads built from the seeded generator.

Allocates the paged caches and per-step buffers with torch (device memory
only), fills the caches through the library's own insert/quantise kernel, and
runs decode steps through the C ABI. Nothing here computes any part of the
method on the host.
"""
from __future__ import annotations

import numpy as np
import torch

from . import msa, synth


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


class DeviceWorkload:
    """All device state of one workload: caches, queries, block table, outputs.

    ``which`` restricts the batch to a subset of requests (keeping their
    seeded streams), so tests can run full-length requests of a large workload.
    ``index_cache=False`` builds a layer without an index cache: one that reuses
    another layer's block selection (``reuse_step``) and writes no index keys.
    """

    def __init__(self, w: synth.Workload, device="cuda", which=None, lens=None, workers: int = 8,
                 index_cache: bool = True):
        self.w = w
        self.has_index = index_cache
        self.device = torch.device(device)
        full_lens = synth.seq_lens(w) if lens is None else np.asarray(lens, dtype=np.int32)
        self.which = list(range(w.batch)) if which is None else list(which)
        self.lens = full_lens[self.which].astype(np.int32)
        B = len(self.which)
        sub = synth.scaled(w, batch=B)
        self.block_table, self.num_pages = synth.page_table(sub, self.lens)
        nb = int(self.block_table.shape[1])
        self.dims = msa.make_dims(B, w.q_len, w.n_heads, w.n_kv_heads, w.n_idx_heads, w.head_dim, w.block_size,
                                  nb, self.num_pages, w.topk, 1, w.softmax_scale)
        dev = self.device
        P, G, I, D, BS, Q, H = self.num_pages, w.n_kv_heads, w.n_idx_heads, w.head_dim, w.block_size, w.q_len, w.n_heads
        if w.kv_dtype == "bf16":
            self.cache = msa.KVCache(msa.BF16, torch.zeros((P, G, BS, D), dtype=torch.bfloat16, device=dev),
                                     torch.zeros((P, G, BS, D), dtype=torch.bfloat16, device=dev))
        elif w.kv_dtype == "fp8":
            s = synth.kv_scale(w)
            self.cache = msa.KVCache(msa.FP8_E4M3, torch.zeros((P, G, BS, D), dtype=torch.uint8, device=dev),
                                     torch.zeros((P, G, BS, D), dtype=torch.uint8, device=dev), None, None, s, s)
        else:
            g = synth.kv_scale(w)
            self.cache = msa.KVCache(msa.NVFP4, torch.zeros((P, G, BS, D // 2), dtype=torch.uint8, device=dev),
                                     torch.zeros((P, G, BS, D // 2), dtype=torch.uint8, device=dev),
                                     torch.zeros((P, G, BS, D // 16), dtype=torch.uint8, device=dev),
                                     torch.zeros((P, G, BS, D // 16), dtype=torch.uint8, device=dev), g, g)
        if not index_cache:
            self.idx_cache = None
            self.q_idx_dtype = self.idx_new_dtype = msa.BF16
        elif w.idx_dtype == "f32":
            self.idx_cache = msa.IndexCache(msa.F32, torch.zeros((P, I, BS, D), dtype=torch.float32, device=dev))
            self.q_idx_dtype = msa.F32
            self.idx_new_dtype = msa.F32
        elif w.idx_dtype == "nvfp4":
            self.idx_cache = msa.IndexCache(msa.NVFP4, torch.zeros((P, I, BS, D // 2), dtype=torch.uint8, device=dev),
                                            None, torch.zeros((P, I, BS, D // 16), dtype=torch.uint8, device=dev),
                                            float(np.float32(synth.NVFP4_IDX_SYNTH_GLOBAL)))
            self.q_idx_dtype = msa.BF16
            self.idx_new_dtype = msa.BF16
        else:
            self.idx_cache = msa.IndexCache(msa.FP8_E4M3, torch.zeros((P, I, BS, D), dtype=torch.uint8, device=dev),
                                            torch.zeros((P, I, BS), dtype=torch.float32, device=dev))
            self.q_idx_dtype = msa.BF16
            self.idx_new_dtype = msa.BF16
        self.flags = torch.zeros(1, dtype=torch.int32, device=dev)
        self.seq_lens_d = torch.from_numpy(self.lens).to(dev)
        self.block_table_d = torch.from_numpy(self.block_table).to(dev)

        q = np.empty((B, Q, H, D), dtype=np.uint16)
        qi = np.empty((B, Q, I, D), dtype=np.float32 if w.idx_dtype == "f32" else np.uint16)
        # the last Q tokens of each request: the tokens a decode step inserts
        new_k = np.empty((B, Q, G, D), dtype=np.uint16)
        new_v = np.empty((B, Q, G, D), dtype=np.uint16)
        new_i = np.empty((B, Q, I, D), dtype=qi.dtype)
        new_slots = np.empty((B, Q), dtype=np.int64)
        for bi, (b, r) in enumerate(synth.requests(w, full_lens, self.which, workers=workers)):
            L = int(full_lens[b])
            q[bi] = r["q"]
            qi[bi] = r["q_idx"]
            slots = synth.slot_mapping(sub, self.block_table, bi, L)
            new_k[bi], new_v[bi], new_i[bi] = r["k"][L - Q:], r["v"][L - Q:], r["idx_k"][L - Q:]
            new_slots[bi] = slots[L - Q:]
            self._insert(r["k"], r["v"], r["idx_k"], slots)
        self.q = _bf16(q).to(dev)
        self.q_idx = (torch.from_numpy(qi) if w.idx_dtype == "f32" else _bf16(qi)).to(dev)
        self.new_k = _bf16(new_k.reshape(B * Q, G, D)).to(dev)
        self.new_v = _bf16(new_v.reshape(B * Q, G, D)).to(dev)
        self.new_idx = ((torch.from_numpy(new_i) if w.idx_dtype == "f32" else _bf16(new_i)).reshape(B * Q, I, D).to(dev)
                        if index_cache else None)
        self.new_slots = torch.from_numpy(new_slots.reshape(-1)).to(dev)
        self.scores = torch.empty((B, Q, I, nb), dtype=torch.float32, device=dev)
        self.selected = torch.empty((B, Q, I, w.topk), dtype=torch.int32, device=dev)
        self.out = torch.empty((B, Q, H, D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
        self._pack_step_inputs()
        self._prep = None
        ws = msa.sparse_gqa_workspace_size(self.dims, self.cache.dtype)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)

    # Per-step inputs: what changes from one decode step to the next.
    STEP_INPUTS = ("q", "q_idx", "new_k", "new_v", "new_idx", "new_slots", "block_table_d", "seq_lens_d")

    def _pack_step_inputs(self):
        """Places the per-step input tensors in one device buffer (256-byte
        aligned views), so that a step's inputs arrive in one host-to-device copy
        of ``step_inputs``."""
        parts = [(n, getattr(self, n)) for n in self.STEP_INPUTS if getattr(self, n) is not None]
        offs, total = [], 0
        for _, t in parts:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(total, dtype=torch.uint8, device=self.device)
        for (n, t), o in zip(parts, offs):
            view = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            view.copy_(t)
            setattr(self, n, view)
        self.step_inputs = buf

    def _insert(self, k, v, idx, slots):
        dev = self.device
        kd = _bf16(k).to(dev)
        vd = _bf16(v).to(dev)
        idd = None
        if self.has_index:
            idd = (torch.from_numpy(idx) if idx.dtype == np.float32 else _bf16(idx)).to(dev)
        sd = torch.from_numpy(slots).to(dev)
        msa.kv_insert_quant(self.dims, kd, vd, idd, self.idx_new_dtype, sd, self.cache, self.idx_cache, self.flags)

    # ------------------------------------------------------------ stages --
    def prepared(self):
        """The four stage calls with their arguments marshalled once (current stream)."""
        if self._prep is None:
            self._prep = dict(
                insert=msa.kv_insert_quant(self.dims, self.new_k, self.new_v, self.new_idx, self.idx_new_dtype,
                                           self.new_slots, self.cache, self.idx_cache, self.flags, prepare=True),
                attend=msa.sparse_gqa_decode(self.dims, self.q, self.cache, self.block_table_d, self.seq_lens_d,
                                             self.selected, self.out, self.lse, self.workspace, self.flags,
                                             prepare=True))
            if self.has_index:
                self._prep.update(select_attend=msa.select_sparse_gqa_decode(
                    self.dims, self.q, self.cache, self.block_table_d, self.seq_lens_d, self.scores, self.selected,
                    self.out, self.lse, self.workspace, self.flags, prepare=True))
            if self.has_index:
                self._prep.update(
                    index=msa.index_score(self.dims, self.q_idx, self.q_idx_dtype, self.idx_cache,
                                          self.block_table_d, self.seq_lens_d, self.scores, self.flags, prepare=True),
                    select=msa.select_blocks(self.dims, self.scores, self.seq_lens_d, self.selected, self.flags,
                                             prepare=True))
            if self.merges_insert:
                self._prep.update(insert_index=msa.insert_index_score(
                    self.dims, self.new_k, self.new_v, self.new_idx, self.new_slots, self.cache, self.q_idx,
                    self.idx_cache, self.block_table_d, self.seq_lens_d, self.scores, self.flags, prepare=True))
        return self._prep

    def insert_step_tokens(self, stream=None):
        if stream is None:
            return self.prepared()["insert"]()
        msa.kv_insert_quant(self.dims, self.new_k, self.new_v, self.new_idx, self.idx_new_dtype, self.new_slots,
                            self.cache, self.idx_cache, self.flags, stream)

    def index_score(self, stream=None):
        if stream is None:
            return self.prepared()["index"]()
        msa.index_score(self.dims, self.q_idx, self.q_idx_dtype, self.idx_cache, self.block_table_d,
                        self.seq_lens_d, self.scores, self.flags, stream)

    def insert_index_score(self, stream=None):
        """The insert and the scoring in one launch (one query position)."""
        if stream is None:
            return self.prepared()["insert_index"]()
        msa.insert_index_score(self.dims, self.new_k, self.new_v, self.new_idx, self.new_slots, self.cache,
                               self.q_idx, self.idx_cache, self.block_table_d, self.seq_lens_d, self.scores,
                               self.flags, stream)

    def select(self, stream=None):
        if stream is None:
            return self.prepared()["select"]()
        msa.select_blocks(self.dims, self.scores, self.seq_lens_d, self.selected, self.flags, stream)

    def attend(self, stream=None, selected=None):
        if stream is None and selected is None:
            return self.prepared()["attend"]()
        msa.sparse_gqa_decode(self.dims, self.q, self.cache, self.block_table_d, self.seq_lens_d,
                              self.selected if selected is None else selected, self.out, self.lse, self.workspace,
                              self.flags, stream)

    def select_attend(self, stream=None):
        """Selection and sparse GQA in one launch (the selection is written to ``selected``)."""
        if stream is None:
            return self.prepared()["select_attend"]()
        msa.select_sparse_gqa_decode(self.dims, self.q, self.cache, self.block_table_d, self.seq_lens_d, self.scores,
                                     self.selected, self.out, self.lse, self.workspace, self.flags, stream)

    @property
    def fuses_selection(self) -> bool:
        """Whether ``step`` selects inside the attention launch: faster where the
        attention CTAs own whole rows (bf16 and FP8 K/V); with NVFP4 K/V the
        rows are split over CTAs and the separate selection launch is faster."""
        return self.w.kv_dtype != "nvfp4"

    @property
    def merges_insert(self) -> bool:
        """Whether ``step`` inserts the new tokens inside the index launch: with one
        query position each request's new token is in its local block, which
        the scoring never reads."""
        return self.has_index and self.w.q_len == 1

    def step(self, stream=None):
        """One decode step: insert this step's tokens, score, select, attend. The
        insert runs inside the index launch and the selection inside the
        attention launch wherever that is faster."""
        if self.merges_insert:
            self.insert_index_score(stream)
        else:
            self.insert_step_tokens(stream)
            self.index_score(stream)
        if self.fuses_selection:
            self.select_attend(stream)
        else:
            self.select(stream)
            self.attend(stream)

    def step_merged(self, stream=None):
        """Insert and scoring in one launch, then selection and attention in one launch."""
        self.insert_index_score(stream)
        self.select_attend(stream)

    def step_separate(self, stream=None):
        """The step with the selection as its own launch."""
        self.insert_step_tokens(stream)
        self.index_score(stream)
        self.select(stream)
        self.attend(stream)

    def step_fused(self, stream=None):
        """The same step with selection and attention in one launch."""
        self.insert_step_tokens(stream)
        self.index_score(stream)
        self.select_attend(stream)

    # ------------------------------------------- fused norm / RoPE / insert --
    def _prologue_state(self):
        if getattr(self, "_pro", None) is None:
            w = self.w
            B, Q = len(self.which), w.q_len
            pos = (self.lens.astype(np.int64)[:, None] - Q + np.arange(Q)[None, :]).astype(np.int32).reshape(-1)
            wts = {n: torch.from_numpy(a).to(self.device) for n, a in synth.norm_weights(w).items()}
            self._pro = dict(
                positions=torch.from_numpy(pos).to(self.device), weights=wts,
                nr=msa.make_norm_rope(wts["q"], wts["k"], wts["idx_q"], wts["idx_k"], synth.PROLOGUE_EPS,
                                      synth.PROLOGUE_THETA),
                q_out=torch.empty((B * Q, w.n_heads, w.head_dim), dtype=torch.bfloat16, device=self.device),
                idx_q_out=torch.empty((B * Q, w.n_idx_heads, w.head_dim), dtype=torch.bfloat16,
                                      device=self.device))
        return self._pro

    def qk_norm_rope_insert(self, stream=None, with_index=None):
        """The fused step in front of the decode path for this step's tokens:
        RMSNorm + RoPE of the queries and keys (and index queries / keys unless
        the layer reuses a selection), K/V/index-key insertion. The queries and
        keys of the workload are taken as the un-normalised projections; the
        normalised queries go to separate buffers (``_prologue_state``)."""
        st = self._prologue_state()
        with_index = self.has_index if with_index is None else with_index
        if with_index and self.w.idx_dtype == "f32":
            raise ValueError("the fused norm/RoPE/insert takes bf16 index projections (FP8 or NVFP4 index cache)")
        B, Q = len(self.which), self.w.q_len
        q = self.q.reshape(B * Q, self.w.n_heads, self.w.head_dim)
        qi = self.q_idx.reshape(B * Q, self.w.n_idx_heads, self.w.head_dim) if with_index else None
        msa.qk_norm_rope_insert(self.dims, q, self.new_k, self.new_v, qi, self.new_idx if with_index else None,
                                st["positions"], self.new_slots, st["nr"], st["q_out"],
                                st["idx_q_out"] if with_index else None, self.cache,
                                self.idx_cache if with_index else None, self.flags, stream)

    def reuse_step(self, selected, stream=None):
        """One decode step of a layer that reuses another layer's selection
        (logical block ids of the same requests): insert this step's K/V only,
        then attend over ``selected``."""
        msa.kv_insert_quant(self.dims, self.new_k, self.new_v, None, self.idx_new_dtype, self.new_slots,
                            self.cache, None, self.flags, stream)
        self.attend(stream if stream is not None else torch.cuda.current_stream(self.device), selected)

    def capture(self, fn) -> torch.cuda.CUDAGraph:
        """Captures ``fn(stream)`` (a step of this workload) into a CUDA graph;
        ``graph.replay()`` then reruns its kernels with the same buffers."""
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(self.device)
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream(self.device))
        torch.cuda.synchronize(self.device)
        return g

    @classmethod
    def layer_like(cls, src: "DeviceWorkload", layer: int, **kw) -> "DeviceWorkload":
        """Another attention layer of the same requests (same lengths, own
        seeded q/K/V, own caches), built without an index cache."""
        w = synth.scaled(src.w, seed=src.w.seed + synth.LAYER_SEED_STRIDE * layer)
        full = np.zeros(src.w.batch, dtype=np.int32)
        full[src.which] = src.lens
        return cls(w, src.device, which=src.which, lens=full, index_cache=False, **kw)

    def check_flags(self) -> int:
        return msa.read_device_flags(self.flags)
