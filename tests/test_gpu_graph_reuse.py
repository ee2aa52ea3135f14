"""A whole decode step replayed from a CUDA graph, and a layer that reuses another
layer's block selection.

"vLLM、AMD Instinct MI355X上でMiniMax M3のボトルネック最適化手法を公開",
question 2: graph execution removes the per-kernel launch cost; question 3:
adjacent sparse layers pick nearly the same blocks, so one layer's top-k
decision serves the next layers, which then write no index keys either.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_07_gb300 import synth
from block_sparse_attention_07_gb300.workload import DeviceWorkload
from oracle import run as orun

import parity

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

GRAPH_CASES = {
    # bf16 KV: every CTA owns whole rows
    "bf16": (synth.scaled(W["b32_32k"], batch=3, ctx=2000), None),
    # NVFP4 KV: rows split over CTAs and merged by the last arriver (tickets)
    "nvfp4_split_rows": (synth.scaled(W["nvfp4_256k"], batch=2, ctx=3000), "tickets"),
    # NVFP4 KV: each row split over a thread-block cluster (the automatic choice here)
    "nvfp4_cluster": (synth.scaled(W["nvfp4_256k"], batch=2, ctx=3000), None),
    # NVFP4 index keys, 8 positions
    "spec_fp4idx": (synth.scaled(W["spec8"], batch=2, ctx=2600, idx_dtype="nvfp4"), None),
}


@pytest.mark.parametrize("name", list(GRAPH_CASES))
def test_graph_replay_matches_eager_and_oracle(name, monkeypatch):
    w, split = GRAPH_CASES[name]
    if split is None:
        monkeypatch.delenv("MSA_NVFP4_SPLIT", raising=False)
    else:
        monkeypatch.setenv("MSA_NVFP4_SPLIT", split)
    dw = parity.build(w)
    dw.step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (dw.scores, dw.selected, dw.out, dw.lse)]
    g = dw.capture(dw.step)
    for _ in range(3):                      # replays reuse the captured split-K tickets
        dw.scores.fill_(7.0)
        dw.selected.fill_(-7)
        dw.out.zero_()
        dw.lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip((dw.scores, dw.selected, dw.out, dw.lse), eager):
            assert torch.equal(a, b)
    assert dw.check_flags() == 0
    parity.verify_workload(dw, w, synth.seq_lens(w), run_step=False)


REUSE_CASES = {
    "bf16": synth.scaled(W["b32_32k"], batch=2, ctx=2500),
    "nvfp4": synth.scaled(W["nvfp4_256k"], batch=2, ctx=2200),
    "spec8": synth.scaled(W["spec8"], batch=2, ctx=2100),
}


@pytest.mark.parametrize("name", list(REUSE_CASES))
@pytest.mark.parametrize("graph", [False, True])
def test_layer_reusing_selection(name, graph):
    w = REUSE_CASES[name]
    src = parity.build(w)
    src.step()
    layer = DeviceWorkload.layer_like(src, 1)
    assert layer.idx_cache is None
    if graph:
        g = layer.capture(lambda st: layer.reuse_step(src.selected, st))
        g.replay()
        g.replay()
    else:
        layer.reuse_step(src.selected)
    torch.cuda.synchronize()
    assert layer.check_flags() == 0 and src.check_flags() == 0
    sel = src.selected.cpu().numpy()
    out = layer.out.float().cpu().numpy()
    lse = layer.lse.cpu().numpy()
    kg, vg = parity.kv_globals(w)
    lens = synth.seq_lens(w)
    for bi, b in enumerate(layer.which):
        L = int(lens[b])
        req = synth.request(layer.w, b, L)          # the layer's own q, K, V
        ora = orun.run_request(req, L, w.topk, w.softmax_scale, w.block_size, w.idx_dtype, w.kv_dtype, kg, vg,
                               sel=sel[bi], idx_global=parity.idx_global(w))
        parity.check_attention(out[bi], lse[bi], ora["out"], ora["lse"], f"{w.name} layer 1 b={b}")
    # a different layer really attends over different data
    assert not torch.equal(layer.out, src.out)


def test_two_streams_at_once(monkeypatch):
    """Two independent decode steps in flight on two streams at once: an NVFP4
    one whose rows are merged through tickets, and a bf16 one. Each has its own
    workspace and caches, and both must still match the oracle and repeat
    bit for bit."""
    monkeypatch.setenv("MSA_NVFP4_SPLIT", "tickets")
    wa = synth.scaled(W["nvfp4_256k"], batch=2, ctx=3000)
    wb = synth.scaled(W["b32_32k"], batch=3, ctx=2000)
    da, db = parity.build(wa), parity.build(wb)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    firsts = None
    for it in range(4):
        with torch.cuda.stream(sa):
            da.step_separate(sa)
        with torch.cuda.stream(sb):
            db.step_fused(sb)
        torch.cuda.synchronize()
        now = [t.clone() for t in (da.out, da.lse, db.out, db.lse)]
        if firsts is None:
            firsts = now
        else:
            for x, y in zip(firsts, now):
                assert torch.equal(x, y)
    parity.verify_workload(da, wa, synth.seq_lens(wa), run_step=False)
    parity.verify_workload(db, wb, synth.seq_lens(wb), run_step=False)


def test_graph_replays_after_many_direct_calls():
    """The index launch hands out its last blocks from a queue slot; a captured
    graph keeps its slot while more than 64 direct calls cycle through theirs,
    and two captured graphs replay in turn, each equal to an eager step."""
    w = synth.scaled(W["b32_32k"], batch=3, ctx=2600)
    dw = parity.build(w)
    dw.step()
    torch.cuda.synchronize()
    eager = dw.scores.clone()
    g1 = dw.capture(dw.step)
    g2 = dw.capture(dw.step)
    for _ in range(70):                     # direct calls through every direct-call slot
        dw.index_score()
    torch.cuda.synchronize()
    for g in (g1, g2, g1, g2):
        dw.scores.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dw.scores, eager)
    assert dw.check_flags() == 0
