"""The README's Python example runs as written, and its output matches the
oracle on the selection the GPU made."""
import os
import re

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example():
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    m = re.search(r"## Python example.*?```python\n(.*?)```", text, flags=re.S)
    assert m, "README has no Python example"
    return m.group(1)


def test_readme_example_runs_and_matches_the_oracle():
    import torch
    from oracle import msa as omsa

    import parity

    env = {}
    exec(compile(_example(), "README.md", "exec"), env)
    torch.cuda.synchronize()
    lens, NB = env["lens"], env["NB"]
    k = env["k"].float().cpu().numpy()
    v = env["v"].float().cpu().numpy()
    q = env["q"].float().cpu().numpy()
    sel = env["selected"].cpu().numpy()
    out = env["out"].float().cpu().numpy()
    lse = env["lse"].cpu().numpy()
    start = 0
    for b, L in enumerate(lens):
        K, V = k[start:start + L].astype(np.float64), v[start:start + L].astype(np.float64)
        start += L
        o, l = omsa.sparse_gqa(q[b].astype(np.float64), K, V, L, sel[b], 1.0 / np.sqrt(128.0), 128)
        parity.check_attention(out[b], lse[b], o, l, f"README example b={b}")
    # each row: the local block plus 15 others, ascending, none past the local block
    for b, L in enumerate(lens):
        ell = (L - 1) // 128
        for g in range(4):
            row = sel[b, 0, g]
            assert row[-1] == ell and len(set(row.tolist())) == 16 and (np.diff(row) > 0).all() and row[0] >= 0
    assert (sel < NB).all()
