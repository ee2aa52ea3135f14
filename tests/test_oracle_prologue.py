"""Pins of the oracle's norm / rotary-embedding step (oracle/prologue.py):
rotation invariants (identity at position 0, norm preservation per pair,
composition, the relative-position identity), the half-split pairing on a
closed form, RMSNorm against torch's own rms_norm and its invariants, and the
bf16 rounding on exact ties and on values just past a tie."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import prologue as P


def _x(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_rope_identity_at_position_zero():
    x = _x((3, 5, 128), 1)
    assert np.array_equal(P.rope(x, np.zeros(3), 10000.0), x)


def test_rope_preserves_each_pair_norm():
    x = _x((4, 2, 128), 2)
    pos = np.array([1, 77, 4095, 262143])
    y = P.rope(x, pos, 10000.0)
    n_in = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_out = y[..., :64] ** 2 + y[..., 64:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12, atol=1e-12)


def test_rope_composition_and_relative_position():
    q = _x((1, 1, 128), 3)
    k = _x((1, 1, 128), 4)
    a, b = 1234, 567
    comp = P.rope(P.rope(q, np.array([a]), 1e4), np.array([b]), 1e4)
    np.testing.assert_allclose(comp, P.rope(q, np.array([a + b]), 1e4), rtol=1e-9, atol=1e-9)
    # <R_p q, R_s k> depends only on p - s
    for p, s in ((900, 100), (5000, 4200), (65535, 64735)):
        lhs = np.sum(P.rope(q, np.array([p]), 1e4) * P.rope(k, np.array([s]), 1e4))
        rhs = np.sum(P.rope(q, np.array([p - s]), 1e4) * k)
        assert lhs == pytest.approx(rhs, rel=1e-9, abs=1e-9)


def test_rope_half_split_pairing_closed_form():
    """Dim i pairs with dim i + 64 and turns by pos * theta^(-2i/128)."""
    D, theta, pos = 128, 500.0, 3
    for i in (0, 1, 17, 63):
        x = np.zeros((1, 1, D))
        x[0, 0, i] = 1.0
        y = P.rope(x, np.array([pos]), theta)[0, 0]
        phi = pos * theta ** (-2.0 * i / D)
        want = np.zeros(D)
        want[i], want[i + 64] = np.cos(phi), np.sin(phi)
        np.testing.assert_allclose(y, want, atol=1e-15)


def test_rms_norm_matches_torch_and_invariants():
    x = _x((6, 3, 128), 5) * 3.0
    w = 1.0 + 0.1 * _x((128,), 6)
    eps = 1e-6
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(w), eps).numpy()
    np.testing.assert_allclose(P.rms_norm(x, w, eps), ref, rtol=1e-12, atol=1e-12)
    y = P.rms_norm(x, np.ones(128), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-12)
    np.testing.assert_allclose(P.rms_norm(7.5 * x, w, 0.0), P.rms_norm(x, w, 0.0), rtol=1e-12)


def test_bf16_rounding_ties_and_near_ties():
    one = 1.0
    ulp = 2.0 ** -7                                   # bf16 spacing at 1
    vals = np.array([one + ulp / 2,                    # exact tie -> even (1.0)
                     one + 3 * ulp / 2,                # exact tie -> even (1 + 2 ulp)
                     one + ulp / 2 + 2.0 ** -40,       # past the tie (its fp32 rounding is the tie) -> up
                     one + ulp / 2 - 2.0 ** -40,       # short of the tie -> down
                     -(one + ulp / 2 + 2.0 ** -40)])
    got = F.bf16_to_f64(P.to_bf16(vals))
    np.testing.assert_array_equal(got, [one, one + 2 * ulp, one + ulp, one, -(one + ulp)])
