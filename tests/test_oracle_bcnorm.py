"""Pins of the B, C prologue oracle (oracle/bcnorm.py) by properties of its definition.

A wrong normalisation axis (ranks instead of state entries), a missing square root, the bias
added before the norm or the weight applied before it each break one of these."""
import numpy as np

from oracle.bcnorm import bc_prologue, bc_prologue_layout


def _v(seed, shape):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape) * 3.0


def test_unit_weight_no_bias_gives_unit_rms_over_state_entries():
    v = _v(1, (5, 4, 16))                       # [T, R, N]
    out = bc_prologue(v, np.ones(16), np.zeros(16), eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(out ** 2, axis=-1)), 1.0, rtol=1e-13)
    # each (token, rank) vector keeps its direction
    cos = np.sum(out * v, -1) / (np.linalg.norm(out, axis=-1) * np.linalg.norm(v, axis=-1))
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)


def test_epsilon_closed_form():
    v = _v(2, (3, 2, 8))
    eps = 0.5
    out = bc_prologue(v, np.ones(8), np.zeros(8), eps)
    ms = np.mean(v * v, -1)
    np.testing.assert_allclose(np.mean(out ** 2, -1), ms / (ms + eps), rtol=1e-13)


def test_scale_invariance():
    v = _v(3, (4, 2, 12))
    w, b = _v(4, 12), _v(5, 12)
    np.testing.assert_allclose(bc_prologue(7.5 * v, w, b, 0.0), bc_prologue(v, w, b, 0.0), rtol=1e-13)


def test_bias_is_added_after_the_norm_and_weight_scales_it():
    v = _v(6, (3, 1, 10))
    w, b = _v(7, 10), _v(8, 10)
    base = bc_prologue(v, np.ones(10), np.zeros(10), 1e-6)
    np.testing.assert_allclose(bc_prologue(v, w, b, 1e-6), base * w + b, rtol=1e-13, atol=1e-13)


def test_layout_uses_each_heads_bias():
    v = _v(9, (2, 3, 4, 2, 6))                  # [B, T, H, R, N]
    w, b = _v(10, 6), _v(11, (4, 6))
    out = bc_prologue_layout(v, w, b, 1e-6)
    for h in range(4):
        np.testing.assert_allclose(out[:, :, h], bc_prologue(v[:, :, h], w, b[h], 1e-6), rtol=1e-14)
