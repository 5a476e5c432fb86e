"""Oracle for the B, C prologue of the Mamba-3 block -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` may import this module; nothing on the CUDA path does.

What it computes (paper section 3.4, "BC / QK normalisation" and "B, C bias"; the aipaper.cc
summary, architecture item 3): after the B and C projections, an RMS normalisation (the
QKNorm of Transformers, called BCNorm), then a learnable, head-specific, channel-wise bias.
The pages do not print the formula; the readings taken here:

  * the RMS is taken over the N state entries of each (token, head, rank) vector;
  * the normalised vector is scaled by a learnable weight w[n] shared by heads and ranks;
  * the bias b[h, n] is per head and state index, shared by the ranks, added after the norm;
  * epsilon is an argument (the pages give none):

        out[n] = v[n] / sqrt(mean_n v^2 + eps) * w[n] + b[h, n]

The output feeds the SSM core unchanged (``oracle.scan``), before the rotation.  Pinned in
tests/test_oracle_bcnorm.py by properties of the definition (unit RMS, scale invariance,
bias shift, weight scaling), not by re-typing it.
"""
from __future__ import annotations

import numpy as np


def bc_prologue(v, w, b, eps: float):
    """v [..., R, N] raw projection output of one head (any leading axes); w [N]; b [N] (this
    head's bias).  Returns the normalised, scaled and shifted values, float64."""
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * np.asarray(w, np.float64) + np.asarray(b, np.float64)


def bc_prologue_layout(v, w, b, eps: float):
    """The library layout: v [B, T, H, R, N]; w [N]; b [H, N]."""
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    for h in range(v.shape[2]):
        out[:, :, h] = bc_prologue(v[:, :, h], w, np.asarray(b)[h], eps)
    return out
