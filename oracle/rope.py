"""Rotary position embedding with per-document positions. TEST INFRASTRUCTURE ONLY.

The pages place it right before attention: the attention-layer pseudo code
under Figure 1 of the XTuner page "序列并行" ("Sequence parallel") applies
``apply_rotary_pos_emb(q, k, cos, sin)`` to q and k after the qkv projection;
the page "Sample Packing: attention problems of long-sequence LLM training"
(section 4.1) notes that packed documents need their position ids reset at
every document start (Megatron's ``reset_position_id``); the InternEvo page
"Data loading and flow" (section "Fetching data from the Dataloader") gives
those positions as ``indexes`` (position inside the current segment).

Readings where the pages are silent (listed in the design notes):

* the rotation is the common "rotate-half" form: channel j of a head is paired
  with channel j + d/2, j < d/2, and rotated by the angle p * theta_j with
  theta_j = base ** (-2 j / d); base (rope_theta) defaults to 10000;
* the gradient of the rotation with respect to its input is the rotation by
  -p * theta_j (an orthogonal map's transpose), used for dQ / dK.

Plain fp64 numpy: the angle, its cosine and sine and the rotation are written
out as the definition states.
"""
import numpy as np


def inv_freq(d, base=10000.0):
    """theta_j = base^(-2j/d), j = 0 .. d/2 - 1, in fp64."""
    j = np.arange(d // 2, dtype=np.float64)
    return base ** (-2.0 * j / d)


def rope(x, positions, base=10000.0, inverse=False):
    """x [T, H, d] (any float type), positions [T] integers -> fp64 [T, H, d]:
    x'_j = x_j cos(a) - x_{j+d/2} sin(a), x'_{j+d/2} = x_{j+d/2} cos(a) + x_j sin(a),
    a = p * theta_j (or -p * theta_j for the inverse)."""
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    a = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq(d, base)[None, :]   # [T, d/2]
    if inverse:
        a = -a
    c, s = np.cos(a)[:, None, :], np.sin(a)[:, None, :]
    lo, hi = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
