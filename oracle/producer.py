"""fp64 oracle of the attention-input producer (TEST INFRASTRUCTURE, not product code).

Only the test suite and the benchmark's CPU-baseline leg may import this module.  It
shares nothing with the CUDA library: plain numpy in double precision.

What it computes, for each new token row of a fused QKV projection (the steps that come
right before attention on the hf2q "Current Inference Path" page, section 3: Q norm and
K norm (RmsNorm), V unit norm, RoPE apply, KV cache append; and the lattice-inference
DESIGN page's fused_qk_norm_rope kernel: an RMS norm over head_dim followed by RoPE over
head_dim / 2 rotation pairs):

- RMS norm of one head vector x (length D) with weight w:
      y = x / sqrt(mean(x^2) + eps) * w
  (the unit norm of V is the same with w = 1);
- rotary position embedding, the "neox" pairing the hf2q page names (RopeVariant Neox):
  element i < D/2 pairs with element i + D/2 and both rotate by
      theta_i = p * base^(-2 i / D)
  at absolute position p:
      (a, b) -> (a cos theta_i - b sin theta_i,  a sin theta_i + b cos theta_i);
- Q heads and K heads are normed (q_w, k_w) and rotated; V heads are copied, or unit
  normed when v_unit_norm is set (Gemma 4).

Readings where the pages are silent (the build's): the norm weight multiplies directly
(no 1 + w offset); eps is added to the mean square inside the square root; every
element of a head is rotated (no partial rotary factor); position p of new row t of
sequence b is pos[b] + t.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def rms_norm(x, w, eps):
    """x [..., D], w [D] or None (unit norm)."""
    x = _f64(x)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if w is None else y * _f64(w)


def rope_neox(x, positions, base):
    """x [..., T, H, D] with positions [..., T] (broadcast over heads)."""
    x = _f64(x)
    D = x.shape[-1]
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / D)
    theta = _f64(positions)[..., None, None] * inv_freq  # [..., T, 1, half]
    c, s = np.cos(theta), np.sin(theta)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def qkv_norm_rope(qkv, pos, *, n_heads, n_kv_heads, head_dim, q_w, k_w, eps, base,
                  v_unit_norm=False):
    """qkv [B, T, (Hq + 2 Hkv) * D] (the fused projection's rows), pos [B] (the first new
    row's position).  Returns q [B, T, Hq, D] and the new cache rows k, v [B, T, Hkv, D]."""
    x = _f64(qkv)
    B, T, _ = x.shape
    Hq, Hkv, D = n_heads, n_kv_heads, head_dim
    q = x[..., :Hq * D].reshape(B, T, Hq, D)
    k = x[..., Hq * D:(Hq + Hkv) * D].reshape(B, T, Hkv, D)
    v = x[..., (Hq + Hkv) * D:].reshape(B, T, Hkv, D)
    positions = _f64(pos)[:, None] + np.arange(T, dtype=np.float64)[None, :]  # [B, T]
    q = rope_neox(rms_norm(q, q_w, eps), positions, base)
    k = rope_neox(rms_norm(k, k_w, eps), positions, base)
    v = rms_norm(v, None, eps) if v_unit_norm else v.copy()
    return q, k, v
