"""Checks that pin the producer oracle (oracle/producer.py) to facts other than itself.

Each ``pin_*`` takes a module-like object with ``rms_norm``, ``rope_neox`` and
``qkv_norm_rope`` and raises AssertionError on a disagreement with the mathematics:

- hand-derived closed forms (tests/golden/producer_cases.json);
- a per-element loop in plain Python floats (math.cos, math.sin), a separate code path
  from the oracle's vectorised numpy;
- invariants: RoPE is a rotation (it keeps each head's length), the product of a rotated
  query and a rotated key depends only on their distance, position 0 changes nothing;
  the RMS norm output has mean square ms / (ms + eps) and does not change when the input
  is scaled (eps = 0).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "producer_cases.json")


def _close(a, b, tol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, "%s: shape %s vs %s" % (what, a.shape, b.shape)
    err = np.abs(a - b).max() if a.size else 0.0
    assert err <= tol, "%s: max abs error %.3e > %.1e" % (what, err, tol)


def pin_golden(prod):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        y = prod.rope_neox(prod.rms_norm(np.array(c["x"], float)[None, None], c["w"], c["eps"]),
                           np.array([c["pos"]], float), c["base"])
        _close(y[0, 0], c["y"], 1e-12, c["name"])


def _loop_reference(x, pos, w, eps, base):
    """One head vector, element by element, in Python floats."""
    D = len(x)
    ms = sum(v * v for v in x) / D
    r = math.sqrt(ms + eps)
    y = [x[i] / r * w[i] for i in range(D)]
    out = list(y)
    for i in range(D // 2):
        th = pos * base ** (-2.0 * i / D)
        a, b = y[i], y[i + D // 2]
        out[i] = a * math.cos(th) - b * math.sin(th)
        out[i + D // 2] = a * math.sin(th) + b * math.cos(th)
    return out


def pin_loop_reference(prod):
    rng = np.random.default_rng(21)
    for D in (2, 8, 80, 128):
        for pos in (0, 3, 1000, 50000):
            x = rng.standard_normal(D)
            w = rng.standard_normal(D)
            eps = 1e-6 if D != 8 else 0.3
            got = prod.rope_neox(prod.rms_norm(x[None, None], w, eps), np.array([pos], float),
                                 1e6)[0, 0]
            _close(got, _loop_reference(list(x), pos, list(w), eps, 1e6), 1e-9,
                   "loop reference D%d pos%d" % (D, pos))


def pin_rope_is_a_rotation(prod):
    rng = np.random.default_rng(22)
    x = rng.standard_normal((2, 5, 3, 64))
    pos = np.array([[0, 7, 100, 4095, 65536], [1, 2, 3, 4, 5]], float)
    y = prod.rope_neox(x, pos, 1e4)
    _close(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), 1e-10, "lengths kept")
    _close(prod.rope_neox(x[:, :1], pos[:, :1] * 0, 1e4), x[:, :1], 0.0, "position 0")


def pin_rope_depends_on_distance(prod):
    """<rope(q, m), rope(k, n)> = <rope(q, m + s), rope(k, n + s)>: the property RoPE exists
    for.  A wrong pairing, sign or frequency breaks it."""
    rng = np.random.default_rng(23)
    q = rng.standard_normal((1, 1, 1, 128))
    k = rng.standard_normal((1, 1, 1, 128))
    for m, n, s in ((5, 2, 100), (0, 37, 1000), (300, 299, 12345)):
        a = np.sum(prod.rope_neox(q, np.array([[m]], float), 1e6) *
                   prod.rope_neox(k, np.array([[n]], float), 1e6))
        b = np.sum(prod.rope_neox(q, np.array([[m + s]], float), 1e6) *
                   prod.rope_neox(k, np.array([[n + s]], float), 1e6))
        assert abs(a - b) < 1e-9, "rotated product moved with the shift: %r vs %r" % (a, b)


def pin_rms_norm_invariants(prod):
    rng = np.random.default_rng(24)
    x = rng.standard_normal((4, 3, 96)) * 3.0
    ones = np.ones(96)
    y = prod.rms_norm(x, ones, 0.0)
    _close(np.mean(y * y, axis=-1), np.ones((4, 3)), 1e-12, "unit mean square")
    _close(prod.rms_norm(7.5 * x, ones, 0.0), y, 1e-12, "scale invariance")
    eps = 0.25
    ms = np.mean(x * x, axis=-1)
    y = prod.rms_norm(x, None, eps)
    _close(np.mean(y * y, axis=-1), ms / (ms + eps), 1e-12, "eps inside the root")


def pin_qkv_split(prod):
    """The fused row splits into Q, K, V heads in that order; V is copied unless unit
    normed; Q and K go through norm and RoPE with their own weights."""
    rng = np.random.default_rng(25)
    B, T, Hq, Hkv, D = 2, 3, 4, 2, 8
    x = rng.standard_normal((B, T, (Hq + 2 * Hkv) * D))
    qw, kw = rng.standard_normal(D), rng.standard_normal(D)
    pos = np.array([10, 0])
    q, k, v = prod.qkv_norm_rope(x, pos, n_heads=Hq, n_kv_heads=Hkv, head_dim=D, q_w=qw, k_w=kw,
                                 eps=1e-6, base=1e4)
    positions = pos[:, None] + np.arange(T)[None, :]
    xq = x[..., :Hq * D].reshape(B, T, Hq, D)
    xk = x[..., Hq * D:(Hq + Hkv) * D].reshape(B, T, Hkv, D)
    xv = x[..., (Hq + Hkv) * D:].reshape(B, T, Hkv, D)
    for b in range(B):
        for t in range(T):
            for h in range(Hq):
                _close(q[b, t, h], _loop_reference(list(xq[b, t, h]), positions[b, t], list(qw),
                                                   1e-6, 1e4), 1e-9, "q head")
            for h in range(Hkv):
                _close(k[b, t, h], _loop_reference(list(xk[b, t, h]), positions[b, t], list(kw),
                                                   1e-6, 1e4), 1e-9, "k head")
    _close(v, xv, 0.0, "v copied")
    _, _, vn = prod.qkv_norm_rope(x, pos, n_heads=Hq, n_kv_heads=Hkv, head_dim=D, q_w=qw,
                                  k_w=kw, eps=1e-6, base=1e4, v_unit_norm=True)
    _close(np.mean(vn * vn, axis=-1), np.mean(xv * xv, axis=-1) /
           (np.mean(xv * xv, axis=-1) + 1e-6), 1e-12, "v unit norm")


ALL_PINS = [pin_golden, pin_loop_reference, pin_rope_is_a_rotation, pin_rope_depends_on_distance,
            pin_rms_norm_invariants, pin_qkv_split]
