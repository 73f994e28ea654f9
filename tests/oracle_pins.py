"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes an oracle object (``.prefill`` / ``.decode``) and raises
AssertionError when the oracle disagrees with the mathematics:

- hand-derived closed-form cases (tests/golden/closed_form_cases.json);
- brute force on tiny inputs: the full score matrix materialised with an explicitly
  built visible-key matrix and the softmax taken in extended precision (long double),
  a separate code path from the oracle's row loop;
- closed forms: one visible key returns that value row exactly; identical keys and a
  zero scale return the mean of the visible values, lse = s + ln n; a softcap far above
  every score changes nothing;
- invariants: GQA equals multi-head attention with the KV heads repeated, a sliding
  window equals full attention with a materialised -inf mask, a decode step equals
  the last prefill row, adding a vector to every key shifts lse by scale*q.c and
  leaves the output alone, and (without a causal mask) jointly permuting the key and
  value rows changes nothing.

The same functions run against deliberately broken copies of the oracle in
test_oracle.py, to show that a plausible mistake fails at least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "closed_form_cases.json")


def _rng(seed):
    return np.random.default_rng(seed)


def golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


# ------------------------------------------------------------------------------------
# brute force, written independently of the oracle's loops

def visible_matrix(S, L, causal, window):
    """[S, L] boolean: row i (absolute position i + L - S) may read key j.

    Built by ranges rather than by testing each pair: with causal masking the row
    reads keys up to and including its own position; a window of W keeps only the
    last W positions up to the row's own; without causal masking keys after the
    row's position stay readable."""
    vis = np.zeros((S, L), dtype=bool)
    for i in range(S):
        pos = i + L - S
        last = min(pos, L - 1) if causal else L - 1
        first = max(0, pos - window + 1) if window > 0 else 0
        if last >= first:
            vis[i, first:last + 1] = True
    return vis


def brute_force(q, k, v, causal, window, scale, softcap=0.0):
    """Materialised softmax attention in long double.  q [B,S,Hq,D], k/v [B,L,Hkv,D];
    with softcap > 0 every scaled score s becomes softcap * tanh(s / softcap)."""
    B, S, Hq, D = q.shape
    L, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    ld = np.longdouble
    k_rep = np.repeat(k.astype(ld), G, axis=2)  # head h reads k_rep[..., h, :]
    v_rep = np.repeat(v.astype(ld), G, axis=2)
    vis = visible_matrix(S, L, causal, window)
    out = np.zeros((B, S, Hq, D), dtype=ld)
    lse = np.zeros((B, S, Hq), dtype=ld)
    for b in range(B):
        for h in range(Hq):
            scores = ld(scale) * np.einsum("sd,ld->sl", q[b, :, h, :].astype(ld),
                                           k_rep[b, :, h, :])
            if softcap > 0:
                scores = ld(softcap) * np.tanh(scores / ld(softcap))
            scores = np.where(vis, scores, ld(-np.inf))
            for i in range(S):
                if not vis[i].any():
                    out[b, i, h] = 0
                    lse[b, i, h] = -np.inf
                    continue
                m = scores[i].max()
                e = np.exp(scores[i] - m)
                z = e.sum()
                out[b, i, h] = (e[:, None] * v_rep[b, :, h, :]).sum(axis=0) / z
                lse[b, i, h] = m + np.log(z)
    return out, lse


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, "%s: shape %s vs %s" % (what, a.shape, b.shape)
    inf_a, inf_b = np.isneginf(a), np.isneginf(b)
    assert (inf_a == inf_b).all(), "%s: -inf pattern differs" % what
    fin = ~inf_a
    err = np.abs(a[fin] - b[fin]).max() if fin.any() else 0.0
    assert err <= tol, "%s: max abs error %.3e > %.1e" % (what, err, tol)


# ------------------------------------------------------------------------------------
# pins

def pin_golden(orc):
    for c in golden_cases():
        q = np.array(c["q"], dtype=np.float64)[None]
        k = np.array(c["k"], dtype=np.float64)[None]
        v = np.array(c["v"], dtype=np.float64)[None]
        out, lse = orc.prefill(q, k, v, causal=c["causal"], window=c["window"],
                               scale=c["scale"], softcap=c.get("softcap", 0.0))
        _close(out[0], np.array(c["out"]), 1e-12, c["name"] + " out")
        _close(lse[0], np.array(c["lse"]), 1e-12, c["name"] + " lse")


BRUTE_CASES = [
    # B, S, L, Hq, Hkv, D, causal, window
    (1, 1, 1, 1, 1, 1, True, 0),
    (1, 4, 4, 2, 1, 3, True, 0),
    (2, 5, 8, 4, 2, 4, True, 0),
    (1, 8, 8, 6, 2, 2, True, 3),
    (2, 3, 7, 3, 3, 5, False, 0),
    (1, 6, 6, 4, 1, 4, False, 2),
    (1, 7, 5, 2, 2, 3, True, 0),     # S > L: the first rows see no key
    (2, 8, 8, 8, 4, 1, True, 1),
    (1, 5, 8, 5, 1, 4, True, 4),
]

# (case, softcap): brute-force cases rerun with a score cap well inside the score range
BRUTE_SOFTCAP = [(1, 0.5), (2, 1.3), (3, 0.8), (5, 2.0), (8, 0.3)]


def pin_brute_force(orc):
    for n, (B, S, L, Hq, Hkv, D, causal, window) in enumerate(BRUTE_CASES):
        r = _rng(100 + n)
        q = r.standard_normal((B, S, Hq, D))
        k = r.standard_normal((B, L, Hkv, D))
        v = r.standard_normal((B, L, Hkv, D))
        scale = 1.0 / math.sqrt(D) if n % 2 else 0.7
        out, lse = orc.prefill(q, k, v, causal=causal, window=window, scale=scale)
        bo, bl = brute_force(q, k, v, causal, window, scale)
        _close(out, bo, 1e-12, "brute force case %d out" % n)
        _close(lse, bl, 1e-12, "brute force case %d lse" % n)
    for n, cap in BRUTE_SOFTCAP:
        B, S, L, Hq, Hkv, D, causal, window = BRUTE_CASES[n]
        r = _rng(300 + n)
        q = 2.0 * r.standard_normal((B, S, Hq, D))  # scores of several units: the cap bites
        k = r.standard_normal((B, L, Hkv, D))
        v = r.standard_normal((B, L, Hkv, D))
        out, lse = orc.prefill(q, k, v, causal=causal, window=window, scale=0.9, softcap=cap)
        bo, bl = brute_force(q, k, v, causal, window, 0.9, softcap=cap)
        _close(out, bo, 1e-12, "brute force softcap case %d out" % n)
        _close(lse, bl, 1e-12, "brute force softcap case %d lse" % n)


def pin_softcap_far_above_scores_is_no_cap(orc):
    """tanh(x) = x - x^3/3 + ...: with every |s| <= 10 and a cap of 1e6 the capped score
    differs from s by under 1e-9, so the result must match the uncapped one."""
    r = _rng(11)
    q = r.standard_normal((2, 6, 4, 8))
    k = r.standard_normal((2, 6, 2, 8))
    v = r.standard_normal((2, 6, 2, 8))
    a_out, a_lse = orc.prefill(q, k, v, causal=True, window=0, scale=0.35)
    b_out, b_lse = orc.prefill(q, k, v, causal=True, window=0, scale=0.35, softcap=1e6)
    _close(b_out, a_out, 1e-8, "huge softcap out")
    _close(b_lse, a_lse, 1e-8, "huge softcap lse")


def pin_single_visible_key(orc):
    """Window 1 with causal masking: each row reads only its own key, so out is that
    value row exactly and lse is its scaled score."""
    r = _rng(7)
    B, S, Hq, Hkv, D = 2, 9, 4, 2, 8
    q = r.standard_normal((B, S, Hq, D))
    k = r.standard_normal((B, S, Hkv, D))
    v = r.standard_normal((B, S, Hkv, D))
    scale = 0.3
    out, lse = orc.prefill(q, k, v, causal=True, window=1, scale=scale)
    G = Hq // Hkv
    for h in range(Hq):
        assert np.array_equal(out[:, :, h, :], v[:, :, h // G, :]), "single key: out != v"
        s = scale * np.einsum("bsd,bsd->bs", q[:, :, h, :], k[:, :, h // G, :])
        _close(lse[:, :, h], s, 1e-13, "single key lse")


def pin_identical_keys(orc):
    """All keys equal: every visible key has the same score s, the weights are 1/n,
    out is the mean of the visible values and lse = s + ln n."""
    r = _rng(8)
    B, S, Hq, Hkv, D = 1, 12, 3, 1, 6
    q = r.standard_normal((B, S, Hq, D))
    krow = r.standard_normal(D)
    k = np.broadcast_to(krow, (B, S, Hkv, D)).copy()
    v = r.standard_normal((B, S, Hkv, D))
    scale, W = 0.5, 5
    out, lse = orc.prefill(q, k, v, causal=True, window=W, scale=scale)
    for i in range(S):
        lo = max(0, i - W + 1)
        n = i - lo + 1
        mean = v[0, lo:i + 1, 0, :].mean(axis=0)
        for h in range(Hq):
            _close(out[0, i, h], mean, 1e-13, "identical keys out")
            s = scale * float(q[0, i, h] @ krow)
            _close(lse[0, i, h], s + math.log(n), 1e-13, "identical keys lse")


def pin_zero_scale(orc):
    """scale 0: uniform weights over the visible keys, lse = ln n."""
    r = _rng(9)
    B, S, L, Hq, Hkv, D = 2, 6, 10, 2, 2, 4
    q = r.standard_normal((B, S, Hq, D))
    k = r.standard_normal((B, L, Hkv, D))
    v = r.standard_normal((B, L, Hkv, D))
    out, lse = orc.prefill(q, k, v, causal=True, window=0, scale=0.0)
    for b in range(B):
        for i in range(S):
            n = i + L - S + 1
            for h in range(Hq):
                _close(out[b, i, h], v[b, :n, h, :].mean(axis=0), 1e-13, "zero scale out")
                _close(lse[b, i, h], math.log(n), 1e-13, "zero scale lse")


def pin_gqa_is_repeated_mha(orc):
    r = _rng(10)
    B, S, L, Hkv, G, D = 2, 7, 9, 2, 3, 5
    q = r.standard_normal((B, S, Hkv * G, D))
    k = r.standard_normal((B, L, Hkv, D))
    v = r.standard_normal((B, L, Hkv, D))
    for causal, window in ((True, 0), (True, 3), (False, 0)):
        out, lse = orc.prefill(q, k, v, causal=causal, window=window, scale=0.4)
        k_rep = np.stack([k[:, :, h // G, :] for h in range(Hkv * G)], axis=2)
        v_rep = np.stack([v[:, :, h // G, :] for h in range(Hkv * G)], axis=2)
        out2, lse2 = orc.prefill(q, k_rep, v_rep, causal=causal, window=window, scale=0.4)
        _close(out, out2, 1e-14, "gqa vs repeated out")
        _close(lse, lse2, 1e-14, "gqa vs repeated lse")


def pin_window_is_masked_softmax(orc):
    """Sliding window against plain fp64 softmax with a materialised -inf mask built
    from the distance |p - j| rather than from ranges."""
    r = _rng(11)
    B, S, Hq, D, W = 1, 40, 2, 8, 7
    q = r.standard_normal((B, S, Hq, D))
    k = r.standard_normal((B, S, 1, D))
    v = r.standard_normal((B, S, 1, D))
    pos = np.arange(S)[:, None]
    key = np.arange(S)[None, :]
    for causal in (True, False):
        dist = pos - key
        mask = np.where(dist < W, 0.0, -np.inf)
        if causal:
            mask = np.where(dist >= 0, mask, -np.inf)
        out, lse = orc.prefill(q, k, v, causal=causal, window=W, scale=0.35)
        for h in range(Hq):
            s = 0.35 * q[0, :, h, :] @ k[0, :, 0, :].T + mask
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            ref = (e @ v[0, :, 0, :]) / e.sum(axis=1, keepdims=True)
            ref_lse = m[:, 0] + np.log(e.sum(axis=1))
            _close(out[0, :, h], ref, 1e-12, "window out")
            _close(lse[0, :, h], ref_lse, 1e-12, "window lse")


def pin_decode_is_last_prefill_row(orc):
    r = _rng(12)
    B, L, Hq, Hkv, D = 3, 11, 4, 2, 6
    q_all = r.standard_normal((B, L, Hq, D))
    k = r.standard_normal((B, L, Hkv, D))
    v = r.standard_normal((B, L, Hkv, D))
    for window in (0, 4):
        out, lse = orc.prefill(q_all, k, v, causal=True, window=window, scale=0.45)
        dout, dlse = orc.decode(q_all[:, -1], k, v, [L] * B, window=window, scale=0.45)
        _close(dout, out[:, -1], 1e-14, "decode vs last prefill row out")
        _close(dlse, lse[:, -1], 1e-14, "decode vs last prefill row lse")
    # per-sequence lengths: sequence b at length n equals prefill over its first n keys
    lens = [4, 11, 1]
    dout, dlse = orc.decode(q_all[:, 0], k, v, lens, window=0, scale=0.45)
    for b, n in enumerate(lens):
        o, l = orc.prefill(q_all[b:b + 1, :1], k[b:b + 1, :n], v[b:b + 1, :n], causal=False,
                           window=0, scale=0.45)
        _close(dout[b], o[0, 0], 1e-14, "decode length %d out" % n)
        _close(dlse[b], l[0, 0], 1e-14, "decode length %d lse" % n)


def pin_key_shift(orc):
    """k_j -> k_j + c adds scale*q.c to every score of the row: out unchanged,
    lse shifted by that amount."""
    r = _rng(13)
    B, S, Hq, Hkv, D = 1, 10, 4, 2, 7
    q = r.standard_normal((B, S, Hq, D))
    k = r.standard_normal((B, S, Hkv, D))
    v = r.standard_normal((B, S, Hkv, D))
    c = r.standard_normal((Hkv, D))
    out, lse = orc.prefill(q, k, v, causal=True, window=0, scale=0.6)
    out2, lse2 = orc.prefill(q, k + c[None, None], v, causal=True, window=0, scale=0.6)
    _close(out2, out, 1e-12, "key shift out")
    G = Hq // Hkv
    shift = np.stack([0.6 * q[:, :, h, :] @ c[h // G] for h in range(Hq)], axis=2)
    _close(lse2, lse + shift, 1e-12, "key shift lse")


def pin_key_permutation(orc):
    r = _rng(14)
    B, S, L, Hq, Hkv, D = 2, 5, 9, 2, 1, 4
    q = r.standard_normal((B, S, Hq, D))
    k = r.standard_normal((B, L, Hkv, D))
    v = r.standard_normal((B, L, Hkv, D))
    perm = r.permutation(L)
    out, lse = orc.prefill(q, k, v, causal=False, window=0, scale=0.5)
    out2, lse2 = orc.prefill(q, k[:, perm], v[:, perm], causal=False, window=0, scale=0.5)
    _close(out2, out, 1e-13, "permutation out")
    _close(lse2, lse, 1e-13, "permutation lse")


ALL_PINS = [pin_golden, pin_brute_force, pin_single_visible_key, pin_identical_keys,
            pin_zero_scale, pin_gqa_is_repeated_mha, pin_window_is_masked_softmax,
            pin_decode_is_last_prefill_row, pin_key_shift, pin_key_permutation,
            pin_softcap_far_above_scores_is_no_cap]
