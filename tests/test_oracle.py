"""The fp64 oracle against its pins (CPU only)."""
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS, golden_cases


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle(oracle.build_library())


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_golden_fixture_is_nontrivial():
    cases = golden_cases()
    assert len(cases) >= 4
    assert any(c["window"] > 0 for c in cases)
    assert any(c["Hq"] > c["Hkv"] for c in cases)


def test_row_subset_equals_full(orc):
    r = np.random.default_rng(1)
    B, S, Hq, Hkv, D = 2, 13, 4, 2, 8
    q = r.standard_normal((B, S, Hq, D))
    k = r.standard_normal((B, S, Hkv, D))
    v = r.standard_normal((B, S, Hkv, D))
    out, lse = orc.prefill(q, k, v, causal=True, window=5, scale=0.3)
    rows = [0, 5, 12, 13, 25]
    o2, l2 = orc.prefill(q, k, v, causal=True, window=5, scale=0.3, rows=rows)
    flat_o, flat_l = out.reshape(B * S, Hq, D), lse.reshape(B * S, Hq)
    assert np.array_equal(o2, flat_o[rows]) and np.array_equal(l2, flat_l[rows])


def test_thread_count_does_not_change_bits(orc):
    r = np.random.default_rng(2)
    q = r.standard_normal((2, 30, 6, 16))
    k = r.standard_normal((2, 30, 2, 16))
    v = r.standard_normal((2, 30, 2, 16))
    a = orc.prefill(q, k, v, causal=True, window=0, scale=0.25, threads=1)
    b = orc.prefill(q, k, v, causal=True, window=0, scale=0.25, threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rows_without_keys(orc):
    """More query rows than keys under causal masking: rows at negative positions read
    nothing, giving out = 0 and lse = -inf."""
    r = np.random.default_rng(3)
    q = r.standard_normal((1, 6, 1, 4))
    k = r.standard_normal((1, 3, 1, 4))
    v = r.standard_normal((1, 3, 1, 4))
    out, lse = orc.prefill(q, k, v, causal=True, window=0, scale=1.0)
    assert np.all(out[0, :3] == 0) and np.all(np.isneginf(lse[0, :3]))
    assert np.all(np.isfinite(lse[0, 3:]))


def test_bad_arguments_raise(orc):
    q = np.zeros((1, 2, 3, 4))
    k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        orc.prefill(q, k, k, causal=True, window=0, scale=1.0)  # 3 % 2 != 0


def test_kv_append_oracle():
    r = np.random.default_rng(4)
    kc = r.standard_normal((2, 8, 2, 4))
    vc = r.standard_normal((2, 8, 2, 4))
    kn = r.standard_normal((2, 3, 2, 4))
    vn = r.standard_normal((2, 3, 2, 4))
    k2, v2 = oracle.kv_append(kc, vc, kn, vn, [0, 5])
    assert np.array_equal(k2[0, :3], kn[0]) and np.array_equal(k2[1, 5:8], kn[1])
    assert np.array_equal(v2[0, 3:], vc[0, 3:]) and np.array_equal(v2[1, :5], vc[1, :5])
    with pytest.raises(IndexError):
        oracle.kv_append(kc, vc, kn, vn, [0, 6])


def test_kv_append_ring_without_wrap_is_the_linear_append():
    """Rows that stay inside the ring land where the linear append puts them."""
    r = np.random.default_rng(5)
    kc, vc = r.standard_normal((2, 8, 2, 4)), r.standard_normal((2, 8, 2, 4))
    kn, vn = r.standard_normal((2, 3, 2, 4)), r.standard_normal((2, 3, 2, 4))
    lin = oracle.kv_append(kc, vc, kn, vn, [0, 5])
    ring = oracle.kv_append_ring(kc, vc, kn, vn, [0, 5])
    assert np.array_equal(lin[0], ring[0]) and np.array_equal(lin[1], ring[1])


def test_kv_append_ring_keeps_the_last_positions():
    """Appending a history chunk by chunk into a ring of C rows leaves, in row r, the
    latest position j with j % C == r (found here by scanning the history backwards),
    and the value rows travel with their key rows."""
    r = np.random.default_rng(6)
    B, C, H, D, n_total, chunk = 2, 7, 2, 3, 40, 5
    kh = r.standard_normal((B, n_total, H, D))
    vh = r.standard_normal((B, n_total, H, D))
    kc = np.full((B, C, H, D), np.nan)
    vc = np.full((B, C, H, D), np.nan)
    for p0 in range(0, n_total, chunk):
        kc, vc = oracle.kv_append_ring(kc, vc, kh[:, p0:p0 + chunk], vh[:, p0:p0 + chunk],
                                       [p0, p0])
        n = p0 + chunk
        for row in range(C):
            latest = next((j for j in range(n - 1, -1, -1) if j % C == row), None)
            if latest is None:
                assert np.isnan(kc[:, row]).all() and np.isnan(vc[:, row]).all()
            else:
                assert np.array_equal(kc[:, row], kh[:, latest])
                assert np.array_equal(vc[:, row], vh[:, latest])
    # a chunk longer than the ring, or a negative position, is refused
    with pytest.raises(IndexError):
        oracle.kv_append_ring(kc, vc, kh[:, :C + 1], vh[:, :C + 1], [0, 0])
    with pytest.raises(IndexError):
        oracle.kv_append_ring(kc, vc, kh[:, :2], vh[:, :2], [0, -1])


# ------------------------------------------------------------------------------------
# planted mistakes: each edit below is a plausible slip in the oracle's C source; the
# pins must reject every one of them.

MUTATIONS = {
    "gqa_modulo_mapping": ("const int hk = h / G;", "const int hk = h % jb->n_kv_heads;"),
    "causal_excludes_self": ("if (causal && j > p) return 0;",
                             "if (causal && j >= p) return 0;"),
    "window_off_by_one": ("if (window > 0 && p - j >= window) return 0;",
                          "if (window > 0 && p - j > window) return 0;"),
    "top_left_alignment": ("const int p = i + (L - S);", "const int p = i;"),
    "unnormalised_output": ("for (int d = 0; d < D; ++d) orow[d] /= Z;", ""),
    "lse_without_log": ("*lrow = m + log(Z);", "*lrow = m + Z;"),
    "scale_dropped": ("scores[j] = jb->scale * dot;", "scores[j] = dot;"),
    "values_from_keys": ("const double *vrow = jb->v +", "const double *vrow = jb->k +"),
    "max_not_subtracted_in_lse": ("const double w = exp(scores[j] - m);",
                                  "const double w = exp(scores[j]);"),
    "softcap_before_scale": (
        "if (jb->softcap > 0.0) scores[j] = jb->softcap * tanh(scores[j] / jb->softcap);",
        "if (jb->softcap > 0.0) scores[j] = jb->scale * jb->softcap * tanh(dot / jb->softcap);"),
    "softcap_without_multiplier": (
        "if (jb->softcap > 0.0) scores[j] = jb->softcap * tanh(scores[j] / jb->softcap);",
        "if (jb->softcap > 0.0) scores[j] = tanh(scores[j] / jb->softcap);"),
    "wrong_batch_stride": ("(((int64_t)b * L + j) * jb->n_kv_heads + hk) * D;\n        double dot",
                           "(((int64_t)b * S + j) * jb->n_kv_heads + hk) * D;\n        double dot"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTATIONS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation anchor for %s not found exactly once" % name
    tmp = tempfile.mkdtemp(prefix="oracle_mut_")
    try:
        path = os.path.join(tmp, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        bad = oracle.Oracle(oracle.compile_library(path, os.path.join(tmp, "libmut.so")))
        failures = []
        for pin in ALL_PINS:
            try:
                pin(bad)
            except (AssertionError, ValueError, IndexError, FloatingPointError) as e:
                failures.append((pin.__name__, str(e)[:80]))
        assert failures, "planted mistake %s passed every pin" % name
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
