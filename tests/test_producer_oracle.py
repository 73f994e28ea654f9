"""The producer oracle against its pins, and planted mistakes that the pins must catch."""
import importlib.util
import os
import sys
import tempfile

import pytest

from producer_pins import ALL_PINS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "oracle", "producer.py")


def _load(path, name):
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_producer_oracle_pins(pin):
    pin(_load(SOURCE, "producer_under_test"))


MUTATIONS = {
    "interleaved_pairs": ("a, b = x[..., :half], x[..., half:]",
                          "a, b = x[..., 0::2], x[..., 1::2]"),
    "frequency_exponent": ("inv_freq = base ** (-2.0 * i / D)", "inv_freq = base ** (-1.0 * i / D)"),
    "rotation_sign": ("[a * c - b * s, a * s + b * c]", "[a * c + b * s, -a * s + b * c]"),
    "sum_not_mean": ("np.mean(x * x, axis=-1, keepdims=True) + eps",
                     "np.sum(x * x, axis=-1, keepdims=True) + eps"),
    "eps_outside_root": ("y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)",
                         "y = x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps)"),
    "k_uses_q_weight": ("k = rope_neox(rms_norm(k, k_w, eps), positions, base)",
                        "k = rope_neox(rms_norm(k, q_w, eps), positions, base)"),
    "positions_not_offset": (
        "positions = _f64(pos)[:, None] + np.arange(T, dtype=np.float64)[None, :]",
        "positions = np.zeros((B, 1)) + np.arange(T, dtype=np.float64)[None, :]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_producer_pins_reject_planted_mistake(name):
    old, new = MUTATIONS[name]
    with open(SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation anchor for %s not found exactly once" % name
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mut_producer.py")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        bad = _load(path, "mut_producer_" + name)
        failures = []
        for pin in ALL_PINS:
            try:
                pin(bad)
            except (AssertionError, ValueError, IndexError) as e:
                failures.append((pin.__name__, str(e)[:60]))
        assert failures, "planted mistake %s passed every pin" % name
