"""Seeded random shapes through prefill and decode, each against the oracle.

The hand-picked sweeps cover the named configurations and their edges; this one draws
batch, lengths, head counts (GQA group 1..8), head_dim, mask, window, dtype and layout at
random from a fixed seed, so every run checks the same 48 cases and a failure is
reproducible from its id."""
import math
import random

import pytest
import torch

import workloads as W
from gpu_helpers import compare, ensure_library, oracle_decode, oracle_prefill, run_decode, \
    run_prefill

pytestmark = pytest.mark.gpu

HEAD_DIMS = [64, 80, 128, 256, 512]


def _prefill_cases(n=28, seed=20260):
    rng = random.Random(seed)
    cases = []
    for _ in range(n):
        D = rng.choice(HEAD_DIMS)
        G = rng.choice([1, 2, 3, 4, 5, 8])
        Hkv = rng.choice([1, 2]) if D >= 256 else rng.choice([1, 2, 4])
        B = rng.randint(1, 3)
        S = rng.randint(1, 400 if D < 256 else 260)
        L = S + (rng.choice([0, 0, rng.randint(1, 700)]))
        causal = rng.random() < 0.75
        window = rng.choice([0, 0, rng.randint(1, 600)])
        dtype = "f32" if rng.random() < 0.2 else "bf16"
        packed = dtype == "bf16" and S == L and rng.random() < 0.3
        while B * Hkv * G * S * L * D > 4e8:  # keep each oracle run to a second or two
            S, L = max(1, S // 2), max(1, L // 2)
            L = max(L, S)
        cases.append((B, S, L, Hkv * G, Hkv, D, causal, window, packed, dtype))
    return cases


def _decode_cases(n=20, seed=20261):
    rng = random.Random(seed)
    cases = []
    for _ in range(n):
        D = rng.choice(HEAD_DIMS)
        G = rng.choice([1, 2, 4, 5, 8, 16])
        Hkv = rng.choice([1, 2, 4])
        B = rng.randint(1, 40)
        cap = rng.randint(1, 3000)
        lens = [rng.choice([0, rng.randint(1, cap), cap]) for _ in range(B)]
        window = rng.choice([0, 0, rng.randint(1, cap)])
        dtype = "f32" if rng.random() < 0.2 else "bf16"
        while B * Hkv * G * cap * D > 4e8:
            B = max(1, B // 2)
            lens = lens[:B]
        cases.append((B, Hkv * G, Hkv, D, cap, lens, window, dtype))
    return cases


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


@pytest.mark.parametrize("case", _prefill_cases(), ids=lambda c: "B%dS%dL%dH%d-%dD%d%s%s%s-%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n", "w%d" % c[7] if c[7] else "",
    "p" if c[8] else "", c[9]))
def test_random_prefill(case):
    B, S, L, Hq, Hkv, D, causal, window, packed, dtype = case
    inp = W.prefill_inputs(B, S, L, Hq, Hkv, D, dtype=dtype, device="cuda",
                           seed=W.BASE_SEED + S * 7 + L, packed=packed,
                           q_pad=0 if packed else 8, kv_pad=0 if packed else 8)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_prefill(inp, causal=causal, window=window, scale=scale, out_pad=8)
    ref, ref_lse = oracle_prefill(inp, causal=causal, window=window, scale=scale)
    compare(out, ref, dtype, str(case), lse, ref_lse)


@pytest.mark.parametrize("case", _decode_cases(), ids=lambda c: "B%dH%d-%dD%dcap%d%s-%s" % (
    c[0], c[1], c[2], c[3], c[4], "w%d" % c[6] if c[6] else "", c[7]))
def test_random_decode(case):
    B, Hq, Hkv, D, cap, lens, window, dtype = case
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=lens, dtype=dtype, device="cuda",
                         seed=W.BASE_SEED + cap * 3 + B)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_decode(di, window=window, scale=scale)
    ref, ref_lse = oracle_decode(di, window=window, scale=scale)
    compare(out, ref, dtype, str(case), lse, ref_lse)
