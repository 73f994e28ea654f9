"""Seeded random shapes: the CUDA path against the oracle over a wide draw of sizes.

The hand-picked sweeps in the other files pin the named cases (tile boundaries, the
Gemma/Qwen shapes, the merge forms).  These cases are drawn from a fixed seed across the
whole accepted range instead: head_dim 64/80/128/256/512, GQA groups 1-16 (odd ones
too), ragged query and key counts on either side of the 128-row and 32/64-key tiles,
causal and bidirectional masks, sliding windows, chunks of new queries after earlier
keys, packed QKV buffers, the Gemma 2 score cap, and decode batches with empty, short
and long sequences mixed (both merge forms).  Every output element and lse is compared
with the fp64 oracle at the tolerances of the other parity tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import DT, DecodeRun, compare, ensure_library, status_tensor
from gqa_attention_lat_gb300 import binding

pytestmark = pytest.mark.gpu

SEED = 20260213
HEAD_DIMS = (64, 80, 128, 256, 512)
GROUPS = (1, 2, 3, 4, 5, 8, 16)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


def _prefill_cases(n):
    rng = np.random.RandomState(SEED)
    cases = []
    while len(cases) < n:
        D = int(rng.choice(HEAD_DIMS))
        Hkv = int(rng.choice((1, 2, 3)))
        G = int(rng.choice(GROUPS[:5]))
        B = int(rng.randint(1, 4))
        S = int(rng.randint(1, 330))
        packed = bool(rng.rand() < 0.25)
        L = S if packed or rng.rand() < 0.5 else S + int(rng.randint(1, 300))
        causal = bool(rng.rand() < 0.75)
        window = int(rng.randint(1, L + 1)) if rng.rand() < 0.3 else 0
        softcap = float(rng.choice((1.5, 3.0))) if rng.rand() < 0.2 else 0.0
        # keep each oracle pass to a fraction of a second
        if B * S * L * Hkv * G * D > 4e8:
            continue
        cases.append((B, S, L, Hkv * G, Hkv, D, causal, window, softcap, packed))
    return cases


def _decode_cases(n):
    rng = np.random.RandomState(SEED + 1)
    cases = []
    while len(cases) < n:
        D = int(rng.choice(HEAD_DIMS))
        Hkv = int(rng.choice((1, 2, 4, 8)))
        G = int(rng.choice(GROUPS))
        B = int(rng.choice((1, 2, 3, 7, 16, 40, 64)))
        cap = int(rng.choice((1, 31, 64, 200, 1000, 4097, 9000)))
        lens = [int(x) for x in rng.randint(0, cap + 1, size=B)]
        if rng.rand() < 0.5:
            lens[int(rng.randint(B))] = cap  # a full-length sequence among them
        window = int(rng.randint(1, cap + 1)) if rng.rand() < 0.3 else 0
        softcap = float(rng.choice((1.5, 3.0))) if rng.rand() < 0.2 else 0.0
        if sum(lens) * Hkv * G * D > 3e9 / 8:
            continue
        cases.append((B, Hkv * G, Hkv, D, cap, lens, window, softcap))
    return cases


PREFILL = _prefill_cases(48)
DECODE = _decode_cases(48)


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: "B%dS%dL%dH%d-%dD%d%s%s%s%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "", "w%d" % c[7] if c[7] else "",
    "-cap%g" % c[8] if c[8] else "", "-packed" if c[9] else ""))
def test_random_prefill_matches_oracle(case):
    B, S, L, Hq, Hkv, D, causal, window, softcap, packed = case
    inp = W.prefill_inputs(B, S, L, Hq, Hkv, D, dtype="bf16", device="cuda", packed=packed,
                           seed=W.BASE_SEED + 7 * S + L + D)
    scale = (2.0 if softcap else 1.0) / math.sqrt(D)
    out = torch.full((B * S, Hq * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B * S, Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = status_tensor()
    binding_args = (DT["bf16"], inp.q, inp.q.stride(0), inp.k, inp.k.stride(0), inp.v,
                    inp.v.stride(0), out, out.stride(0), lse, B, S, L, Hq, Hkv, D, causal,
                    window, scale)
    if softcap:
        binding.lat_attn_prefill_softcap(*binding_args, softcap, st)
    else:
        binding.lat_attn_prefill(*binding_args, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    ref, ref_lse = oracle.prefill(inp.heads("q"), inp.heads("k"), inp.heads("v"), causal=causal,
                                  window=window, scale=scale, softcap=softcap)
    compare(out.view(B, S, Hq, D), ref, "bf16", str(case), lse.view(B, S, Hq), ref_lse)


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "B%dH%d-%dD%dcap%d%s%s" % (
    c[0], c[1], c[2], c[3], c[4], "w%d" % c[6] if c[6] else "", "-cap%g" % c[7] if c[7] else ""))
def test_random_decode_matches_oracle(case):
    B, Hq, Hkv, D, cap, lens, window, softcap = case
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=lens, device="cuda",
                         seed=W.BASE_SEED + 3 * cap + D + B)
    scale = (2.0 if softcap else 1.0) / math.sqrt(D)
    run = DecodeRun("bf16", B, Hq, Hkv, D, cap)
    out = torch.full((B, Hq * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = status_tensor()
    binding.lat_attn_decode_softcap(DT["bf16"], di.q, di.q.stride(0), di.k_cache, di.v_cache,
                                    Hkv * D, D, cap * Hkv * D, di.kv_lens, cap, out,
                                    out.stride(0), lse, B, Hq, Hkv, D, window, scale, softcap,
                                    run.ws, run.nbytes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    ref, ref_lse = oracle.decode(di.q_heads(), di.cache_heads("k_cache"),
                                 di.cache_heads("v_cache"), di.kv_lens.cpu().tolist(),
                                 window=window, scale=scale, softcap=softcap)
    # sequences with no visible key: out = 0, lse = -inf (the oracle's convention)
    compare(out.view(B, Hq, D), ref, "bf16", str(case), lse, ref_lse)
