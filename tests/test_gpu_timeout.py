"""Failure detection on the GPU without a fault: a bounded pipeline wait that runs out.

Prefill: the test hook loads every tile but the first K tile, so the tensor-core issuer's
wait for that tile can never complete.  Decode: the hook never fills a CTA's first K/V
stage.  Every CTA must give up after the given budget, record LAT_ERR_TIMEOUT in the
status word, drain its copies (and free its tensor memory) and exit; the context stays
usable, which the follow-up call on the same buffers checks.
"""
import math
import time

import pytest
import torch

import workloads as W
from gpu_helpers import (compare, ensure_library, oracle_decode, oracle_prefill, run_prefill,
                         status_tensor)
from gqa_attention_lat_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


@pytest.mark.parametrize("D", [128, 512], ids=["single-CTA", "CTA-pair"])
def test_prefill_wait_times_out_and_context_survives(D):
    """head_dim 128 runs one CTA per item; head_dim 512 with two query heads per KV head
    runs on CTA pairs, where the even CTA waits for the tile and the odd CTA's waits for
    the S it never gets run out in the same way."""
    B, S, Hq, Hkv = 1, 256, 4, 2
    inp = W.prefill_inputs(B, S, S, Hq, Hkv, D, dtype="bf16", device="cuda")
    out = torch.zeros((B * S, Hq * D), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    budget_ns = 20_000_000  # 20 ms per CTA
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.lat_test_prefill_timeout(inp.q, inp.q.stride(0), inp.k, inp.k.stride(0), inp.v,
                                     inp.v.stride(0), out, out.stride(0), B, S, Hq, Hkv, D,
                                     budget_ns, st)
    torch.cuda.synchronize()  # the kernel ends by itself: no fault, no hang
    elapsed = time.perf_counter() - t0
    assert st.item() == binding.LAT_ERR_TIMEOUT
    assert elapsed < 2.0, elapsed  # the budget plus the drain, far below the default 4 s

    # the same buffers, the regular entry point: correct results on a healthy context
    scale = 1.0 / math.sqrt(D)
    got, lse = run_prefill(inp, causal=True, window=0, scale=scale)
    ref, ref_lse = oracle_prefill(inp, causal=True, window=0, scale=scale)
    compare(got, ref, "bf16", "after timeout", lse, ref_lse)


@pytest.mark.parametrize("shape", [(40, 8, 1, 128, 3000), (2, 8, 1, 512, 20000)],
                         ids=["in-kernel-merge", "deferred-merge"])
def test_decode_wait_times_out_and_context_survives(shape):
    """The decode's bounded waits: every CTA's first K/V stage is never filled, so its
    compute warps' wait (and its producer's wait for that stage to come back) must run
    out; the CTA records LAT_ERR_TIMEOUT, drains and exits.  With few units a second
    kernel merges the pieces; it still runs and ends.  Then the same buffers, a
    re-zeroed workspace and the regular entry point give correct results."""
    B, Hq, Hkv, D, cap = shape
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=None, device="cuda",
                         seed=W.BASE_SEED + D)
    nbytes = binding.lat_attn_decode_workspace_size(binding.LAT_BF16, B, Hq, Hkv, D, cap)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.zeros((B, Hq * D), dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.lat_test_decode_timeout(di.q, di.q.stride(0), di.k_cache, di.v_cache, Hkv * D, D,
                                    cap * Hkv * D, di.kv_lens, cap, out, out.stride(0), B, Hq,
                                    Hkv, D, ws, nbytes, 20_000_000, st)
    torch.cuda.synchronize()  # the kernels end by themselves: no fault, no hang
    elapsed = time.perf_counter() - t0
    assert st.item() == binding.LAT_ERR_TIMEOUT
    assert elapsed < 2.0, elapsed

    ws.zero_()
    st2 = status_tensor()
    out2 = torch.full_like(out, float("nan"))
    lse2 = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    binding.lat_attn_decode(binding.LAT_BF16, di.q, di.q.stride(0), di.k_cache, di.v_cache,
                            Hkv * D, D, cap * Hkv * D, di.kv_lens, cap, out2, out2.stride(0),
                            lse2, B, Hq, Hkv, D, 0, 0.125, ws, nbytes, st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    ref, ref_lse = oracle_decode(di, window=0, scale=0.125)
    compare(out2.view(B, Hq, D), ref, "bf16", "decode after timeout", lse2, ref_lse)
