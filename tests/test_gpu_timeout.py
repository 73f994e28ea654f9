"""Failure detection on the GPU without a fault: a bounded pipeline wait that runs out.

The test hook loads every tile but the first K tile, so the tensor-core issuer's wait for
that tile can never complete.  Every CTA must give up after the given budget, record
LAT_ERR_TIMEOUT in the status word, drain its copies, free its tensor memory and exit;
the context stays usable, which the follow-up prefill on the same buffers checks.
"""
import math
import time

import pytest
import torch

import workloads as W
from gpu_helpers import compare, ensure_library, oracle_prefill, run_prefill, status_tensor
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
