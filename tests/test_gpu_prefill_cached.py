"""Chunked prefill against an in-place KV cache: lat_attn_prefill_cached vs the oracle.

A chunk of S new query rows per sequence sits at positions L-S .. L-1 and attends to cache
rows 0 .. L-1 (bottom-right causal alignment); cache slots at or past L hold NaN and must
never reach the result.  The oracle sees the same values with K/V = the cache prefix.
"""
import math

import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import DT, compare, ensure_library, status_tensor
from gqa_attention_lat_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


def run_cached(q, kc, vc, cache_rs, head_stride, seq_stride, B, S, L, Hq, Hkv, D, causal,
               window, scale, dtype):
    out = torch.full((B * S, Hq * D), float("nan"), dtype=W.torch_dtype(dtype), device="cuda")
    lse = torch.full((B * S, Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = status_tensor()
    binding.lat_attn_prefill_cached(DT[dtype], q, q.stride(0), kc, vc, cache_rs, head_stride,
                                    seq_stride, out, out.stride(0), lse, B, S, L, Hq, Hkv, D,
                                    causal, window, scale, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    return out.view(B, S, Hq, D), lse.view(B, S, Hq)


# (B, Hq, Hkv, D, cap, L, S, causal, window, dtype, head_major)
CASES = [
    (2, 8, 2, 128, 600, 357, 100, True, 0, "bf16", False),     # chunk after 257 cached keys
    (3, 16, 8, 64, 300, 300, 300, True, 0, "bf16", True),      # S == L, head-major cache
    (1, 4, 1, 256, 2100, 2050, 200, True, 1024, "bf16", False),  # sliding window
    (1, 4, 4, 80, 260, 200, 1, True, 0, "bf16", True),         # one new row
    (1, 16, 2, 512, 1100, 1000, 256, True, 0, "bf16", False),  # head_dim 512 (split O)
    (2, 8, 4, 128, 512, 384, 130, False, 0, "bf16", False),    # no mask: the chunk sees all
    (2, 8, 2, 64, 2100, 2048, 300, True, 0, "bf16", False),   # 96-key tiles (long range)
    (2, 4, 2, 64, 100, 90, 30, True, 0, "f32", False),
    (1, 4, 2, 64, 96, 70, 70, True, 16, "f32", True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%d-%dD%dcap%dL%dS%d%s%s-%s%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "c" if c[7] else "", "w%d" % c[8] if c[8] else "",
    c[9], "-hm" if c[10] else ""))
def test_prefill_cached_matches_oracle(case):
    B, Hq, Hkv, D, cap, L, S, causal, window, dtype, head_major = case
    seed = W.BASE_SEED + cap + S
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=L, dtype=dtype, device="cuda", seed=seed)
    q = W.normal((B * S, Hq * D), dtype=dtype, device="cuda", seed=seed, role="chunk_q")
    kt, vt = di.cache_heads("k_cache"), di.cache_heads("v_cache")  # [B, cap, Hkv, D]
    if head_major:  # [B, Hkv, cap, D]
        kc = kt.permute(0, 2, 1, 3).contiguous()
        vc = vt.permute(0, 2, 1, 3).contiguous()
        strides = (D, cap * D, Hkv * cap * D)
    else:
        kc, vc = di.k_cache, di.v_cache
        strides = (Hkv * D, D, cap * Hkv * D)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_cached(q, kc, vc, *strides, B, S, L, Hq, Hkv, D, causal, window, scale, dtype)
    ref, ref_lse = oracle.prefill(q.view(B, S, Hq, D), kt[:, :L], vt[:, :L], causal=causal,
                                  window=window, scale=scale)
    compare(out, ref, dtype, str(case), lse, ref_lse)


def test_prefill_cached_equals_prefill_on_contiguous_kv():
    """With a cache that holds exactly L rows per sequence, the two entry points read the
    same bytes and must give bit-identical results."""
    B, Hq, Hkv, D, S, L = 2, 8, 2, 128, 200, 200
    inp = W.prefill_inputs(B, S, L, Hq, Hkv, D, dtype="bf16", device="cuda")
    scale = 0.09
    out_a = torch.empty((B * S, Hq * D), dtype=torch.bfloat16, device="cuda")
    lse_a = torch.empty((B * S, Hq), dtype=torch.float32, device="cuda")
    binding.lat_attn_prefill(binding.LAT_BF16, inp.q, inp.q.stride(0), inp.k, inp.k.stride(0),
                             inp.v, inp.v.stride(0), out_a, out_a.stride(0), lse_a, B, S, L, Hq,
                             Hkv, D, True, 0, scale)
    out_b, lse_b = run_cached(inp.q, inp.k, inp.v, inp.k.stride(0), D, L * inp.k.stride(0), B, S,
                              L, Hq, Hkv, D, True, 0, scale, "bf16")
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(B, S, Hq, D), out_b)
    assert torch.equal(lse_a.view(B, S, Hq), lse_b)


def test_chunked_prefill_workload_full_sampled_rows():
    """The measured chunked prefill at full size (B8, 512 new rows after 1536 cached keys,
    Hq16/8 D64, a 4096-slot token-major cache whose slots past L hold NaN; the bench's own
    inputs), in its 96-key-tile form: sampled rows against the oracle."""
    wl = W.WORKLOADS["qwen3_chunked_prefill"]
    di = W.decode_inputs(wl.B, wl.Hq, wl.Hkv, wl.D, wl.cap, kv_lens=wl.L, dtype=wl.dtype,
                         device="cuda", nan_fill=True)
    q = W.normal((wl.B * wl.S, wl.Hq * wl.D), dtype=wl.dtype, device="cuda", seed=W.BASE_SEED,
                 role="chunk_q")
    out, lse = run_cached(q, di.k_cache, di.v_cache, wl.Hkv * wl.D, wl.D,
                          wl.cap * wl.Hkv * wl.D, wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D,
                          wl.causal, wl.window, wl.scale, wl.dtype)
    rows = W.sample_rows(wl.B * wl.S, wl.S, extra=[95, 96, 127, 128, 255, 256], n_random=256)
    kt, vt = di.cache_heads("k_cache"), di.cache_heads("v_cache")
    ref, ref_lse = oracle.prefill(q.view(wl.B, wl.S, wl.Hq, wl.D), kt[:, :wl.L], vt[:, :wl.L],
                                  causal=wl.causal, window=wl.window, scale=wl.scale, rows=rows)
    idx = torch.tensor(rows, device="cuda")
    compare(out.reshape(wl.B * wl.S, wl.Hq, wl.D)[idx], ref, wl.dtype, wl.name,
            lse.reshape(wl.B * wl.S, wl.Hq)[idx], ref_lse)
