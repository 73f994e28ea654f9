"""Decode and KV-append parity: the CUDA library (through its C ABI) against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (DT, DecodeRun, assert_bits_equal, compare, ensure_library,
                         oracle_decode, oracle_prefill, run_decode, run_prefill, status_tensor)
from gqa_attention_lat_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


# (B, Hq, Hkv, D, cap, kv_lens, window, dtype)
SWEEP = [
    (4, 8, 2, 64, 300, [1, 63, 64, 300], 0, "bf16"),
    (3, 10, 2, 80, 257, [257, 100, 17], 0, "bf16"),
    (5, 16, 4, 128, 1000, [1000, 999, 513, 129, 2], 0, "bf16"),
    (2, 5, 1, 128, 700, [700, 31], 0, "bf16"),            # G = 5
    (2, 8, 1, 256, 900, [900, 450], 0, "bf16"),           # G = 8
    (2, 16, 1, 128, 300, [300, 77], 0, "bf16"),           # G = 16: two head blocks
    (3, 4, 2, 512, 2000, [2000, 1500, 1], 0, "bf16"),
    (2, 8, 8, 64, 64, [64, 5], 0, "bf16"),                # G = 1
    # one long sequence among 39 one-token ones (enough units for the in-kernel merge),
    # cut into many pieces: about 20 (merged from a shared-memory copy of the partials)
    # and about 60 (too many to stage: merged straight from L2)
    (40, 8, 1, 128, 5000, [5000] + [1] * 39, 0, "bf16"),
    (40, 8, 1, 512, 32768, [32768] + [1] * 39, 0, "bf16"),
    # few units, long keys: the stream is cut across every CTA and a second kernel merges
    # the pieces (an empty sequence among them, head_dim 80, a window, G = 16)
    (1, 8, 1, 128, 5000, [5000], 0, "bf16"),
    (1, 8, 1, 512, 32768, [32768], 0, "bf16"),
    (3, 8, 1, 80, 9000, [9000, 0, 4500], 0, "bf16"),
    (2, 8, 1, 64, 40000, [40000, 3], 0, "bf16"),
    (1, 8, 1, 256, 20000, [20000], 700, "bf16"),
    (1, 16, 1, 128, 6000, [6000], 0, "bf16"),
    # sliding window: the visible keys start at a non-zero cache offset
    (4, 8, 2, 128, 3000, [3000, 1024, 1025, 40], 1024, "bf16"),
    (2, 8, 4, 256, 500, [500, 18], 17, "bf16"),
    (2, 4, 2, 64, 100, [100, 1], 1, "bf16"),
    # fp32
    (2, 4, 2, 64, 64, [64, 33], 0, "f32"),
    (2, 8, 2, 80, 200, [200, 7], 50, "f32"),
    (2, 4, 1, 512, 300, [300, 129], 0, "f32"),
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "B%dH%d-%dD%dcap%d%s-%s" % (
    c[0], c[1], c[2], c[3], c[4], "w%d" % c[6] if c[6] else "", c[7]))
def test_decode_sweep(case):
    B, Hq, Hkv, D, cap, lens, window, dtype = case
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=lens, dtype=dtype, device="cuda",
                         seed=W.BASE_SEED + cap)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_decode(di, window=window, scale=scale)
    ref, ref_lse = oracle_decode(di, window=window, scale=scale)
    compare(out, ref, dtype, str(case), lse, ref_lse)


def test_decode_head_major_cache():
    """The hf2q target page's per-layer cache layout [B, Hkv, cap, D]."""
    B, Hq, Hkv, D, cap = 3, 8, 2, 128, 600
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=[600, 300, 5], device="cuda")
    kc = di.cache_heads("k_cache").permute(0, 2, 1, 3).contiguous()  # [B, Hkv, cap, D]
    vc = di.cache_heads("v_cache").permute(0, 2, 1, 3).contiguous()
    run = DecodeRun("bf16", B, Hq, Hkv, D, cap)
    out, lse, st = run(di.q, kc, vc, D, cap * D, Hkv * cap * D, di.kv_lens, cap, B, Hq, Hkv, D,
                       0, 0.1)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref, ref_lse = oracle_decode(di, window=0, scale=0.1)
    compare(out.view(B, Hq, D), ref, "bf16", "head-major", lse, ref_lse)


@pytest.mark.parametrize("B,Hkv", [(6, 2), (32, 8)], ids=["few-units", "many-units"])
def test_decode_workspace_reuse_gives_identical_results(B, Hkv):
    """Calls that reuse a workspace give identical results.  With few units (12 here) the
    stream is cut across every CTA and merged by a second kernel; with many (256) the
    in-kernel merge counters must be back at zero after every call."""
    di = W.decode_inputs(B, 16, Hkv, 128, 2048, kv_lens=None, device="cuda")
    run = DecodeRun("bf16", B, 16, Hkv, 128, 2048)
    a, la = run_decode(di, window=0, scale=0.08, runner=run)
    b, lb = run_decode(di, window=0, scale=0.08, runner=run)
    assert torch.equal(a, b) and torch.equal(la, lb)
    if Hkv == 8:
        units = B * Hkv  # one head block per KV head (16 / 8 = 2 query heads each)
        cnt_off = run.nbytes - (units * 4 + 255) // 256 * 256
        assert run.ws[cnt_off:].eq(0).all()


def test_decode_mixed_staged_and_direct_merges_repeat_identically():
    """CTAs that merge, after their stream, one unit with too many pieces to stage (read
    straight from L2) and one staged from a shared-memory copy.  Ten 40000-key sequences
    cut into ~28 pieces each sit between 3000-key ones cut into ~3, so about 18 CTAs hold
    pieces of both kinds; whichever merge a CTA queues first, each staged copy must be
    waited for on its own barrier phase.  Every launch equals the oracle and the others."""
    lens = [40000, 3000, 1, 1] * 10
    B, Hq, Hkv, D, cap = 40, 8, 1, 128, 40000
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=lens, device="cuda", seed=W.BASE_SEED + 77)
    run = DecodeRun("bf16", B, Hq, Hkv, D, cap)
    first, first_lse = run_decode(di, window=0, scale=0.09, runner=run)
    for _ in range(9):
        out, lse = run_decode(di, window=0, scale=0.09, runner=run)
        assert torch.equal(out, first) and torch.equal(lse, first_lse)
    ref, ref_lse = oracle_decode(di, window=0, scale=0.09)
    compare(first, ref, "bf16", "mixed merges", first_lse, ref_lse)


def test_decode_empty_sequence():
    """kv_len 0: nothing visible, out = 0 and lse = -inf."""
    di = W.decode_inputs(2, 4, 2, 64, 64, kv_lens=[0, 10], device="cuda")
    out, lse = run_decode(di, window=0, scale=0.125)
    assert torch.all(out[0].float() == 0) and torch.all(torch.isneginf(lse[0]))
    ref, ref_lse = oracle_decode(di, window=0, scale=0.125)
    compare(out[1:], ref[1:], "bf16", "empty", lse[1:], ref_lse[1:])


def test_decode_kv_len_over_bound_sets_status():
    di = W.decode_inputs(2, 4, 2, 64, 64, kv_lens=[64, 10], device="cuda")
    run = DecodeRun("bf16", 2, 4, 2, 64, 32)
    out, lse, st = run(di.q, di.k_cache, di.v_cache, 128, 64, 64 * 128, di.kv_lens, 32, 2, 4, 2,
                       64, 0, 0.125)
    torch.cuda.synchronize()
    assert st.item() == binding.LAT_ERR_BOUNDS


def test_decode_workspace_too_small():
    di = W.decode_inputs(2, 4, 2, 64, 64, kv_lens=[64, 10], device="cuda")
    run = DecodeRun("bf16", 2, 4, 2, 64, 64)
    with pytest.raises(binding.LatError) as e:
        binding.lat_attn_decode(binding.LAT_BF16, di.q, di.q.stride(0), di.k_cache, di.v_cache,
                                128, 64, 64 * 128, di.kv_lens, 64,
                                torch.empty_like(di.q), di.q.stride(0), None, 2, 4, 2, 64, 0,
                                0.125, run.ws, run.nbytes - 1)
    assert e.value.status == binding.LAT_ERR_WORKSPACE


@pytest.mark.parametrize("name", ["decode_b32_h32_kv8_d128", "gemma4_global_decode",
                                  "decode_b1_kv2_d128_128k"])
def test_decode_workloads_full(name):
    wl = W.WORKLOADS[name]
    di = W.decode_inputs(wl.B, wl.Hq, wl.Hkv, wl.D, wl.L, kv_lens=wl.kv_lens, dtype=wl.dtype,
                         device="cuda")
    out, lse = run_decode(di, window=wl.window, scale=wl.scale)
    ref, ref_lse = oracle_decode(di, window=wl.window, scale=wl.scale)
    compare(out, ref, wl.dtype, name, lse, ref_lse)


@pytest.mark.parametrize("dtype,D,window", [("bf16", 128, 0), ("bf16", 256, 100),
                                            ("f32", 64, 0)])
def test_decode_equals_last_prefill_row_on_gpu(dtype, D, window):
    B, L, Hq, Hkv = 2, 333, 8, 2
    inp = W.prefill_inputs(B, L, L, Hq, Hkv, D, dtype=dtype, device="cuda")
    pout, plse = run_prefill(inp, causal=True, window=window, scale=0.1)
    cache_k = inp.k.reshape(B, L, Hkv * D).contiguous()
    cache_v = inp.v.reshape(B, L, Hkv * D).contiguous()
    q_last = inp.q.reshape(B, L, Hq * D)[:, -1].contiguous()
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    run = DecodeRun(dtype, B, Hq, Hkv, D, L)
    dout, dlse, st = run(q_last, cache_k, cache_v, Hkv * D, D, L * Hkv * D, lens, L, B, Hq, Hkv,
                         D, window, 0.1)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref, ref_lse = oracle_prefill(inp, causal=True, window=window, scale=0.1)
    compare(dout.view(B, Hq, D), ref[:, -1], dtype, "decode", dlse, ref_lse[:, -1])
    compare(pout[:, -1], ref[:, -1], dtype, "prefill last row", plse[:, -1], ref_lse[:, -1])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_append_then_decode(dtype):
    """lat_kv_append rows into a NaN-filled cache, bit-exact against the oracle's copy,
    then decode over the grown cache."""
    B, Hq, Hkv, D, cap = 3, 8, 2, 128, 256
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=[100, 7, 253], dtype=dtype, device="cuda")
    n_new = 5
    packed = W.normal((B * n_new, (Hq + 2 * Hkv) * D), dtype=dtype, device="cuda",
                      seed=W.BASE_SEED, role="new")
    k_new = packed[:, Hq * D:(Hq + Hkv) * D]
    v_new = packed[:, (Hq + Hkv) * D:]
    pos = torch.tensor([100, 7, 253], dtype=torch.int32, device="cuda")
    before_k = di.k_cache.clone()
    before_v = di.v_cache.clone()
    st = status_tensor()
    # the third sequence does not fit (253 + 5 > 256): skipped whole, status BOUNDS
    binding.lat_kv_append(DT[dtype], di.k_cache, di.v_cache, Hkv * D, D, cap * Hkv * D, cap,
                          k_new, v_new, packed.stride(0), pos, n_new, B, Hkv, D, st)
    torch.cuda.synchronize()
    assert st.item() == binding.LAT_ERR_BOUNDS

    def heads(t, rows):
        return t.reshape(t.shape[0], rows, Hkv, D)[:2].cpu().float().numpy()
    ok_k, ok_v = oracle.kv_append(heads(before_k, cap), heads(before_v, cap),
                                  heads(k_new.reshape(B, n_new, Hkv * D), n_new),
                                  heads(v_new.reshape(B, n_new, Hkv * D), n_new), [100, 7])
    # both caches, bit for bit (the copy is exact in either dtype), NaN pattern included
    assert_bits_equal(di.k_cache[:2].view(2, cap, Hkv, D), ok_k, "K cache")
    assert_bits_equal(di.v_cache[:2].view(2, cap, Hkv, D), ok_v, "V cache")
    # the sequence that did not fit is untouched in both caches
    assert_bits_equal(di.k_cache[2], before_k[2].cpu().float().numpy(), "K cache, skipped")
    assert_bits_equal(di.v_cache[2], before_v[2].cpu().float().numpy(), "V cache, skipped")
    # decode the two grown sequences at their new lengths
    di.kv_lens = torch.tensor([105, 12, 253], dtype=torch.int32, device="cuda")
    out, lse = run_decode(di, window=0, scale=0.1)
    ref, ref_lse = oracle_decode(di, window=0, scale=0.1)
    compare(out, ref, dtype, "append+decode", lse, ref_lse)


def test_tiny_f32_prefill_append_decode():
    """The tiny fp32 workload: causal prefill of 64 tokens, then row 63 appended into a
    cache of capacity 64 holding rows 0..62, then one decode step at kv_len 64."""
    wl = W.WORKLOADS["tiny_f32_prefill"]
    inp = W.prefill_inputs(1, 64, 64, 4, 2, 64, dtype="f32", device="cuda")
    pout, plse = run_prefill(inp, causal=True, window=0, scale=wl.scale)
    cap = 64
    kc = torch.full((1, cap, 128), float("nan"), device="cuda")
    vc = torch.full((1, cap, 128), float("nan"), device="cuda")
    kc[0, :63] = inp.k[:63]
    vc[0, :63] = inp.v[:63]
    pos = torch.tensor([63], dtype=torch.int32, device="cuda")
    st = status_tensor()
    binding.lat_kv_append(binding.LAT_F32, kc, vc, 128, 64, cap * 128, cap, inp.k[63:],
                          inp.v[63:], inp.k.stride(0), pos, 1, 1, 2, 64, st)
    lens = torch.tensor([64], dtype=torch.int32, device="cuda")
    run = DecodeRun("f32", 1, 4, 2, 64, 64)
    dout, dlse, st2 = run(inp.q[63:].contiguous(), kc, vc, 128, 64, cap * 128, lens, 64, 1, 4, 2,
                          64, 0, wl.scale)
    torch.cuda.synchronize()
    assert st.item() == 0 and st2.item() == 0
    ref, ref_lse = oracle_prefill(inp, causal=True, window=0, scale=wl.scale)
    compare(pout, ref, "f32", "tiny prefill", plse, ref_lse)
    compare(dout.view(1, 4, 64), ref[:, -1], "f32", "tiny decode", dlse, ref_lse[:, -1])


def test_decode_large_batch_with_empty_sequences():
    """600 sequences (more units than CTAs), lengths drawn in [0, 300] with zeros forced in:
    empty sequences give out = 0 and lse = -inf, the rest match the oracle."""
    B, Hq, Hkv, D, cap = 600, 8, 2, 128, 300
    g = torch.Generator().manual_seed(W.BASE_SEED + 600)
    lens = torch.randint(0, cap + 1, (B,), generator=g)
    lens[::97] = 0
    lens[1::89] = cap
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=lens.tolist(), dtype="bf16", device="cuda",
                         seed=W.BASE_SEED + 601)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_decode(di, window=0, scale=scale)
    ref, ref_lse = oracle_decode(di, window=0, scale=scale)
    compare(out, ref, "bf16", "B600 with empty sequences", lse, ref_lse)
    empty = (lens == 0).nonzero().flatten().tolist()
    assert empty and torch.all(out[empty].float() == 0)


def test_decode_million_keys():
    """Key streams past 2^20: two sequences, 1048576 and 700001 cached keys (slots past
    each length NaN), every output against the oracle."""
    di = W.decode_inputs(2, 8, 1, 128, 1 << 20, kv_lens=[1 << 20, 700001], dtype="bf16",
                         device="cuda", seed=W.BASE_SEED + 21)
    out, lse = run_decode(di, window=0, scale=1.0 / math.sqrt(128))
    ref, ref_lse = oracle_decode(di, window=0, scale=1.0 / math.sqrt(128))
    compare(out, ref, "bf16", "1M keys", lse, ref_lse)
