"""Prefill parity: the CUDA library (through its C ABI) against the fp64 oracle."""
import math
import zlib

import pytest
import torch

import workloads as W
from gpu_helpers import compare, ensure_library, oracle_prefill, run_prefill, status_tensor
from gqa_attention_lat_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


# (B, S, L, Hq, Hkv, D, causal, window, packed, dtype)
SWEEP = [
    # head_dim sweep, GQA groups 1/2/4/5/8, ragged lengths that span several tiles
    (2, 300, 300, 4, 2, 64, True, 0, False, "bf16"),
    (1, 257, 257, 10, 2, 80, True, 0, False, "bf16"),     # Qwen3-4B-like head_dim 80
    (2, 200, 200, 8, 2, 128, True, 0, True, "bf16"),
    (1, 333, 333, 5, 1, 128, True, 0, False, "bf16"),     # G = 5
    (1, 190, 190, 8, 1, 256, True, 0, False, "bf16"),     # G = 8
    (1, 150, 150, 4, 2, 512, True, 0, False, "bf16"),
    # non-causal, tiny and odd lengths
    (1, 1, 1, 2, 1, 64, False, 0, False, "bf16"),
    (2, 2, 2, 4, 4, 128, False, 0, False, "bf16"),
    (1, 127, 127, 4, 2, 64, False, 0, False, "bf16"),
    (1, 129, 129, 4, 2, 256, False, 0, False, "bf16"),
    # sliding windows: 1 (self only), 17, 1024 (Gemma-4 sliding layers)
    (1, 300, 300, 4, 2, 128, True, 1, False, "bf16"),
    (2, 270, 270, 4, 1, 64, True, 17, False, "bf16"),
    (1, 1100, 1100, 2, 1, 256, True, 1024, False, "bf16"),
    (1, 200, 200, 2, 2, 128, False, 33, False, "bf16"),
    # chunked prefill: fewer queries than keys (bottom-right causal alignment)
    (2, 100, 700, 4, 2, 128, True, 0, False, "bf16"),
    (1, 64, 1000, 8, 2, 64, True, 300, False, "bf16"),
    (1, 130, 600, 4, 1, 512, True, 0, False, "bf16"),
    (1, 1000, 1000, 4, 2, 64, True, 0, True, "bf16"),
    # head_dim 64 with long key ranges (a query tile visits ~1K keys or more): 96-key tiles
    (1, 2500, 2500, 8, 2, 64, True, 0, False, "bf16"),
    (2, 130, 1100, 4, 4, 64, False, 0, False, "bf16"),
    (1, 3000, 3000, 4, 2, 64, True, 1100, True, "bf16"),
    (2, 300, 2048, 4, 1, 64, True, 0, False, "bf16"),
    # head_dim 512 on CTA pairs (even GQA group): two heads per pair, ragged last tiles,
    # a window, no mask, a chunk after cached keys, more items than the GPU has pairs
    (2, 300, 300, 8, 2, 512, True, 0, False, "bf16"),
    (1, 257, 257, 16, 2, 512, True, 0, True, "bf16"),
    (1, 700, 700, 4, 2, 512, True, 200, False, "bf16"),
    (1, 200, 200, 2, 1, 512, False, 0, False, "bf16"),
    (1, 100, 600, 4, 2, 512, True, 0, False, "bf16"),
    (4, 1024, 1024, 8, 2, 512, True, 0, False, "bf16"),
    # head_dim 256 with an odd GQA group: the single-CTA form (even groups run on pairs)
    (1, 300, 300, 3, 1, 256, True, 0, False, "bf16"),
    (2, 260, 400, 6, 2, 256, True, 100, False, "bf16"),
    # head_dim 512 with an odd GQA group: the single-CTA form
    (1, 150, 150, 3, 1, 512, True, 0, False, "bf16"),
    (1, 200, 200, 5, 5, 512, True, 64, False, "bf16"),
    # fp32 (exact CUDA-core path)
    (1, 64, 64, 4, 2, 64, True, 0, False, "f32"),
    (2, 100, 100, 6, 2, 80, True, 7, False, "f32"),
    (1, 50, 120, 4, 4, 256, True, 0, False, "f32"),
    (1, 40, 40, 2, 1, 512, False, 0, False, "f32"),
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "B%dS%dL%dH%d-%dD%d%s%s%s-%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n", "w%d" % c[7] if c[7] else "",
    "p" if c[8] else "", c[9]))
def test_prefill_sweep(case):
    B, S, L, Hq, Hkv, D, causal, window, packed, dtype = case
    inp = W.prefill_inputs(B, S, L, Hq, Hkv, D, dtype=dtype, device="cuda",
                           seed=W.BASE_SEED + zlib.crc32(repr(case).encode()) % 1000, packed=packed,
                           q_pad=0 if packed else 8, kv_pad=0 if packed else 16)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_prefill(inp, causal=causal, window=window, scale=scale, out_pad=8)
    ref, ref_lse = oracle_prefill(inp, causal=causal, window=window, scale=scale)
    compare(out, ref, dtype, str(case), lse, ref_lse)


def test_prefill_without_lse():
    inp = W.prefill_inputs(1, 200, 200, 4, 2, 128, dtype="bf16", device="cuda")
    out, _ = run_prefill(inp, causal=True, window=0, scale=0.1, with_lse=False)
    ref, _ = oracle_prefill(inp, causal=True, window=0, scale=0.1)
    compare(out, ref, "bf16", "no lse")


def test_prefill_is_deterministic():
    inp = W.prefill_inputs(2, 300, 300, 8, 2, 128, dtype="bf16", device="cuda")
    a, la = run_prefill(inp, causal=True, window=0, scale=0.09)
    b, lb = run_prefill(inp, causal=True, window=0, scale=0.09)
    assert torch.equal(a, b) and torch.equal(la, lb)


def _workload_inputs(wl, device="cuda"):
    return W.prefill_inputs(wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D, dtype=wl.dtype, device=device,
                            packed=wl.packed, k_mul=wl.k_mul)


def test_tiny_f32_prefill_full():
    wl = W.WORKLOADS["tiny_f32_prefill"]
    inp = _workload_inputs(wl)
    out, lse = run_prefill(inp, causal=wl.causal, window=wl.window, scale=wl.scale)
    ref, ref_lse = oracle_prefill(inp, causal=wl.causal, window=wl.window, scale=wl.scale)
    compare(out, ref, "f32", wl.name, lse, ref_lse)


def test_qwen3_prefill_full():
    """Packed [4096, 2048] QKV buffer read with row stride 2048, every output compared."""
    wl = W.WORKLOADS["qwen3_0.6b_prefill"]
    inp = _workload_inputs(wl)
    assert inp.q.stride(0) == 2048 and inp.k.stride(0) == 2048
    out, lse = run_prefill(inp, causal=wl.causal, window=wl.window, scale=wl.scale)
    ref, ref_lse = oracle_prefill(inp, causal=wl.causal, window=wl.window, scale=wl.scale)
    compare(out, ref, "bf16", wl.name, lse, ref_lse)


@pytest.mark.parametrize("name", ["gemma4_sliding_prefill", "gemma4_global_prefill"])
def test_gemma4_prefill_sampled_rows(name):
    """Full-size Gemma-4 layer shapes; rows sampled (rows are independent, so each
    sampled row is exact): sequence ends, window and tile boundaries +-1, random rows."""
    wl = W.WORKLOADS[name]
    inp = _workload_inputs(wl)
    out, lse = run_prefill(inp, causal=wl.causal, window=wl.window, scale=wl.scale)
    extra = [64, 128, 256, 1023, 1024, 2048, 4096]
    rows = W.sample_rows(wl.B * wl.S, wl.S, extra=extra, n_random=256)
    ref, ref_lse = oracle_prefill(inp, causal=wl.causal, window=wl.window, scale=wl.scale,
                                  rows=rows)
    idx = torch.tensor(rows, device="cuda")
    got = out.reshape(wl.B * wl.S, wl.Hq, wl.D)[idx]
    got_lse = lse.reshape(wl.B * wl.S, wl.Hq)[idx]
    compare(got, ref, "bf16", name, got_lse, ref_lse)


# Size extremes: a 32K-row causal prefill (rows sampled), and many short sequences (more
# items than the grid has CTAs several times over, every row compared).
@pytest.mark.parametrize("case", [
    (1, 32768, 4, 1, 128, 0),
    (1, 20000, 8, 2, 64, 0),      # head_dim 64 in its 96-key-tile form
    (1, 16384, 4, 2, 256, 4096),
    (1, 131072, 8, 1, 128, 0),    # 128K rows: tile coordinates and item counts at scale
], ids=lambda c: "S%dH%d-%dD%dw%d" % (c[1], c[2], c[3], c[4], c[5]))
def test_prefill_long_sequence_sampled_rows(case):
    B, S, Hq, Hkv, D, window = case
    inp = W.prefill_inputs(B, S, S, Hq, Hkv, D, dtype="bf16", device="cuda",
                           seed=W.BASE_SEED + S + D)
    scale = 1.0 / math.sqrt(D)
    out, lse = run_prefill(inp, causal=True, window=window, scale=scale)
    rows = W.sample_rows(B * S, S, extra=[127, 128, 4095, 4096, S // 2],
                         n_random=256 if S <= 32768 else 24)
    ref, ref_lse = oracle_prefill(inp, causal=True, window=window, scale=scale, rows=rows)
    idx = torch.tensor(rows, device="cuda")
    compare(out.reshape(B * S, Hq, D)[idx], ref, "bf16", str(case),
            lse.reshape(B * S, Hq)[idx], ref_lse)


def test_prefill_many_short_sequences():
    B, S, Hq, Hkv, D = 300, 37, 8, 2, 64
    inp = W.prefill_inputs(B, S, S, Hq, Hkv, D, dtype="bf16", device="cuda", seed=W.BASE_SEED + 3)
    out, lse = run_prefill(inp, causal=True, window=0, scale=0.125)
    ref, ref_lse = oracle_prefill(inp, causal=True, window=0, scale=0.125)
    compare(out, ref, "bf16", "300 x 37 rows", lse, ref_lse)


# Output placement: short ragged sequences (every query tile ends inside its sequence, and
# the next sequence's rows follow at once), an output that is a column window of a wider
# buffer starting 0 or 16 bytes past a 32-byte boundary, and rows after the last sequence.
# Rows and columns outside the window must keep their sentinel.  Covers the tensor-map
# output stores (head_dim 128/256) and the direct row stores in their 32- and 16-byte forms.
@pytest.mark.parametrize("D,Hq,Hkv,col0", [
    (64, 4, 2, 0), (64, 4, 2, 8), (80, 4, 2, 0), (80, 4, 2, 8), (128, 4, 2, 0), (128, 4, 1, 8),
    (256, 3, 1, 0), (256, 2, 2, 8), (512, 4, 2, 0), (512, 4, 2, 8), (512, 3, 1, 0),
], ids=lambda v: str(v))
def test_prefill_output_stays_in_its_window(D, Hq, Hkv, col0):
    B, S = 5, 37
    inp = W.prefill_inputs(B, S, S, Hq, Hkv, D, dtype="bf16", device="cuda",
                           seed=W.BASE_SEED + 11 * D + col0)
    rows, width, tail = B * S, Hq * D, 40
    # row strides of 16-element multiples (col0 0) and of 8 (col0 8)
    full = torch.full((rows + tail, col0 + width + (24 if col0 else 32)), float("nan"),
                      dtype=torch.bfloat16, device="cuda")
    out = full[:rows, col0:col0 + width]
    lse = torch.full((rows, Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = status_tensor()
    binding.lat_attn_prefill(binding.LAT_BF16, inp.q, inp.q.stride(0), inp.k, inp.k.stride(0),
                             inp.v, inp.v.stride(0), out, out.stride(0), lse, B, S, S, Hq, Hkv,
                             D, True, 0, 0.1, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    outside = torch.ones_like(full, dtype=torch.bool)
    outside[:rows, col0:col0 + width] = False
    assert torch.isnan(full[outside].float()).all(), "prefill wrote outside its output"
    ref, ref_lse = oracle_prefill(inp, causal=True, window=0, scale=0.1)
    compare(out.reshape(B, S, Hq, D), ref, "bf16", "D%d col0 %d" % (D, col0),
            lse.reshape(B, S, Hq), ref_lse)
