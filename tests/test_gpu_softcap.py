"""Score softcap (Gemma 2): lat_attn_prefill_softcap / lat_attn_decode_softcap vs the oracle.

Scores are scaled, then capped as softcap * tanh(s / softcap), then go through the
softmax.  Caps here are a few units, well inside the score range, so the cap changes the
result noticeably (checked against the uncapped oracle).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import DT, DecodeRun, compare, ensure_library, oracle_prefill, status_tensor
from gqa_attention_lat_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


def run_prefill_softcap(inp, causal, window, scale, softcap):
    tdt = inp.q.dtype
    out = torch.full((inp.B * inp.S, inp.Hq * inp.D), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((inp.B * inp.S, inp.Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = status_tensor()
    binding.lat_attn_prefill_softcap(DT[inp.dtype], inp.q, inp.q.stride(0), inp.k,
                                     inp.k.stride(0), inp.v, inp.v.stride(0), out, out.stride(0),
                                     lse, inp.B, inp.S, inp.L, inp.Hq, inp.Hkv, inp.D, causal,
                                     window, scale, softcap, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    return out.view(inp.B, inp.S, inp.Hq, inp.D), lse.view(inp.B, inp.S, inp.Hq)


# (B, S, L, Hq, Hkv, D, causal, window, softcap, dtype)
PREFILL = [
    (1, 300, 300, 8, 4, 256, True, 0, 2.0, "bf16"),
    (2, 200, 333, 8, 2, 128, True, 64, 1.5, "bf16"),
    (2, 256, 256, 16, 8, 64, True, 0, 3.0, "bf16"),
    (1, 130, 130, 4, 2, 512, True, 0, 2.5, "bf16"),
    (1, 100, 100, 4, 4, 80, False, 0, 1.0, "bf16"),
    (2, 40, 50, 4, 2, 64, True, 0, 2.0, "f32"),
]


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: "B%dS%dL%dH%d-%dD%d%s%s-cap%g-%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "", "w%d" % c[7] if c[7] else "",
    c[8], c[9]))
def test_prefill_softcap_matches_oracle(case):
    B, S, L, Hq, Hkv, D, causal, window, cap, dtype = case
    inp = W.prefill_inputs(B, S, L, Hq, Hkv, D, dtype=dtype, device="cuda",
                           seed=W.BASE_SEED + 17 * D + S)
    scale = 2.0 / math.sqrt(D)  # scores of a few units: the cap bites
    out, lse = run_prefill_softcap(inp, causal, window, scale, cap)
    ref, ref_lse = oracle.prefill(inp.heads("q"), inp.heads("k"), inp.heads("v"), causal=causal,
                                  window=window, scale=scale, softcap=cap)
    compare(out, ref, dtype, str(case), lse, ref_lse)
    plain, _ = oracle_prefill(inp, causal=causal, window=window, scale=scale)
    assert np.abs(np.asarray(plain) - np.asarray(ref)).max() > 0.05, "cap did not change the result"


def test_prefill_softcap_zero_is_plain_prefill():
    inp = W.prefill_inputs(2, 150, 150, 8, 2, 128, dtype="bf16", device="cuda")
    a, la = run_prefill_softcap(inp, True, 0, 0.09, 0.0)
    out = torch.empty_like(a.view(300, -1))
    lse = torch.empty_like(la.view(300, -1))
    binding.lat_attn_prefill(binding.LAT_BF16, inp.q, inp.q.stride(0), inp.k, inp.k.stride(0),
                             inp.v, inp.v.stride(0), out, out.stride(0), lse, 2, 150, 150, 8, 2,
                             128, True, 0, 0.09)
    torch.cuda.synchronize()
    assert torch.equal(a, out.view_as(a)) and torch.equal(la, lse.view_as(la))


# (B, Hq, Hkv, D, cap, kv_lens, window, softcap, dtype)
DECODE = [
    (4, 8, 2, 128, 1000, [1000, 517, 64, 3], 0, 1.5, "bf16"),
    (3, 16, 2, 512, 700, [700, 350, 1], 0, 2.0, "bf16"),
    (2, 8, 8, 64, 300, [300, 129], 100, 3.0, "bf16"),
    (2, 4, 2, 64, 80, [80, 33], 0, 2.0, "f32"),
]


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "B%dH%d-%dD%dcap%d%s-sc%g-%s" % (
    c[0], c[1], c[2], c[3], c[4], "w%d" % c[6] if c[6] else "", c[7], c[8]))
def test_decode_softcap_matches_oracle(case):
    B, Hq, Hkv, D, cap, lens, window, softcap, dtype = case
    di = W.decode_inputs(B, Hq, Hkv, D, cap, kv_lens=lens, dtype=dtype, device="cuda",
                         seed=W.BASE_SEED + cap + 1)
    scale = 2.0 / math.sqrt(D)
    run = DecodeRun(dtype, B, Hq, Hkv, D, cap)
    out = torch.full((B, Hq * D), float("nan"), dtype=di.q.dtype, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = status_tensor()
    binding.lat_attn_decode_softcap(DT[dtype], di.q, di.q.stride(0), di.k_cache, di.v_cache,
                                    Hkv * D, D, cap * Hkv * D, di.kv_lens, cap, out,
                                    out.stride(0), lse, B, Hq, Hkv, D, window, scale, softcap,
                                    run.ws, run.nbytes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    ref, ref_lse = oracle.decode(di.q_heads(), di.cache_heads("k_cache"),
                                 di.cache_heads("v_cache"), di.kv_lens.cpu().tolist(),
                                 window=window, scale=scale, softcap=softcap)
    compare(out.view(B, Hq, D), ref, dtype, str(case), lse, ref_lse)


# The bf16 kernels form the capped score as cap * log2(e) * tanh(y) through
# tanh y = 1 - 2 / (1 + e^{2y}) with the hardware exp2; its error is absolute, a few 1e-7
# of tanh.  Checked against the exact value (fp64 tanh of the same fp32 factors) and
# against CUDA's own tanhf (torch.tanh on the device), over raw dot products from 1e-30 to
# 1e30, both signs, zero and the infinities (which must give exactly +-cap * log2(e)).
@pytest.mark.parametrize("scale,softcap", [(0.0625, 50.0), (0.0884, 30.0), (1.0, 2.0),
                                           (0.5, 1e-3)])
def test_capped_score_matches_tanh(scale, softcap):
    g = torch.Generator().manual_seed(W.BASE_SEED + 77)
    parts = [torch.randn(50000, generator=g, dtype=torch.float64) * s
             for s in (1e-3, 0.1, 1.0, 30.0, 300.0, 3000.0)]
    parts.append(torch.tensor([0.0, 1e-30, -1e-30, 1e-7, -1e-7, 1e30, -1e30]))
    raw = torch.cat(parts).float()
    special = torch.tensor([math.inf, -math.inf])
    raw_all = torch.cat([raw, special]).cuda()
    out = torch.full_like(raw_all, math.nan)
    binding.lat_test_capped_scores(raw_all, raw_all.numel(), scale, softcap, out)
    torch.cuda.synchronize()
    raw_over_cap = np.float32(np.float32(scale) / np.float32(softcap))
    cap_log2 = np.float32(np.float32(softcap) * np.float32(1.4426950408889634))
    y64 = raw.double() * float(raw_over_cap)
    exact = float(cap_log2) * torch.tanh(y64)
    got = out[:-2].cpu().double()
    bound = 1e-6 * float(cap_log2)
    err = (got - exact).abs().max().item()
    assert err <= bound, "capped score off by %.3g (bound %.3g)" % (err, bound)
    cuda_tanh = float(cap_log2) * torch.tanh(raw.cuda() * raw_over_cap.item()).cpu().double()
    err_cuda = (got - cuda_tanh).abs().max().item()
    assert err_cuda <= bound, "capped score vs tanhf off by %.3g" % err_cuda
    assert out[-2].item() == pytest.approx(float(cap_log2), abs=0.0)
    assert out[-1].item() == pytest.approx(-float(cap_log2), abs=0.0)
    assert torch.isfinite(out).all()


def test_capped_score_rejects_bad_arguments():
    x = torch.zeros(4, device="cuda")
    for scale, softcap in [(0.1, 0.0), (0.1, -1.0), (math.inf, 5.0), (math.nan, 5.0)]:
        with pytest.raises(Exception):
            binding.lat_test_capped_scores(x, 4, scale, softcap, x)


def test_softcap_prefill_workload_full_sampled_rows():
    """The measured capped prefill at full size (B1 S8192 Hq16/8 D256, cap 50, the bench's
    own inputs): sampled rows (sequence ends, tile boundaries, random rows) against the
    oracle's fp64 tanh."""
    wl = W.WORKLOADS["gemma2_softcap_prefill"]
    inp = W.prefill_inputs(wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D, dtype=wl.dtype, device="cuda",
                           packed=wl.packed, k_mul=wl.k_mul)
    out, lse = run_prefill_softcap(inp, wl.causal, wl.window, wl.scale, wl.softcap)
    rows = W.sample_rows(wl.B * wl.S, wl.S, extra=[127, 128, 4095, 4096], n_random=256)
    ref, ref_lse = oracle.prefill(inp.heads("q"), inp.heads("k"), inp.heads("v"),
                                  causal=wl.causal, window=wl.window, scale=wl.scale, rows=rows,
                                  softcap=wl.softcap)
    idx = torch.tensor(rows, device="cuda")
    compare(out.reshape(wl.B * wl.S, wl.Hq, wl.D)[idx], ref, wl.dtype, wl.name,
            lse.reshape(wl.B * wl.S, wl.Hq)[idx], ref_lse)
