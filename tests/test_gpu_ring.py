"""Ring-buffer caches for sliding-window layers: lat_attn_decode_ring / lat_kv_append_ring.

A ring of C rows keeps the last C positions (position j in row j % C).  The visible keys
of a decode step are the last W positions, which may wrap past the end of the ring.
Rows holding positions outside the window are filled with NaN, so any read of them
shows up in the output.  The oracle sees the same keys laid out linearly.
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


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


def make_ring(B, Hkv, D, C, W_, lens, dtype, seed):
    """Ring caches [B, C, Hkv*D] whose rows hold the last C positions of each sequence,
    NaN where a row's position is outside the window; also the linear history the oracle
    reads ([B, max_len, Hkv, D], position j at index j)."""
    n_max = max(max(lens), 1)
    hist = W.normal((B, n_max, Hkv * D), dtype=dtype, device="cpu", seed=seed, role="cache")
    kr = torch.full((B, C, Hkv * D), float("nan"), dtype=hist.dtype)
    vr = torch.full((B, C, Hkv * D), float("nan"), dtype=hist.dtype)
    vh = W.normal((B, n_max, Hkv * D), dtype=dtype, device="cpu", seed=seed, role="new")
    for b, n in enumerate(lens):
        for j in range(max(0, n - W_), n):
            kr[b, j % C] = hist[b, j]
            vr[b, j % C] = vh[b, j]
    return (kr.cuda(), vr.cuda(), hist.view(B, n_max, Hkv, D), vh.view(B, n_max, Hkv, D))


def run_ring(q, kr, vr, C, lens_t, max_len, B, Hq, Hkv, D, window, scale, dtype):
    run = DecodeRun(dtype, B, Hq, Hkv, D, C)  # the ring bounds the scratch layout
    out = torch.full((B, Hq * D), float("nan"), dtype=q.dtype, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = status_tensor()
    binding.lat_attn_decode_ring(DT[dtype], q, q.stride(0), kr, vr, Hkv * D, D, C * Hkv * D, C,
                                 lens_t, max_len, out, out.stride(0), lse, B, Hq, Hkv, D,
                                 window, scale, run.ws, run.nbytes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    return out.view(B, Hq, D), lse


# (B, Hq, Hkv, D, C, window, lens, dtype)
CASES = [
    (5, 8, 2, 128, 256, 200, [1100, 255, 256, 57, 400], "bf16"),   # wraps, edges, short
    (3, 16, 8, 64, 1024, 1024, [5000, 1024, 1500], "bf16"),        # window = whole ring
    (2, 8, 1, 256, 300, 257, [10000, 299], "bf16"),
    (2, 16, 2, 512, 128, 100, [333, 90], "bf16"),
    (2, 4, 2, 64, 64, 50, [130, 20], "f32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%d-%dD%dC%dW%d-%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[7]))
def test_ring_decode_matches_oracle(case):
    B, Hq, Hkv, D, C, Wn, lens, dtype = case
    seed = W.BASE_SEED + C + D
    kr, vr, kh, vh = make_ring(B, Hkv, D, C, Wn, lens, dtype, seed)
    q = W.normal((B, Hq * D), dtype=dtype, device="cuda", seed=seed, role="q")
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    out, lse = run_ring(q, kr, vr, C, lens_t, max(lens), B, Hq, Hkv, D, Wn, scale, dtype)
    ref, ref_lse = oracle.decode(q.view(B, Hq, D), kh, vh, lens, window=Wn, scale=scale)
    compare(out, ref, dtype, str(case), lse, ref_lse)


def test_ring_append_then_decode_follows_the_history():
    """Append chunks of 37 rows into a 96-row ring (wrapping several times) and decode
    after each; every step must match the oracle over the linear history."""
    B, Hq, Hkv, D, C, Wn = 2, 8, 2, 128, 96, 80
    steps, chunk = 7, 37
    total = steps * chunk
    kh = W.normal((B, total, Hkv * D), dtype="bf16", device="cuda", seed=5, role="k")
    vh = W.normal((B, total, Hkv * D), dtype="bf16", device="cuda", seed=5, role="v")
    q = W.normal((B, Hq * D), dtype="bf16", device="cuda", seed=5, role="q")
    kr = torch.full((B, C, Hkv * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vr = torch.full_like(kr, float("nan"))
    st = status_tensor()
    scale = 0.1
    for s in range(steps):
        p0 = s * chunk
        pos = torch.full((B,), p0, dtype=torch.int32, device="cuda")
        kn = kh[:, p0:p0 + chunk].contiguous()
        vn = vh[:, p0:p0 + chunk].contiguous()
        binding.lat_kv_append_ring(binding.LAT_BF16, kr, vr, Hkv * D, D, C * Hkv * D, C, kn, vn,
                                   Hkv * D, pos, chunk, B, Hkv, D, st)
        n = p0 + chunk
        lens_t = torch.full((B,), n, dtype=torch.int32, device="cuda")
        out, lse = run_ring(q, kr, vr, C, lens_t, total, B, Hq, Hkv, D, Wn, scale, "bf16")
        assert int(st.item()) == 0
        ref, ref_lse = oracle.decode(q.view(B, Hq, D), kh.view(B, total, Hkv, D).cpu(),
                                     vh.view(B, total, Hkv, D).cpu(), [n] * B, window=Wn,
                                     scale=scale)
        compare(out, ref, "bf16", "step %d (length %d)" % (s, n), lse, ref_lse)
    # every ring row was written by the last append or an earlier one, none left NaN
    assert not torch.isnan(kr.float()).any()
