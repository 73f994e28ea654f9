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
from gpu_helpers import DT, DecodeRun, assert_bits_equal, compare, ensure_library, status_tensor
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
    # the oracle's ring, appended alongside and compared bit for bit after every append
    ok_k = np.full((B, C, Hkv, D), np.nan)
    ok_v = np.full((B, C, Hkv, D), np.nan)
    st = status_tensor()
    scale = 0.1
    for s in range(steps):
        p0 = s * chunk
        pos = torch.full((B,), p0, dtype=torch.int32, device="cuda")
        kn = kh[:, p0:p0 + chunk].contiguous()
        vn = vh[:, p0:p0 + chunk].contiguous()
        binding.lat_kv_append_ring(binding.LAT_BF16, kr, vr, Hkv * D, D, C * Hkv * D, C, kn, vn,
                                   Hkv * D, pos, chunk, B, Hkv, D, st)
        ok_k, ok_v = oracle.kv_append_ring(
            ok_k, ok_v, kn.view(B, chunk, Hkv, D).cpu().float().numpy(),
            vn.view(B, chunk, Hkv, D).cpu().float().numpy(), [p0] * B)
        torch.cuda.synchronize()
        assert_bits_equal(kr.view(B, C, Hkv, D), ok_k, "K ring after append %d" % s)
        assert_bits_equal(vr.view(B, C, Hkv, D), ok_v, "V ring after append %d" % s)
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


@pytest.mark.parametrize("dtype,head_major", [("bf16", False), ("f32", False), ("bf16", True)])
def test_ring_append_bit_exact(dtype, head_major):
    """lat_kv_append_ring against the oracle's ring copy, bit for bit in both caches:
    sequences at different positions (one chunk wrapping past the end of the ring, one
    starting exactly on a multiple of it), token-major and head-major cache layouts."""
    B, Hkv, D, C, n_new = 3, 2, 64, 40, 9
    pos = [35, 80, 3]  # 35..43 wraps; 80 = 2C lands on row 0
    if head_major:  # [B, Hkv, C, D]: rows D apart, heads C*D apart
        rs, hs, ss = D, C * D, Hkv * C * D
    else:           # [B, C, Hkv*D]
        rs, hs, ss = Hkv * D, D, C * Hkv * D
    tdt = W.torch_dtype(dtype)
    kc = torch.full((B * ss,), float("nan"), dtype=tdt, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    kn = W.normal((B * n_new, Hkv * D), dtype=dtype, device="cuda", seed=21, role="k")
    vn = W.normal((B * n_new, Hkv * D), dtype=dtype, device="cuda", seed=21, role="v")
    st = status_tensor()
    binding.lat_kv_append_ring(DT[dtype], kc, vc, rs, hs, ss, C, kn, vn, Hkv * D,
                               torch.tensor(pos, dtype=torch.int32, device="cuda"), n_new, B,
                               Hkv, D, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    def as_rows(t):  # [B, C, Hkv, D] whatever the layout
        v = t.view(B, Hkv, C, D).permute(0, 2, 1, 3) if head_major else t.view(B, C, Hkv, D)
        return v
    empty = np.full((B, C, Hkv, D), np.nan)
    ok_k, ok_v = oracle.kv_append_ring(empty, empty, kn.view(B, n_new, Hkv, D).cpu().float().numpy(),
                                       vn.view(B, n_new, Hkv, D).cpu().float().numpy(), pos)
    assert_bits_equal(as_rows(kc), ok_k, "K ring")
    assert_bits_equal(as_rows(vc), ok_v, "V ring")


def test_ring_decode_workload_full():
    """The measured ring workload at full size (B32 Hq16/8 D256, a 1024-row ring, window
    1024, absolute lengths up to 32768, the bench's own inputs): every output against the
    oracle over each sequence's visible positions gathered from the ring in order."""
    wl = W.WORKLOADS["gemma4_sliding_decode_ring"]
    di = W.ring_decode_inputs(wl.B, wl.Hq, wl.Hkv, wl.D, wl.ring, wl.max_len, dtype=wl.dtype,
                              device="cuda")
    out, lse = run_ring(di.q, di.k_cache, di.v_cache, wl.ring, di.kv_lens, wl.max_len, wl.B,
                        wl.Hq, wl.Hkv, wl.D, wl.window, wl.scale, wl.dtype)
    lens = di.kv_lens.cpu().tolist()
    vis = [min(n, wl.window) for n in lens]
    kr = di.k_cache.cpu().view(wl.B, wl.ring, wl.Hkv, wl.D)
    vr = di.v_cache.cpu().view(wl.B, wl.ring, wl.Hkv, wl.D)
    kl = torch.zeros((wl.B, max(vis), wl.Hkv, wl.D), dtype=kr.dtype)
    vl = torch.zeros_like(kl)
    for b, (n, m) in enumerate(zip(lens, vis)):
        rows = torch.tensor([p % wl.ring for p in range(n - m, n)])
        kl[b, :m] = kr[b, rows]
        vl[b, :m] = vr[b, rows]
    ref, ref_lse = oracle.decode(di.q.cpu().view(wl.B, wl.Hq, wl.D), kl, vl, vis, window=0,
                                 scale=wl.scale)
    compare(out, ref, wl.dtype, wl.name, lse, ref_lse)
