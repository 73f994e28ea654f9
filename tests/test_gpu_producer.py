"""The fused attention-input producer (Q/K RMS norm, neox RoPE, V, cache append) on the GPU
against the fp64 producer oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import DT, ensure_library, status_tensor
from gqa_attention_lat_gb300 import binding
from oracle import producer

pytestmark = pytest.mark.gpu

# The producer's outputs are not averages (|y| reaches ~10 with N(0,1) norm weights), so
# the bound for a bf16 output is its one rounding from fp32: half a bf16 ulp, at most
# 2^-8 |y|, plus an absolute 1e-4 for the fp32 arithmetic before it (cancellation in
# a cos - b sin).  fp32 outputs: 1e-4 absolute.
def _bound(ref, dtype):
    if dtype == "bf16":
        return np.abs(ref) * 2.0 ** -8 + 1e-4
    return np.full_like(ref, 1e-4)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


def _check(got, ref, dtype, what):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what + ": non-finite output"
    over = err > _bound(ref, dtype)
    assert not over.any(), "%s: %d elements over the bound, worst err %.3g at |ref| %.3g" % (
        what, int(over.sum()), err.max(), float(np.abs(ref).flat[int(np.argmax(err))]))


# (B, T, Hq, Hkv, D, cap, pos, base, v_unit_norm, dtype, head_major)
CASES = [
    (2, 5, 16, 8, 64, 64, [0, 40], 1e6, False, "bf16", False),
    (3, 1, 32, 8, 128, 5000, [4095, 17, 4999], 1e6, False, "bf16", False),  # decode-step rows
    (1, 33, 8, 2, 256, 300, [200], 1e4, True, "bf16", True),                # V unit norm
    (2, 4, 16, 2, 512, 4096, [1000, 3000], 1e6, False, "bf16", False),
    (1, 7, 4, 4, 80, 16, [3], 1e4, False, "bf16", True),
    (2, 3, 4, 2, 64, 40, [10, 0], 1e4, True, "f32", False),
    (1, 2, 8, 2, 128, 70000, [65535], 5e5, False, "f32", False),           # long position
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dT%dH%d-%dD%dcap%d-%s%s%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[9], "-vn" if c[8] else "", "-hm" if c[10] else ""))
def test_producer_matches_oracle(case):
    B, T, Hq, Hkv, D, cap, pos, base, vnorm, dtype, head_major = case
    seed = W.BASE_SEED + D + cap
    width = (Hq + 2 * Hkv) * D
    qkv = W.normal((B * T, width + 16), dtype=dtype, device="cuda", seed=seed, role="new")
    qkv_v = qkv[:, :width]  # row stride larger than the row
    qw = W.normal((D,), dtype=dtype, device="cuda", seed=seed, role="q", mul=0.5)
    kw = W.normal((D,), dtype=dtype, device="cuda", seed=seed, role="k", mul=0.5)
    tdt = W.torch_dtype(dtype)
    if head_major:  # [B, Hkv, cap, D]
        kc = torch.full((B, Hkv, cap, D), float("nan"), dtype=tdt, device="cuda")
        strides = (D, cap * D, Hkv * cap * D)
    else:           # [B, cap, Hkv * D]
        kc = torch.full((B, cap, Hkv * D), float("nan"), dtype=tdt, device="cuda")
        strides = (Hkv * D, D, cap * Hkv * D)
    vc = torch.full_like(kc, float("nan"))
    q_out = torch.full((B * T, Hq * D), float("nan"), dtype=tdt, device="cuda")
    pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
    st = status_tensor()
    eps = 1e-6
    binding.lat_qkv_norm_rope_append(DT[dtype], qkv_v, qkv.stride(0), qw, kw, eps, base, vnorm,
                                     q_out, q_out.stride(0), kc, vc, *strides, cap, pos_t, T, B, Hq,
                                     Hkv, D, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rq, rk, rv = producer.qkv_norm_rope(qkv_v.reshape(B, T, width), pos, n_heads=Hq,
                                        n_kv_heads=Hkv, head_dim=D, q_w=qw, k_w=kw, eps=eps,
                                        base=base, v_unit_norm=vnorm)
    _check(q_out.view(B, T, Hq, D), rq, dtype, "q")
    if head_major:
        kview = lambda c, b: c[b].permute(1, 0, 2)           # [cap, Hkv, D]
    else:
        kview = lambda c, b: c[b].view(cap, Hkv, D)
    for b in range(B):
        rows = slice(pos[b], pos[b] + T)
        _check(kview(kc, b)[rows], rk[b], dtype, "k rows of sequence %d" % b)
        _check(kview(vc, b)[rows], rv[b], dtype, "v rows of sequence %d" % b)
        # nothing outside the new rows was written
        rest = torch.ones(cap, dtype=torch.bool)
        rest[rows] = False
        assert torch.isnan(kview(kc, b)[rest].float()).all()


def test_producer_skips_a_sequence_out_of_range():
    B, T, Hq, Hkv, D, cap = 2, 4, 8, 2, 64, 32
    qkv = W.normal((B * T, (Hq + 2 * Hkv) * D), dtype="bf16", device="cuda", seed=3, role="new")
    kc = torch.full((B, cap, Hkv * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    q_out = torch.full((B * T, Hq * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([0, 30], dtype=torch.int32, device="cuda")  # 30 + 4 > 32
    st = status_tensor()
    binding.lat_qkv_norm_rope_append(binding.LAT_BF16, qkv, qkv.stride(0), None, None, 1e-6, 1e4,
                                     False, q_out, q_out.stride(0), kc, vc, Hkv * D, D,
                                     cap * Hkv * D, cap, pos, T, B, Hq, Hkv, D, st)
    torch.cuda.synchronize()
    assert st.item() == binding.LAT_ERR_BOUNDS
    assert not torch.isnan(kc[0, :T].float()).any()          # sequence 0 written
    assert torch.isnan(kc[1].float()).all()                  # sequence 1 skipped whole
    assert torch.isnan(q_out[T:].float()).all()


def test_producer_full_workload():
    """The benchmark's producer workload at full size (every row checked): 8 sequences of
    512 new rows of a Qwen3-0.6B-shaped fused QKV projection, appended at positions
    0..511 of a 4096-slot token-major cache."""
    wl = W.WORKLOADS["qwen3_qkv_producer"]
    B, T, Hq, Hkv, D, cap = wl.B, wl.S, wl.Hq, wl.Hkv, wl.D, wl.cap
    width = (Hq + 2 * Hkv) * D
    qkv = W.normal((B * T, width), dtype="bf16", device="cuda", seed=W.BASE_SEED, role="new")
    qw = W.normal((D,), dtype="bf16", device="cuda", seed=W.BASE_SEED, role="q")
    kw = W.normal((D,), dtype="bf16", device="cuda", seed=W.BASE_SEED, role="k")
    kc = torch.full((B, cap, Hkv * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    q_out = torch.empty((B * T, Hq * D), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = status_tensor()
    binding.lat_qkv_norm_rope_append(binding.LAT_BF16, qkv, qkv.stride(0), qw, kw, 1e-6, 1e6,
                                     False, q_out, q_out.stride(0), kc, vc, Hkv * D, D,
                                     cap * Hkv * D, cap, pos, T, B, Hq, Hkv, D, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rq, rk, rv = producer.qkv_norm_rope(qkv.reshape(B, T, width), [0] * B, n_heads=Hq,
                                        n_kv_heads=Hkv, head_dim=D, q_w=qw, k_w=kw, eps=1e-6,
                                        base=1e6)
    _check(q_out.view(B, T, Hq, D), rq, "bf16", "q")
    _check(kc[:, :T].reshape(B, T, Hkv, D), rk, "bf16", "k rows")
    _check(vc[:, :T].reshape(B, T, Hkv, D), rv, "bf16", "v rows")
    assert torch.isnan(kc[:, T:].float()).all() and torch.isnan(vc[:, T:].float()).all()


# (D, pos, T, base): rows far out, where fp32 can no longer hold p * freq exactly; the
# last case crosses 2^24, where positions stop being exact in fp32 at all.  fp32 outputs,
# so an angle error above ~1e-5 rad would show.  One sequence, one KV head: the caches
# hold pos + T rows (up to 4.3 GB each).
FAR = [
    (64, 5_000_003, 5, 1e4),
    (80, 9_999_998, 3, 1e4),       # the general kernel
    (64, (1 << 24) - 3, 6, 1e4),   # crosses 2^24
]


@pytest.mark.parametrize("case", FAR, ids=lambda c: "D%d-pos%d" % (c[0], c[1]))
def test_producer_far_positions(case):
    D, p0, T, base = case
    Hq, Hkv, cap = 2, 1, case[1] + case[2]
    width = (Hq + 2 * Hkv) * D
    qkv = W.normal((T, width), dtype="f32", device="cuda", seed=W.BASE_SEED + D, role="new")
    kc = torch.full((1, cap, Hkv * D), float("nan"), dtype=torch.float32, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    q_out = torch.empty((T, Hq * D), dtype=torch.float32, device="cuda")
    pos = torch.tensor([p0], dtype=torch.int32, device="cuda")
    st = status_tensor()
    binding.lat_qkv_norm_rope_append(binding.LAT_F32, qkv, qkv.stride(0), None, None, 1e-6, base,
                                     False, q_out, q_out.stride(0), kc, vc, Hkv * D, D,
                                     cap * Hkv * D, cap, pos, T, 1, Hq, Hkv, D, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rq, rk, rv = producer.qkv_norm_rope(qkv.reshape(1, T, width), [p0], n_heads=Hq,
                                        n_kv_heads=Hkv, head_dim=D, q_w=None, k_w=None,
                                        eps=1e-6, base=base)
    _check(q_out.view(1, T, Hq, D), rq, "f32", "q")
    _check(kc[:, p0:p0 + T].reshape(1, T, Hkv, D), rk, "f32", "k rows")
    _check(vc[:, p0:p0 + T].reshape(1, T, Hkv, D), rv, "f32", "v rows")
    del kc, vc
    torch.cuda.empty_cache()
