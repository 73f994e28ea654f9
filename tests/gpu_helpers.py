"""Helpers for the GPU parity tests: run the CUDA library through its C ABI on seeded
inputs, run the oracle on the same values, compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gqa_attention_lat_gb300 import binding
from gqa_attention_lat_gb300.build import build_library

# parity bars: fp32 inputs max-abs 1e-4; bf16 inputs (oracle fed the bf16 values)
# max-abs 2e-2 and mean-abs 2e-3; log-sum-exp 1e-3
TOL = {"f32": dict(max_abs=1e-4, mean_abs=1e-4), "bf16": dict(max_abs=2e-2, mean_abs=2e-3)}
LSE_TOL = 1e-3

DT = {"f32": binding.LAT_F32, "bf16": binding.LAT_BF16}


def ensure_library():
    build_library()
    binding.library()


def status_tensor(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)


def compare(got, ref, dtype, what, lse_got=None, lse_ref=None):
    """got: GPU output (any float tensor/array), ref: float64 oracle array."""
    g = got.detach().float().cpu().numpy().astype(np.float64) if hasattr(got, "detach") else got
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, "%s: shape %s vs %s" % (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    err = np.abs(g - ref)
    tol = TOL[dtype]
    assert err.max() <= tol["max_abs"], "%s: max abs err %.3e > %.1e" % (what, err.max(), tol["max_abs"])
    assert err.mean() <= tol["mean_abs"], "%s: mean abs err %.3e > %.1e" % (what, err.mean(), tol["mean_abs"])
    if lse_got is not None:
        lg = lse_got.detach().double().cpu().numpy()
        lr = np.asarray(lse_ref, dtype=np.float64)
        assert lg.shape == lr.shape
        inf_g, inf_r = np.isneginf(lg), np.isneginf(lr)
        assert (inf_g == inf_r).all(), "%s: lse -inf pattern differs" % what
        fin = ~inf_r
        if fin.any():
            le = np.abs(lg[fin] - lr[fin]).max()
            assert le <= LSE_TOL, "%s: lse max abs err %.3e > %.1e" % (what, le, LSE_TOL)
    return float(err.max()), float(err.mean())


def assert_bits_equal(got, ref, what):
    """Byte work (cache appends) is exact: every element equal to the expected value and
    NaN exactly where the expected array holds NaN.  `got` is a torch tensor whose
    values convert to float64 exactly (bf16 or fp32), `ref` a float array."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, "%s: shape %s vs %s" % (what, g.shape, r.shape)
    assert np.array_equal(np.isnan(g), np.isnan(r)), "%s: NaN pattern differs" % what
    fin = ~np.isnan(r)
    bad = np.count_nonzero(g[fin] != r[fin])
    assert bad == 0, "%s: %d elements differ" % (what, bad)


def run_prefill(inp, *, causal, window, scale, out_pad=0, with_lse=True, stream=None):
    """Run lat_attn_prefill on PrefillInputs; returns (out [B,S,Hq,D], lse [B,S,Hq])."""
    dev = inp.q.device
    tdt = inp.q.dtype
    rows = inp.B * inp.S
    width = inp.Hq * inp.D
    out_full = torch.full((rows, width + out_pad), float("nan"), dtype=tdt, device=dev)
    out = out_full[:, :width]
    lse = torch.full((rows, inp.Hq), float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    st = status_tensor(dev)
    binding.lat_attn_prefill(DT[inp.dtype], inp.q, inp.q.stride(0), inp.k, inp.k.stride(0),
                             inp.v, inp.v.stride(0), out, out.stride(0), lse, inp.B, inp.S,
                             inp.L, inp.Hq, inp.Hkv, inp.D, causal, window, scale, st,
                             stream=stream)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    if out_pad:
        assert torch.isnan(out_full[:, width:].float()).all(), "prefill wrote past the row"
    o = out.reshape(inp.B, inp.S, inp.Hq, inp.D)
    l = lse.reshape(inp.B, inp.S, inp.Hq) if with_lse else None
    return o, l


def oracle_prefill(inp, *, causal, window, scale, rows=None):
    return oracle.prefill(inp.heads("q"), inp.heads("k"), inp.heads("v"), causal=causal,
                          window=window, scale=scale, rows=rows)


class DecodeRun:
    """Owns a zeroed decode workspace sized for one shape."""

    def __init__(self, dtype, B, Hq, Hkv, D, max_kv_len, device="cuda"):
        self.dt = DT[dtype]
        self.nbytes = binding.lat_attn_decode_workspace_size(self.dt, B, Hq, Hkv, D, max_kv_len)
        self.ws = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)

    def __call__(self, q, k_cache, v_cache, cache_rs, cache_head_stride, cache_seq_stride,
                 kv_lens, max_kv_len, B, Hq, Hkv, D, window, scale, out=None, lse=None,
                 status=None, stream=None):
        dev = q.device
        if out is None:
            out = torch.full((B, Hq * D), float("nan"), dtype=q.dtype, device=dev)
        if lse is None:
            lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
        st = status if status is not None else status_tensor(dev)
        binding.lat_attn_decode(self.dt, q, q.stride(0), k_cache, v_cache, cache_rs,
                                cache_head_stride, cache_seq_stride, kv_lens, max_kv_len, out,
                                out.stride(0), lse, B, Hq, Hkv, D, window, scale, self.ws,
                                self.nbytes, st, stream=stream)
        return out, lse, st


def run_decode(di, *, window, scale, max_kv_len=None, runner=None):
    """Run lat_attn_decode on DecodeInputs (token-major cache)."""
    mk = di.cap if max_kv_len is None else max_kv_len
    runner = runner or DecodeRun(di.dtype, di.B, di.Hq, di.Hkv, di.D, mk, di.q.device)
    out, lse, st = runner(di.q, di.k_cache, di.v_cache, di.Hkv * di.D, di.D,
                          di.cap * di.Hkv * di.D, di.kv_lens, mk, di.B, di.Hq, di.Hkv, di.D,
                          window, scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d" % int(st.item())
    return out.view(di.B, di.Hq, di.D), lse


def oracle_decode(di, *, window, scale):
    return oracle.decode(di.q_heads(), di.cache_heads("k_cache"), di.cache_heads("v_cache"),
                         di.kv_lens.cpu().tolist(), window=window, scale=scale)
