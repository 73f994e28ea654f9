"""Seeded synthetic inputs and the named attention workloads.

This module draws random numbers and lays tensors out; it holds none of the attention
arithmetic.  Both sides of every parity check -- the CUDA library and the fp64 oracle --
consume the tensors it returns (the oracle gets the same values, upcast exactly).

All values are i.i.d. N(0, 1) drawn in fp32 from a seeded torch generator and, for
bf16 workloads, rounded to bf16 (round-to-nearest-even, torch's conversion).  Unused
KV-cache slots are filled with NaN so that any read of them poisons the result.

The named workloads follow the model shapes the pages give: Qwen3 attention shapes on
the lattice-inference DESIGN page ("Model Compatibility Matrix": head_dim 64/80/128,
GQA groups 2/2/4/5) and Gemma 4 layer shapes on the hf2q "Current Inference Path"
page (section 2 step 1: 16 heads, sliding window 1024, sliding layers head_dim 256
with 8 KV heads, global layers head_dim 512 with 2 KV heads).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BASE_SEED = 0x1A7A77

# independent generator streams per tensor role
_STREAM = {"q": 1, "k": 2, "v": 3, "kv_len": 4, "cache": 5, "new": 6, "pos": 7, "rows": 8,
           "chunk_q": 9}


def torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(device, seed: int, role: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1000003 + _STREAM[role]) & 0x7FFFFFFFFFFFFFFF)
    return g


def normal(shape, *, dtype: str, device, seed: int, role: str, mul: float = 1.0):
    """N(0,1) in fp32 (times `mul`, applied before rounding), then cast to `dtype`."""
    x = torch.randn(shape, generator=_gen(device, seed, role), device=device,
                    dtype=torch.float32)
    if mul != 1.0:
        x.mul_(mul)
    return x.to(torch_dtype(dtype))


@dataclass
class PrefillInputs:
    """Q/K/V as 2-D row views [rows, row_stride] plus the shape of the problem."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    B: int
    S: int
    L: int
    Hq: int
    Hkv: int
    D: int
    dtype: str
    packed: torch.Tensor | None = None  # the parent buffer when Q/K/V share one

    def heads(self, which: str) -> torch.Tensor:
        """The logical [B, rows, H, D] view of q, k or v (no copy)."""
        t = getattr(self, which)
        rows, H = (self.S, self.Hq) if which == "q" else (self.L, self.Hkv)
        return t.as_strided((self.B, rows, H, self.D),
                            (rows * t.stride(0), t.stride(0), self.D, 1))


def prefill_inputs(B, S, L, Hq, Hkv, D, *, dtype="bf16", device="cpu", seed=BASE_SEED,
                   packed=False, k_mul=1.0, q_pad=0, kv_pad=0) -> PrefillInputs:
    """Prefill inputs.

    packed=True puts Q, K and V side by side in one [B*S, (Hq + 2*Hkv)*D] buffer, as a
    fused QKV projection writes them (weight shape [q_dim + 2*kv_dim, hidden], INV-7 on
    the lattice-inference DESIGN page); Q/K/V are then column slices read with the
    parent's row stride (the rlx-metal DESIGN page, "Cross-crate contract": per-tensor
    q/k/v row strides let attention read straight from the parent QKV buffer).
    q_pad / kv_pad add unused columns to each row of separate buffers, so the row
    stride exceeds the data width.
    """
    if packed:
        if S != L:
            raise ValueError("a packed QKV buffer needs seq_len == kv_len")
        W = (Hq + 2 * Hkv) * D
        buf = torch.empty((B * S, W), dtype=torch_dtype(dtype), device=device)
        buf[:, :Hq * D] = normal((B * S, Hq * D), dtype=dtype, device=device, seed=seed,
                                 role="q")
        buf[:, Hq * D:(Hq + Hkv) * D] = normal((B * S, Hkv * D), dtype=dtype, device=device,
                                               seed=seed, role="k", mul=k_mul)
        buf[:, (Hq + Hkv) * D:] = normal((B * S, Hkv * D), dtype=dtype, device=device,
                                         seed=seed, role="v")
        q = buf[:, :Hq * D]
        k = buf[:, Hq * D:(Hq + Hkv) * D]
        v = buf[:, (Hq + Hkv) * D:]
        return PrefillInputs(q, k, v, B, S, L, Hq, Hkv, D, dtype, packed=buf)

    def rows(n, H, role, pad, mul=1.0):
        full = torch.full((n, H * D + pad), float("nan"), dtype=torch_dtype(dtype),
                          device=device)
        full[:, :H * D] = normal((n, H * D), dtype=dtype, device=device, seed=seed,
                                 role=role, mul=mul)
        return full[:, :H * D]

    q = rows(B * S, Hq, "q", q_pad)
    k = rows(B * L, Hkv, "k", kv_pad, k_mul)
    v = rows(B * L, Hkv, "v", kv_pad)
    return PrefillInputs(q, k, v, B, S, L, Hq, Hkv, D, dtype)


@dataclass
class DecodeInputs:
    """One query token per sequence and a token-major KV cache [B, cap, Hkv*D]."""
    q: torch.Tensor            # [B, Hq*D]
    k_cache: torch.Tensor      # [B, cap, Hkv*D]
    v_cache: torch.Tensor
    kv_lens: torch.Tensor      # int32 [B]
    B: int
    Hq: int
    Hkv: int
    D: int
    cap: int
    dtype: str

    def q_heads(self):
        return self.q.view(self.B, self.Hq, self.D)

    def cache_heads(self, which: str):
        t = getattr(self, which)
        return t.view(self.B, self.cap, self.Hkv, self.D)


def decode_inputs(B, Hq, Hkv, D, cap, *, kv_lens=None, dtype="bf16", device="cpu",
                  seed=BASE_SEED, nan_fill=True) -> DecodeInputs:
    """Decode inputs.  kv_lens None draws each length uniformly from [1, cap]; an int
    gives every sequence that length; a list gives them one by one.  Slots at or past
    a sequence's length hold NaN when nan_fill is set."""
    if kv_lens is None:
        lens = torch.randint(1, cap + 1, (B,), generator=_gen("cpu", seed, "kv_len"),
                             dtype=torch.int64).to(torch.int32)
    elif isinstance(kv_lens, int):
        lens = torch.full((B,), kv_lens, dtype=torch.int32)
    else:
        lens = torch.tensor(list(kv_lens), dtype=torch.int32)
    q = normal((B, Hq * D), dtype=dtype, device=device, seed=seed, role="q")
    kc = normal((B, cap, Hkv * D), dtype=dtype, device=device, seed=seed, role="k")
    vc = normal((B, cap, Hkv * D), dtype=dtype, device=device, seed=seed, role="v")
    if nan_fill:
        for b in range(B):
            n = int(lens[b])
            kc[b, n:] = float("nan")
            vc[b, n:] = float("nan")
    return DecodeInputs(q, kc, vc, lens.to(device), B, Hq, Hkv, D, cap, dtype)


def ring_decode_inputs(B, Hq, Hkv, D, ring, max_len, *, dtype="bf16", device="cpu",
                       seed=BASE_SEED) -> DecodeInputs:
    """Decode inputs over a ring cache of `ring` rows per sequence (every row holds some
    earlier position, so none is NaN); lengths are absolute, uniform in [1, max_len]."""
    lens = torch.randint(1, max_len + 1, (B,), generator=_gen("cpu", seed, "kv_len"),
                         dtype=torch.int64).to(torch.int32)
    q = normal((B, Hq * D), dtype=dtype, device=device, seed=seed, role="q")
    kc = normal((B, ring, Hkv * D), dtype=dtype, device=device, seed=seed, role="k")
    vc = normal((B, ring, Hkv * D), dtype=dtype, device=device, seed=seed, role="v")
    return DecodeInputs(q, kc, vc, lens.to(device), B, Hq, Hkv, D, ring, dtype)


def sample_rows(n_rows_total: int, S: int, *, extra=(), n_random=256, seed=BASE_SEED):
    """A deterministic subset of query rows (flattened b*S + i) for large workloads:
    the first and last 4 rows of each sequence, the listed in-sequence positions
    (e.g. window and tile boundaries, each +-1) and `n_random` seeded random rows."""
    B = n_rows_total // S
    picks = set()
    for b in range(B):
        for i in list(range(4)) + list(range(S - 4, S)):
            picks.add(b * S + i)
        for e in extra:
            for i in (e - 1, e, e + 1):
                if 0 <= i < S:
                    picks.add(b * S + i)
    g = _gen("cpu", seed, "rows")
    picks.update(torch.randint(0, n_rows_total, (n_random,), generator=g).tolist())
    return sorted(picks)


# ----------------------------------------------------------------------------------
# Named workloads

@dataclass
class Workload:
    name: str
    kind: str             # "prefill", "prefill_cached", "decode" or "producer"
    dtype: str
    B: int
    Hq: int
    Hkv: int
    D: int
    S: int = 1            # prefill query length
    L: int = 0            # prefill key length (>= S) / decode cache capacity
    cap: int = 0          # prefill_cached: cache capacity (rows per sequence)
    softcap: float = 0.0  # > 0: Gemma 2 score cap softcap * tanh(s / softcap)
    ring: int = 0         # decode: > 0, a ring cache of L = ring rows; lengths up to max_len
    max_len: int = 0
    causal: bool = True
    window: int = 0
    packed: bool = False
    k_mul: float = 1.0
    kv_lens: object = None  # decode: None (uniform draw), int or list
    scale: float = field(default=0.0)

    def __post_init__(self):
        if self.scale == 0.0:
            self.scale = 1.0 / math.sqrt(self.D)


WORKLOADS = {
    # tiny fp32: causal prefill and one decode step at kv_len 64
    "tiny_f32_prefill": Workload("tiny_f32_prefill", "prefill", "f32", 1, 4, 2, 64, S=64, L=64),
    "tiny_f32_decode": Workload("tiny_f32_decode", "decode", "f32", 1, 4, 2, 64, L=64,
                                kv_lens=64),
    # Qwen3-0.6B-shaped prefill read from one packed QKV buffer
    "qwen3_0.6b_prefill": Workload("qwen3_0.6b_prefill", "prefill", "bf16", 8, 16, 8, 64,
                                   S=512, L=512, packed=True),
    # decode over a 4096-slot cache, lengths uniform in [1, 4096]
    "decode_b32_h32_kv8_d128": Workload("decode_b32_h32_kv8_d128", "decode", "bf16", 32, 32,
                                        8, 128, L=4096, kv_lens=None),
    # Gemma-4 sliding layer: head_dim 256, 8 KV heads, window 1024, K scaled by 0.5
    "gemma4_sliding_prefill": Workload("gemma4_sliding_prefill", "prefill", "bf16", 2, 16, 8,
                                       256, S=8192, L=8192, window=1024, k_mul=0.5),
    # Gemma-4 global layer: head_dim 512, 2 KV heads
    "gemma4_global_prefill": Workload("gemma4_global_prefill", "prefill", "bf16", 1, 16, 2,
                                      512, S=8192, L=8192),
    "gemma4_global_decode": Workload("gemma4_global_decode", "decode", "bf16", 8, 16, 2, 512,
                                     L=32768, kv_lens=32768),
    # Gemma-2-shaped global layer with its attention score cap of 50
    "gemma2_softcap_prefill": Workload("gemma2_softcap_prefill", "prefill", "bf16", 1, 16, 8,
                                       256, S=8192, L=8192, softcap=50.0),
    # Gemma-4 sliding layer decode over a 1024-row ring cache, absolute lengths up to 32768
    "gemma4_sliding_decode_ring": Workload("gemma4_sliding_decode_ring", "decode", "bf16", 32,
                                           16, 8, 256, L=1024, window=1024, ring=1024,
                                           max_len=32768),
    # the attention-input producer on the Qwen3-0.6B prefill rows: Q/K RMS norm, RoPE
    # (base 1e6), V copy, append into a token-major 4096-slot cache
    "qwen3_qkv_producer": Workload("qwen3_qkv_producer", "producer", "bf16", 8, 16, 8, 64,
                                   S=512, L=512, cap=4096),
    # one long sequence: 16 query heads over 2 KV heads, head_dim 128, 131072 cached
    # tokens -- two work units only, so the key stream must be cut finely to keep every
    # SM busy
    "decode_b1_kv2_d128_128k": Workload("decode_b1_kv2_d128_128k", "decode", "bf16", 1, 16, 2,
                                        128, L=131072, kv_lens=131072),
    # chunked prefill against the decode cache: 512 new rows after 1536 cached keys, read
    # from a token-major 4096-slot cache (Qwen3-0.6B attention shape)
    "qwen3_chunked_prefill": Workload("qwen3_chunked_prefill", "prefill_cached", "bf16", 8, 16,
                                      8, 64, S=512, L=2048, cap=4096),
}
