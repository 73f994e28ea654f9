"""lat_attn_decode_static: decode for callers that cannot allocate device memory.

Callers inside a host framework that owns all device memory, or on a path where an
allocation's implicit synchronisation is not acceptable, cannot hand lat_attn_decode a
workspace.  This entry point keeps its split-KV scratch in a fixed array in the library's
own device memory instead.  These checks call it through the C ABI and compare it with
lat_attn_decode (which gets a freshly allocated workspace) and with the fp64 oracle, on
two calls in a row with different shapes, so the second call runs over whatever the
first left in the shared array.  This file is collected last on purpose.
"""
import pytest
import torch

import workloads as W
from gpu_helpers import DecodeRun, compare, ensure_library, oracle_decode, status_tensor
from gqa_attention_lat_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    ensure_library()


def _decode_both(di, window, scale):
    B, Hq, Hkv, D, cap = di.B, di.Hq, di.Hkv, di.D, di.cap
    run = DecodeRun(di.dtype, B, Hq, Hkv, D, cap)
    ref_out, ref_lse, st = run(di.q, di.k_cache, di.v_cache, Hkv * D, D, cap * Hkv * D,
                               di.kv_lens, cap, B, Hq, Hkv, D, window, scale)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    st2 = status_tensor()
    binding.lat_attn_decode_static(binding.LAT_BF16 if di.dtype == "bf16" else binding.LAT_F32,
                                   di.q, di.q.stride(0), di.k_cache, di.v_cache, Hkv * D, D,
                                   cap * Hkv * D, di.kv_lens, cap, out, out.stride(0), lse, B, Hq,
                                   Hkv, D, window, scale, st2)
    torch.cuda.synchronize()
    assert st.item() == 0 and st2.item() == 0
    return out, lse, ref_out, ref_lse


def test_static_scratch_decode_matches_workspace_decode_twice():
    first = W.decode_inputs(4, 16, 2, 128, 3000, kv_lens=[3000, 1500, 17, 1], device="cuda",
                            seed=W.BASE_SEED + 11)
    second = W.decode_inputs(3, 8, 2, 64, 1000, kv_lens=[1000, 999, 500], device="cuda",
                             seed=W.BASE_SEED + 12)
    for di, window in ((first, 0), (second, 100)):
        scale = 1.0 / di.D ** 0.5
        out, lse, ref_out, ref_lse = _decode_both(di, window, scale)
        out = out.view(di.B, di.Hq, di.D)
        compare(out, ref_out.view(di.B, di.Hq, di.D).double().cpu().numpy(), di.dtype,
                "static scratch vs workspace", lse, ref_lse.double().cpu().numpy())
        orc_out, orc_lse = oracle_decode(di, window=window, scale=scale)
        compare(out, orc_out, di.dtype, "static scratch vs oracle", lse, orc_lse)


def test_static_scratch_rejects_shapes_beyond_its_maximum():
    # Every pointer is NULL: the size check answers first; were it ever moved behind the
    # argument checks, the NULL pointers would be refused with INVALID_ARG instead, and
    # nothing would launch either way.
    with pytest.raises(binding.LatError) as e:
        binding.lat_attn_decode_static(binding.LAT_BF16, None, 16 * 512, None, None, 2 * 512,
                                       512, 32768 * 2 * 512, None, 32768, None, 16 * 512, None,
                                       1024, 16, 2, 512, 0, 0.04)
    assert e.value.status == binding.LAT_ERR_WORKSPACE
