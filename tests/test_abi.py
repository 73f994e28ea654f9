"""The C ABI without a GPU: the library builds, loads, exports every declared symbol, and
rejects bad arguments on the host before touching CUDA."""
import ctypes
import glob
import os
import re

import pytest

import torch

from gqa_attention_lat_gb300 import binding
from gqa_attention_lat_gb300.build import INCLUDE, build_library

LAT_F32, LAT_BF16 = binding.LAT_F32, binding.LAT_BF16

# These checks hand the library addresses that are never valid device memory and rely on
# the host rejecting the call before any launch.  They run only where no GPU is visible,
# so that a change in the order of the checks can never launch on them.
no_device = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake-pointer host checks run only without a GPU")


@pytest.fixture(scope="module")
def lib():
    path = build_library()
    return binding.library(path)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(INCLUDE, "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names.update(re.findall(r"\b(lat_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_headers_declare_the_three_calls():
    names = declared_functions()
    for n in ("lat_attn_prefill", "lat_attn_decode", "lat_kv_append",
              "lat_attn_decode_workspace_size", "lat_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) <= set(binding._SIGNATURES)


def test_status_strings(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert binding.lat_status_string(code) == name
    assert binding.lat_status_string(99) == "LAT_ERR_UNKNOWN"


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced


def _prefill(**kw):
    args = dict(dt=LAT_BF16, q=FAKE, q_rs=2048, k=FAKE, k_rs=2048, v=FAKE, v_rs=2048, out=FAKE,
                out_rs=1024, lse=None, batch=1, seq_len=4, kv_len=4, n_heads=16, n_kv_heads=8,
                head_dim=64, causal=1, window=0, scale=0.125)
    args.update(kw)
    return binding.lat_attn_prefill(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(n_heads=12, n_kv_heads=8), binding.LAT_ERR_INVALID_ARG),   # 12 % 8 != 0
    (dict(head_dim=96, q_rs=4096, out_rs=4096), binding.LAT_ERR_UNSUPPORTED),
    (dict(head_dim=32), binding.LAT_ERR_UNSUPPORTED),
    (dict(kv_len=3), binding.LAT_ERR_INVALID_ARG),                   # kv_len < seq_len
    (dict(batch=-1), binding.LAT_ERR_INVALID_ARG),
    (dict(q=None), binding.LAT_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), binding.LAT_ERR_INVALID_ARG),                  # bf16 misaligned
    (dict(k_rs=2044), binding.LAT_ERR_INVALID_ARG),                   # stride % 8
    (dict(q_rs=512), binding.LAT_ERR_INVALID_ARG),                    # row narrower than heads
    (dict(dt=7), binding.LAT_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.LAT_ERR_INVALID_ARG),
    (dict(batch=65536), binding.LAT_ERR_UNSUPPORTED),
    # 65535 sequences x 32768 heads x 1 query tile = 2^31 - 2^15 items: past the 2^30 the
    # kernel numbers in int32 (each factor alone is within its own limit)
    (dict(batch=65535, n_heads=32768, n_kv_heads=32768, q_rs=32768 * 64, k_rs=32768 * 64,
          v_rs=32768 * 64, out_rs=32768 * 64), binding.LAT_ERR_UNSUPPORTED),
    # head_dim 512 has two items per query tile and head: 65535 x 16384 x 2 > 2^30
    (dict(batch=65535, n_heads=16384, n_kv_heads=16384, head_dim=512, q_rs=16384 * 512,
          k_rs=16384 * 512, v_rs=16384 * 512, out_rs=16384 * 512), binding.LAT_ERR_UNSUPPORTED),
])
@no_device
def test_prefill_rejects_on_host(lib, kw, code):
    with pytest.raises(binding.LatError) as e:
        _prefill(**kw)
    assert e.value.status == code


@no_device
def test_prefill_empty_is_a_no_op(lib):
    _prefill(batch=0)
    _prefill(seq_len=0, kv_len=0)


def _decode(**kw):
    args = dict(dt=LAT_BF16, q=FAKE, q_rs=4096, k_cache=FAKE, v_cache=FAKE, cache_rs=1024,
                cache_head_stride=128, cache_seq_stride=4096 * 1024, kv_lens=FAKE,
                max_kv_len=4096, out=FAKE, out_rs=4096, lse=None, batch=32, n_heads=32,
                n_kv_heads=8, head_dim=128, window=0, scale=0.088, workspace=FAKE,
                workspace_bytes=1 << 30)
    args.update(kw)
    return binding.lat_attn_decode(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(n_heads=30), binding.LAT_ERR_INVALID_ARG),
    (dict(head_dim=100, q_rs=3200, out_rs=3200), binding.LAT_ERR_UNSUPPORTED),
    (dict(kv_lens=None), binding.LAT_ERR_INVALID_ARG),
    (dict(max_kv_len=-1), binding.LAT_ERR_INVALID_ARG),
    (dict(cache_rs=0), binding.LAT_ERR_INVALID_ARG),
    (dict(cache_rs=1020), binding.LAT_ERR_INVALID_ARG),               # bf16 stride % 8
    (dict(k_cache=FAKE + 4), binding.LAT_ERR_INVALID_ARG),
    (dict(out=FAKE + 8), binding.LAT_ERR_INVALID_ARG),                # bf16 output misaligned
    (dict(out_rs=4100), binding.LAT_ERR_INVALID_ARG),                 # not a multiple of 8
    (dict(batch=65536), binding.LAT_ERR_UNSUPPORTED),
    # 65535 sequences x 129 KV heads (one head block each) = 8.45M units >= 2^23, the
    # unit field of the split-KV merge tickets
    (dict(batch=65535, n_heads=129, n_kv_heads=129, q_rs=129 * 128, out_rs=129 * 128,
          cache_rs=129 * 128, cache_seq_stride=4096 * 129 * 128), binding.LAT_ERR_UNSUPPORTED),
])
@no_device
def test_decode_rejects_on_host(lib, kw, code):
    with pytest.raises(binding.LatError) as e:
        _decode(**kw)
    assert e.value.status == code


@no_device
def test_decode_empty_batch_is_a_no_op(lib):
    _decode(batch=0)


def test_workspace_size_rejects_bad_shapes(lib):
    assert binding.lat_attn_decode_workspace_size(LAT_F32, 8, 16, 8, 64, 100) == 0
    assert binding.lat_attn_decode_workspace_size(LAT_BF16, 8, 15, 8, 64, 100) == 0
    assert binding.lat_attn_decode_workspace_size(LAT_BF16, 8, 16, 8, 96, 100) == 0


@pytest.mark.parametrize("cap", [-1.0, float("inf"), float("nan")])
@no_device
def test_softcap_must_be_finite_and_non_negative(lib, cap):
    with pytest.raises(binding.LatError) as e:
        binding.lat_attn_prefill_softcap(LAT_BF16, FAKE, 1024, FAKE, 512, FAKE, 512, FAKE, 1024,
                                         None, 1, 4, 4, 16, 8, 64, 1, 0, 0.125, cap)
    assert e.value.status == binding.LAT_ERR_INVALID_ARG
    with pytest.raises(binding.LatError) as e:
        binding.lat_attn_decode_softcap(LAT_BF16, FAKE, 4096, FAKE, FAKE, 1024, 128,
                                        4096 * 1024, FAKE, 4096, FAKE, 4096, None, 32, 32, 8,
                                        128, 0, 0.088, cap, FAKE, 1 << 30)
    assert e.value.status == binding.LAT_ERR_INVALID_ARG


@pytest.mark.parametrize("window,ring,code", [
    (0, 256, binding.LAT_ERR_INVALID_ARG),      # a ring needs a window
    (300, 256, binding.LAT_ERR_INVALID_ARG),    # the window must fit in the ring
    (100, 0, binding.LAT_ERR_INVALID_ARG),      # no ring
])
@no_device
def test_ring_decode_rejects_on_host(lib, window, ring, code):
    with pytest.raises(binding.LatError) as e:
        binding.lat_attn_decode_ring(LAT_BF16, FAKE, 4096, FAKE, FAKE, 1024, 128, 256 * 1024,
                                     ring, FAKE, 100000, FAKE, 4096, None, 32, 32, 8, 128,
                                     window, 0.088, FAKE, 1 << 30)
    assert e.value.status == code


@no_device
def test_ring_append_rejects_more_rows_than_the_ring(lib):
    with pytest.raises(binding.LatError) as e:
        binding.lat_kv_append_ring(LAT_BF16, FAKE, FAKE, 1024, 128, 64 * 1024, 64, FAKE, FAKE,
                                   1024, FAKE, 65, 2, 8, 128)
    assert e.value.status == binding.LAT_ERR_INVALID_ARG


def _prefill_cached(**kw):
    args = dict(dt=LAT_BF16, q=FAKE, q_rs=1024, k_cache=FAKE, v_cache=FAKE, cache_rs=512,
                cache_head_stride=128, cache_seq_stride=512 * 4096, out=FAKE, out_rs=1024,
                lse=None, batch=2, seq_len=64, kv_len=300, n_heads=8, n_kv_heads=4,
                head_dim=128, causal=1, window=0, scale=0.088)
    args.update(kw)
    return binding.lat_attn_prefill_cached(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(kv_len=10), binding.LAT_ERR_INVALID_ARG),                    # kv_len < seq_len
    (dict(n_heads=6), binding.LAT_ERR_INVALID_ARG),
    (dict(head_dim=96, q_rs=768, out_rs=768), binding.LAT_ERR_UNSUPPORTED),
    (dict(k_cache=None), binding.LAT_ERR_INVALID_ARG),
    (dict(cache_seq_stride=0), binding.LAT_ERR_INVALID_ARG),
    (dict(cache_head_stride=100), binding.LAT_ERR_INVALID_ARG),        # bf16 stride % 8
    (dict(v_cache=FAKE + 8), binding.LAT_ERR_INVALID_ARG),            # bf16 misaligned
    (dict(scale=float("inf")), binding.LAT_ERR_INVALID_ARG),
])
@no_device
def test_prefill_cached_rejects_on_host(lib, kw, code):
    with pytest.raises(binding.LatError) as e:
        _prefill_cached(**kw)
    assert e.value.status == code


@no_device
def test_prefill_cached_empty_is_a_no_op(lib):
    _prefill_cached(seq_len=0)
    _prefill_cached(batch=0)


def _append(**kw):
    args = dict(dt=LAT_BF16, k_cache=FAKE, v_cache=FAKE, cache_rs=1024, cache_head_stride=128,
                cache_seq_stride=1024 * 64, capacity=64, k_new=FAKE, v_new=FAKE, new_rs=1024,
                pos=FAKE, n_new=1, batch=2, n_kv_heads=8, head_dim=128)
    args.update(kw)
    return binding.lat_kv_append(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(n_kv_heads=0), binding.LAT_ERR_INVALID_ARG),
    (dict(n_new=-1), binding.LAT_ERR_INVALID_ARG),
    (dict(head_dim=48), binding.LAT_ERR_UNSUPPORTED),
    (dict(pos=None), binding.LAT_ERR_INVALID_ARG),
    (dict(new_rs=512), binding.LAT_ERR_INVALID_ARG),
])
@no_device
def test_append_rejects_on_host(lib, kw, code):
    with pytest.raises(binding.LatError) as e:
        _append(**kw)
    assert e.value.status == code


@no_device
def test_append_nothing_is_a_no_op(lib):
    _append(n_new=0)
    _append(batch=0)


def _producer(**kw):
    args = dict(dt=LAT_BF16, qkv=FAKE, qkv_rs=32 * 128, q_norm_w=FAKE, k_norm_w=FAKE, eps=1e-6,
                rope_base=1e6, v_unit_norm=False, q_out=FAKE, q_out_rs=16 * 128, k_cache=FAKE,
                v_cache=FAKE, cache_rs=1024, cache_head_stride=128, cache_seq_stride=1024 * 64,
                capacity=64, pos=FAKE, n_new=4, batch=2, n_heads=16, n_kv_heads=8,
                head_dim=128)
    args.update(kw)
    return binding.lat_qkv_norm_rope_append(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(dt=7), binding.LAT_ERR_INVALID_ARG),
    (dict(n_heads=12, n_kv_heads=8), binding.LAT_ERR_INVALID_ARG),
    (dict(head_dim=48), binding.LAT_ERR_UNSUPPORTED),
    (dict(eps=-1e-6), binding.LAT_ERR_INVALID_ARG),
    (dict(eps=float("nan")), binding.LAT_ERR_INVALID_ARG),
    (dict(rope_base=1.0), binding.LAT_ERR_INVALID_ARG),
    (dict(rope_base=float("inf")), binding.LAT_ERR_INVALID_ARG),
    (dict(qkv_rs=31 * 128), binding.LAT_ERR_INVALID_ARG),   # shorter than Hq + 2 Hkv heads
    (dict(q_out_rs=15 * 128), binding.LAT_ERR_INVALID_ARG),
    (dict(pos=None), binding.LAT_ERR_INVALID_ARG),
    (dict(k_cache=None), binding.LAT_ERR_INVALID_ARG),
    (dict(cache_rs=0), binding.LAT_ERR_INVALID_ARG),
    (dict(batch=-1), binding.LAT_ERR_INVALID_ARG),
])
@no_device
def test_producer_rejects_on_host(lib, kw, code):
    with pytest.raises(binding.LatError) as e:
        _producer(**kw)
    assert e.value.status == code


@no_device
def test_producer_nothing_is_a_no_op(lib):
    _producer(n_new=0)
    _producer(batch=0)


def test_library_is_sm103a_only():
    from gqa_attention_lat_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
