"""lat_attn: fused grouped-query attention for one GB300 GPU (sm_103a).

The compute lives in the CUDA library ``liblat_attn.so`` (C ABI in include/lat_attn.h);
this package is its ctypes binding plus the nvcc build step.  Importing the package does
not load the library; the first call does, and raises if it is missing.
"""
from .binding import (LAT_BF16, LAT_ERR_BOUNDS, LAT_ERR_CUDA, LAT_ERR_INVALID_ARG,
                      LAT_ERR_TIMEOUT, LAT_ERR_UNSUPPORTED, LAT_ERR_WORKSPACE, LAT_F32, LAT_OK,
                      LatError, lat_attn_decode, lat_attn_decode_workspace_size,
                      lat_attn_prefill, lat_kv_append, lat_status_string, library)

__all__ = ["LAT_BF16", "LAT_F32", "LAT_OK", "LAT_ERR_INVALID_ARG", "LAT_ERR_UNSUPPORTED",
           "LAT_ERR_WORKSPACE", "LAT_ERR_CUDA", "LAT_ERR_BOUNDS", "LAT_ERR_TIMEOUT",
           "LatError", "lat_attn_prefill", "lat_attn_decode", "lat_attn_decode_workspace_size",
           "lat_kv_append", "lat_status_string", "library"]
