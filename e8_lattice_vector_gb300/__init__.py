"""E8 lattice KV-cache compression for GB300 (sm_103a).

The codec runs in libnq (hand-written CUDA, C ABI in include/nq.h); this
package is its thin Python binding.  Nothing here computes the method on the
CPU: when the library is missing, calls raise.
"""
from .codec import (CodecParams, RopeTable, code_histogram, compress_kv, compress_kv_layers, decompress_kv,
                    decompress_kv_layers, decompress_kv_static, e8_nearest, get_status, layer_profile, plan,
                    plan_layers, roundtrip_kv, roundtrip_kv_layers, sections, shape_of, static_workspace_bytes,
                    workspace)

__all__ = ["CodecParams", "RopeTable", "code_histogram", "compress_kv", "compress_kv_layers", "decompress_kv",
           "decompress_kv_layers", "decompress_kv_static", "e8_nearest", "get_status", "layer_profile", "plan",
           "plan_layers", "roundtrip_kv", "roundtrip_kv_layers", "sections", "shape_of", "static_workspace_bytes",
           "workspace"]
