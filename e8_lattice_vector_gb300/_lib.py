"""ctypes binding of libnq (include/nq.h).

Argument marshalling only: torch tensors are passed as raw device pointers
together with the current CUDA stream; every step of the codec runs in the
library's kernels.  If the library is missing the first call raises -- there
is no fallback path.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libnq.so")

NQ_OK, NQ_ERR_ARG, NQ_ERR_UNSUPPORTED, NQ_ERR_SIZE, NQ_ERR_CUDA = range(5)
NQ_HIST_BINS = 274
FORMAT_VERSION = 1


class Shape(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("batch", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("tokens", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class Params(ctypes.Structure):
    _fields_ = [("key_bits", ctypes.c_int32), ("value_bits", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("strict", ctypes.c_int32),
                ("delta_chunk", ctypes.c_int32), ("rope_theta", ctypes.c_float)]


class Layout(ctypes.Structure):
    _fields_ = [("version", ctypes.c_uint32), ("padded_dim", ctypes.c_uint32),
                ("tokens_padded", ctypes.c_uint32), ("reserved", ctypes.c_uint32), ("rows", ctypes.c_uint64),
                ("k_idx_row_bytes", ctypes.c_uint64), ("v_idx_row_bytes", ctypes.c_uint64),
                ("scales_per_row", ctypes.c_uint64),
                ("k_idx", ctypes.c_uint64), ("k_coset", ctypes.c_uint64), ("k_scale", ctypes.c_uint64),
                ("v_idx", ctypes.c_uint64), ("v_coset", ctypes.c_uint64), ("v_scale", ctypes.c_uint64),
                ("total_bytes", ctypes.c_uint64), ("workspace_bytes", ctypes.c_uint64)]


# name -> (restype, argtypes); the exported C ABI, in header order
class LayerBits(ctypes.Structure):
    _fields_ = [("key_bits", ctypes.c_int32), ("value_bits", ctypes.c_int32)]


_LB = ctypes.POINTER(LayerBits)
_U64P = ctypes.POINTER(ctypes.c_uint64)

SIGNATURES = {
    "nq_plan": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Params), ctypes.POINTER(Layout)]),
    "nq_rope_table": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                     ctypes.c_void_p]),
    "nq_compress_kv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.POINTER(Shape), ctypes.POINTER(Params), ctypes.c_void_p,
                                      ctypes.c_size_t, ctypes.c_void_p]),
    "nq_decompress_kv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                        ctypes.POINTER(Shape), ctypes.POINTER(Params), ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nq_decompress_kv_static": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                               ctypes.POINTER(Shape), ctypes.POINTER(Params), ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p]),
    "nq_get_status": (ctypes.c_int, [ctypes.c_void_p]),
    "nq_roundtrip_kv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.POINTER(Shape), ctypes.POINTER(Params), ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "nq_plan_layers": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Params), _LB, _U64P, _U64P, _U64P]),
    "nq_compress_kv_layers": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.POINTER(Shape), ctypes.POINTER(Params), _LB, ctypes.c_void_p,
                                             ctypes.c_size_t, ctypes.c_void_p]),
    "nq_decompress_kv_layers": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                               ctypes.POINTER(Shape), ctypes.POINTER(Params), _LB, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nq_roundtrip_kv_layers": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.POINTER(Shape), ctypes.POINTER(Params), _LB, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]),
    "nq_code_histogram": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(Shape),
                                         ctypes.POINTER(Params), ctypes.c_void_p, ctypes.c_void_p]),
    "nq_e8_nearest": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_void_p]),
    "nq_strerror": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


class NQError(RuntimeError):
    def __init__(self, fn, status):
        msg = lib().nq_strerror(status).decode()
        super().__init__("%s failed with status %d: %s" % (fn, status, msg))
        self.status = status


def lib():
    """Load libnq.so (raises OSError when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError("libnq.so not built (%s); run e8_lattice_vector_gb300/build.py" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(fn, status):
    if status != NQ_OK:
        raise NQError(fn, status)
