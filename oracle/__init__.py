"""CPU oracle for E8 lattice KV-cache compression (ctypes over plain C).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library and never imports it.

All array arguments are numpy arrays; binary16 data travels as ``uint16`` bit
patterns so that nothing here depends on a numpy float16 rounding path.
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        sigs = {
            "orc_padded_dim": (_I, [_I]),
            "orc_h2f": (_F, [ctypes.c_uint16]),
            "orc_f2h_rn": (ctypes.c_uint16, [_F]),
            "orc_rope_table": (None, [_P, _I, _I, _F, _P]),
            "orc_rope_remove": (None, [_P, _I, _P]),
            "orc_rope_apply": (None, [_P, _I, _P]),
            "orc_fwht": (None, [_P, _I]),
            "orc_fwht_forward": (None, [_P, _I]),
            "orc_group_scale": (ctypes.c_uint16, [_F, _I, _I]),
            "orc_e8_block": (_I, [_P, _I, _I, _P]),
            "orc_e8_nearest": (None, [_P, _P, _I64, _I, _I]),
            "orc_encode_row": (None, [_P, _P, _I, _I, _I, _I, _P, _P, _P]),
            "orc_decode_row": (None, [_P, ctypes.c_uint16, _P, _P, _I, _I, _I, _P]),
            "orc_delta_row": (None, [_P, _P, _P, ctypes.c_uint16, _I, _I]),
            "orc_undelta_row": (None, [_P, _P, _P, ctypes.c_uint16, _I, _I]),
            "orc_compress_tensor": (None, [_P, _I64, _I, _I, _P, _I, _I, _I, _I, _P, _P, _P]),
            "orc_decompress_tensor": (None, [_P, _P, _P, _I64, _I, _I, _P, _I, _I, _I, _I, _P]),
            "orc_joint_pack_row": (None, [_P, ctypes.c_uint16, _I, _I]),
            "orc_joint_split_row": (ctypes.c_uint16, [_P, _I, _I]),
            "orc_code_histogram": (None, [_P, _P, _I64, _I, _I, _P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def padded_dim(head_dim):
    return lib().orc_padded_dim(int(head_dim))


def h2f(bits):
    bits = _c(bits, np.uint16)
    return np.array([lib().orc_h2f(int(b)) for b in bits.ravel()], dtype=np.float32).reshape(bits.shape)


def f2h(x):
    x = _c(x, np.float32)
    return np.array([lib().orc_f2h_rn(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def rope_table(tokens, head_dim, theta, positions=None):
    """[tokens, head_dim/2, 2] float32 (cos, sin) table."""
    cs = np.zeros((tokens, head_dim // 2, 2), dtype=np.float32)
    pos = None if positions is None else _c(positions, np.int32)
    lib().orc_rope_table(_ptr(pos), int(tokens), int(head_dim), float(theta), _ptr(cs))
    return cs


def rope_remove(x, cs_row):
    x = _c(x, np.float32).copy()
    lib().orc_rope_remove(_ptr(x), x.shape[-1], _ptr(_c(cs_row, np.float32)))
    return x


def rope_apply(x, cs_row):
    x = _c(x, np.float32).copy()
    lib().orc_rope_apply(_ptr(x), x.shape[-1], _ptr(_c(cs_row, np.float32)))
    return x


def fwht(x):
    x = _c(x, np.float32).copy()
    lib().orc_fwht(_ptr(x), x.shape[-1])
    return x


def fwht_forward(x):
    x = _c(x, np.float32).copy()
    lib().orc_fwht_forward(_ptr(x), x.shape[-1])
    return x


def group_scale(amax, bits, dp):
    return lib().orc_group_scale(float(amax), int(bits), int(dp))


def e8_nearest(u, strict, bits):
    """Nearest codebook point for each 8-block; u has shape [..., 8]."""
    u = _c(u, np.float32)
    r = np.empty_like(u)
    n = u.size // 8
    lib().orc_e8_nearest(_ptr(u), _ptr(r), n, int(strict), int(bits))
    return r


def e8_block(u, strict, bits):
    u = _c(u, np.float32)
    r = np.empty(8, dtype=np.float32)
    c = lib().orc_e8_block(_ptr(u), int(strict), int(bits), _ptr(r))
    return r, c


def row_bytes(head_dim, bits):
    return padded_dim(head_dim) * bits // 8


def compress_tensor(x_bits, tokens, head_dim, bits, group, strict, delta_chunk, cs=None):
    """x_bits: uint16 [slices, tokens, head_dim].  Returns (idx, coset, scales)."""
    x_bits = _c(x_bits, np.uint16)
    slices = x_bits.size // (tokens * head_dim) if tokens * head_dim else 0
    dp = padded_dim(head_dim)
    rows = slices * tokens
    idx = np.zeros((rows, dp * bits // 8), dtype=np.uint8)
    coset = np.zeros(rows, dtype=np.uint16)
    scales = np.zeros((rows, dp // group), dtype=np.uint16)
    csa = None if cs is None else _c(cs, np.float32)
    lib().orc_compress_tensor(_ptr(x_bits), slices, int(tokens), int(head_dim), _ptr(csa),
                              int(bits), int(group), int(strict), int(delta_chunk),
                              _ptr(idx), _ptr(coset), _ptr(scales))
    return idx, coset, scales


def decompress_tensor(idx, coset, scales, slices, tokens, head_dim, bits, group, delta_chunk, cs=None,
                      joint=False):
    idx = _c(idx, np.uint8)
    coset = _c(coset, np.uint16)
    scales = _c(scales, np.uint16)
    out = np.zeros((slices, tokens, head_dim), dtype=np.uint16)
    csa = None if cs is None else _c(cs, np.float32)
    lib().orc_decompress_tensor(_ptr(idx), _ptr(coset), _ptr(scales), int(slices), int(tokens),
                                int(head_dim), _ptr(csa), int(bits), int(group), int(delta_chunk),
                                int(bool(joint)), _ptr(out))
    return out


def joint_pack_row(idx, coset, dp, bits):
    idx = _c(idx, np.uint8).copy()
    lib().orc_joint_pack_row(_ptr(idx), int(coset), int(dp), int(bits))
    return idx


def joint_split_row(idx, dp, bits):
    idx = _c(idx, np.uint8).copy()
    c = lib().orc_joint_split_row(_ptr(idx), int(dp), int(bits))
    return idx, int(c)


def encode_row(x_bits, head_dim, bits, group, strict, cs_row=None):
    x_bits = _c(x_bits, np.uint16)
    dp = padded_dim(head_dim)
    idx = np.zeros(dp * bits // 8, dtype=np.uint8)
    coset = np.zeros(1, dtype=np.uint16)
    scales = np.zeros(dp // group, dtype=np.uint16)
    csr = None if cs_row is None else _c(cs_row, np.float32)
    lib().orc_encode_row(_ptr(x_bits), _ptr(csr), int(head_dim), int(bits), int(group), int(strict),
                         _ptr(idx), _ptr(coset), _ptr(scales))
    return idx, int(coset[0]), scales


def decode_row(idx, coset, scales, head_dim, bits, group, cs_row=None):
    out = np.zeros(head_dim, dtype=np.uint16)
    csr = None if cs_row is None else _c(cs_row, np.float32)
    lib().orc_decode_row(_ptr(_c(idx, np.uint8)), int(coset), _ptr(_c(scales, np.uint16)), _ptr(csr),
                         int(head_dim), int(bits), int(group), _ptr(out))
    return out


def delta_row(idx, coset, prev_idx, prev_coset, dp, bits):
    idx = _c(idx, np.uint8).copy()
    c = np.array([coset], dtype=np.uint16)
    lib().orc_delta_row(_ptr(idx), _ptr(c), _ptr(_c(prev_idx, np.uint8)), int(prev_coset), int(dp), int(bits))
    return idx, int(c[0])


def undelta_row(idx, coset, prev_idx, prev_coset, dp, bits):
    idx = _c(idx, np.uint8).copy()
    c = np.array([coset], dtype=np.uint16)
    lib().orc_undelta_row(_ptr(idx), _ptr(c), _ptr(_c(prev_idx, np.uint8)), int(prev_coset), int(dp), int(bits))
    return idx, int(c[0])


def code_histogram(idx, coset, head_dim, bits):
    """Counts (274 uint64) of field values, idx bytes and coset bits over the
    record rows idx [rows, Dp*b/8], coset [rows]."""
    idx = _c(idx, np.uint8)
    coset = None if coset is None else _c(coset, np.uint16)
    counts = np.zeros(274, dtype=np.uint64)
    rows = idx.shape[0] if idx.ndim == 2 else 0
    lib().orc_code_histogram(_ptr(idx), _ptr(coset), int(rows), padded_dim(head_dim), int(bits), _ptr(counts))
    return counts
