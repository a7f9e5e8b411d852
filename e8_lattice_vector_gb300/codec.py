"""Python face of libnq: E8 lattice KV-cache compression on the GPU.

    params = CodecParams(key_bits=2, value_bits=2, strict=False, rope_theta=5e5)
    rope = RopeTable.build(tokens, head_dim, params.rope_theta, device="cuda")
    buf = compress_kv(K, V, params, rope)           # uint8 device buffer
    K2, V2 = decompress_kv(buf, shape_of(K), params, rope)

K and V are contiguous fp16 CUDA tensors [layers, batch, kv_heads, tokens,
head_dim] (a 4-D [layers, kv_heads, tokens, head_dim] tensor means batch 1).
All work is enqueued on the current torch CUDA stream.
"""
import ctypes
from dataclasses import dataclass

import torch

from . import _lib

__all__ = ["CodecParams", "RopeTable", "plan", "shape_of", "compress_kv", "decompress_kv",
           "e8_nearest", "sections", "workspace", "get_status"]


@dataclass(frozen=True)
class CodecParams:
    key_bits: int = 2
    value_bits: int = 2
    group_size: int = 64
    strict: int = 0  # 0 relaxed, 1 strict, 2 strict in the joint 8b-bit format (no coset words)
    delta_chunk: int = 0
    rope_theta: float = 1e4

    def c(self):
        return _lib.Params(self.key_bits, self.value_bits, self.group_size, int(self.strict),
                           self.delta_chunk, float(self.rope_theta))


def shape_of(x):
    """nq shape tuple (layers, batch, kv_heads, tokens, head_dim) of a K/V tensor."""
    if x.dim() == 4:
        L, H, T, D = x.shape
        return (L, 1, H, T, D)
    if x.dim() == 5:
        return tuple(x.shape)
    raise ValueError("K/V must be 4-D [L,H,T,D] or 5-D [L,B,H,T,D], got %s" % (tuple(x.shape),))


def _cshape(shape):
    return _lib.Shape(*[int(v) for v in shape])


def plan(shape, params):
    lay = _lib.Layout()
    _lib.check("nq_plan", _lib.lib().nq_plan(ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), ctypes_ref(lay)))
    return lay


def ctypes_ref(obj):
    return ctypes.byref(obj)


def _stream_handle(device):
    return ctypes_void(torch.cuda.current_stream(device).cuda_stream)


def ctypes_void(v):
    return ctypes.c_void_p(int(v))


class RopeTable:
    """Device copy of the (cos, sin) table that nq_rope_table builds on the host
    for given positions, theta and head_dim.  Build once, reuse for every call
    on those tokens."""

    def __init__(self, host, device_tensor, tokens, head_dim, theta):
        self.host = host
        self.device = device_tensor
        self.tokens, self.head_dim, self.theta = tokens, head_dim, theta

    @staticmethod
    def host_table(tokens, head_dim, theta, positions=None):
        """[head_dim/4, tokens, 4] float32: plane q holds (cos, sin) of pairs 2q
        and 2q+1 for every token."""
        host = torch.empty((head_dim // 4, tokens, 4), dtype=torch.float32)
        pos = None
        if positions is not None:
            pos = torch.as_tensor(positions, dtype=torch.int32).contiguous()
            if pos.numel() != tokens:
                raise ValueError("positions must have `tokens` entries")
        st = _lib.lib().nq_rope_table(None if pos is None else ctypes_void(pos.data_ptr()), int(tokens),
                                      int(head_dim), float(theta), ctypes_void(host.data_ptr()))
        _lib.check("nq_rope_table", st)
        return host

    @classmethod
    def build(cls, tokens, head_dim, theta, positions=None, device="cuda"):
        host = cls.host_table(tokens, head_dim, theta, positions)
        return cls(host, host.to(device), tokens, head_dim, theta)

    def pairs(self):
        """The table as [tokens, head_dim/2, (cos, sin)] (numpy), token-major."""
        h = self.host.numpy()
        return h.transpose(1, 0, 2).reshape(self.tokens, self.head_dim // 2, 2)


def _rope_ptr(rope, params, tokens, head_dim, device):
    if params.rope_theta <= 0:
        return None
    if rope is None:
        raise ValueError("rope_theta > 0 needs a RopeTable for these tokens")
    if rope.tokens != tokens or rope.head_dim != head_dim or rope.theta != params.rope_theta:
        raise ValueError("RopeTable (%d tokens, head_dim %d, theta %g) does not match the call"
                         % (rope.tokens, rope.head_dim, rope.theta))
    if rope.device.device != device:
        raise ValueError("RopeTable is on %s; the call runs on %s" % (rope.device.device, device))
    return ctypes_void(rope.device.data_ptr())


def _on(device):
    """The library sizes its grids and launches on the current device: make it
    the tensors' device for the duration of a call."""
    return torch.cuda.device(device)


def _call(device, name, *args):
    """One library call with `device` current (the library sizes its grids and
    sets kernel attributes on the current device); raises on a bad status."""
    with _on(device):
        st = getattr(_lib.lib(), name)(*args)
    _lib.check(name, st)


def _check_kv(x, name):
    if not (x.is_cuda and x.dtype == torch.float16 and x.is_contiguous()):
        raise ValueError("%s must be a contiguous fp16 CUDA tensor" % name)


def _check_buf(buf, name="buf"):
    if not (buf.is_cuda and buf.dtype == torch.uint8 and buf.is_contiguous()):
        raise ValueError("%s must be a contiguous uint8 CUDA tensor" % name)


def _check_like(x, shape, device, name):
    """An fp16 tensor the library writes or reads as `shape` on `device`."""
    _check_kv(x, name)
    if shape_of(x) != shape:
        raise ValueError("%s has shape %s; the call's shape is %s" % (name, shape_of(x), shape))
    if x.device != device:
        raise ValueError("%s is on %s; the call runs on %s" % (name, x.device, device))


def _norm_shape(shape):
    """(layers, batch, kv_heads, tokens, head_dim); a 4-D shape means batch 1."""
    shape = tuple(int(v) for v in shape)
    if len(shape) == 4:
        return (shape[0], 1, shape[1], shape[2], shape[3])
    if len(shape) != 5:
        raise ValueError("shape must be [L,B,H,T,D] or [L,H,T,D], got %s" % (shape,))
    return shape


def _kv_shape(K, V):
    _check_kv(K, "K")
    shape = shape_of(K)
    _check_like(V, shape, K.device, "V")
    return shape


def compress_kv(K, V, params, rope=None, out=None):
    """Compress K and V; returns (or fills) a uint8 device buffer of
    plan(...).total_bytes bytes."""
    shape = _kv_shape(K, V)
    lay = plan(shape, params)
    if out is None:
        out = torch.empty(max(int(lay.total_bytes), 16), dtype=torch.uint8, device=K.device)
    _check_buf(out, "out")
    if out.device != K.device:
        raise ValueError("out is on %s; the call runs on %s" % (out.device, K.device))
    rp = _rope_ptr(rope, params, shape[3], shape[4], K.device)
    _call(K.device, "nq_compress_kv", ctypes_void(K.data_ptr()), ctypes_void(V.data_ptr()), rp,
          ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), ctypes_void(out.data_ptr()), int(out.numel()),
          _stream_handle(K.device))
    return out


def workspace(nbytes, device):
    """A device workspace of `nbytes` bytes (None when nothing is needed): the
    scratch that decompression with a temporal delta uses.  Reuse it across
    calls on one stream."""
    if nbytes <= 0:
        return None
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def _ws_args(ws, need, device):
    if need <= 0:
        return None, 0
    if ws is None:
        raise ValueError("this call needs a workspace of %d bytes" % need)
    _check_buf(ws, "workspace")
    if ws.device != device:
        raise ValueError("workspace is on %s; the call runs on %s" % (ws.device, device))
    if ws.numel() < need:
        raise ValueError("workspace has %d bytes; the call needs %d" % (ws.numel(), need))
    return ctypes_void(ws.data_ptr()), int(ws.numel())


def decompress_kv(buf, shape, params, rope=None, K_out=None, V_out=None, ws=None):
    """Decompress a buffer produced by compress_kv; returns (K, V) fp16 tensors
    of `shape` ([L,B,H,T,D]).  ws: the workspace (see workspace()) that a
    temporal delta needs, allocated here when not given."""
    shape = _norm_shape(shape)
    _check_buf(buf)
    if K_out is None:
        K_out = torch.empty(shape, dtype=torch.float16, device=buf.device)
    if V_out is None:
        V_out = torch.empty(shape, dtype=torch.float16, device=buf.device)
    _check_like(K_out, shape, buf.device, "K_out")
    _check_like(V_out, shape, buf.device, "V_out")
    rp = _rope_ptr(rope, params, shape[3], shape[4], buf.device)
    need = int(plan(shape, params).workspace_bytes)
    if ws is None and need > 0:
        ws = workspace(need, buf.device)
    wp, wn = _ws_args(ws, need, buf.device)
    _call(buf.device, "nq_decompress_kv", ctypes_void(buf.data_ptr()), int(buf.numel()), rp,
          ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), ctypes_void(K_out.data_ptr()),
          ctypes_void(V_out.data_ptr()), wp, wn, _stream_handle(buf.device))
    return K_out, V_out


def decompress_kv_static(buf, shape, params, rope, K_out, V_out):
    """decompress_kv through nq_decompress_kv_static: the delta scratch is the
    library's static device array, so nothing is allocated, here or in the
    library (K_out and V_out are required).  Raises NQError (NQ_ERR_SIZE) when
    the call needs more scratch than the array holds
    (plan(...).workspace_bytes > static_workspace_bytes())."""
    shape = _norm_shape(shape)
    _check_buf(buf)
    _check_like(K_out, shape, buf.device, "K_out")
    _check_like(V_out, shape, buf.device, "V_out")
    rp = _rope_ptr(rope, params, shape[3], shape[4], buf.device)
    _call(buf.device, "nq_decompress_kv_static", ctypes_void(buf.data_ptr()), int(buf.numel()), rp,
          ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), ctypes_void(K_out.data_ptr()),
          ctypes_void(V_out.data_ptr()), _stream_handle(buf.device))
    return K_out, V_out


def static_workspace_bytes():
    """Size of the static scratch behind decompress_kv_static (the header's
    NQ_STATIC_WORKSPACE_BYTES)."""
    return 8 << 20


def get_status(device=None):
    """The deferred status of the work enqueued on the device's current
    stream (waits for it): raises NQError when the stream or an earlier launch
    failed."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _call(dev, "nq_get_status", _stream_handle(dev))


def roundtrip_kv(K, V, params, rope=None, K_out=None, V_out=None):
    """decompress_kv(compress_kv(K, V)) in one pass, without the compressed
    buffer; returns (K_out, V_out).  Passing K_out=K, V_out=V reconstructs the
    cache in place."""
    shape = _kv_shape(K, V)
    if K_out is None:
        K_out = torch.empty_like(K)
    if V_out is None:
        V_out = torch.empty_like(V)
    _check_like(K_out, shape, K.device, "K_out")
    _check_like(V_out, shape, K.device, "V_out")
    rp = _rope_ptr(rope, params, shape[3], shape[4], K.device)
    _call(K.device, "nq_roundtrip_kv", ctypes_void(K.data_ptr()), ctypes_void(V.data_ptr()), rp,
          ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), ctypes_void(K_out.data_ptr()),
          ctypes_void(V_out.data_ptr()), _stream_handle(K.device))
    return K_out, V_out


def _layer_table(layer_bits, layers):
    lb = list(layer_bits)
    if len(lb) != layers:
        raise ValueError("layer_bits needs one (key_bits, value_bits) entry per layer")
    arr = (_lib.LayerBits * max(layers, 1))()
    for i, (kb, vb) in enumerate(lb):
        arr[i].key_bits, arr[i].value_bits = int(kb), int(vb)
    return arr


def layer_profile(layers, key_bits=3, value_bits=2, protect_boundary=0):
    """A per-layer table: the first and last `protect_boundary` layers kept in
    fp16 ((0, 0)), the others at (key_bits, value_bits)."""
    keep = set(range(min(protect_boundary, layers))) | set(range(max(layers - protect_boundary, 0), layers))
    return [(0, 0) if l in keep else (key_bits, value_bits) for l in range(layers)]


def _plan_layers3(shape, params, layer_bits):
    shape = _norm_shape(shape)
    table = _layer_table(layer_bits, shape[0])
    offs = (ctypes.c_uint64 * max(shape[0], 1))()
    total = ctypes.c_uint64(0)
    ws = ctypes.c_uint64(0)
    st = _lib.lib().nq_plan_layers(ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), table, offs,
                                   ctypes.byref(total), ctypes.byref(ws))
    _lib.check("nq_plan_layers", st)
    return [int(offs[i]) for i in range(shape[0])], int(total.value), int(ws.value)


def plan_layers(shape, params, layer_bits):
    """(offsets per layer, total bytes) of the per-layer buffer."""
    offs, total, _ = _plan_layers3(shape, params, layer_bits)
    return offs, total


def compress_kv_layers(K, V, params, layer_bits, rope=None, out=None):
    """Compress with a per-layer table of (key_bits, value_bits); (0, 0) keeps
    a layer in fp16.  Returns (or fills) the uint8 device buffer."""
    shape = _kv_shape(K, V)
    _, total = plan_layers(shape, params, layer_bits)
    if out is None:
        out = torch.empty(max(total, 16), dtype=torch.uint8, device=K.device)
    _check_buf(out, "out")
    if out.device != K.device:
        raise ValueError("out is on %s; the call runs on %s" % (out.device, K.device))
    rp = _rope_ptr(rope, params, shape[3], shape[4], K.device)
    _call(K.device, "nq_compress_kv_layers", ctypes_void(K.data_ptr()), ctypes_void(V.data_ptr()), rp,
          ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), _layer_table(layer_bits, shape[0]),
          ctypes_void(out.data_ptr()), int(out.numel()), _stream_handle(K.device))
    return out


def decompress_kv_layers(buf, shape, params, layer_bits, rope=None, K_out=None, V_out=None, ws=None):
    shape = _norm_shape(shape)
    _check_buf(buf)
    if K_out is None:
        K_out = torch.empty(shape, dtype=torch.float16, device=buf.device)
    if V_out is None:
        V_out = torch.empty(shape, dtype=torch.float16, device=buf.device)
    _check_like(K_out, shape, buf.device, "K_out")
    _check_like(V_out, shape, buf.device, "V_out")
    rp = _rope_ptr(rope, params, shape[3], shape[4], buf.device)
    _, _, need = _plan_layers3(shape, params, layer_bits)
    if ws is None and need > 0:
        ws = workspace(need, buf.device)
    wp, wn = _ws_args(ws, need, buf.device)
    _call(buf.device, "nq_decompress_kv_layers", ctypes_void(buf.data_ptr()), int(buf.numel()), rp,
          ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), _layer_table(layer_bits, shape[0]),
          ctypes_void(K_out.data_ptr()), ctypes_void(V_out.data_ptr()), wp, wn, _stream_handle(buf.device))
    return K_out, V_out


def roundtrip_kv_layers(K, V, params, layer_bits, rope=None, K_out=None, V_out=None):
    shape = _kv_shape(K, V)
    K_out = torch.empty_like(K) if K_out is None else K_out
    V_out = torch.empty_like(V) if V_out is None else V_out
    _check_like(K_out, shape, K.device, "K_out")
    _check_like(V_out, shape, K.device, "V_out")
    rp = _rope_ptr(rope, params, shape[3], shape[4], K.device)
    _call(K.device, "nq_roundtrip_kv_layers", ctypes_void(K.data_ptr()), ctypes_void(V.data_ptr()), rp,
          ctypes_ref(_cshape(shape)), ctypes_ref(params.c()), _layer_table(layer_bits, shape[0]),
          ctypes_void(K_out.data_ptr()), ctypes_void(V_out.data_ptr()), _stream_handle(K.device))
    return K_out, V_out


def code_histogram(buf, shape, params, counts=None):
    """Symbol counts of a compressed buffer: int64 device tensor [2, 274] (K, V)
    of field values [0, 16), idx bytes [16, 272) and coset bits [272, 274)."""
    shape = _norm_shape(shape)
    _check_buf(buf)
    if counts is None:
        counts = torch.empty((2, _lib.NQ_HIST_BINS), dtype=torch.int64, device=buf.device)
    if not (counts.is_cuda and counts.dtype == torch.int64 and counts.is_contiguous()
            and counts.numel() == 2 * _lib.NQ_HIST_BINS):
        raise ValueError("counts must be a contiguous int64 CUDA tensor of 2 * 274 entries")
    _call(buf.device, "nq_code_histogram", ctypes_void(buf.data_ptr()), int(buf.numel()), ctypes_ref(_cshape(shape)),
          ctypes_ref(params.c()), ctypes_void(counts.data_ptr()), _stream_handle(buf.device))
    return counts


def e8_nearest(u, strict, bits):
    """Nearest E8 codebook point of each 8-block of a float32 CUDA tensor [..., 8]."""
    if not (u.is_cuda and u.dtype == torch.float32 and u.is_contiguous() and u.shape[-1] == 8):
        raise ValueError("u must be a contiguous float32 CUDA tensor [..., 8]")
    out = torch.empty_like(u)
    _call(u.device, "nq_e8_nearest", ctypes_void(u.data_ptr()), ctypes_void(out.data_ptr()), u.numel() // 8,
          int(bool(strict)), int(bits), _stream_handle(u.device))
    return out


def sections(buf, lay, tokens=None):
    """Views of the six sections of a compressed buffer (uint8 idx rows, int16
    coset words, fp16 scales), following the layout from plan().  Rows are
    record rows (slices * tokens_padded); with `tokens` given, the views are
    [slices, tokens, ...] with the padding rows dropped."""
    rows = int(lay.rows)
    tp = int(lay.tokens_padded)

    def view(off, nbytes):
        return buf[int(off): int(off) + nbytes]

    def shape(x):
        if tokens is None or tp == 0:
            return x
        return x.view(rows // tp, tp, *x.shape[1:])[:, :tokens]

    out = {}
    for t, rb in (("k", int(lay.k_idx_row_bytes)), ("v", int(lay.v_idx_row_bytes))):
        out[t + "_idx"] = shape(view(getattr(lay, t + "_idx"), rows * rb).view(rows, rb))
        # the joint format (strict = 2) has an empty coset section
        has_coset = int(getattr(lay, t + "_scale")) - int(getattr(lay, t + "_coset")) >= rows * 2
        nc = rows if has_coset else 0
        cos = view(getattr(lay, t + "_coset"), nc * 2).view(torch.int16)
        out[t + "_coset"] = shape(cos) if has_coset else cos
        spr = int(lay.scales_per_row)
        out[t + "_scale"] = shape(view(getattr(lay, t + "_scale"), rows * spr * 2).view(torch.float16).view(rows, spr))
    return out
