"""Host-side checks of libnq that need no GPU: the library loads, exports every
symbol include/nq.h declares, and its host-only entry points (layout, RoPE
table, argument validation) behave as specified."""
import contextlib
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nq():
    from e8_lattice_vector_gb300 import build as nqbuild

    nqbuild.build()
    from e8_lattice_vector_gb300 import _lib

    return _lib


def _declared_functions():
    with open(os.path.join(ROOT, "include", "nq.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(nq_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(nq):
    names = _declared_functions()
    assert len(names) >= 6
    L = nq.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(nq.SIGNATURES)


def test_strerror(nq):
    L = nq.lib()
    for s in range(5):
        assert L.nq_strerror(s)
    assert b"unknown" in L.nq_strerror(99)


def _plan(nq, shape, **kw):
    p = dict(key_bits=3, value_bits=2, group_size=64, strict=0, delta_chunk=0, rope_theta=1e4)
    p.update(kw)
    lay = nq.Layout()
    st = nq.lib().nq_plan(ctypes.byref(nq.Shape(*shape)), ctypes.byref(nq.Params(**p)), ctypes.byref(lay))
    return st, lay


@pytest.mark.parametrize("shape,kb,vb,g", [((1, 1, 8, 512, 128), 3, 2, 64), ((2, 2, 3, 77, 96), 3, 2, 32),
                                           ((1, 1, 1, 5, 64), 4, 4, 64), ((3, 1, 2, 100, 128), 2, 2, 128)])
def test_plan_sizes_match_oracle_format(nq, orc, shape, kb, vb, g):
    st, lay = _plan(nq, shape, key_bits=kb, value_bits=vb, group_size=g)
    assert st == 0
    slices = int(np.prod(shape[:3]))
    tp = (shape[3] + 31) // 32 * 32
    rows = slices * tp
    D = shape[4]
    dp = orc.padded_dim(D)
    assert lay.version == 1 and lay.padded_dim == dp and lay.tokens_padded == tp and lay.rows == rows
    x = np.zeros((slices, shape[3], D), np.uint16)
    for off, bits in (("k", kb), ("v", vb)):
        idx, cos_, sc = orc.compress_tensor(x, shape[3], D, bits, g, 0, 0)
        assert getattr(lay, off + "_idx_row_bytes") == idx.shape[1]
        assert lay.scales_per_row == sc.shape[1]
    offs = [lay.k_idx, lay.k_coset, lay.k_scale, lay.v_idx, lay.v_coset, lay.v_scale, lay.total_bytes]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert lay.k_coset - lay.k_idx >= rows * lay.k_idx_row_bytes
    assert lay.total_bytes - lay.v_scale >= rows * lay.scales_per_row * 2


def test_plan_rejects_bad_arguments(nq):
    ok = (1, 1, 8, 64, 128)
    assert _plan(nq, ok)[0] == 0
    assert _plan(nq, (1, 1, 8, 64, 80))[0] == nq.NQ_ERR_UNSUPPORTED
    assert _plan(nq, (1, 1, 8, 64, 256))[0] == nq.NQ_ERR_UNSUPPORTED
    assert _plan(nq, ok, key_bits=1)[0] == nq.NQ_ERR_UNSUPPORTED
    assert _plan(nq, ok, value_bits=5)[0] == nq.NQ_ERR_UNSUPPORTED
    assert _plan(nq, ok, group_size=48)[0] == nq.NQ_ERR_UNSUPPORTED
    assert _plan(nq, (1, 1, 8, 64, 64), group_size=128)[0] == nq.NQ_ERR_UNSUPPORTED
    assert _plan(nq, ok, delta_chunk=40)[0] == nq.NQ_ERR_ARG
    assert _plan(nq, ok, delta_chunk=-32)[0] == nq.NQ_ERR_ARG
    assert _plan(nq, ok, strict=3)[0] == nq.NQ_ERR_ARG
    assert _plan(nq, ok, strict=-1)[0] == nq.NQ_ERR_ARG
    assert _plan(nq, (1, -1, 8, 64, 128))[0] == nq.NQ_ERR_ARG
    assert _plan(nq, ok, rope_theta=float("inf"))[0] == nq.NQ_ERR_ARG
    st, lay = _plan(nq, (0, 1, 8, 64, 128))
    assert st == 0 and lay.rows == 0


def test_compress_validates_before_touching_the_gpu(nq):
    """Error paths return before any CUDA call (so they run without a GPU)."""
    L = nq.lib()
    shape = nq.Shape(1, 1, 8, 64, 128)
    good = nq.Params(2, 2, 64, 0, 0, 1e4)
    p16 = ctypes.c_void_p(16)
    # null pointers
    assert L.nq_compress_kv(None, p16, p16, ctypes.byref(shape), ctypes.byref(good), p16, 1 << 30, None) == nq.NQ_ERR_ARG
    # rope on but no table
    assert L.nq_compress_kv(p16, p16, None, ctypes.byref(shape), ctypes.byref(good), p16, 1 << 30, None) == nq.NQ_ERR_ARG
    # misaligned
    p17 = ctypes.c_void_p(17)
    assert L.nq_compress_kv(p17, p16, p16, ctypes.byref(shape), ctypes.byref(good), p16, 1 << 30, None) == nq.NQ_ERR_ARG
    # output too small
    assert L.nq_compress_kv(p16, p16, p16, ctypes.byref(shape), ctypes.byref(good), p16, 100, None) == nq.NQ_ERR_SIZE
    assert L.nq_decompress_kv(p16, 100, p16, ctypes.byref(shape), ctypes.byref(good), p16, p16, None, 0,
                              None) == nq.NQ_ERR_SIZE
    # with a long delta chain the workspace is required, aligned and large enough
    shape = nq.Shape(1, 1, 8, 4096, 128)
    dlt = nq.Params(2, 2, 64, 0, 4096, 1e4)
    lay = nq.Layout()
    assert L.nq_plan(ctypes.byref(shape), ctypes.byref(dlt), ctypes.byref(lay)) == 0 and lay.workspace_bytes > 0
    big = 1 << 30
    sh, dp = ctypes.byref(shape), ctypes.byref(dlt)
    assert L.nq_decompress_kv(p16, big, p16, sh, dp, p16, p16, None, big, None) == nq.NQ_ERR_ARG
    assert L.nq_decompress_kv(p16, big, p16, sh, dp, p16, p16, ctypes.c_void_p(24), big, None) == nq.NQ_ERR_ARG
    assert L.nq_decompress_kv(p16, big, p16, sh, dp, p16, p16, p16, lay.workspace_bytes - 1, None) == nq.NQ_ERR_SIZE
    bad = nq.Params(2, 7, 64, 0, 0, 1e4)
    assert L.nq_compress_kv(p16, p16, p16, ctypes.byref(shape), ctypes.byref(bad), p16, 1 << 30, None) == nq.NQ_ERR_UNSUPPORTED
    # empty tensors are a no-op
    empty = nq.Shape(1, 1, 8, 0, 128)
    assert L.nq_compress_kv(None, None, None, ctypes.byref(empty), ctypes.byref(good), None, 0, None) == 0
    assert L.nq_e8_nearest(None, None, 0, 1, 2, None) == 0
    # the histogram validates before its first CUDA call
    cnt = ctypes.c_void_p(64)
    assert L.nq_code_histogram(p16, 1 << 30, sh := ctypes.byref(shape), ctypes.byref(good), None, None) == nq.NQ_ERR_ARG
    assert L.nq_code_histogram(p16, 1 << 30, sh, ctypes.byref(good), ctypes.c_void_p(12), None) == nq.NQ_ERR_ARG
    assert L.nq_code_histogram(p17, 1 << 30, sh, ctypes.byref(good), cnt, None) == nq.NQ_ERR_ARG
    assert L.nq_code_histogram(p16, 100, sh, ctypes.byref(good), cnt, None) == nq.NQ_ERR_SIZE
    # the one-pass round trip validates the same way
    sh = ctypes.byref(shape)
    assert L.nq_roundtrip_kv(p16, p16, p16, sh, ctypes.byref(good), None, p16, None) == nq.NQ_ERR_ARG
    assert L.nq_roundtrip_kv(p16, p16, None, sh, ctypes.byref(good), p16, p16, None) == nq.NQ_ERR_ARG
    assert L.nq_roundtrip_kv(p16, p16, p16, sh, ctypes.byref(good), p16, p17, None) == nq.NQ_ERR_ARG
    assert L.nq_roundtrip_kv(p16, p16, p16, sh, ctypes.byref(bad), p16, p16, None) == nq.NQ_ERR_UNSUPPORTED
    assert L.nq_roundtrip_kv(None, None, None, ctypes.byref(empty), ctypes.byref(good), None, None, None) == 0
    assert L.nq_e8_nearest(p16, p16, 5, 1, 5, None) == nq.NQ_ERR_UNSUPPORTED
    assert L.nq_e8_nearest(p16, p16, -1, 1, 2, None) == nq.NQ_ERR_ARG


@pytest.mark.parametrize("T,D,theta", [(512, 128, 1e4), (2048, 96, 1e4), (300, 128, 5e5), (1000, 64, 1e6)])
def test_rope_table_equals_oracle_bit_for_bit(nq, orc, T, D, theta):
    host = np.zeros((D // 4, T, 4), np.float32)
    st = nq.lib().nq_rope_table(None, T, D, theta, host.ctypes.data_as(ctypes.c_void_p))
    assert st == 0
    ref = orc.rope_table(T, D, theta)  # [T, D/2, (cos, sin)]
    got = host.transpose(1, 0, 2).reshape(T, D // 2, 2)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_rope_table_positions_and_errors(nq, orc):
    pos = np.array([5, 0, 131071, 77], np.int32)
    host = np.zeros((32, 4, 4), np.float32)
    L = nq.lib()
    assert L.nq_rope_table(pos.ctypes.data_as(ctypes.c_void_p), 4, 128, 1e6, host.ctypes.data_as(ctypes.c_void_p)) == 0
    assert np.array_equal(host.transpose(1, 0, 2).reshape(4, 64, 2), orc.rope_table(4, 128, 1e6, positions=pos))
    assert L.nq_rope_table(None, 4, 127, 1e4, host.ctypes.data_as(ctypes.c_void_p)) == nq.NQ_ERR_ARG
    assert L.nq_rope_table(None, 4, 128, 0.0, host.ctypes.data_as(ctypes.c_void_p)) == nq.NQ_ERR_ARG
    assert L.nq_rope_table(None, 4, 128, 1e4, None) == nq.NQ_ERR_ARG


def test_package_has_no_cpu_path():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "e8_lattice_vector_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert "import oracle" not in src and "from oracle" not in src and "nq_oracle" not in src, f


def test_plan_layers_parts(nq):
    """One 256-aligned part per layer: the single-layer buffer of the layer's bit
    widths, or the layer's K and V in fp16."""
    import e8_lattice_vector_gb300 as pkg
    from e8_lattice_vector_gb300 import CodecParams

    shape = (5, 2, 3, 77, 96)
    p = CodecParams(3, 2, 64, False, 64, 1e4)
    table = [(0, 0), (3, 2), (2, 2), (4, 3), (0, 0)]
    offs, total = pkg.plan_layers(shape, p, table)
    one = (1,) + shape[1:]
    raw = 2 * 2 * 3 * 77 * 96 * 2
    expect, off = [], 0
    for kb, vb in table:
        expect.append(off)
        size = raw if kb == 0 else int(pkg.plan(one, CodecParams(kb, vb, 64, False, 64, 1e4)).total_bytes)
        off = (off + size + 255) // 256 * 256
    assert offs == expect and total == off
    assert pkg.layer_profile(6, 3, 2, protect_boundary=2) == [(0, 0), (0, 0), (3, 2), (3, 2), (0, 0), (0, 0)]


def test_layers_validate_before_touching_the_gpu(nq):
    L = nq.lib()
    shape = nq.Shape(2, 1, 8, 64, 128)
    good = nq.Params(2, 2, 64, 0, 0, 1e4)
    offs = (ctypes.c_uint64 * 2)()
    total = ctypes.c_uint64()
    ok = (nq.LayerBits * 2)(nq.LayerBits(3, 2), nq.LayerBits(0, 0))
    half = (nq.LayerBits * 2)(nq.LayerBits(3, 0), nq.LayerBits(2, 2))
    sh, pr = ctypes.byref(shape), ctypes.byref(good)
    ws = ctypes.c_uint64(7)
    assert L.nq_plan_layers(sh, pr, ok, offs, ctypes.byref(total), ctypes.byref(ws)) == 0 and total.value > 0
    assert ws.value == 0  # no delta, no workspace
    assert L.nq_plan_layers(sh, pr, ok, offs, ctypes.byref(total), None) == 0
    assert L.nq_plan_layers(sh, pr, half, offs, ctypes.byref(total), None) == nq.NQ_ERR_UNSUPPORTED
    assert L.nq_plan_layers(sh, pr, None, offs, ctypes.byref(total), None) == nq.NQ_ERR_ARG
    p16 = ctypes.c_void_p(16)
    assert L.nq_compress_kv_layers(None, p16, p16, sh, pr, ok, p16, 1 << 30, None) == nq.NQ_ERR_ARG
    assert L.nq_compress_kv_layers(p16, p16, p16, sh, pr, ok, p16, 100, None) == nq.NQ_ERR_SIZE
    assert L.nq_decompress_kv_layers(p16, 100, p16, sh, pr, ok, p16, p16, None, 0, None) == nq.NQ_ERR_SIZE
    dlt = nq.Params(2, 2, 64, 0, 4096, 1e4)
    sh = ctypes.byref(nq.Shape(2, 1, 8, 4096, 128))
    assert L.nq_plan_layers(sh, ctypes.byref(dlt), ok, offs, ctypes.byref(total), ctypes.byref(ws)) == 0
    assert ws.value > 0  # the compressed layer's workspace
    assert L.nq_decompress_kv_layers(p16, 1 << 30, p16, sh, ctypes.byref(dlt), ok, p16, p16, p16, ws.value - 1,
                                     None) == nq.NQ_ERR_SIZE
    assert L.nq_roundtrip_kv_layers(p16, p16, p16, sh, pr, half, p16, p16, None) == nq.NQ_ERR_UNSUPPORTED
    empty = nq.Shape(0, 1, 8, 64, 128)
    assert L.nq_compress_kv_layers(None, None, None, ctypes.byref(empty), pr, None, None, 0, None) == 0
    # a kept first layer: the missing or misaligned RoPE table is refused before its copies are enqueued
    p17 = ctypes.c_void_p(17)
    for table in (None, p17):
        assert L.nq_compress_kv_layers(p16, p16, table, sh, pr, ok_kept_first := (nq.LayerBits * 2)(
            nq.LayerBits(0, 0), nq.LayerBits(2, 2)), p16, 1 << 30, None) == nq.NQ_ERR_ARG
        assert L.nq_decompress_kv_layers(p16, 1 << 30, table, sh, pr, ok_kept_first, p16, p16, None, 0,
                                         None) == nq.NQ_ERR_ARG
        assert L.nq_roundtrip_kv_layers(p16, p16, table, sh, pr, ok_kept_first, p16, p16, None) == nq.NQ_ERR_ARG


def test_plan_joint_format_has_no_coset_words(nq):
    shape = (2, 1, 4, 100, 128)
    st1, l1 = _plan(nq, shape, strict=1)
    st2, l2 = _plan(nq, shape, strict=2)
    assert st1 == 0 and st2 == 0
    assert l2.k_scale == l2.k_coset and l2.v_scale == l2.v_coset
    assert l2.k_idx_row_bytes == l1.k_idx_row_bytes  # 8b bits per block either way
    rows = l1.rows
    assert l1.total_bytes - l2.total_bytes >= 2 * (rows * 2 // 256 * 256)


class _FakeCuda:
    """Stand-in for a CUDA tensor: the binding's argument checks read only
    these attributes, and every case below is rejected before any CUDA call."""

    def __init__(self, shape, dtype, device="cuda:0", contiguous=True):
        import torch

        self.shape = torch.Size(shape)
        self.dtype = dtype
        self.device = torch.device(device)
        self.is_cuda = True
        self._contiguous = contiguous

    def dim(self):
        return len(self.shape)

    def is_contiguous(self):
        return self._contiguous

    def numel(self):
        n = 1
        for v in self.shape:
            n *= v
        return n

    def data_ptr(self):
        return 256


def test_binding_rejects_mismatched_outputs_before_the_gpu():
    import torch

    import e8_lattice_vector_gb300 as nq
    from e8_lattice_vector_gb300 import CodecParams, codec

    p = CodecParams(2, 2, 64, 0, 0, 0.0)
    shp = (2, 1, 8, 64, 128)
    K = _FakeCuda(shp, torch.float16)
    buf = _FakeCuda((1 << 20,), torch.uint8)

    def raises(fn, text):
        with pytest.raises(ValueError, match=text):
            fn()

    raises(lambda: nq.compress_kv(K, _FakeCuda((2, 1, 8, 32, 128), torch.float16), p), "V has shape")
    raises(lambda: nq.compress_kv(K, _FakeCuda(shp, torch.float16, "cuda:1"), p), "V is on")
    raises(lambda: nq.compress_kv(K, K, p, out=_FakeCuda((1 << 20,), torch.float32)), "out must be")
    raises(lambda: nq.compress_kv(K, K, p, out=_FakeCuda((1 << 20,), torch.uint8, "cuda:1")), "out is on")
    small = _FakeCuda((2, 1, 8, 32, 128), torch.float16)
    raises(lambda: nq.decompress_kv(buf, shp, p, K_out=small, V_out=K), "K_out has shape")
    raises(lambda: nq.decompress_kv(buf, shp, p, K_out=K, V_out=_FakeCuda(shp, torch.float16, "cuda:1")),
           "V_out is on")
    raises(lambda: nq.decompress_kv(_FakeCuda((1 << 20,), torch.int32), shp, p, K_out=K, V_out=K), "buf must be")
    raises(lambda: nq.decompress_kv(buf, shp, p, K_out=_FakeCuda(shp, torch.float16, contiguous=False), V_out=K),
           "K_out must be")
    raises(lambda: nq.roundtrip_kv(K, K, p, K_out=small, V_out=K), "K_out has shape")
    table = [(2, 2), (0, 0)]
    raises(lambda: nq.roundtrip_kv_layers(K, small, p, table), "V has shape")
    raises(lambda: nq.decompress_kv_layers(buf, shp, p, table, K_out=K, V_out=small), "V_out has shape")
    raises(lambda: nq.code_histogram(_FakeCuda((64,), torch.float16), shp, p), "buf must be")
    # 4-D shapes mean batch 1; anything else is refused
    assert codec._norm_shape((2, 8, 64, 128)) == (2, 1, 8, 64, 128)
    raises(lambda: codec._norm_shape((8, 64, 128)), "shape must be")
    # a 4-D K with a 4-D output of the same cache passes the shape check (then stops at V's device)
    K4 = _FakeCuda((2, 8, 64, 128), torch.float16)
    raises(lambda: nq.roundtrip_kv(K4, _FakeCuda((2, 8, 64, 128), torch.float16, "cuda:1"), p), "V is on")


def test_binding_passes_valid_calls_through_to_the_library(monkeypatch):
    """The call shapes the benchmark, smoke check and parity tests use (5-D and
    4-D caches, per-layer slices as outputs, in-place round trips) pass the
    argument checks and reach the C entry point once each."""
    import torch

    import e8_lattice_vector_gb300 as nq
    from e8_lattice_vector_gb300 import CodecParams, _lib, codec

    real = _lib.lib()
    calls = []

    class _Recorder:
        def __getattr__(self, name):
            if name.startswith("nq_plan"):
                return getattr(real, name)  # host-only sizing

            def entry(*args):
                calls.append(name)
                return 0

            return entry

    monkeypatch.setattr(_lib, "lib", lambda: _Recorder())
    monkeypatch.setattr(codec, "_stream_handle", lambda device: None)
    monkeypatch.setattr(codec, "_on", lambda device: contextlib.nullcontext())
    p = CodecParams(2, 2, 64, 0, 0, 0.0)
    shp = (2, 1, 8, 64, 128)
    K, V = _FakeCuda(shp, torch.float16), _FakeCuda(shp, torch.float16)
    lay = nq.plan(shp, p)
    buf = _FakeCuda((int(lay.total_bytes),), torch.uint8)
    nq.compress_kv(K, V, p, out=buf)
    nq.decompress_kv(buf, shp, p, K_out=K, V_out=V)
    nq.roundtrip_kv(K, V, p, K_out=K, V_out=V)
    lshape = (1,) + shp[1:]  # one layer of the cache into a slice of the outputs
    lbuf = _FakeCuda((int(nq.plan(lshape, p).total_bytes),), torch.uint8)
    nq.compress_kv(_FakeCuda(lshape, torch.float16), _FakeCuda(lshape, torch.float16), p, out=lbuf)
    nq.decompress_kv(lbuf, lshape, p, K_out=_FakeCuda(lshape, torch.float16), V_out=_FakeCuda(lshape, torch.float16))
    K4 = _FakeCuda((2, 8, 64, 128), torch.float16)
    nq.roundtrip_kv(K4, _FakeCuda((2, 8, 64, 128), torch.float16), p, K_out=K4, V_out=_FakeCuda(shp, torch.float16))
    table = [(2, 2), (0, 0)]
    _, total = nq.plan_layers(shp, p, table)
    nbuf = _FakeCuda((total,), torch.uint8)
    nq.compress_kv_layers(K, V, p, table, out=nbuf)
    nq.decompress_kv_layers(nbuf, shp, p, table, K_out=K, V_out=V)
    nq.roundtrip_kv_layers(K, V, p, table, K_out=K, V_out=V)
    nq.code_histogram(buf, shp, p, counts=_FakeCuda((2, _lib.NQ_HIST_BINS), torch.int64))
    assert calls == ["nq_compress_kv", "nq_decompress_kv", "nq_roundtrip_kv", "nq_compress_kv", "nq_decompress_kv",
                     "nq_roundtrip_kv", "nq_compress_kv_layers", "nq_decompress_kv_layers", "nq_roundtrip_kv_layers",
                     "nq_code_histogram"]


def test_binding_rejects_a_rope_table_on_another_device():
    """The RoPE table must live on the call's device (a table on another GPU
    would be read across devices by the kernels)."""
    import torch

    import e8_lattice_vector_gb300 as nq
    from e8_lattice_vector_gb300 import CodecParams

    p = CodecParams(2, 2, 64, 0, 0, 1e4)
    shp = (2, 1, 8, 64, 128)
    K = _FakeCuda(shp, torch.float16, "cuda:1")
    table = nq.RopeTable(None, _FakeCuda((32, 64, 4), torch.float32, "cuda:0"), 64, 128, 1e4)
    buf = _FakeCuda((1 << 24,), torch.uint8, "cuda:1")
    for fn in (lambda: nq.compress_kv(K, K, p, table, out=buf),
               lambda: nq.decompress_kv(buf, shp, p, table, K_out=K, V_out=K),
               lambda: nq.roundtrip_kv(K, K, p, table, K_out=K, V_out=K),
               lambda: nq.roundtrip_kv_layers(K, K, p, [(2, 2), (0, 0)], table, K_out=K, V_out=K)):
        with pytest.raises(ValueError, match="RopeTable is on cuda:0; the call runs on cuda:1"):
            fn()


def test_workspace_plan_and_status_without_a_gpu(nq):
    """Decompression walks delta chains in runs of up to 32 record tiles (32
    rows; 16 at head_dim 64); only chains longer than one run need the
    workspace: per run a slot of the idx row words plus a coset word for its
    total and one for its starting sum.  nq_get_status answers through the C
    ABI without a GPU (an error status, not a crash)."""
    L = nq.lib()
    for D, rows, kb, vb, chunk in ((128, 32, 3, 2, 96), (128, 32, 3, 2, 1024), (96, 32, 2, 2, 2048),
                                   (64, 16, 4, 2, 4096)):
        shape = nq.Shape(2, 1, 3, 1000, D)
        lay = nq.Layout()
        assert L.nq_plan(ctypes.byref(shape), ctypes.byref(nq.Params(kb, vb, 64, 0, 0, 1e4)), ctypes.byref(lay)) == 0
        assert lay.workspace_bytes == 0
        assert L.nq_plan(ctypes.byref(shape), ctypes.byref(nq.Params(kb, vb, 64, 0, chunk, 1e4)),
                         ctypes.byref(lay)) == 0
        tiles = (1000 + rows - 1) // rows
        tpc = chunk // rows
        gpc = (min(tpc, tiles) + 31) // 32
        if gpc == 1:
            assert lay.workspace_bytes == 0, (D, chunk)
            continue
        groups = 6 * ((tiles + tpc - 1) // tpc) * gpc
        dp = 64 if D == 64 else 128
        slot = (dp * max(kb, vb) // 32 + 1 + 3) // 4 * 4 * 4
        assert lay.workspace_bytes >= 2 * groups * slot
        assert lay.workspace_bytes % 256 == 0
    import torch

    assert L.nq_get_status(None) == (nq.NQ_OK if torch.cuda.is_available() else nq.NQ_ERR_CUDA)
