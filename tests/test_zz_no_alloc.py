"""nq_decompress_kv_static (delta scratch in a static device array, no
allocation) against nq_decompress_kv (caller workspace): the same outputs,
bit for bit, on two calls in a row.  Collected last on purpose: it must pass
after every other test has used the library on the same device, as well as
alone."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (shape, key_bits, value_bits, strict, delta_chunk, rope_theta, seed): single
# delta chains longer than 32 record tiles, so the static scratch is used
CASES = [
    ((1, 1, 3, 3000, 128), 3, 2, 0, 3008, 1e4, 11),
    ((1, 2, 2, 2100, 96), 2, 2, 1, 2112, 1e4, 12),
]


@pytest.fixture(scope="module")
def nq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from e8_lattice_vector_gb300 import build as nqbuild

    nqbuild.build()
    import e8_lattice_vector_gb300 as nq

    return nq


def _cache(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    K = (torch.randn(shape, generator=g, device="cuda") * 1.5).to(torch.float16)
    V = torch.randn(shape, generator=g, device="cuda").to(torch.float16)
    return K, V


@pytest.mark.gpu
def test_static_scratch_matches_the_workspace_call_twice_in_a_row(nq):
    runs = []
    for shape, kb, vb, strict, delta, theta, seed in CASES:
        p = nq.CodecParams(kb, vb, 64, strict, delta, theta)
        assert nq.plan(shape, p).workspace_bytes > 0, "the case must need the scratch"
        assert nq.plan(shape, p).workspace_bytes <= nq.static_workspace_bytes()
        K, V = _cache(shape, seed)
        rope = nq.RopeTable.build(shape[3], shape[4], theta)
        buf = nq.compress_kv(K, V, p, rope)
        Kw, Vw = nq.decompress_kv(buf, shape, p, rope)
        runs.append((shape, p, rope, buf, Kw, Vw))
    torch.cuda.synchronize()
    outs = []
    for shape, p, rope, buf, _, _ in runs:  # back to back on one stream, no sync between
        Ks = torch.full(shape, float("nan"), dtype=torch.float16, device="cuda")
        Vs = torch.full(shape, float("nan"), dtype=torch.float16, device="cuda")
        nq.decompress_kv_static(buf, shape, p, rope, Ks, Vs)
        outs.append((Ks, Vs))
    nq.get_status()
    for (shape, _, _, _, Kw, Vw), (Ks, Vs) in zip(runs, outs):
        assert torch.equal(Ks.view(torch.int16), Kw.view(torch.int16)), shape
        assert torch.equal(Vs.view(torch.int16), Vw.view(torch.int16)), shape


@pytest.mark.gpu
def test_static_scratch_without_a_delta(nq):
    shape = (2, 1, 2, 700, 64)
    p = nq.CodecParams(2, 3, 32, 0, 0, 5e5)
    K, V = _cache(shape, 13)
    rope = nq.RopeTable.build(shape[3], shape[4], 5e5)
    buf = nq.compress_kv(K, V, p, rope)
    Kw, Vw = nq.decompress_kv(buf, shape, p, rope)
    Ks, Vs = torch.empty_like(Kw), torch.empty_like(Vw)
    nq.decompress_kv_static(buf, shape, p, rope, Ks, Vs)
    nq.get_status()
    assert torch.equal(Ks.view(torch.int16), Kw.view(torch.int16))
    assert torch.equal(Vs.view(torch.int16), Vw.view(torch.int16))


def test_static_scratch_size_matches_the_header():
    with open(os.path.join(ROOT, "include", "nq.h")) as f:
        m = re.search(r"#define NQ_STATIC_WORKSPACE_BYTES \((\d+)u << (\d+)\)", f.read())
    assert m, "NQ_STATIC_WORKSPACE_BYTES not found"
    import e8_lattice_vector_gb300 as nq

    assert nq.static_workspace_bytes() == int(m.group(1)) << int(m.group(2))


def test_static_scratch_rejects_a_cache_that_needs_more():
    """Host-side: the size check comes before any CUDA call, so it runs without
    a GPU."""
    from e8_lattice_vector_gb300 import _lib, build as nqbuild
    from e8_lattice_vector_gb300.codec import CodecParams, _cshape, plan, static_workspace_bytes

    nqbuild.build()
    big = (64, 1, 8, 131072, 128)  # single 4-bit chains on 512 slices
    p = CodecParams(4, 4, 64, 0, 131072, 0.0)
    assert plan(big, p).workspace_bytes > static_workspace_bytes()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call returns first
    st = _lib.lib().nq_decompress_kv_static(fake, 1 << 40, None, ctypes.byref(_cshape(big)), ctypes.byref(p.c()),
                                            fake, fake, None)
    assert st == 3  # NQ_ERR_SIZE
    # a cache that fits goes on to the usual argument checks (null outputs)
    small = (1, 1, 2, 4096, 128)
    ps = CodecParams(2, 2, 64, 0, 4096, 0.0)
    assert 0 < plan(small, ps).workspace_bytes <= static_workspace_bytes()
    st = _lib.lib().nq_decompress_kv_static(None, 1 << 30, None, ctypes.byref(_cshape(small)), ctypes.byref(ps.c()),
                                            None, None, None)
    assert st in (1, 4)  # NQ_ERR_ARG, or NQ_ERR_CUDA where no device answers the scratch look-up
