"""GPU (libnq, through its C ABI) against the CPU oracle on the same seeded
inputs.  Codes, coset words and scales must be bit-exact; reconstructions
within max |diff| <= 1e-3 and MSE(gpu, oracle) / mean(oracle^2) <= 1e-5."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

RECON_ATOL = 1e-3
RECON_REL_MSE = 1e-5


@pytest.fixture(scope="module")
def nq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from e8_lattice_vector_gb300 import build as nqbuild

    nqbuild.build()
    import e8_lattice_vector_gb300 as nq

    return nq


def _bits(x):
    """fp16 tensor -> numpy uint16 bit patterns."""
    return x.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle_compress(orc, K, V, params):
    L, B, H, T, D = K.shape
    cs = orc.rope_table(T, D, params.rope_theta) if params.rope_theta > 0 else None
    k = orc.compress_tensor(_bits(K).reshape(-1, T, D), T, D, params.key_bits, params.group_size,
                            int(params.strict), params.delta_chunk, cs)
    v = orc.compress_tensor(_bits(V).reshape(-1, T, D), T, D, params.value_bits, params.group_size,
                            int(params.strict), params.delta_chunk, None)
    return k, v, cs


def _gpu_sections(nq, buf, shape, params):
    """Sections as logical rows [slices * tokens, ...]; checks the padding
    rows of every slice are zero."""
    lay = nq.plan(shape, params)
    T = shape[3]
    full = nq.sections(buf, lay)
    tp = int(lay.tokens_padded)
    out = {}
    for t in ("k", "v"):
        arrs = []
        for key in ("_idx", "_coset", "_scale"):
            a = full[t + key]
            a = a.contiguous().view(torch.int16) if a.dtype == torch.float16 else a
            a = a.cpu().numpy()
            a = a.reshape(a.shape[0] // tp, tp, *a.shape[1:]) if tp else a.reshape(0, 0, *a.shape[1:])
            assert not np.any(a[:, T:]), t + key + " padding rows are not zero"
            a = a[:, :T].reshape(-1, *a.shape[2:])
            arrs.append(a.view(np.uint16) if a.dtype == np.int16 else a)
        out[t] = tuple(arrs)
    return out


def _same_values(gpu_bits, ref_bits):
    """Equal fp16 values (the sign of a zero may differ: the two-thread
    decompression produces some coordinates as the negation of a difference,
    which turns the oracle's -0 / +0 into the other zero)."""
    return np.array_equal(gpu_bits.view(np.float16), ref_bits.view(np.float16))


def _assert_recon(gpu_bits, ref_bits):
    g = gpu_bits.view(np.float16).astype(np.float64)
    r = ref_bits.view(np.float16).astype(np.float64)
    assert np.max(np.abs(g - r)) <= RECON_ATOL
    denom = max(np.mean(r ** 2), 1e-30)
    assert np.mean((g - r) ** 2) / denom <= RECON_REL_MSE


def _round_trip_check(nq, orc, K, V, params, expect_exact_recon=True):
    shape = tuple(K.shape)
    L, B, H, T, D = shape
    rope = nq.RopeTable.build(T, D, params.rope_theta) if params.rope_theta > 0 else None
    buf = nq.compress_kv(K, V, params, rope)
    (k_ref, v_ref, cs) = _oracle_compress(orc, K, V, params)
    got = _gpu_sections(nq, buf, shape, params)
    joint = int(params.strict) == 2  # no coset words: the block codes carry the coset bits
    for name, ref in (("k", k_ref), ("v", v_ref)):
        gi, gc, gs = got[name]
        ri, rc, rs = ref
        assert np.array_equal(gs, rs), name + " scales"
        if joint:
            assert gc.size == 0 and not rc.any(), name + " coset section"
        else:
            assert np.array_equal(gc, rc), name + " coset words"
        assert np.array_equal(gi, ri), name + " idx"
    K2, V2 = nq.decompress_kv(buf, shape, params, rope)
    torch.cuda.synchronize()
    kd = orc.decompress_tensor(*k_ref, L * B * H, T, D, params.key_bits, params.group_size,
                               params.delta_chunk, cs, joint=joint)
    vd = orc.decompress_tensor(*v_ref, L * B * H, T, D, params.value_bits, params.group_size,
                               params.delta_chunk, None, joint=joint)
    for g, r in ((K2, kd), (V2, vd)):
        gb = _bits(g).reshape(r.shape)
        _assert_recon(gb, r)
        if expect_exact_recon:
            assert _same_values(gb, r)
    # symbol statistics of the buffer equal the oracle's counts over its records
    counts = nq.code_histogram(buf, shape, params).cpu().numpy().astype(np.uint64)
    for n, (ref, bits) in enumerate(((k_ref, params.key_bits), (v_ref, params.value_bits))):
        ref_counts = orc.code_histogram(ref[0], None if joint else ref[1], D, bits)
        assert np.array_equal(counts[n], ref_counts), ("histogram", n)
    # the one-pass round trip reconstructs the same values
    K3, V3 = nq.roundtrip_kv(K, V, params, rope)
    torch.cuda.synchronize()
    for g3, r in ((K3, kd), (V3, vd)):
        gb = _bits(g3).reshape(r.shape)
        _assert_recon(gb, r)
        if expect_exact_recon:
            assert _same_values(gb, r)
    return buf


# ---------------------------------------------------------------- decoder


@pytest.mark.parametrize("bits", [0, 2, 3, 4])
@pytest.mark.parametrize("strict", [1, 0])
def test_e8_nearest_bit_exact(nq, orc, bits, strict):
    rng = np.random.default_rng(40 + bits + 7 * strict)
    h = ((1 << bits) - 1) / 2 if bits else 3.0
    u = rng.uniform(-1.1 * h, 1.1 * h, size=(50000, 8)).astype(np.float32)
    u[:3000] = np.round(u[:3000] * 2) / 2  # ties
    u[3000:4000] = 0.0
    u[4000:4500] = -0.0
    if bits:
        u[4500:5000] = np.clip(u[4500:5000], -h, h)  # on the box edge
    got = nq.e8_nearest(torch.from_numpy(u).cuda(), strict, bits).cpu().numpy()
    ref = orc.e8_nearest(u, strict, bits)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)) or np.array_equal(got, ref)
    mism = np.nonzero(np.any(got != ref, axis=1))[0]
    assert mism.size == 0, (mism[:5], u[mism[:1]], got[mism[:1]], ref[mism[:1]])


def _near_tie_blocks(rng, bits, strict, n):
    """Blocks whose two coset distances (after the parity fix-ups) differ by at
    most a few 1e-5: one coordinate's residual is set so that, in exact
    arithmetic, sum|u - rint(u)| - 2 + fix-up costs lands near zero (exact ties
    included).  Only the inputs are made here; the expected points are the
    oracle's."""
    h = ((1 << bits) - 1) / 2
    hi0 = (1 << bits) // 2 - 1
    out = []
    while len(out) < n:
        u = rng.uniform(-h * 0.98, h * 0.98, 8)
        r0 = np.rint(u)
        e0 = r0 - u
        e1 = e0 - np.copysign(0.5, e0)
        s0 = np.minimum(np.abs(e0), hi0 - np.abs(u))
        odd0 = int(r0.sum()) & 1
        odd1 = bool(strict) and (int(round((u + e1 - 0.5).sum())) & 1)
        gap = np.abs(e0).sum() - 2 + (1 - 2 * s0.max()) * odd0 - (1 - 2 * np.abs(e1).max()) * odd1
        ks = [k for k in range(8) if s0[k] != s0.max() and abs(e1[k]) != np.abs(e1).max()
              and 0.05 < abs(e0[k]) < 0.45 and abs(u[k]) < hi0]
        if not ks:
            continue
        na = abs(e0[ks[0]]) - gap + rng.choice([0.0, rng.uniform(-3e-5, 3e-5), rng.uniform(-1e-6, 1e-6)])
        if not 0.01 < na < 0.49:
            continue
        u[ks[0]] = r0[ks[0]] - np.sign(e0[ks[0]]) * na
        out.append(u)
    return np.asarray(out, dtype=np.float32)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("strict", [0, 1])
def test_e8_nearest_near_ties(nq, orc, bits, strict):
    """Coset choices decided by less than the fp32 rounding of the distances."""
    rng = np.random.default_rng(90 + bits + 7 * strict)
    u = _near_tie_blocks(rng, bits, strict, 20000)
    got = nq.e8_nearest(torch.from_numpy(u).cuda(), strict, bits).cpu().numpy()
    ref = orc.e8_nearest(u, strict, bits)
    mism = np.nonzero(np.any(got != ref, axis=1))[0]
    assert mism.size == 0, (mism[:5], u[mism[:1]], got[mism[:1]], ref[mism[:1]])


# ------------------------------------------------------------- tiny cache


def test_tiny_cache_full_parity(nq, orc):
    from e8_lattice_vector_gb300.synth import CONFIGS, make_cache

    cfg = CONFIGS["tiny"]
    K, V = make_cache(cfg, device="cuda")
    for params in cfg.modes:
        _round_trip_check(nq, orc, K, V, params)


# ------------------------------------------------- combinations, ragged tails


COMBOS = [
    # shape [L,B,H,T,D], key_bits, value_bits, group, strict, delta, theta
    ((2, 1, 3, 77, 128), 3, 2, 64, 0, 0, 1e4),
    ((2, 1, 3, 77, 128), 2, 2, 64, 1, 0, 1e4),
    ((1, 2, 2, 130, 128), 4, 3, 32, 1, 32, 5e5),
    ((1, 2, 2, 130, 128), 2, 4, 128, 0, 64, 1e6),
    ((2, 2, 2, 100, 96), 3, 2, 64, 0, 32, 1e4),
    ((1, 1, 4, 65, 96), 2, 3, 128, 1, 0, 1e4),
    ((1, 1, 4, 65, 64), 3, 2, 64, 1, 32, 1e4),
    ((1, 1, 3, 40, 64), 4, 2, 32, 0, 0, 0.0),
    ((1, 1, 2, 300, 128), 3, 2, 64, 1, 256, 1e4),
    ((1, 1, 2, 33, 128), 2, 2, 64, 0, 512, 1e4),
    # long delta chains: decompression chains tiles by the look-back; chains longer than a
    # compression segment start their segments with a halo tile
    ((1, 1, 3, 1000, 128), 3, 2, 64, 0, 1024, 1e4),
    ((1, 1, 3, 3000, 128), 2, 2, 64, 0, 3008, 1e4),
    ((1, 2, 2, 2100, 96), 3, 2, 64, 1, 2112, 1e4),
    ((1, 1, 2, 1500, 64), 2, 3, 64, 1, 1504, 5e5),
    ((1, 1, 3, 500, 64), 4, 2, 32, 0, 512, 5e5),
    # three-bit values along a long chain (the value decoder's column carry from the workspace)
    ((1, 1, 3, 1100, 96), 2, 3, 32, 0, 1120, 5e5),
    # strict joint format (no coset words)
    ((2, 1, 3, 77, 128), 2, 2, 64, 2, 0, 1e4),
    ((1, 2, 2, 130, 128), 3, 4, 32, 2, 32, 5e5),
    ((2, 2, 2, 100, 96), 3, 2, 64, 2, 32, 1e4),
    ((1, 1, 4, 65, 64), 4, 3, 64, 2, 0, 1e4),
    # joint format along long chains: three-bit keys and values, four-bit keys
    ((1, 1, 2, 2100, 128), 3, 3, 64, 2, 2112, 1e4),
    ((1, 1, 2, 1300, 128), 4, 2, 64, 2, 1312, 5e5),
]


@pytest.mark.parametrize("shape,kb,vb,g,strict,delta,theta", COMBOS)
def test_combinations_parity(nq, orc, shape, kb, vb, g, strict, delta, theta):
    from e8_lattice_vector_gb300 import CodecParams

    torch.manual_seed(hash((shape, kb, vb, g, strict, delta)) % (1 << 31))
    K = (torch.randn(shape, device="cuda") * torch.exp(torch.randn(shape[-1], device="cuda") * 0.7)).half()
    V = torch.randn(shape, device="cuda").half()
    params = CodecParams(kb, vb, g, int(strict), delta, theta)
    _round_trip_check(nq, orc, K, V, params)


# -------------------------------------------------------------- edge cases


def _edge_inputs(kind, shape):
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    if kind == "zeros":
        return torch.zeros(shape, device="cuda").half(), torch.zeros(shape, device="cuda").half()
    if kind == "neg_zeros":
        z = torch.full(shape, -0.0, device="cuda").half()
        return z, z.clone()
    if kind == "constant":  # every group's scale is exact: the general (clamping) path
        return torch.full(shape, 0.75, device="cuda").half(), torch.full(shape, -3.0, device="cuda").half()
    if kind == "fp16_max":
        x = torch.randn(shape, generator=g, device="cuda").sign() * 65504.0
        return x.half(), (x * 0.5).half()
    if kind == "tiny":  # subnormal fp16 inputs and scales
        x = torch.randn(shape, generator=g, device="cuda") * 1e-6
        return x.half(), (x * 0.01).half()
    if kind == "sparse":
        x = torch.randn(shape, generator=g, device="cuda")
        x = torch.where(torch.rand(shape, generator=g, device="cuda") < 0.9, torch.zeros_like(x), x)
        return x.half(), (x * 3).half()
    if kind == "quantized":  # values on a coarse grid: many exact ties
        x = torch.round(torch.randn(shape, generator=g, device="cuda") * 4) / 4
        return x.half(), torch.round(torch.randn(shape, generator=g, device="cuda")).half()
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["zeros", "neg_zeros", "constant", "fp16_max", "tiny", "sparse", "quantized"])
@pytest.mark.parametrize("strict", [1, 0, 2])
def test_edge_cases_parity(nq, orc, kind, strict):
    from e8_lattice_vector_gb300 import CodecParams

    shape = (1, 1, 2, 45, 128)
    K, V = _edge_inputs(kind, shape)
    for kb, vb in ((3, 2), (2, 2), (4, 4)):
        params = CodecParams(kb, vb, 64, int(strict), 32, 1e4)
        _round_trip_check(nq, orc, K, V, params)


@pytest.mark.parametrize("T", [1, 2, 31, 32, 33])
def test_short_sequences(nq, orc, T):
    from e8_lattice_vector_gb300 import CodecParams

    shape = (1, 1, 3, T, 128)
    K = torch.randn(shape, device="cuda").half()
    V = torch.randn(shape, device="cuda").half()
    _round_trip_check(nq, orc, K, V, CodecParams(3, 2, 64, False, 32, 1e4))


@pytest.mark.parametrize("shape,theta", [((2, 1, 3, 77, 128), 1e4), ((1, 2, 5, 45, 64), 5e5),
                                         ((1, 1, 4, 70, 96), 1e4), ((1, 1, 2, 33, 128), 0.0)])
def test_roundtrip_in_place(nq, orc, shape, theta):
    """nq_roundtrip_kv with the outputs aliasing the inputs."""
    from e8_lattice_vector_gb300 import CodecParams

    params = CodecParams(key_bits=3, value_bits=2, group_size=64, strict=False, delta_chunk=0, rope_theta=theta)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    K = (torch.randn(shape, generator=g, device="cuda") * 2).to(torch.float16)
    V = torch.randn(shape, generator=g, device="cuda").to(torch.float16)
    rope = nq.RopeTable.build(shape[3], shape[4], theta) if theta > 0 else None
    K2, V2 = nq.decompress_kv(nq.compress_kv(K, V, params, rope), shape, params, rope)
    Kc, Vc = K.clone(), V.clone()
    nq.roundtrip_kv(Kc, Vc, params, rope, K_out=Kc, V_out=Vc)
    torch.cuda.synchronize()
    assert bool((Kc == K2).all()) and bool((Vc == V2).all())


def test_per_layer_bits_and_kept_layers(nq, orc):
    """A per-layer table with kept (fp16) layers and mixed bit widths: every
    compressed part equals the oracle's compression of that layer alone, kept
    parts are the layer's bytes, and both directions reproduce the oracle."""
    from e8_lattice_vector_gb300 import CodecParams

    shape = (5, 1, 3, 77, 128)
    table = [(0, 0), (3, 2), (2, 2), (4, 3), (0, 0)]
    params = CodecParams(3, 2, 64, True, 64, 1e4)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    K = (torch.randn(shape, generator=g, device="cuda") * 3).to(torch.float16)
    V = torch.randn(shape, generator=g, device="cuda").to(torch.float16)
    rope = nq.RopeTable.build(shape[3], shape[4], params.rope_theta)
    buf = nq.compress_kv_layers(K, V, params, table, rope)
    offs, total = nq.plan_layers(shape, params, table)
    K2, V2 = nq.decompress_kv_layers(buf, shape, params, table, rope)
    K3, V3 = nq.roundtrip_kv_layers(K, V, params, table, rope)
    torch.cuda.synchronize()
    one = (1,) + shape[1:]
    raw = K[0].numel() * 2
    for l, (kb, vb) in enumerate(table):
        part = buf[offs[l]:]
        if kb == 0:
            assert torch.equal(part[:raw], K[l].contiguous().view(-1).view(torch.uint8))
            assert torch.equal(part[raw:2 * raw], V[l].contiguous().view(-1).view(torch.uint8))
            assert torch.equal(K2[l], K[l]) and torch.equal(V2[l], V[l]) and torch.equal(K3[l], K[l])
            continue
        p = CodecParams(kb, vb, params.group_size, params.strict, params.delta_chunk, params.rope_theta)
        got = _gpu_sections(nq, part, one, p)
        k_ref, v_ref, cs = _oracle_compress(orc, K[l:l + 1], V[l:l + 1], p)
        for name, ref in (("k", k_ref), ("v", v_ref)):
            for a, b in zip(got[name], ref):
                assert np.array_equal(a, b), (l, name)
        kd = orc.decompress_tensor(*k_ref, 3, 77, 128, kb, 64, params.delta_chunk, cs)
        vd = orc.decompress_tensor(*v_ref, 3, 77, 128, vb, 64, params.delta_chunk, None)
        for out2, out3, ref in ((K2[l], K3[l], kd), (V2[l], V3[l], vd)):
            assert _same_values(_bits(out2).reshape(ref.shape), ref)
            assert _same_values(_bits(out3).reshape(ref.shape), ref)


def test_empty_cache_is_noop(nq):
    from e8_lattice_vector_gb300 import CodecParams

    K = torch.zeros((2, 1, 8, 0, 128), device="cuda").half()
    buf = nq.compress_kv(K, K.clone(), CodecParams(), nq.RopeTable.build(0, 128, 1e4))
    K2, V2 = nq.decompress_kv(buf, K.shape, CodecParams(), nq.RopeTable.build(0, 128, 1e4))
    assert K2.numel() == 0
    K3, V3 = nq.roundtrip_kv(K, K.clone(), CodecParams(), nq.RopeTable.build(0, 128, 1e4))
    assert K3.numel() == 0


# ------------------------------------------- full-size caches, sampled rows


def _sample_rows(rng, cfg, n):
    rows = cfg.rows
    pick = rng.choice(rows, size=n, replace=False)
    # always include chunk boundaries and the first/last token of a slice
    T = cfg.tokens
    extra = np.array([0, T - 1, T, rows - 1, 255 if T > 256 else 1, 256 if T > 256 else 1])
    return np.unique(np.concatenate([pick, extra]) % rows)


def _full_size_check(nq, orc, cfg, K, V, params, rows, cs):
    """One codec mode on a full-size cache: the sampled rows' records against
    the oracle's encoding of those rows (delta rows against the oracle's
    encoding of the previous token too), the sampled reconstructions against
    the oracle's decoding, and the one-pass round trip against
    decompress(compress(.)) on every element.  cs: the oracle's own RoPE
    table [tokens, head_dim/2, 2]."""
    T, D = cfg.tokens, cfg.head_dim
    rope = nq.RopeTable.build(T, D, params.rope_theta)
    buf = nq.compress_kv(K, V, params, rope)
    lay = nq.plan(cfg.shape, params)
    tp = int(lay.tokens_padded)
    full = nq.sections(buf, lay)
    rec = torch.from_numpy((rows // T) * tp + rows % T).cuda()  # record rows of the sampled tokens
    got = {}
    for t in ("k", "v"):
        got[t] = (full[t + "_idx"][rec].cpu().numpy(),
                  full[t + "_coset"][rec].cpu().numpy().view(np.uint16),
                  full[t + "_scale"][rec].contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    Kf = K.view(-1, D)
    Vf = V.view(-1, D)
    rows_t = torch.from_numpy(rows).cuda()
    prev_t = torch.from_numpy(np.maximum(rows - 1, 0)).cuda()
    for name_t, X, bits, rope_on in (("k", Kf, params.key_bits, True), ("v", Vf, params.value_bits, False)):
        xr = _bits(X[rows_t])
        xp = _bits(X[prev_t])
        gi, gc, gs = got[name_t]
        for n, r in enumerate(rows):
            t = int(r % T)
            csr = cs[t] if rope_on else None
            idx, cw, sc = orc.encode_row(xr[n], D, bits, params.group_size, int(params.strict), csr)
            if params.delta_chunk and t % params.delta_chunk != 0:
                pidx, pcw, _ = orc.encode_row(xp[n], D, bits, params.group_size, int(params.strict),
                                              cs[t - 1] if rope_on else None)
                idx, cw = orc.delta_row(idx, cw, pidx, pcw, orc.padded_dim(D), bits)
            assert np.array_equal(gs[n], sc), (name_t, r)
            assert gc[n] == cw, (name_t, r)
            assert np.array_equal(gi[n], idx), (name_t, r)
    # decompression of the same rows against the oracle's decoding of its own
    # encoding of the raw rows (the GPU side restores them through the delta chain)
    K2, V2 = nq.decompress_kv(buf, cfg.shape, params, rope)
    for name_t, X2, bits, rope_on in (("k", K2, params.key_bits, True), ("v", V2, params.value_bits, False)):
        xr2 = _bits(X2.view(-1, D)[rows_t])
        xr = _bits((K if name_t == "k" else V).view(-1, D)[rows_t])
        ref = np.empty_like(xr2)
        for n, r in enumerate(rows):
            t = int(r % T)
            csr = cs[t] if rope_on else None
            idx, cw, sc = orc.encode_row(xr[n], D, bits, params.group_size, int(params.strict), csr)
            ref[n] = orc.decode_row(idx, cw, sc, D, bits, params.group_size, csr)
        _assert_recon(xr2, ref)
        assert _same_values(xr2, ref)
    # the one-pass round trip equals decompress(compress(.)) everywhere
    K3, V3 = nq.roundtrip_kv(K, V, params, rope)
    assert bool((K3 == K2).all()) and bool((V3 == V2).all())
    del buf, K2, V2, K3, V3
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["mistral7b", "phi3mini", "llama31_8b", "qwen25_14b", "llama32_1b"])
def test_full_size_sampled_parity(nq, orc, name):
    """Each full-size cache in every codec mode it is served in, compressed and
    decompressed by the same library calls the benchmark times; a sample of
    rows re-computed one by one by the oracle, with the oracle's own RoPE
    table."""
    from e8_lattice_vector_gb300.synth import CONFIGS, make_cache

    cfg = CONFIGS[name]
    K, V = make_cache(cfg, device="cuda")
    rows = _sample_rows(np.random.default_rng(1234), cfg, 600)
    cs = orc.rope_table(cfg.tokens, cfg.head_dim, cfg.theta)
    for params in cfg.modes:
        assert params.rope_theta == cfg.theta
        _full_size_check(nq, orc, cfg, K, V, params, rows, cs)


@pytest.mark.parametrize("name,kb,vb", [("mistral7b", 2, 2), ("phi3mini", 3, 2), ("llama32_1b", 2, 2),
                                        ("qwen25_14b", 3, 2), ("many_short_slices", 3, 2)])
def test_full_size_single_chain_delta(nq, orc, name, kb, vb):
    """The pages' temporal delta as one chain per slice (delta_chunk >= tokens)
    on a full-size cache: sampled rows deep in the chain (their predecessors
    span many tiles) are checked against the oracle, and their reconstructions
    need every earlier delta row of the slice.  The Qwen2.5-14B shape is the
    benchmarked single-chain case; the last one (6144 slices of 1536 tokens,
    two runs per chain, the second one short) has the most runs."""
    import dataclasses

    from e8_lattice_vector_gb300 import CodecParams
    from e8_lattice_vector_gb300.synth import CONFIGS, make_cache

    if name == "many_short_slices":
        cfg = dataclasses.replace(CONFIGS["mistral7b"], name=name, layers=24, batch=1, kv_heads=256, tokens=1536)
    else:
        cfg = CONFIGS[name]
    K, V = make_cache(cfg, device="cuda")
    T = cfg.tokens
    chain = (T + 31) // 32 * 32
    rng = np.random.default_rng(4321)
    rows = _sample_rows(rng, cfg, 400)
    # the last tokens of a few slices depend on the whole chain
    ends = (rng.choice(cfg.rows // T, size=8, replace=False) + 1) * T - 1
    rows = np.unique(np.concatenate([rows, ends, ends - 33]))
    cs = orc.rope_table(T, cfg.head_dim, cfg.theta)
    params = CodecParams(kb, vb, 64, 0, chain, cfg.theta)
    _full_size_check(nq, orc, cfg, K, V, params, rows, cs)


def test_long_chains_on_a_user_stream_back_to_back(nq):
    """Long delta chains decompressed on a non-default stream, three calls in
    a row into different outputs with one workspace and no synchronisation in
    between (the value run totals of each call run on the library's side
    stream): every result equals the one decompressed alone on the default
    stream."""
    from e8_lattice_vector_gb300 import CodecParams

    shape = (2, 1, 4, 3000, 128)
    p = CodecParams(3, 2, 64, 0, 3008, 1e4)
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    caches = [((torch.randn(shape, generator=g, device="cuda") * 2).half(),
               torch.randn(shape, generator=g, device="cuda").half()) for _ in range(3)]
    rope = nq.RopeTable.build(shape[3], shape[4], p.rope_theta)
    bufs = [nq.compress_kv(K, V, p, rope) for K, V in caches]
    ref = [nq.decompress_kv(b, shape, p, rope) for b in bufs]
    torch.cuda.synchronize()
    ws = nq.workspace(int(nq.plan(shape, p).workspace_bytes), "cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        outs = [nq.decompress_kv(b, shape, p, rope, ws=ws) for b in bufs]
    s.synchronize()
    for (Kr, Vr), (Ko, Vo) in zip(ref, outs):
        assert torch.equal(Kr.view(torch.int16), Ko.view(torch.int16))
        assert torch.equal(Vr.view(torch.int16), Vo.view(torch.int16))


@pytest.mark.parametrize("name,kb,vb", [("mistral7b", 2, 2), ("phi3mini", 3, 2)])
def test_full_size_joint_format(nq, orc, name, kb, vb):
    """The strict joint format on a full-size cache: sampled rows re-encoded by
    the oracle (strict decode, then the joint packing), no coset section, and
    the sampled reconstructions equal the oracle's."""
    from e8_lattice_vector_gb300 import CodecParams
    from e8_lattice_vector_gb300.synth import CONFIGS, make_cache

    cfg = CONFIGS[name]
    K, V = make_cache(cfg, device="cuda")
    T, D = cfg.tokens, cfg.head_dim
    params = CodecParams(kb, vb, 64, 2, 0, cfg.theta)
    rope = nq.RopeTable.build(T, D, params.rope_theta)
    cs = orc.rope_table(T, D, params.rope_theta)  # the oracle's own table
    buf = nq.compress_kv(K, V, params, rope)
    lay = nq.plan(cfg.shape, params)
    assert lay.k_coset == lay.k_scale and lay.v_coset == lay.v_scale
    tp = int(lay.tokens_padded)
    full = nq.sections(buf, lay)
    rows = _sample_rows(np.random.default_rng(99), cfg, 400)
    rec = torch.from_numpy((rows // T) * tp + rows % T).cuda()
    K2, V2 = nq.decompress_kv(buf, cfg.shape, params, rope)
    dp = orc.padded_dim(D)
    for t_name, X, X2, bits, rope_on in (("k", K, K2, kb, True), ("v", V, V2, vb, False)):
        gi = full[t_name + "_idx"][rec].cpu().numpy()
        gs = full[t_name + "_scale"][rec].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        sel = torch.from_numpy(rows).cuda()
        xr = _bits(X.view(-1, D)[sel])
        xr2 = _bits(X2.view(-1, D)[sel])
        for n, r in enumerate(rows):
            csr = cs[int(r % T)] if rope_on else None
            idx, cw, sc = orc.encode_row(xr[n], D, bits, 64, 1, csr)
            assert np.array_equal(gs[n], sc), (t_name, r)
            assert np.array_equal(gi[n], orc.joint_pack_row(idx, cw, dp, bits)), (t_name, r)
            ref = orc.decode_row(idx, cw, sc, D, bits, 64, csr)
            assert _same_values(xr2[n], ref), (t_name, r)
    del buf, K2, V2
    torch.cuda.empty_cache()


def test_entropy_report_on_the_tiny_cache(nq):
    """The entropy report runs end to end on device counts: every field of every
    real row is counted, and order-0 entropies stay within [0, b] bits."""
    from e8_lattice_vector_gb300 import CodecParams
    from e8_lattice_vector_gb300.entropy import report
    from e8_lattice_vector_gb300.synth import CONFIGS, make_cache

    cfg = CONFIGS["tiny"]
    K, V = make_cache(cfg, device="cuda")
    rope = nq.RopeTable.build(cfg.tokens, cfg.head_dim, 1e4)
    for delta in (0, 32):
        p = CodecParams(3, 2, 64, 0, delta, 1e4)
        rep = report(K, V, p, rope)
        for t, bits in (("k", 3), ("v", 2)):
            r = rep[t]
            assert r["fields"] == cfg.rows * 128
            assert 0.0 < r["field_entropy_bits"] <= bits
            assert 0.0 <= r["byte_entropy_bits_per_byte"] <= 8.0
            assert r["raw_bits_per_coord"] == pytest.approx(bits + 1 / 8 + 16 * 2 / 128)


def test_delta_status_clean_after_calls(nq):
    """A delta-coded round trip through a reused workspace decodes the same
    twice, and the stream reports no error."""
    from e8_lattice_vector_gb300 import CodecParams

    shape = (1, 1, 4, 700, 128)
    p = CodecParams(3, 2, 64, 0, 704, 1e4)
    K = torch.randn(shape, device="cuda").half()
    V = torch.randn(shape, device="cuda").half()
    rope = nq.RopeTable.build(700, 128, 1e4)
    ws = nq.workspace(int(nq.plan(shape, p).workspace_bytes), K.device)
    buf = nq.compress_kv(K, V, p, rope)
    a = nq.decompress_kv(buf, shape, p, rope, ws=ws)
    b = nq.decompress_kv(buf, shape, p, rope, ws=ws)
    nq.get_status()  # raises on a deferred error
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
