"""Pins for the CPU oracle: it is checked against what the pages and the
mathematics fix, never against itself or against the CUDA path.

Each test names what it pins.  Brute force uses float64 arithmetic over
explicit enumerations (or an exhaustive per-coordinate dynamic program over
the same candidate sets), which shares nothing with the oracle's decoder.
"""
import itertools
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e8_constants.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ------------------------------------------------------------ brute force


def _dp_min(values, costs, par):
    """Exhaustive minimum over per-coordinate candidates, split by the parity
    of the summed integer parts.  values/costs/par: [N, 8, m] arrays.
    Returns (best_even, best_odd) float64 [N]."""
    inf = np.full(costs.shape[0], np.inf)
    best0, best1 = np.zeros(costs.shape[0]), inf.copy()
    for j in range(8):
        c = costs[:, j, :]
        p = par[:, j, :]
        ev = np.where(p == 0, c, np.inf).min(axis=1)
        od = np.where(p == 1, c, np.inf).min(axis=1)
        best0, best1 = np.minimum(best0 + ev, best1 + od), np.minimum(best0 + od, best1 + ev)
    return best0, best1


def _candidates(u, half, bits):
    """Candidate coordinate values per block.  Box codes: every value of the
    coset inside the box; unbounded: a window of 6 values around u."""
    u = u.astype(np.float64)
    N = u.shape[0]
    if bits:
        L = 1 << bits
        if half:
            vals = np.arange(-(L - 1) / 2, (L - 1) / 2 + 0.5, 1.0)
        else:
            vals = np.arange(-(L // 2 - 1), L // 2 - 1 + 0.5, 1.0)
        v = np.broadcast_to(vals, (N, 8, vals.size)).copy()
    else:
        base = np.floor(u) + (0.5 if half else 0.0)
        v = base[:, :, None] + np.arange(-3, 3)[None, None, :]
    costs = (u[:, :, None] - v) ** 2
    ints = v - 0.5 if half else v
    par = np.mod(np.rint(ints).astype(np.int64), 2)
    return v, costs, par


def brute_min_dist(u, strict, bits):
    _, c0, p0 = _candidates(u, False, bits)
    _, c1, p1 = _candidates(u, True, bits)
    i_even, _ = _dp_min(None, c0, p0)
    h_even, h_odd = _dp_min(None, c1, p1)
    half = h_even if strict else np.minimum(h_even, h_odd)
    return np.minimum(i_even, half)


def enumerate_codebook(strict, bits):
    """Every point of the box codebook (small bit widths only)."""
    L = 1 << bits
    pts = []
    ivals = np.arange(-(L // 2 - 1), L // 2)
    for p in itertools.product(ivals, repeat=8):
        if sum(p) % 2 == 0:
            pts.append(p)
    hvals = np.arange(-(L - 1) / 2, (L - 1) / 2 + 0.5, 1.0)
    for p in itertools.product(hvals, repeat=8):
        if not strict or int(round(sum(x - 0.5 for x in p))) % 2 == 0:
            pts.append(p)
    return np.array(pts, dtype=np.float64)


def in_codebook(r, strict, bits):
    r = r.astype(np.float64)
    frac = r - np.floor(r)
    is_int = np.all(frac == 0.0, axis=1)
    is_half = np.all(frac == 0.5, axis=1)
    ok = is_int | is_half
    s_int = np.rint(r.sum(axis=1)).astype(np.int64)
    s_half = np.rint((r - 0.5).sum(axis=1)).astype(np.int64)
    ok &= ~is_int | (s_int % 2 == 0)
    if strict:
        ok &= ~is_half | (s_half % 2 == 0)
    if bits:
        L = 1 << bits
        ok &= ~is_int | np.all(np.abs(r) <= L // 2 - 1, axis=1)
        ok &= ~is_half | np.all(np.abs(r) <= (L - 1) / 2, axis=1)
    return ok


# ------------------------------------------------------------- T1 decoder


@pytest.mark.parametrize("strict", [1, 0])
def test_t1_unbounded_matches_brute_force(orc, strict):
    rng = np.random.default_rng(11 + strict)
    u = rng.uniform(-3, 3, size=(20000, 8)).astype(np.float32)
    r = orc.e8_nearest(u, strict, 0)
    assert in_codebook(r, strict, 0).all()
    d_orc = ((u.astype(np.float64) - r) ** 2).sum(axis=1)
    d_min = brute_min_dist(u, strict, 0)
    assert np.all(d_orc <= d_min + 1e-5), np.max(d_orc - d_min)


def test_t1_dp_agrees_with_full_enumeration(orc):
    """The factorised brute force itself against a plain enumeration (b = 2)."""
    rng = np.random.default_rng(3)
    u = rng.uniform(-1.6, 1.6, size=(60, 8)).astype(np.float32)
    for strict in (1, 0):
        cb = enumerate_codebook(strict, 2)
        d_enum = ((u.astype(np.float64)[:, None, :] - cb[None]) ** 2).sum(-1).min(axis=1)
        assert np.allclose(d_enum, brute_min_dist(u, strict, 2), atol=1e-12)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("strict", [1, 0])
def test_t1_box_codes_match_brute_force(orc, bits, strict):
    rng = np.random.default_rng(100 * bits + strict)
    h = ((1 << bits) - 1) / 2
    # inside the box, on its edges, and a little beyond it
    u = rng.uniform(-1.05 * h, 1.05 * h, size=(4000, 8)).astype(np.float32)
    u[:200] = np.round(u[:200] * 2) / 2  # exact half-integers / integers: tie cases
    r = orc.e8_nearest(u, strict, bits)
    assert in_codebook(r, strict, bits).all()
    d_orc = ((u.astype(np.float64) - r) ** 2).sum(axis=1)
    d_min = brute_min_dist(u, strict, bits)
    assert np.all(d_orc <= d_min + 1e-5), np.max(d_orc - d_min)


def test_t1_tie_rules(orc):
    # integer coset rounds half to even: 0.5 -> 0, 1.5 -> 2 (unbounded)
    r, c = orc.e8_block(np.array([0.5, 1.5, 0, 0, 0, 0, 0, 0], np.float32), 1, 0)
    # both cosets are at distance 0.5; the tie goes to the integer coset
    assert c == 0 and list(r) == [0, 2, 0, 0, 0, 0, 0, 0]
    # the half-integer point of an integer u is u - 1/2 (ceil(u) - 1/2)
    r, c = orc.e8_block(np.array([0.5, 0.5, 0.5, 0.5, 0.5, 0.5, 0.5, 2.0], np.float32), 0, 0)
    assert c == 1 and list(r) == [0.5] * 7 + [1.5]
    # parity fix-up moves the coordinate farthest from its rounding, toward u
    r, c = orc.e8_block(np.array([0.1, 0.2, 0.3, 0.4, 0, 0, 0, 1.0], np.float32), 1, 0)
    assert c == 0 and list(r) == [0, 0, 0, 1, 0, 0, 0, 1]
    # equal scores: the lowest index is moved
    r, c = orc.e8_block(np.array([0.3, 0.3, 0, 0, 0, 0, 0, 1.0], np.float32), 1, 0)
    assert c == 0 and list(r) == [1, 0, 0, 0, 0, 0, 0, 1]


def test_t1_fixup_at_box_edge_steps_inward(orc):
    # b = 2, integer box [-1, 1]: u = (1.2, 0, ..., 0) rounds to 1 (odd); stepping
    # toward u would leave the box, so the cheapest legal change is chosen.
    u = np.array([1.2, 0.05, 0, 0, 0, 0, 0, 0], np.float32)
    r = orc.e8_nearest(u[None], 1, 2)[0]
    d = ((u.astype(np.float64) - r) ** 2).sum()
    assert d <= brute_min_dist(u[None], 1, 2)[0] + 1e-6
    assert np.all(np.abs(r) <= 1.5)


# ---------------------------------------------------------- T2 invariants


def test_t2_lattice_invariants_and_covering_radius(orc):
    g = _golden()
    rng = np.random.default_rng(5)
    u = rng.normal(0, 3, size=(50000, 8)).astype(np.float32)
    for strict in (1, 0):
        r = orc.e8_nearest(u, strict, 0)
        assert in_codebook(r, strict, 0).all()
        d = ((u.astype(np.float64) - r) ** 2).sum(axis=1)
        assert d.max() <= g["covering_radius_sq_e8"]["value"] + 1e-5


def test_t2_norm2_shell_counts(orc):
    """Points of squared norm 2 that each decoder keeps as fixed points."""
    g = _golden()
    ints = []
    for i, j in itertools.combinations(range(8), 2):
        for si in (-1, 1):
            for sj in (-1, 1):
                v = np.zeros(8)
                v[i], v[j] = si, sj
                ints.append(v)
    halves = [np.array(s) * 0.5 for s in itertools.product((-1, 1), repeat=8)]
    assert len(ints) == 112 and len(halves) == 256
    for strict, key in ((1, "norm2_shell_strict"), (0, "norm2_shell_relaxed")):
        fi = sum(np.array_equal(orc.e8_nearest(v.astype(np.float32)[None], strict, 0)[0], v) for v in ints)
        fh = sum(np.array_equal(orc.e8_nearest(v.astype(np.float32)[None], strict, 0)[0], v) for v in halves)
        assert fi == g[key]["integer_coset"]
        assert fh == g[key]["half_coset"]
    assert 112 + 128 == g["kissing_number"]["value"]


# ------------------------------------------------------------- T3 Hadamard


@pytest.mark.parametrize("n", [8, 64, 128])
@pytest.mark.parametrize("order", ["textbook", "forward"])
def test_t3_fwht_is_sylvester_hadamard(orc, n, order):
    f = orc.fwht if order == "textbook" else orc.fwht_forward
    H = np.stack([f(np.eye(n, dtype=np.float32)[j]) for j in range(n)], axis=1)
    i = np.arange(n)
    pop = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    assert np.array_equal(H, (-1.0) ** pop)
    assert np.array_equal(H @ H, n * np.eye(n))


def test_t3_fwht_involution_and_matrix_product(orc):
    rng = np.random.default_rng(7)
    n = 128
    xi = rng.integers(-1000, 1000, size=n).astype(np.float32)
    assert np.array_equal(orc.fwht(orc.fwht(xi)), n * xi)  # exact on integers
    assert np.array_equal(orc.fwht(orc.fwht_forward(xi)), n * xi)
    x = rng.normal(size=n).astype(np.float32)
    i = np.arange(n)
    H = (-1.0) ** np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    ref = H @ x.astype(np.float64)
    for f in (orc.fwht, orc.fwht_forward):
        assert np.allclose(f(x), ref, rtol=0, atol=1e-5 * np.abs(x).sum())
    # the two orders round differently somewhere (otherwise the order would not matter)
    xs = rng.normal(size=(200, n)).astype(np.float32) * 10.0 ** rng.integers(-3, 4, size=(200, 1))
    assert any(not np.array_equal(orc.fwht(v), orc.fwht_forward(v)) for v in xs)


def test_t3_zero_padded_round_trip(orc):
    rng = np.random.default_rng(8)
    x = np.zeros(128, np.float32)
    x[:96] = rng.integers(-50, 50, size=96)
    y = orc.fwht(x)
    back = orc.fwht(y) / 128
    assert np.array_equal(back[:96], x[:96]) and np.all(back[96:] == 0)


# ----------------------------------------------------------------- T4 RoPE


@pytest.mark.parametrize("theta", [1e4, 5e5, 1e6])
@pytest.mark.parametrize("D", [96, 128])
def test_t4_rope_table_closed_form(orc, theta, D):
    pos = np.array([0, 1, 2, 17, 511, 4095, 32767, 131071], np.int32)
    cs = orc.rope_table(len(pos), D, theta, positions=pos)
    i = np.arange(D // 2)
    ang = pos[:, None].astype(np.float64) * np.power(float(theta), -2.0 * i / D)[None, :]
    # within one float32 ulp of the double-precision value
    assert np.allclose(cs[..., 0], np.cos(ang), rtol=0, atol=1.2e-7)
    assert np.allclose(cs[..., 1], np.sin(ang), rtol=0, atol=1.2e-7)
    assert np.all(cs[0, :, 0] == 1.0) and np.all(cs[0, :, 1] == 0.0)
    assert np.array_equal(cs[:, 0, 0], np.cos(pos.astype(np.float64)).astype(np.float32))


def test_t4_rope_apply_matches_rotate_half_convention(orc):
    """apply == q*cos + rotate_half(q)*sin with rotate_half(q) = (-q2, q1)."""
    rng = np.random.default_rng(9)
    D = 128
    cs = orc.rope_table(64, D, 1e4)
    for t in (0, 5, 63):
        q = rng.normal(size=D).astype(np.float32)
        c = np.concatenate([cs[t, :, 0], cs[t, :, 0]]).astype(np.float64)
        s = np.concatenate([cs[t, :, 1], cs[t, :, 1]]).astype(np.float64)
        rot = np.concatenate([-q[D // 2:], q[: D // 2]]).astype(np.float64)
        ref = q * c + rot * s
        assert np.allclose(orc.rope_apply(q, cs[t]), ref, atol=1e-6)


@pytest.mark.parametrize("theta", [1e4, 5e5, 1e6])
def test_t4_rope_remove_inverts_apply(orc, theta):
    rng = np.random.default_rng(10)
    D = 128
    pos = np.array([0, 1, 1000, 65535, 131071], np.int32)
    cs = orc.rope_table(len(pos), D, theta, positions=pos)
    for t in range(len(pos)):
        x = rng.normal(size=D).astype(np.float32) * 3
        y = orc.rope_apply(x, cs[t])
        back = orc.rope_remove(y, cs[t])
        pair = np.sqrt(x[: D // 2] ** 2 + x[D // 2:] ** 2)
        pair = np.concatenate([pair, pair])
        assert np.all(np.abs(back - x) <= 4 * np.finfo(np.float32).eps * pair + 1e-30)
        n0 = x[: D // 2].astype(np.float64) ** 2 + x[D // 2:].astype(np.float64) ** 2
        n1 = y[: D // 2].astype(np.float64) ** 2 + y[D // 2:].astype(np.float64) ** 2
        assert np.allclose(n0, n1, rtol=1e-6)
        if pos[t] == 0:
            assert np.array_equal(y, x)


# ------------------------------------------------------------- binary16


def test_h2f_all_codes_match_ieee(orc):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.h2f(codes)
    ref = codes.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f2h_round_to_nearest_even(orc):
    rng = np.random.default_rng(12)
    x = np.concatenate([
        rng.normal(size=4000) * 10.0 ** rng.integers(-9, 5, size=4000),
        np.arange(0, 2049, dtype=np.float64) * 2.0 ** -25,  # subnormal ties
        [65504, 65519.99, 65520, 70000, -65520, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -0.0, 0.0],
    ]).astype(np.float32)
    ours = orc.f2h(x)
    with np.errstate(over="ignore"):  # the inputs past 65520 overflow to infinity on purpose
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ----------------------------------------------------------- group scale


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("dp", [64, 128])
def test_group_scale_is_smallest_non_clipping_half(orc, bits, dp):
    step = dp * ((1 << bits) - 1) / 2
    halves = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    rng = np.random.default_rng(13)
    amax = np.concatenate([
        np.abs(rng.normal(size=300)) * 10.0 ** rng.integers(-8, 7, size=300),
        halves[rng.integers(1, halves.size, size=100)] * step,  # exactly representable
        [0.0, 1e-30, 2.0 ** -24 * step, 1.0, dp * 65504.0 * 1.41421],  # largest reachable
    ]).astype(np.float32)
    for a in amax:
        v = orc.group_scale(a, bits, dp)
        ok = halves * step >= np.float64(a)
        expect = int(np.argmax(ok))
        assert v == expect, (a, v, expect)


# ----------------------------------------------------- T5 Figure-1 shape


def test_t5_e8_mse_gain_over_integer_lattice(orc):
    """Equal point density (det 1), high resolution: the mean squared error per
    dimension of the E8 decoder is the normalized second moment G(E8); Z^8 gives
    1/12.  A wrong decoder (dropped fix-up, wrong coset choice) is far off."""
    g = _golden()["normalized_second_moment_e8"]
    G = g["numerator"] / g["denominator"]
    rng = np.random.default_rng(14)
    u = rng.uniform(-40, 40, size=(200000, 8)).astype(np.float32)
    r = orc.e8_nearest(u, 1, 0)
    mse_e8 = ((u.astype(np.float64) - r) ** 2).mean()
    mse_z = ((u.astype(np.float64) - np.rint(u)) ** 2).mean()
    assert abs(mse_e8 - G) < 0.01 * G, mse_e8
    assert abs(mse_z - 1 / 12) < 0.01 / 12
    gain_db = 10 * np.log10(mse_z / mse_e8)
    assert abs(gain_db - 10 * np.log10((1 / 12) / G)) < 0.06, gain_db


@pytest.mark.parametrize("bits", [2, 3])
def test_t5_relaxed_box_never_worse_than_scalar(orc, bits):
    """The relaxed box codebook contains the scalar b-bit half-integer grid, so
    per block it is never farther than scalar b-bit absmax quantisation."""
    rng = np.random.default_rng(15 + bits)
    h = ((1 << bits) - 1) / 2
    u = rng.uniform(-h, h, size=(20000, 8)).astype(np.float32)
    r = orc.e8_nearest(u, 0, bits)
    scalar = np.clip(np.ceil(u) - 0.5, -h, h)
    d_r = ((u.astype(np.float64) - r) ** 2).sum(1)
    d_s = ((u.astype(np.float64) - scalar) ** 2).sum(1)
    assert np.all(d_r <= d_s + 1e-6)


# ------------------------------------------------------------- T7 format


def _rand_fp16(rng, shape, scale=1.0):
    return (rng.normal(size=shape) * scale).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_t7_delta_round_trip_and_field_ranges(orc, bits):
    rng = np.random.default_rng(16 + bits)
    slices, T, D, G = 3, 77, 128, 64
    x = _rand_fp16(rng, (slices, T, D))
    idx, cos_, sc = orc.compress_tensor(x, T, D, bits, G, 1, 0)
    idx_d, cos_d, sc_d = orc.compress_tensor(x, T, D, bits, G, 1, 32)
    assert np.array_equal(sc, sc_d)
    a = orc.decompress_tensor(idx, cos_, sc, slices, T, D, bits, G, 0)
    b = orc.decompress_tensor(idx_d, cos_d, sc_d, slices, T, D, bits, G, 32)
    assert np.array_equal(a, b)
    # chunk starts are stored raw
    rows = np.arange(slices * T) % T
    assert np.array_equal(idx[rows % 32 == 0], idx_d[rows % 32 == 0])
    # every field < L; integer-coset fields <= L - 2
    L = 1 << bits
    bitsarr = np.unpackbits(idx, axis=1, bitorder="little").reshape(idx.shape[0], D, bits)
    fields = (bitsarr * (1 << np.arange(bits))).sum(-1)
    assert fields.max() <= L - 1
    coset_bit = (cos_[:, None] >> (np.arange(D) // 8)[None, :]) & 1
    assert np.all(fields[coset_bit == 0] <= L - 2)


def _unpack_fields(idx, bits, n):
    """b-bit fields of packed rows (field i at bit i*b, LSB first), [rows, n]."""
    a = np.unpackbits(np.atleast_2d(np.asarray(idx, np.uint8)), axis=1, bitorder="little")[:, : n * bits]
    return (a.reshape(a.shape[0], n, bits) * (1 << np.arange(bits))).sum(-1)


# Hand-computed forward differences d = (cur - prev) mod 2^b, field by field, at
# the start of the row (the rest of the 128 fields are zero in both rows).
DELTA_CASES = {
    2: ([0, 3, 1, 2, 3, 0, 2, 1], [3, 0, 2, 2, 1, 1, 3, 0], [1, 3, 3, 0, 2, 3, 3, 1]),
    3: ([0, 7, 2, 5, 6, 1, 4, 3], [7, 0, 5, 5, 2, 6, 4, 1], [1, 7, 5, 0, 4, 3, 0, 2]),
    4: ([0, 15, 3, 9, 14, 6, 8, 1], [15, 0, 12, 9, 2, 11, 8, 4], [1, 15, 7, 0, 12, 11, 0, 13]),
}


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_t7_delta_row_hand_built(orc, bits):
    """Temporal delta ("Negative results", entropy-coded indices entry: subtract
    the previous token's index): every field of the delta row is the current
    code minus the previous token's code modulo 2^b, wrap-around included, and
    the coset word is XORed.  The expected rows are packed here independently
    of the oracle.  A field-wise XOR, a reversed difference or a carry between
    fields fails this."""
    cur, prev, want = (list(v) + [0] * (128 - len(v)) for v in DELTA_CASES[bits])
    d, cw = orc.delta_row(_pack_fields(cur, bits), 0xA5C3, _pack_fields(prev, bits), 0x0FF0, 128, bits)
    assert list(_unpack_fields(d, bits, 128)[0]) == want
    assert np.array_equal(d, _pack_fields(want, bits))
    assert cw == 0xA5C3 ^ 0x0FF0 == 0xAA33
    back, c2 = orc.undelta_row(_pack_fields(want, bits), 0xAA33, _pack_fields(prev, bits), 0x0FF0, 128, bits)
    assert np.array_equal(back, _pack_fields(cur, bits)) and c2 == 0xA5C3


@pytest.mark.parametrize("bits,chunk", [(2, 32), (3, 64), (4, 512)])
def test_t7_delta_tensor_is_difference_of_raw_codes(orc, bits, chunk):
    """Along the tokens of a slice, every delta row holds the raw codes of its
    token minus those of the token before (not minus the previous stored
    delta), each chunk's first token is stored raw, scales are untouched, and
    chunk >= tokens is one chain per slice."""
    rng = np.random.default_rng(30 + bits)
    slices, T, D, G = 2, 100, 128, 64
    x = _rand_fp16(rng, (slices, T, D))
    raw_i, raw_c, raw_s = orc.compress_tensor(x, T, D, bits, G, 0, 0)
    del_i, del_c, del_s = orc.compress_tensor(x, T, D, bits, G, 0, chunk)
    assert np.array_equal(raw_s, del_s)
    L = 1 << bits
    f_raw = _unpack_fields(raw_i, bits, D).reshape(slices, T, D)
    f_del = _unpack_fields(del_i, bits, D).reshape(slices, T, D)
    c_raw = raw_c.reshape(slices, T)
    c_del = del_c.reshape(slices, T)
    for t in range(T):
        if t % chunk == 0:
            assert np.array_equal(f_del[:, t], f_raw[:, t]) and np.array_equal(c_del[:, t], c_raw[:, t])
        else:
            assert np.array_equal(f_del[:, t], (f_raw[:, t] - f_raw[:, t - 1]) % L), t
            assert np.array_equal(c_del[:, t], c_raw[:, t] ^ c_raw[:, t - 1]), t


def test_t7_delta_row_inverse(orc):
    rng = np.random.default_rng(17)
    for bits in (2, 3, 4):
        rb = 128 * bits // 8
        a = rng.integers(0, 256, size=rb).astype(np.uint8)
        p = rng.integers(0, 256, size=rb).astype(np.uint8)
        d, c = orc.delta_row(a, 0x1234, p, 0x0F0F, 128, bits)
        back, c2 = orc.undelta_row(d, c, p, 0x0F0F, 128, bits)
        assert np.array_equal(back, a) and c2 == 0x1234


# ------------------------------------------- whole-row error bound (glue pin)


@pytest.mark.parametrize("strict", [1, 0])
@pytest.mark.parametrize("bits,D,G", [(2, 128, 64), (3, 128, 64), (3, 96, 64), (2, 128, 128), (4, 64, 32)])
def test_row_reconstruction_error_bound(orc, strict, bits, D, G):
    """||x - x_hat||^2 <= dp * sum_g sc_g^2 * (blocks in g) * c, c = 2 for the
    relaxed code (it contains the scalar grid) and 4 for the strict one (one
    fix-up step costs at most 2 more), plus binary16 output rounding.  Catches a
    wrong Hadamard normalisation, scale divisor, code offset or packing."""
    rng = np.random.default_rng(18 + bits + D + strict)
    dp = orc.padded_dim(D)
    c_blk = 4.0 if strict else 2.0
    for trial in range(60):
        x = _rand_fp16(rng, D, scale=float(10.0 ** rng.integers(-3, 3)))
        idx, cw, sc = orc.encode_row(x, D, bits, G, strict)
        xh = orc.decode_row(idx, cw, sc, D, bits, G)
        xf = x.view(np.float16).astype(np.float64)
        xhf = xh.view(np.float16).astype(np.float64)
        scf = sc.view(np.float16).astype(np.float64)
        bound = dp * (scf ** 2).sum() * (G // 8) * c_blk
        err = ((xf - xhf) ** 2).sum()
        slack = ((np.abs(xhf) + np.abs(xf)) * 2.0 ** -10).__pow__(2).sum() + 1e-12
        assert err <= bound * (1 + 1e-4) + slack, (trial, err, bound)


def test_row_exact_codebook_points_round_trip(orc):
    """A row whose transform lands exactly on codebook points is reproduced."""
    rng = np.random.default_rng(19)
    bits, D, G = 3, 128, 64
    for trial in range(20):
        r = orc.e8_nearest(rng.uniform(-3.4, 3.4, size=(16, 8)).astype(np.float32), 0, bits).ravel()
        # one whole half-integer block per group reaches the box edge, so the
        # group scale comes out exactly sc
        r[0:8] = [3.5, -0.5, 0.5, 0.5, -0.5, 0.5, 1.5, -2.5]
        r[64:72] = [-3.5, 0.5, 2.5, -1.5, 0.5, 0.5, -0.5, 0.5]
        sc = 2.0 ** -6
        x = orc.fwht((r * sc).astype(np.float32))  # x = H (r * sc), exact here
        xb = x.astype(np.float16).view(np.uint16)
        assert np.array_equal(xb.view(np.float16).astype(np.float32), x)  # exact in fp16
        idx, cw, scl = orc.encode_row(xb, D, bits, G, 0)
        xh = orc.decode_row(idx, cw, scl, D, bits, G)
        assert np.array_equal(xh, xb)


def test_decode_saturates_at_fp16_max(orc):
    """A cache of +-65504 values reconstructs to finite values (no infinities)."""
    rng = np.random.default_rng(20)
    x = (np.sign(rng.normal(size=128)) * 65504.0).astype(np.float16).view(np.uint16)
    for bits in (2, 3, 4):
        idx, cw, sc = orc.encode_row(x, 128, bits, 64, 1)
        xh = orc.decode_row(idx, cw, sc, 128, bits, 64).view(np.float16)
        assert np.all(np.isfinite(xh)) and np.max(np.abs(xh.astype(np.float64))) <= 65504.0


# ------------------------------------------------ symbol statistics (report)


def _pack_fields(fields, bits):
    """LSB-first packing of b-bit fields (field i at bit i*b), written out here
    independently of the oracle."""
    nbits = len(fields) * bits
    out = np.zeros((nbits + 7) // 8, dtype=np.uint8)
    for i, f in enumerate(fields):
        for q in range(bits):
            if (int(f) >> q) & 1:
                b = i * bits + q
                out[b >> 3] |= np.uint8(1 << (b & 7))
    return out


def test_code_histogram_hand_built_rows(orc):
    """Rows whose field, byte and coset-bit counts are known by construction."""
    # b = 2, Dp = 64: fields 0,1,2,3 repeating -> every byte is 0b11100100
    idx = np.full((3, 16), 0xE4, np.uint8)
    coset = np.array([0x00FF, 0x0000, 0x000F], np.uint16)
    c = orc.code_histogram(idx, coset, 64, 2)
    assert list(c[:4]) == [48, 48, 48, 48] and not c[4:16].any()
    assert c[16 + 0xE4] == 48 and c[16:272].sum() == 48
    assert list(c[272:274]) == [12, 12]  # 8 + 0 + 4 half-coset blocks of 24
    # b = 3, Dp = 128: field i = i mod 8, fields straddle byte boundaries
    row = _pack_fields([i % 8 for i in range(128)], 3)
    c = orc.code_histogram(row[None, :], np.array([0xAAAA], np.uint16), 128, 3)
    assert list(c[:8]) == [16] * 8 and not c[8:16].any()
    assert c[16:272].sum() == 48
    # the byte pattern of 8 fields 0..7 (24 bits) repeats every 3 bytes
    assert all(c[16 + int(row[j])] == 16 for j in range(3))
    assert list(c[272:274]) == [8, 8]


def test_code_histogram_totals_on_compressed_rows(orc):
    rng = np.random.default_rng(21)
    for D, bits in ((128, 2), (96, 3), (64, 4)):
        x = rng.normal(size=(2, 40, D)).astype(np.float16).view(np.uint16)
        idx, coset, _ = orc.compress_tensor(x, 40, D, bits, 32, 1, 32)
        c = orc.code_histogram(idx, coset, D, bits)
        dp = orc.padded_dim(D)
        assert c[:16].sum() == 80 * dp and c[16:272].sum() == 80 * dp * bits // 8
        assert c[272:274].sum() == 80 * dp // 8
        assert not c[1 << bits:16].any()


def test_entropy_bits_closed_forms():
    from e8_lattice_vector_gb300.entropy import entropy_bits

    assert entropy_bits([5, 5, 5, 5]) == 2.0
    assert entropy_bits([7, 0, 0]) == 0.0
    assert abs(entropy_bits([1, 3]) - (2 - 0.75 * np.log2(3))) < 1e-12


# ------------------------------------------------ strict joint format (8b bits)


def _strict_box_points(bits):
    """Every point of strict E8 inside the b-bit box, as (fields, coset)."""
    import itertools

    L = 1 << bits
    hi0 = L // 2 - 1
    pts = []
    for r in itertools.product(range(-hi0, hi0 + 1), repeat=8):
        if sum(r) % 2 == 0:
            pts.append(([v + hi0 for v in r], 0))
    for m in itertools.product(range(L), repeat=8):
        # half-integer coordinates m - (L-1)/2: their sum is sum(m) - 4(L-1), even iff sum(m) is
        if sum(m) % 2 == 0:
            pts.append((list(m), 1))
    return pts


def test_joint_format_is_a_bijection_b2(orc):
    """All 3281 + 32768 strict box points at b = 2 get distinct 16-bit codes and
    split back to themselves."""
    pts = _strict_box_points(2)
    assert len(pts) == 3281 + 32768
    codes = set()
    for fields, c in pts:
        row = _pack_fields(fields, 2)
        j = orc.joint_pack_row(row, c, 8, 2)
        code = int(j[0]) | (int(j[1]) << 8)
        codes.add(code)
        back, c2 = orc.joint_split_row(j, 8, 2)
        assert c2 == c and np.array_equal(back, row)
    assert len(codes) == len(pts) and max(codes) < 1 << 16


def test_joint_format_round_trips_strict_decodes(orc):
    """Strict decodes at b = 3, 4 survive pack -> split; relaxed parity would
    not always (its half coset has odd sums)."""
    rng = np.random.default_rng(23)
    for bits in (3, 4):
        h = ((1 << bits) - 1) / 2
        u = rng.uniform(-h, h, size=(4000, 8)).astype(np.float32)
        for strict in (1, 0):
            r = orc.e8_nearest(u, strict, bits)
            bad = 0
            for blk in r:
                half = blk[0] != np.floor(blk[0])
                off = h if half else (1 << bits) // 2 - 1
                fields = [int(v + off) for v in blk]
                row = _pack_fields(fields, bits)
                back, c = orc.joint_split_row(orc.joint_pack_row(row, int(half), 8, bits), 8, bits)
                bad += (not np.array_equal(back, row)) or c != int(half)
            if strict:
                assert bad == 0
            else:
                assert bad > 0


def test_joint_tensor_equals_strict_tensor(orc):
    """compress(strict = 2) then decompress(joint) reconstructs exactly what
    strict = 1 does, with and without the delta; the scales are the same."""
    rng = np.random.default_rng(24)
    for D, bits, delta in ((128, 2, 0), (96, 3, 32), (64, 4, 64)):
        x = (rng.normal(size=(2, 70, D)) * 2).astype(np.float16).view(np.uint16)
        i1, c1, s1 = orc.compress_tensor(x, 70, D, bits, 64 if D > 64 else 32, 1, delta)
        i2, c2, s2 = orc.compress_tensor(x, 70, D, bits, 64 if D > 64 else 32, 2, delta)
        assert np.array_equal(s1, s2) and not c2.any()
        g = 64 if D > 64 else 32
        a = orc.decompress_tensor(i1, c1, s1, 2, 70, D, bits, g, delta)
        b = orc.decompress_tensor(i2, c2, s2, 2, 70, D, bits, g, delta, joint=True)
        assert np.array_equal(a, b)
