"""Host restatements of the index arithmetic the kernels use in strength-reduced
form, checked against the plain definitions they replace, and of the
power-of-two tie test of the E8 fast path (nq_device.cuh: TileWalkT,
PairTileAddr, e8_fast; nq_encode.cuh: load_pair_tile; the table stagers of
nq_compress.cu, nq_decompress.cu, nq_roundtrip.cu).  No GPU needed."""
import itertools
from fractions import Fraction

import numpy as np


def swz16(r, q):
    """16-row tile, 128-byte swizzle: chunk q of row r."""
    return ((q >> 3) << 11) + (r << 7) + (((q & 7) ^ (r & 7)) << 4)


def pair_chunk(dp, hf, c):
    """Global 16-byte chunk of the thread's slot chunk c in the two-thread layout."""
    q = dp // 4
    return hf * (q // 8) + c if c < q // 8 else dp // 16 + hf * (q // 8) + (c - q // 8)


def test_pair_tile_addr_split():
    # base(r) + chunk immediate, the lane's swizzle bits x0 = (hf * dp/32) ^ (r & 7)
    for dp in (64, 128):
        for hf in (0, 1):
            for r in range(16):
                base, x0 = r << 7, ((hf * (dp // 32)) ^ (r & 7)) << 4
                for c in range(dp // 16):
                    cp = c if c < dp // 32 else c + dp // 16 - dp // 32
                    assert base + ((cp >> 3) << 11) + (x0 ^ ((cp & 7) << 4)) == swz16(r, pair_chunk(dp, hf, c))


def test_full_tile_loader_split():
    # copy i of a lane is chunk g = lane + 32 i; destination = d0 + (RS i << 7) + (x0 ^ (RS (i % PER) << 4))
    for cpr in (8, 16):
        rs, per = 32 // cpr, 8 // (32 // cpr)
        for lane in range(32):
            c, r0 = lane % cpr, lane // cpr
            d0, x0 = ((c >> 3) << 11) + (r0 << 7), ((c & 7) ^ r0) << 4
            for i in range(cpr // 2):
                g = lane + 32 * i
                assert d0 + ((rs * i) << 7) + (x0 ^ ((rs * (i % per)) << 4)) == swz16(g // cpr, g % cpr)


def test_table_stagers_cover_the_same_copies():
    # (plane, token row) pairs each thread copies: strided loop over g versus one token row per thread
    for d, rows, threads in ((128, 16, 256), (64, 16, 256), (128, 32, 128), (96, 32, 128), (64, 32, 128),
                             (128, 16, 512), (64, 16, 512)):
        qs = threads // rows
        for t in range(threads):
            old = [(g // rows, g % rows) for g in range(t, (d // 4) * rows, threads)]
            new = [(t // rows + qs * j, t % rows) for j in range((d // 4 + qs - 1) // qs)
                   if (d // 4) % qs == 0 or t // rows + qs * j < d // 4]
            assert new == old


class _WalkByDivision:
    def __init__(self, first, step, slices, tokens, chunk, rows):
        self.step, self.chunk, self.tokens, self.rows = step, chunk, tokens, rows
        self.nchunks = (tokens + chunk - 1) // chunk
        self.items = slices * self.nchunks
        self.set(first)

    def set(self, it):
        self.item = it
        if it < self.items:
            self.slice = it // self.nchunks
            self.t_begin = (it - self.slice * self.nchunks) * self.chunk
            self.t_end = min(self.t_begin + self.chunk, self.tokens)
            self.t0 = self.t_begin

    def valid(self):
        return self.item < self.items

    def next(self):
        self.t0 += self.rows
        if self.t0 >= self.t_end:
            self.set(self.item + self.step)


class _WalkByCarry:
    def __init__(self, first, step, slices, tokens, chunk, rows):
        self.slices, self.chunk, self.tokens, self.rows = slices, chunk, tokens, rows
        self.nchunks = (tokens + chunk - 1) // chunk
        self.slice, self.c, self.dslice, self.dc = slices, 0, 0, 0
        if self.nchunks > 0:
            self.slice, self.c = divmod(first, self.nchunks)
            self.dslice, self.dc = divmod(step, self.nchunks)
        self.t0 = self.c * chunk

    def valid(self):
        return self.slice < self.slices

    def t_begin(self):
        return self.c * self.chunk

    def t_end(self):
        return min(self.c * self.chunk + self.chunk, self.tokens)

    def next(self):
        self.t0 += self.rows
        if self.t0 >= self.t_end():
            self.slice += self.dslice
            self.c += self.dc
            if self.c >= self.nchunks:
                self.c -= self.nchunks
                self.slice += 1
            self.t0 = self.c * self.chunk


def test_tile_walk_by_carry_matches_division():
    for tokens in (0, 1, 15, 16, 17, 33, 100, 512):
        for chunk in (16, 32, 256):
            for slices in (1, 3, 17):
                for step in (1, 2, 7, 152, 2432):
                    for first in sorted({0, 1, step - 1, min(step, 5)}):
                        a = _WalkByDivision(first, step, slices, tokens, chunk, 16)
                        b = _WalkByCarry(first, step, slices, tokens, chunk, 16)
                        for _ in range(2000):
                            assert a.valid() == b.valid()
                            if not a.valid():
                                break
                            assert (a.slice, a.t0, a.t_begin, a.t_end) == (b.slice, b.t0, b.t_begin(), b.t_end())
                            a.next()
                            b.next()


def test_single_power_of_two_tie_test():
    """For b <= 3: fma(G_hi, L^4, G_lo) over any nonempty signed set of the terms
    L^j / 2 (j < 4 in G_lo, L^(j-4) / 2 in G_hi) is exact in fp32 and is a
    power of two exactly when the set has one term."""
    for b in (2, 3):
        L = 1 << b
        for signs in itertools.product((-1, 0, 1), repeat=8):
            if not any(signs):
                continue
            gx, gy = np.float32(0), np.float32(0)
            for j, s in enumerate(signs):
                if s and j < 4:
                    gx = np.float32(gx + np.float32(s * L ** j / 2))
                elif s:
                    gy = np.float32(gy + np.float32(s * L ** (j - 4) / 2))
            t = np.float32(float(gy) * L ** 4 + float(gx))
            exact = sum(s * Fraction(L ** j, 2) for j, s in enumerate(signs))
            assert Fraction(float(t)) == exact
            pow2 = (np.array(t, np.float32).view(np.uint32) & 0x7FFFFF) == 0
            assert pow2 == (sum(1 for s in signs if s) == 1)
