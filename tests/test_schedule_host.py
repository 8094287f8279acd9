"""Arithmetic of the tensor-core kernels' tile schedule, restated in Python.

The device code hands each CTA pair units p, p + pairs, ... and decodes a unit into a
token (M) tile, a vocabulary (N) group and, for a split dH launch, a K part: the part
slowest, then bands of `band` tiles of the first-walked dimension, inside a band that
dimension fastest.  The forward's planner picks the vocabulary tiles per unit from the
makespan of that order.  These tests restate both formulas and check the properties the
kernels rely on: the decode maps the units one-to-one onto every (tile, group, part),
never outside the valid ranges, and the planner's closed-form makespan equals the load of
the most loaded pair counted unit by unit.  They check the scheme, not the compiled code
(the GPU parity tests cover that)."""
import random


def cdiv(a, b):
    return (a + b - 1) // b


def decode(order, band, k_split, m_tiles, n_groups, u):
    ks = 0
    if k_split > 1:
        per_part = m_tiles * n_groups
        ks, u = divmod(u, per_part)
    fast, slow = (m_tiles, n_groups) if order == 0 else (n_groups, m_tiles)
    if 0 < band < fast:
        per_band = band * slow
        b, r = divmod(u, per_band)
        width = min(band, fast - b * band)
        sl, f = divmod(r, width)
        f += b * band
    else:
        sl, f = divmod(u, fast)
    mt, g = (f, sl) if order == 0 else (sl, f)
    return mt, g, ks


def k_range(ks, k_split, k_blocks):
    k_split = max(k_split, 1)
    return ks * k_blocks // k_split, (ks + 1) * k_blocks // k_split


def count_congruent(lo, hi, r, mod):
    if hi <= lo:
        return 0
    upto = lambda x: 0 if x <= r else (x - 1 - r) // mod + 1
    return upto(hi) - upto(lo)


def lse_makespan(m_tiles, v_tiles, G, band, pairs, max_bands_exact=64):
    ng = cdiv(v_tiles, G)
    units = m_tiles * ng
    last = v_tiles - (ng - 1) * G
    bw = band if (0 < band < m_tiles and cdiv(m_tiles, band) <= max_bands_exact) else m_tiles
    t = 0
    for p in range(pairs):
        tail, b0 = 0, 0
        while b0 < m_tiles:
            w = min(bw, m_tiles - b0)
            start = b0 * ng + (ng - 1) * w
            tail += count_congruent(start, start + w, p, pairs)
            b0 += bw
        t = max(t, G * count_congruent(0, units, p, pairs) - (G - last) * tail)
    return t


def test_decode_is_a_bijection_onto_the_valid_tiles():
    rng = random.Random(7)
    for _ in range(600):
        order = rng.choice([0, 1])
        band = rng.choice([0, 1, 5, 16, 64])
        k_split = rng.choice([0, 1, 2, 3, 4])
        m_tiles = rng.choice([1, 2, 15, 16, 17, 32, 33, 128])
        n_groups = rng.randint(1, 70)
        parts = max(k_split, 1)
        seen = set()
        for u in range(parts * m_tiles * n_groups):
            mt, g, ks = decode(order, band, k_split, m_tiles, n_groups, u)
            assert 0 <= mt < m_tiles and 0 <= g < n_groups and 0 <= ks < parts
            seen.add((mt, g, ks))
        assert len(seen) == parts * m_tiles * n_groups


def test_k_parts_cover_the_k_range_once_and_are_never_empty():
    for k_blocks in range(1, 200):
        for k_split in range(1, 5):
            if k_split > k_blocks:  # the host never splits into more parts than K blocks
                continue
            ranges = [k_range(ks, k_split, k_blocks) for ks in range(k_split)]
            assert ranges[0][0] == 0 and ranges[-1][1] == k_blocks
            assert all(a < b for a, b in ranges)
            assert all(ranges[i][1] == ranges[i + 1][0] for i in range(k_split - 1))


def test_planner_makespan_equals_the_unit_by_unit_load():
    rng = random.Random(11)
    checked = 0
    for _ in range(1500):
        m = rng.choice([1, 2, 15, 16, 17, 31, 32, 33, 64, 100, 128, 129, 500])
        v = rng.randint(1, 1200)
        G = rng.randint(4, 8)
        band = rng.choice([0, 1, 5, 16, 64])
        pairs = rng.choice([1, 7, 13, 76])
        if not (band <= 0 or band >= m or cdiv(m, band) <= 64):
            continue  # past 64 bands the planner counts the tail as if unbanded
        ng = cdiv(v, G)
        load = [0] * pairs
        for u in range(m * ng):
            mt, g, _ = decode(0, band, 1, m, ng, u)
            load[u % pairs] += min(G, v - g * G)
        assert lse_makespan(m, v, G, band, pairs) == max(load)
        checked += 1
    assert checked > 1000
