"""A host model of the split softmax the attention kernels run ("DeepSeek-V4 deep dive",
section 3.4, Eq. 27: one softmax over the window and the compressed keys, with the
per-head sink in the denominator), in the arithmetic the kernels use: each 128-key
tile keeps its base-2 maximum m, its sum l of exp2(z - m) and its output as O / l
rounded to bf16; the merge starts from the sink and rescales in fp32, a tile entering
with weight exp2(m - M) * l.  Checked against the softmax written out in fp64: the
error stays within the bf16 rounding of the partials, whatever the values' scale, and
empty tiles drop out."""

import numpy as np

LOG2E = 1.4426950408889634


def _bf16(x):
    """fp32 -> bf16 (round to nearest even), returned as fp32."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _tile_partial(z, v):
    """z: [n] logits (already times the softmax scale), v: [n, d].  Returns fp32 m (base
    2), l and bf16 O / l, as a tile stores them; an empty tile gives (-inf, 0, 0)."""
    if len(z) == 0:
        return np.float32(-np.inf), np.float32(0), np.zeros(v.shape[1], np.float32)
    t = np.float32(z * LOG2E)
    m = t.max()
    p = np.exp2(t - m).astype(np.float32)
    l = p.sum(dtype=np.float32)
    o = (p[:, None] * v).sum(0, dtype=np.float32)
    return m, l, _bf16(o * np.float32(1.0 / l))


def _merge(parts, sink):
    """The combine's order: the sink first, then batches of eight tiles."""
    M = np.float32(sink * LOG2E) if sink is not None else np.float32(-np.inf)
    L = np.float32(1.0 if sink is not None else 0.0)
    o = np.zeros(parts[0][2].shape, np.float32)
    for s0 in range(0, len(parts), 8):
        batch = parts[s0:s0 + 8]
        Mb = max([M] + [m for m, _, _ in batch])
        if Mb == -np.inf:
            continue
        f = np.float32(0) if M == -np.inf else np.exp2(np.float32(M - Mb))
        L, o = L * f, o * f
        for m, l, ov in batch:
            if m == -np.inf:
                continue
            g = np.float32(np.exp2(np.float32(m - Mb)) * l)
            L, o = L + g, o + g * ov
        M = Mb
    return o * np.float32(1.0 / L) if L > 0 else o


def _exact(z, v, sink):
    zz = np.concatenate([z, [sink]]) if sink is not None else z
    e = np.exp(zz - zz.max())
    return (e[:len(z), None] * v).sum(0) / e.sum()


def _split(n, rs):
    """Tile sizes: 128-key tiles with some left empty or ragged (padding, -1 entries)."""
    sizes = []
    while n > 0:
        s = int(min(n, rs.choice([128, 128, 128, 77, 0, 1])))
        sizes.append(s)
        n -= s
    return sizes + [0]


def test_merge_matches_the_softmax_within_the_partials_rounding():
    rs = np.random.default_rng(5)
    for case in range(40):
        n, d = int(rs.integers(1, 700)), 64
        scale = 10.0 ** rs.uniform(-3, 30)             # any bf16-representable scale
        v = _bf16(rs.standard_normal((n, d)).astype(np.float32) * np.float32(scale))
        z = (rs.standard_normal(n) * rs.uniform(0.1, 6)).astype(np.float32)
        sink = float(rs.standard_normal()) if case % 3 else None
        sizes = _split(n, rs)
        parts, i = [], 0
        for s in sizes:
            parts.append(_tile_partial(z[i:i + s], v[i:i + s]))
            i += s
        got = _merge(parts, sink).astype(np.float64)
        ref = _exact(z.astype(np.float64), v.astype(np.float64), sink)
        vmax = float(np.abs(v).max())
        # bf16 partials: 2^-9 of each |O / l| <= max|v| (weights sum to at most 1); the
        # fp32 sums and exp2 add well under that
        assert np.all(np.isfinite(got)), case
        assert np.max(np.abs(got - ref)) <= (2.0 ** -9 + 2.0 ** -16) * vmax, case


def test_empty_tiles_drop_out_and_an_empty_list_gives_zero():
    rs = np.random.default_rng(6)
    v = rs.standard_normal((130, 16)).astype(np.float32)
    z = rs.standard_normal(130).astype(np.float32)
    full = [_tile_partial(z[:128], v[:128]), _tile_partial(z[128:], v[128:])]
    with_empty = [full[0], _tile_partial(z[:0], v[:0]), full[1], _tile_partial(z[:0], v[:0])]
    assert np.array_equal(_merge(full, 0.3), _merge(with_empty, 0.3))
    nothing = [_tile_partial(z[:0], v[:0])] * 3
    assert np.array_equal(_merge(nothing, 0.3), np.zeros(16, np.float32))
    assert np.array_equal(_merge(nothing, None), np.zeros(16, np.float32))


def test_normalised_partials_keep_the_values_range():
    """O / l lies within the tile's values, so it cannot overflow where they do not; an
    unnormalised O (up to 128 times the largest value) would overflow f16 at values of a
    few hundred."""
    v = np.full((128, 8), 600.0, np.float32)
    z = np.zeros(128, np.float32)
    m, l, ov = _tile_partial(z, v)
    assert l == 128 and np.all(ov == 600.0)
    with np.errstate(over="ignore"):
        assert np.all(np.isinf((l * ov).astype(np.float16)))
