"""Pins for the oracle's decode-step state update and YaRN table (CPU only)."""

import numpy as np
import pytest

from oracle import compress, decode_state, rope


def _stream(ratio, overlap, T, D, seed, zero_bias=False):
    rs = np.random.default_rng(seed)
    coff = 2 if overlap else 1
    kv = rs.standard_normal((T, coff, D)).astype(np.float32)
    gate = (1.5 * rs.standard_normal((T, coff, D))).astype(np.float32)
    ape = np.zeros((ratio, coff * D), np.float32) if zero_bias else \
        (0.5 * rs.standard_normal((ratio, coff * D))).astype(np.float32)
    nw = rs.uniform(0.5, 1.5, D).astype(np.float32)
    return kv, gate, ape, nw


@pytest.mark.parametrize("ratio,overlap,zero_bias", [(4, True, False), (128, False, False), (2, False, True),
                                                     (1, False, True), (4, False, False)])
def test_streamed_decode_equals_whole_sequence(ratio, overlap, zero_bias):
    """Pushing the tokens one decode step at a time emits, bit for bit, the entries the
    whole-sequence compressor computes, each at the step that completes its block."""
    T, D = ratio * 9 + (ratio - 1), 64
    kv, gate, ape, nw = _stream(ratio, overlap, T, D, seed=ratio, zero_bias=zero_bias)
    st = decode_state.CompressorState(ratio, overlap, D)
    got = {}
    for p in range(T):
        out = st.push(p, kv[p], gate[p], ape, norm_w=nw, yarn=rope.YARN_V4)
        if out is not None:
            j, e = out
            assert p == (j + 1) * ratio - 1          # emitted exactly when its block completes
            got[j] = e
    n = T // ratio
    assert sorted(got) == list(range(n))
    whole = compress.compress_contract(kv[:n * ratio], gate[:n * ratio], ape, ratio, overlap, norm_w=nw,
                                       rope_cs=rope.table(np.arange(n) * ratio, yarn=rope.YARN_V4))
    assert np.array_equal(np.stack([got[j] for j in range(n)]), whole)


def test_thousand_token_prompt_state(golden):
    """After 1,000 tokens: a CSA compressor has written 250 entries and still holds
    tokens 996-999 for the next entry's overlap; an HCA compressor has written 7 entries
    (tokens 0-895) and holds the 104 pending tokens 896-999."""
    g = golden["thousand_token_prompt"]
    T, D = g["tokens"], 64
    kv4, gate4, ape4, _ = _stream(4, True, T, D, seed=1)
    kv128, gate128, ape128, _ = _stream(128, False, T, D, seed=2)
    csa = decode_state.CompressorState(4, True, D)
    hca = decode_state.CompressorState(128, False, D)
    n4, n128 = [], []
    for p in range(T):
        if csa.push(p, kv4[p], gate4[p], ape4) is not None:
            n4.append(p)
        if hca.push(p, kv128[p], gate128[p], ape128) is not None:
            n128.append(p)
    assert len(n4) == g["csa_entries"] and len(n128) == g["hca_entries"]
    assert n128[-1] + 1 - 128 * len(n128) == 0 and n128[-1] == g["hca_covered_tokens"][1]
    k0, k1 = g["csa_overlap_kept_tokens"]
    assert np.array_equal(csa.kv[:4], kv4[k0:k1 + 1])          # the previous-block slots
    pend = T - 128 * len(n128)
    assert pend == g["hca_pending"]
    assert np.array_equal(hca.kv[:pend], kv128[T - pend:])       # tokens 896-999 wait in slots 0-103


def test_first_block_sees_an_empty_previous_block():
    """A fresh state's previous-block slots (kv 0, score -inf) weigh nothing: the first
    entry equals pooling the first block's own half-1 tokens alone."""
    D = 64
    kv, gate, ape, _ = _stream(4, True, 4, D, seed=3)
    st = decode_state.CompressorState(4, True, D)
    for p in range(4):
        out = st.push(p, kv[p], gate[p], ape)
    s = gate[:, 1].astype(np.float64) + ape[:, D:].astype(np.float64)
    w = np.exp(s - s.max(0)) / np.exp(s - s.max(0)).sum(0)
    assert np.allclose(out[1], (w * kv[:, 1]).sum(0), rtol=0, atol=3e-6)


def test_window_row_is_normalised_and_rotated_to_its_position():
    rs = np.random.default_rng(4)
    D, p = 512, 300_000
    x = rs.standard_normal(D).astype(np.float32)
    nw = rs.uniform(0.5, 1.5, D).astype(np.float32)
    slot, row = decode_state.window_row(x, p, norm_w=nw, yarn=rope.YARN_V4)
    assert slot == p % 128
    y = x.astype(np.float64) / np.sqrt(np.mean(x.astype(np.float64) ** 2) + 1e-6) * nw
    ref = rope.rotate_fp64(y, rope.angles([p], yarn=rope.YARN_V4)[0])
    assert np.allclose(row, ref, rtol=0, atol=2e-5 * np.abs(ref).max())


def test_yarn_pairs_follow_the_printed_split(golden):
    g = golden["yarn_split"]
    yarn = dict(factor=g["factor"], original=g["original_max_position_embeddings"],
                beta_fast=g["beta_fast"], beta_slow=g["beta_slow"])
    assert yarn == {kk: rope.YARN_V4[kk] for kk in yarn}
    assert g["original_max_position_embeddings"] * g["factor"] == g["max_position_embeddings"]
    f0 = rope.inv_freq(g["base"])
    f = rope.inv_freq(g["base"], yarn=yarn)
    ratio = f / f0
    u0, u1 = g["unchanged_pairs"]
    b0, b1 = g["blended_pairs"]
    d0, d1 = g["divided_pairs"]
    assert np.all(ratio[u0:u1 + 1] == 1.0)
    assert np.all((ratio[b0:b1 + 1] < 1.0) & (ratio[b0:b1 + 1] > 1.0 / g["factor"]))
    assert np.all(np.diff(ratio[b0:b1 + 1]) < 0)                   # a monotone ramp between them
    assert np.allclose(ratio[d0:d1 + 1], 1.0 / g["factor"], rtol=1e-15)
    for k, lam in g["wavelength_tokens_about"].items():
        assert abs(2 * np.pi / f0[int(k)] - lam) <= 0.05 * lam
    # the plain table is the one without YaRN
    assert np.array_equal(rope.table([12345]), rope.table([12345], yarn=None))
    assert not np.array_equal(rope.table([1_000_000]), rope.table([1_000_000], yarn=yarn))


def test_product_rope_tables_equal_the_oracle_tables():
    """The library's host table (cskv_rope_table, an input of the CUDA path) and the oracle's
    table agree bit for bit, with and without YaRN, on the edges and 4,096 random positions."""
    import compressed_sparse_attention_kv_gb300 as cskv
    pos = np.concatenate([[0, 1, 2, 127, 4096, 65535, 65536, 524287, 1048575],
                          np.random.default_rng(9).integers(0, 1 << 21, 4096)])
    assert np.array_equal(cskv.rope_table(pos), rope.table(pos))
    assert np.array_equal(cskv.rope_table(pos, yarn=cskv.YARN_V4), rope.table(pos, yarn=rope.YARN_V4))
