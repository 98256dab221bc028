"""Pins for the oracle's compressor, exp_own and RoPE (CPU only)."""

import math

import numpy as np
import pytest

from oracle import compress, expo, rope


def _toy(golden):
    g = golden["compressor_toy_block"]
    v = np.array(g["values"], np.float64)
    sa = np.array([0, 0, 0, math.log(5.0)])
    sb = np.array(g["channel_B_scores"], np.float64)
    kv = np.stack([v, v], axis=-1)[:, None, :]          # [T=4, coff=1, D=2]
    gate = np.stack([sa, sb], axis=-1)[:, None, :]
    ape = np.zeros((4, 2))
    return g, kv, gate, ape


def test_toy_block_definition(golden):
    g, kv, gate, ape = _toy(golden)
    out = compress.compress_fp64(kv, gate, ape, ratio=4, overlap=False)
    assert out.shape == (1, 2)
    assert out[0, 0] == pytest.approx(g["channel_A_entry"], abs=1e-12)
    assert out[0, 1] == pytest.approx(g["channel_B_entry"], abs=1e-12)
    # the printed weights
    w = np.exp(gate[:, 0, 0]) / np.exp(gate[:, 0, 0]).sum()
    assert np.allclose(w, g["channel_A_weights"], atol=1e-12)


def test_toy_block_contract(golden):
    g, kv, gate, ape = _toy(golden)
    out = compress.compress_contract(kv.astype(np.float32), gate.astype(np.float32),
                                     ape.astype(np.float32), ratio=4, overlap=False)
    assert out[0, 0] == pytest.approx(g["channel_A_entry"], rel=4e-7)
    assert out[0, 1] == g["channel_B_entry"]          # equal weights: exact


def test_equal_gates_give_mean_and_dominant_gate_gives_token():
    rs = np.random.default_rng(0)
    kv = rs.standard_normal((128, 1, 64)).astype(np.float32)
    gate = np.full((128, 1, 64), 0.75, np.float32)
    ape = np.zeros((128, 64), np.float32)
    out = compress.compress_contract(kv, gate, ape, ratio=128, overlap=False)
    assert np.allclose(out[0], kv[:, 0].astype(np.float64).mean(0), atol=2e-6)
    gate2 = np.zeros((128, 1, 64), np.float32)
    gate2[37] = 60.0
    out2 = compress.compress_contract(kv, gate2, ape, ratio=128, overlap=False)
    assert np.array_equal(out2[0], kv[37, 0])


def test_v41_ratio1_entry_is_the_token():
    """The V4.1 decoder compressor keeps one entry per position (m = 1, no overlap,
    no slot bias): the softmax over a single slot is 1, so the pooled entry is the
    token's projected value itself, in the definition and bit for bit in the contract."""
    rs = np.random.default_rng(2)
    kv = rs.standard_normal((40, 1, 32)).astype(np.float32)
    gate = (3 * rs.standard_normal((40, 1, 32))).astype(np.float32)
    ape = np.zeros((1, 32), np.float32)
    assert np.array_equal(compress.compress_fp64(kv, gate, ape, ratio=1, overlap=False), kv[:, 0])
    assert np.array_equal(compress.compress_contract(kv, gate, ape, ratio=1, overlap=False), kv[:, 0])


def test_v41_ratio2_pairs_are_a_logistic_blend():
    """The V4.1 encoder compressor merges 2 adjacent positions (m = 2, no overlap, no
    slot bias): entry i = v_{2i} * sigma(g_{2i} - g_{2i+1}) + v_{2i+1} * sigma(g_{2i+1} - g_{2i})
    per channel (a two-way softmax is a logistic function), and a dominant gate on one
    token of the pair returns that token."""
    rs = np.random.default_rng(3)
    T, D = 64, 16
    kv = rs.standard_normal((T, 1, D))
    gate = 2 * rs.standard_normal((T, 1, D))
    ape = np.zeros((2, D))
    out = compress.compress_fp64(kv, gate, ape, ratio=2, overlap=False)
    v0, v1 = kv[0::2, 0], kv[1::2, 0]
    g0, g1 = gate[0::2, 0], gate[1::2, 0]
    sig = 1.0 / (1.0 + np.exp(g1 - g0))
    assert np.allclose(out, v0 * sig + v1 * (1.0 - sig), rtol=0, atol=1e-12)
    c32 = compress.compress_contract(kv.astype(np.float32), gate.astype(np.float32), ape.astype(np.float32),
                                     ratio=2, overlap=False)
    assert np.allclose(c32, out, rtol=0, atol=4e-6 * np.abs(kv).max())
    g2 = np.zeros((T, 1, D), np.float32)
    g2[2 * 5 + 1] = 80.0                      # the second token of pair 5
    g2[2 * 9] = 80.0                          # the first token of pair 9
    c = compress.compress_contract(kv.astype(np.float32), g2, ape.astype(np.float32), ratio=2, overlap=False)
    assert np.array_equal(c[5], kv[11, 0].astype(np.float32))
    assert np.array_equal(c[9], kv[18, 0].astype(np.float32))
    assert np.array_equal(c[3], ((kv[6, 0].astype(np.float32) + kv[7, 0].astype(np.float32)) / np.float32(2))
                          .astype(np.float32))


def test_ten_token_prompt_overlap_structure(golden):
    g = golden["ten_token_prompt"]
    T = g["tokens"]
    rs = np.random.default_rng(1)
    D = 16
    kv = rs.standard_normal((T, 2, D))
    gate = rs.standard_normal((T, 2, D))
    ape = rs.standard_normal((4, 2 * D))
    done = (T // 4) * 4                   # the compressor only sees completed blocks
    base = compress.compress_fp64(kv[:done], gate[:done], ape, 4, True)
    assert base.shape[0] == len(g["csa_entries"])
    for e in g["csa_entries"]:
        lo, hi = e["tokens"]
        assert e["position"] == e["entry"] * 4
        for tok in range(T):
            kv2 = kv.copy()
            kv2[tok] += 1.0
            out = compress.compress_fp64(kv2[:done], gate[:done], ape, 4, True)
            changed = not np.allclose(out[e["entry"]], base[e["entry"]])
            assert changed == (lo <= tok <= hi), (e, tok)
    assert (T // 128) == g["hca_entries"]
    assert list(range(done, T)) == g["csa_pending"]


def test_first_entry_reads_nothing_before_the_sequence():
    rs = np.random.default_rng(2)
    D = 32
    kv = rs.standard_normal((8, 2, D))
    gate = rs.standard_normal((8, 2, D))
    ape = rs.standard_normal((4, 2 * D))
    out = compress.compress_fp64(kv, gate, ape, 4, True)
    # entry 0 == plain pooling of tokens 0..3 through channel half 1 with ape[:, D:]
    alone = compress.compress_fp64(kv[:4, 1:2], gate[:4, 1:2], ape[:, D:], 4, False)
    assert np.allclose(out[0], alone[0], atol=1e-14)


def test_chunked_equals_whole_bit_exact():
    rs = np.random.default_rng(3)
    D = 64
    T = 64
    kv = rs.standard_normal((T, 2, D)).astype(np.float32)
    gate = rs.standard_normal((T, 2, D)).astype(np.float32)
    ape = rs.standard_normal((4, 2 * D)).astype(np.float32)
    nw = rs.uniform(0.5, 1.5, D).astype(np.float32)
    cs = rope.table(np.arange(T // 4) * 4)
    whole = compress.compress_contract(kv, gate, ape, 4, True, norm_w=nw, rope_cs=cs)
    a = compress.compress_contract(kv[:32], gate[:32], ape, 4, True, norm_w=nw, rope_cs=cs[:8])
    b = compress.compress_contract(kv[32:], gate[32:], ape, 4, True, prev_kv=kv[28:32],
                                   prev_gate=gate[28:32], norm_w=nw, rope_cs=cs[8:])
    assert np.array_equal(whole, np.concatenate([a, b]))


@pytest.mark.parametrize("ratio,overlap", [(4, True), (128, False)])
def test_contract_close_to_definition(ratio, overlap):
    rs = np.random.default_rng(4)
    D = 512
    T = ratio * 6
    coff = 2 if overlap else 1
    kv = rs.standard_normal((T, coff, D)).astype(np.float32)
    gate = rs.standard_normal((T, coff, D)).astype(np.float32)
    ape = (0.5 * rs.standard_normal((ratio, coff * D))).astype(np.float32)
    nw = rs.uniform(0.5, 1.5, D).astype(np.float32)
    pos = np.arange(T // ratio) * ratio + 1000
    c32 = compress.compress_contract(kv, gate, ape, ratio, overlap, norm_w=nw, eps=1e-6,
                                     rope_cs=rope.table(pos))
    c64 = compress.compress_fp64(kv, gate, ape, ratio, overlap, norm_w=nw, eps=1e-6, positions=pos)
    assert np.max(np.abs(c32 - c64)) < 3e-6 * np.max(np.abs(c64))


def test_rmsnorm_unit_weight_gives_unit_rms():
    rs = np.random.default_rng(5)
    kv = (3.0 * rs.standard_normal((16, 1, 512)))
    gate = rs.standard_normal((16, 1, 512))
    out = compress.compress_fp64(kv, gate, np.zeros((4, 512)), 4, False, norm_w=np.ones(512), eps=0.0)
    assert np.allclose(np.sqrt(np.mean(out ** 2, axis=-1)), 1.0, atol=1e-12)


def test_pairwise_sum_order():
    # recursive halves: (1 + 2^-24) + (0 + 2^-24) = 1 in fp32; an interleaved order would give 1 + 2^-23
    v = np.array([1.0, 2.0 ** -24, 0.0, 2.0 ** -24], np.float32)
    assert compress.pairwise_sum_f32(v) == np.float32(1.0)
    ints = np.arange(512, dtype=np.float32)
    assert compress.pairwise_sum_f32(ints) == 511 * 512 / 2


def test_thousand_token_counts(golden):
    g = golden["thousand_token_prompt"]
    T = g["tokens"]
    assert T // 4 == g["csa_entries"]
    assert T // 128 == g["hca_entries"]
    assert [0, (T // 128) * 128 - 1] == g["hca_covered_tokens"]
    assert T - (T // 128) * 128 == g["hca_pending"]


# ---------------------------------------------------------------- exp_own

def test_exp_own_accuracy_and_edges():
    x = np.linspace(-87.0, 0.0, 400001).astype(np.float32)
    got = expo.exp_own(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - ref) / ulp) <= 2.0
    assert expo.exp_own(np.float32(0.0)) == 1.0
    assert expo.exp_own(np.float32(-np.inf)) == 0.0
    assert expo.exp_own(np.float32(-110.0)) == 0.0
    assert np.all(np.diff(got) >= 0)
    assert float(expo.LN2_HI) * 65536 == round(float(expo.LN2_HI) * 65536)
    assert abs(float(expo.LN2_HI) + float(expo.LN2_LO) - math.log(2.0)) < 1e-12


# ---------------------------------------------------------------- RoPE

def test_rope_relative_example(golden):
    g = golden["rope_relative"]
    th = math.radians(g["theta_degrees"])
    u = np.zeros((1, 512))
    u[0, -64] = 1.0                           # pair 0 of the rope dims, along the first axis
    for shift in (0, g["shift"]):
        key = rope.rotate_fp64(u, np.full((1, 32), th * (g["key_position"] + shift)))
        back = rope.rotate_fp64(key, np.full((1, 32), th * (g["query_position"] + shift)), inverse=True)
        ang = math.degrees(math.atan2(back[0, -63], back[0, -64]))
        assert ang == pytest.approx(g["net_degrees"], abs=1e-9)


def test_rope_table_and_frequencies():
    t = rope.table(np.array([0, 1, 12345]))
    assert np.array_equal(t[0, :, 0], np.ones(32, np.float32)) and np.all(t[0, :, 1] == 0)
    f = rope.inv_freq()
    assert f[0] == 1.0 and f[-1] == pytest.approx(160000.0 ** (-62 / 64))
    assert t[1, 0, 0] == np.float32(math.cos(1.0)) and t[1, 0, 1] == np.float32(math.sin(1.0))
    # fp32 contract rotation preserves pair norms to rounding
    y = np.random.default_rng(6).standard_normal((3, 512)).astype(np.float32)
    r = rope.rotate_table_fp32(y, t)
    n0 = np.hypot(y[:, -64::2], y[:, -63::2])
    n1 = np.hypot(r[:, -64::2], r[:, -63::2])
    assert np.allclose(n0, n1, rtol=1e-6) and np.array_equal(y[:, :448], r[:, :448])


# ---------------------------------------------------------------- overlap halves

@pytest.mark.parametrize("render", ["fp64", "contract"])
def test_overlap_channel_halves_by_perturbation(render):
    """"DeepSeek-V4 deep dive", section 4.2 (the overlap transform): every token feeds two
    entries - the next block's entry through channel half 0 (as part of its previous
    block) and its own block's entry through half 1.  So perturbing half 0 of token 4i+j
    may change entry i+1 only (and must change it), and perturbing half 1 may change
    entry i only (and must change it).  The halves are perturbed one at a time."""
    rs = np.random.default_rng(12)
    D, T = 8, 24
    kv = rs.standard_normal((T, 2, D)).astype(np.float32)
    gate = rs.standard_normal((T, 2, D)).astype(np.float32)
    ape = rs.standard_normal((4, 2 * D)).astype(np.float32)
    run = ((lambda k, g, a: compress.compress_fp64(k, g, a, 4, True)) if render == "fp64"
           else (lambda k, g, a: compress.compress_contract(k, g, a, 4, True)))
    base = run(kv, gate, ape)
    n = T // 4
    for tok in range(T):
        i = tok // 4
        for half, expect in ((0, i + 1), (1, i)):
            kv2 = kv.copy()
            kv2[tok, half] += np.float32(0.75)
            out = run(kv2, gate, ape)
            changed = [e for e in range(n) if not np.array_equal(out[e], base[e])]
            want = [expect] if expect < n else []
            assert changed == want, (render, tok, half, changed, want)


def test_overlap_slot_bias_halves_pick_the_right_tokens():
    """The slot bias is added before the overlap transform (section 4.2): slots 0-3 (the
    previous block, channel half 0) carry ape[:, :D], slots 4-7 (the entry's own block,
    half 1) carry ape[:, D:].  A dominant bias on one slot of one half makes that slot's
    token win the softmax, so the pooled channel equals that token's value in that half:
    ape[j, c] (half 0) gives token 4(i-1)+j's half-0 value to entry i >= 1, and
    ape[j, D + c] gives token 4i+j's half-1 value to entry i."""
    rs = np.random.default_rng(13)
    D, T = 16, 20
    kv = rs.standard_normal((T, 2, D)).astype(np.float32)
    gate = (0.1 * rs.standard_normal((T, 2, D))).astype(np.float32)
    for j in range(4):
        for c in (0, 5, D - 1):
            for half in (0, 1):
                ape = np.zeros((4, 2 * D), np.float32)
                ape[j, half * D + c] = 80.0
                for render in (compress.compress_fp64, compress.compress_contract):
                    out = render(kv, gate, ape, 4, True)
                    for i in range(T // 4):
                        if half == 0:
                            if i == 0:
                                continue      # no previous block: its slots weigh nothing
                            want = kv[4 * (i - 1) + j, 0, c]
                        else:
                            want = kv[4 * i + j, 1, c]
                        assert np.float32(out[i, c]) == want, (render.__name__, j, c, half, i)
