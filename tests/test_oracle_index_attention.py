"""Pins for the oracle's indexer, top-k and attention (CPU only)."""

import itertools

import numpy as np
import pytest
import torch

from oracle import attention, codecs, indexer, rope


# ---------------------------------------------------------------- indexer / top-k

def test_tiny_csa_selection(golden):
    g = golden["tiny_csa_selection"]
    t = g["query_position"]
    n = int(indexer.visible_entries(t + 1, g["ratio"]))
    assert n == g["visible_blocks"]
    # one head, w = 1, scores scaled to integers: 0.1, 0.9, 0, 0.4, 0.7 -> 1, 9, 0, 4, 7
    q = np.zeros((1, 128))
    q[0, 0] = 1.0
    keys = np.zeros((n, 128))
    keys[:, 0] = [round(10 * s) for s in g["block_scores"]]
    top, I = indexer.index_topk(q, np.ones(1), keys, t + 1, g["ratio"], g["k"], fp8_keys=False)
    assert set(top.tolist()) == set(g["top_blocks"])
    wpos = attention.window_positions(t, window=g["window"])
    assert [wpos[0], wpos[-1]] == g["window_positions"]
    assert len(wpos) + len(attention.compressed_ids(t + 1, g["ratio"], top)) == g["keys"]


def _brute_topk(scores, k):
    n = len(scores)
    winners = []
    for S in itertools.combinations(range(n), min(k, n)):
        inside = set(S)
        ok = all(scores[i] > scores[j] or (scores[i] == scores[j] and i < j)
                 for i in inside for j in range(n) if j not in inside)
        if ok:
            winners.append(sorted(S))
    assert len(winners) == 1
    return winners[0]


def test_topk_brute_force_with_ties():
    rs = np.random.default_rng(0)
    for trial in range(300):
        n = int(rs.integers(1, 9))
        k = int(rs.integers(1, 7))
        scores = rs.integers(0, 4, n).astype(np.float64)     # many exact ties
        got = indexer.select_topk(scores, k)
        want = _brute_topk(scores, k)
        assert got[:len(want)].tolist() == want
        assert np.all(got[len(want):] == -1)


def test_scores_brute_force_loops():
    rs = np.random.default_rng(1)
    q = rs.standard_normal((3, 8))
    w = rs.uniform(-1, 1, 3)
    k = rs.standard_normal((5, 8))
    I = indexer.scores_fp64(q, w, k)
    for j in range(5):
        ref = 0.0
        for h in range(3):
            d = sum(q[h, i] * k[j, i] for i in range(8))
            ref += w[h] * (d if d > 0 else 0.0)
        assert I[j] == pytest.approx(ref, rel=1e-12, abs=1e-12)


def test_query_coding_is_per_head_fp8():
    rs = np.random.default_rng(2)
    q = (rs.standard_normal((64, 128)) * np.exp2(rs.integers(-5, 5, (64, 1)))).astype(np.float32)
    qh = indexer.quantize_queries(q)
    c, s = codecs.encode_q_perhead(q)
    assert s.shape == (64,)
    ratio = np.abs(q).max(-1) / codecs.e8m0_decode(s)
    assert np.all((ratio > 224) & (ratio <= 448))
    assert np.all(np.abs(qh - q) <= np.maximum(np.abs(q) * 2.0 ** -4, codecs.e8m0_decode(s)[:, None] * 2.0 ** -10))


def test_visibility_counts(golden):
    g = golden["query_10000"]
    t = g["query_position"]
    assert indexer.visible_entries(t + 1, 4) == g["csa_visible"]
    wpos = attention.window_positions(t)
    assert (wpos[0], wpos[-1]) == (g["window_first"], g["window_last"])
    assert attention.key_count(t + 1, 4, k=g["pro_topk"]) == g["csa_keys"]
    assert indexer.visible_entries(t + 1, 128) == g["hca_entries"]
    assert attention.key_count(t + 1, 128) == g["hca_keys"]
    h = golden["query_1000_hca"]
    t = h["query_position"]
    n = int(indexer.visible_entries(t + 1, 128))
    assert n == h["entries"] and (n - 1) * 128 == h["last_entry_rope_position"]
    assert t + 1 - n * 128 == h["pending_tokens"]
    assert attention.window_positions(t)[0] == h["window_first"]
    assert attention.key_count(t + 1, 128) == h["keys"]


def test_key_count_tables(golden):
    g = golden["key_counts"]
    c = g["csa_1m"]
    assert indexer.visible_entries(c["context"], 4) == c["entries"]
    assert attention.key_count(c["context"], 4, k=c["pro_k"]) == c["pro_keys"]
    assert attention.key_count(c["context"], 4, k=c["flash_k"]) == c["flash_keys"]
    for row in g["hca"]:
        assert attention.key_count(row["context"], 128) == row["keys"]
    s = golden["sparsity_threshold"]
    for m in ("flash", "pro"):
        p = s[m]["position"]
        assert indexer.visible_entries(p + 1, 4) == s[m]["visible"] == s[m]["k"] + 1
        assert indexer.visible_entries(p, 4) <= s[m]["k"]


# ---------------------------------------------------------------- attention

def _marker_keys(logits):
    """Keys whose logit against q = e_0 is given and whose dims 1+j mark key j."""
    keys = np.zeros((len(logits), 512))
    keys[:, 0] = logits
    for j in range(len(logits)):
        keys[j, 1 + j] = 1.0
    q = np.zeros((1, 512))
    q[0, 0] = 1.0
    return q, keys


def test_sink_example(golden):
    g = golden["sink_example"]
    q, keys = _marker_keys(g["logits"])
    tol = g["print_precision"]
    o = attention.decode_attention_fp64(q, 500, keys, np.zeros((0, 512)), None, 1.0)
    assert np.allclose(o[0, 1:4], g["weights_without_sink"], atol=tol)
    o = attention.decode_attention_fp64(q, 500, keys, np.zeros((0, 512)), np.array([g["sink_logit"]]), 1.0)
    assert np.allclose(o[0, 1:4], g["weights_with_sink"], atol=tol)
    assert o[0, 1:4].sum() == pytest.approx(g["sum_with_sink"], abs=tol)


def _sdpa(q, keys, scale, sink=None):
    """torch SDPA (fp64, CPU) with K = V = keys; a sink becomes a zero key with a logit bias."""
    H = q.shape[0]
    K = torch.from_numpy(keys)[None, None].expand(1, H, -1, -1)
    Q = torch.from_numpy(q)[None, :, None, :]
    mask = None
    if sink is not None:
        K = torch.cat([K, torch.zeros(1, H, 1, keys.shape[1], dtype=torch.float64)], dim=2)
        mask = torch.zeros(1, H, 1, K.shape[2], dtype=torch.float64)
        mask[0, :, 0, -1] = torch.from_numpy(np.asarray(sink, np.float64))
    out = torch.nn.functional.scaled_dot_product_attention(Q, K, K, attn_mask=mask, scale=scale)
    return out[0, :, 0].numpy()


def _no_rope(x):
    x = np.array(x, np.float64)
    x[..., -64:] = 0.0
    return x


@pytest.mark.parametrize("with_sink", [False, True])
def test_window_only_is_textbook_mqa(with_sink):
    rs = np.random.default_rng(3)
    H = 8
    q = _no_rope(rs.standard_normal((H, 512)))
    ring = _no_rope(rs.standard_normal((128, 512)))
    sink = rs.standard_normal(H) if with_sink else None
    t = 300
    o = attention.request_attention(q, t + 1, 4, ring, np.zeros((0, 512)), np.full(16, -1), sink, 512 ** -0.5)
    ref = _sdpa(q, ring[attention.window_positions(t) % 128], 512 ** -0.5, sink)
    assert np.allclose(o, ref, atol=1e-12)


def test_hca_is_dense_over_window_and_entries():
    rs = np.random.default_rng(4)
    H = 4
    ctx = 128 * 9 + 17
    q = _no_rope(rs.standard_normal((H, 512)))
    ring = _no_rope(rs.standard_normal((128, 512)))
    ents = _no_rope(rs.standard_normal((20, 512)))
    sink = rs.standard_normal(H)
    o = attention.request_attention(q, ctx, 128, ring, ents, None, sink, 0.05)
    t = ctx - 1
    keys = np.concatenate([ring[attention.window_positions(t) % 128], ents[:ctx // 128]])
    assert np.allclose(o, _sdpa(q, keys, 0.05, sink), atol=1e-12)


def test_short_context_window_is_padded():
    rs = np.random.default_rng(5)
    q = _no_rope(rs.standard_normal((2, 512)))
    ring = _no_rope(rs.standard_normal((128, 512)))
    ents = _no_rope(rs.standard_normal((2, 512)))
    o = attention.request_attention(q, 10, 4, ring, ents, np.array([1, -1, 0, -1]), None, 0.1)
    assert attention.window_positions(9).tolist() == list(range(10))
    assert attention.key_count(10, 4, k=4) == 12
    assert np.allclose(o, _sdpa(q, np.concatenate([ring[:10], ents[[1, 0]]]), 0.1), atol=1e-12)


def test_duplicates_are_kept_and_minus_one_is_skipped():
    rs = np.random.default_rng(6)
    H = 3
    q = _no_rope(rs.standard_normal((H, 512)))
    ring = _no_rope(rs.standard_normal((128, 512)))
    ents = _no_rope(rs.standard_normal((8, 512)))
    t = 40
    dup = attention.request_attention(q, t + 1, 4, ring, ents, np.array([2, 5, 5, -1, -1]), None, 0.07)
    # two copies of key 5 == one copy whose logit is larger by ln 2
    keys = np.concatenate([ring[:t + 1], ents[[2, 5]]])
    z = (q @ keys.T) * 0.07
    z[:, -1] += np.log(2.0)
    p = np.exp(z - z.max(1, keepdims=True))
    ref = (p @ keys) / p.sum(1, keepdims=True)
    assert np.allclose(dup, ref, atol=1e-12)


def test_rope_shift_invariance():
    """Shifting every position by D leaves the output unchanged (relative positions only)."""
    rs = np.random.default_rng(7)
    H = 4
    q = rs.standard_normal((H, 512))
    u_win = rs.standard_normal((128, 512))
    u_ent = rs.standard_normal((6, 512))
    ent_pos = np.array([0, 4, 8, 12, 16, 20])
    sink = rs.standard_normal(H)

    def run(shift):
        t = 300 + shift
        wpos = attention.window_positions(t)
        win = rope.rotate_fp64(u_win, rope.angles(wpos))
        ents = rope.rotate_fp64(u_ent, rope.angles(ent_pos + shift))
        return attention.decode_attention_fp64(q, t, win, ents, sink, 512 ** -0.5)

    a, b = run(0), run(100)
    assert np.allclose(a, b, atol=1e-9)
    # the test is sensitive: moving only the query changes the output
    t = 300
    wpos = attention.window_positions(t)
    win = rope.rotate_fp64(u_win, rope.angles(wpos))
    ents = rope.rotate_fp64(u_ent, rope.angles(ent_pos))
    c = attention.decode_attention_fp64(q, t + 7, win, ents, sink, 512 ** -0.5)
    assert not np.allclose(a, c, atol=1e-3)
