"""The seeded input generator (CPU): reproducible streams, pages that regenerate alone,
the named workloads' shapes, valid shuffled page tables, and the stated value
distributions."""

import numpy as np

from compressed_sparse_attention_kv_gb300 import synth


def test_streams_are_reproducible_and_distinct():
    a = synth.normal(7, (synth.T_MAIN, 3, 5), (64, 512))
    b = synth.normal(7, (synth.T_MAIN, 3, 5), (64, 512))
    c = synth.normal(7, (synth.T_MAIN, 3, 6), (64, 512))
    d = synth.normal(8, (synth.T_MAIN, 3, 5), (64, 512))
    assert a.dtype == np.float32 and np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_a_page_regenerates_alone():
    """Any page of a request equals the same rows of the whole request's values, and a
    sampled-row request returns exactly the pages holding those rows."""
    w = synth.custom_workload("t", 5, [4 * (64 * 7 + 10), 4 * 64 * 3], 4, 16, 16, 4, synth.FMT_FP8, synth.FMT_FP8,
                              synth.FMT_FP8_PAGESPLIT)
    whole = synth.request_values(w, 0, "main")
    assert whole.shape == (int(w.pages_per_req()[0]) * 64, 512)
    for p in (0, 3, int(w.pages_per_req()[0]) - 1):
        assert np.array_equal(synth.main_page_values(w, 0, p), whole[64 * p:64 * (p + 1)])
    some = synth.request_values(w, 0, "main", rows=[5, 70, 71, 200])
    assert sorted(some) == [0, 1, 3]
    for p, v in some.items():
        assert np.array_equal(v, whole[64 * p:64 * (p + 1)])
    keys = synth.request_values(w, 1, "index")
    assert keys.shape == (64 * 3, 128)
    assert not np.array_equal(keys[:64], synth.index_page_values(w, 0, 0))


def test_named_workloads_have_the_stated_shapes():
    t = synth.workload("tiny_csa")
    assert (t.B, int(t.ctx_len[0]), int(t.n_entries[0]), t.k, t.H, t.Hi) == (1, 4096, 1024, 512, 16, 4)
    h = synth.workload("hca_128k")
    assert (h.B, h.ratio, h.k, int(h.n_entries[0])) == (32, 128, None, 1024)
    c = synth.workload("csa_1m")
    assert (c.B, c.max_ctx, int(c.n_entries[0]), c.k, c.H, c.Hi) == (8, 1 << 20, 262144, 512, 64, 64)
    assert c.key_fmt == synth.FMT_FP8_PAGESPLIT and c.main_fmt == synth.FMT_FP8
    m = synth.workload("mixed_mxfp4")
    assert m.B == 64 and m.main_fmt == synth.FMT_FP4
    assert m.ctx_len.min() >= 32768 and m.ctx_len.max() <= 524288
    assert len(np.unique(m.ctx_len)) > 32                         # a real length mix
    assert np.array_equal(m.ctx_len, synth.workload("mixed_mxfp4").ctx_len)
    small = synth.workload("csa_1m", batch=2)
    assert small.B == 2 and np.array_equal(small.ctx_len, c.ctx_len[:2])


def test_page_tables_are_a_shuffled_partition_of_the_pool():
    w = synth.workload("mixed_mxfp4", batch=9)
    for lane in ("main", "index"):
        bt, num_pages = synth.page_tables(w, lane)
        ppr = w.pages_per_req()
        assert num_pages == int(ppr.sum()) and bt.shape == (9, int(ppr.max()))
        owned = np.concatenate([bt[b, :ppr[b]] for b in range(9)])
        assert np.array_equal(np.sort(owned), np.arange(num_pages))   # every page once
        for b in range(9):
            assert np.all(bt[b, ppr[b]:] == -1)
        assert not np.array_equal(owned, np.arange(num_pages))        # shuffled
    assert not np.array_equal(synth.page_tables(w, "main")[0], synth.page_tables(w, "index")[0])


def test_value_distributions():
    w = synth.workload("csa_1m")
    q, qi, wt, sink = synth.queries(w)
    assert q.shape == (8, 64, 512) and qi.shape == (8, 64, 128) and wt.shape == (8, 64) and sink.shape == (64,)
    for x in (q, qi, synth.index_page_values(w, 0, 0), synth.swa_values(w, 0)):
        assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05
    assert wt.min() >= 0.0 and wt.max() < 1.0 and abs(float(wt.mean()) - 0.5) < 0.05
    ape, nw = synth.compressor_params(3, 4, True, 512)
    assert ape.shape == (4, 1024) and abs(float(ape.std()) - 0.5) < 0.03
    assert nw.shape == (512,) and nw.min() >= 0.5 and nw.max() <= 1.5
    kv, gate = synth.compressor_tokens(3, 64, 4, True, 512)
    assert kv.shape == (64, 2, 512) and gate.shape == (64, 2, 512)
    pk, pg = synth.compressor_prev(3, 4, 512)
    assert pk.shape == (4, 2, 512) and not np.array_equal(pk, kv[:4])


def test_integer_inputs_are_small_integers():
    q, k, wt = synth.integer_index_inputs(11, 2, 8, 100)
    assert np.all(q == np.round(q)) and np.abs(q).max() <= 3
    assert np.all(k == np.round(k)) and np.abs(k).max() <= 3
    assert np.all(wt * 8 == np.round(wt * 8)) and wt.min() >= 0 and wt.max() <= 7 / 8
