"""The seeded input generators: splitmix64 known answers, row layouts of the
five workloads, and the shape and range of every generated input."""
import numpy as np

from engram_hashed_gram_gb300 import synth


def test_splitmix64_known_answers():
    # the first outputs of splitmix64 seeded with 0 (Vigna's splitmix64.c)
    got = synth.draw64(0, np.arange(3))
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert synth.mix64_int(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_workload_row_totals():
    want = [100_776, 25_169_534, 402_659_764, 100_667_472, 384_016_682, 100_776, 25_169_534, 100_667_472]
    assert [w.num_rows() for w in synth.WORKLOADS] == want


def test_mxfp8_inputs():
    """The MXFP8 workloads: E8M0 table scales (the fp32 scales' stream
    positions, rounded to powers of two), and an FP8 weight whose values have
    about the bf16 weight's spread N(0, 1/K)."""
    w = synth.workload("tiny_1x16_mxfp8")
    assert (w.scale_block, w.scale_fmt, w.wkv_fmt) == (32, 1, 1)
    rows = np.arange(0, 2000, 7)
    _, s32 = synth.table_rows(w.seed, rows, w.head_dim, 32)
    _, s8 = synth.table_rows(w.seed, rows, w.head_dim, 32, scale_fmt=1)
    assert s8.dtype == np.uint8
    assert np.all(np.abs(np.log2(s32.astype(np.float64)) - (s8.astype(np.float64) - 127)) <= 0.5 + 1e-9)
    codes, scales = synth.make_wkv_mxfp8(w, rows_per_chunk=4096)
    assert codes.shape == (w.N, w.K) and scales.shape == (w.N, w.K // 32)
    assert set(np.unique(scales).tolist()) == {120, 121}
    assert not np.any((codes & 0x7F) == 0x7F)                   # no NaN codes
    from oracle import engram_oracle as O
    W = O.mxfp8_weight(codes[:256], scales[:256])
    assert abs(W.std() * np.sqrt(w.K) - 1.0) < 0.1


def test_table_rows_deterministic_and_chunk_independent():
    rows = np.array([0, 1, 5, 99, 100_775, 7])
    c1, s1 = synth.table_rows(3, rows)
    c2, s2 = synth.table_rows(3, rows[::-1])
    assert np.array_equal(c1, c2[::-1]) and np.array_equal(s1, s2[::-1])
    ct, st = synth.host_table(3, 120, chunk=17)
    c3, s3 = synth.table_rows(3, np.arange(120))
    assert np.array_equal(ct, c3) and np.array_equal(st, s3)
    c4, _ = synth.table_rows(4, rows)
    assert not np.array_equal(c1, c4)


def test_quantile_tables():
    ct = synth.code_quantile_table()
    assert ct.dtype == np.uint8 and ct.size == 65536
    assert not np.any((ct & 0x7F) == 0x7F)              # never NaN
    st = synth.scale_quantile_table()
    assert st.dtype == np.float32 and np.all(st > 0)
    assert abs(float(np.median(st)) - 1.0) < 1e-3
    assert abs(float(np.log(st.astype(np.float64)).std()) - 0.5) < 0.01


def test_hash_ids_in_their_column_ranges():
    for i in range(4):
        w = synth.workload(i)
        lengths, offsets = w.layout()
        ids = synth.make_hash_ids(w, lengths, offsets).reshape(w.M, w.n_cols)
        lo, hi = offsets, offsets + lengths
        assert np.all(ids >= lo[None]) and np.all(ids < hi[None])
    w = synth.workload("prefill_1x4096_zipf")
    ids = synth.make_hash_ids(w).reshape(w.M, w.n_cols)
    top = np.unique(ids[:, 0], return_counts=True)[1].max()
    assert top > 0.05 * w.M                              # Zipf: a hot row per column
    w = synth.workload("decode_512x1_skew")
    ids = synth.make_hash_ids(w).reshape(w.M, w.n_cols)
    # 256 of the 512 draws come from 1,024 hot rows: about 30 repeats; uniform draws over
    # 25M rows repeat almost never
    assert np.unique(ids[:, 0]).size < w.M - 10


def test_masks():
    assert synth.make_mask(synth.workload(0)) is None
    m = synth.make_mask(synth.workload("prefill_1x4096_zipf")).reshape(-1)
    off = np.flatnonzero(m == 0)
    assert off.size == 410 and off[-1] - off[0] == 409
    w4 = synth.WORKLOADS[4]
    m4 = synth.make_mask(w4)
    assert m4.shape == (2, 8192) and int((m4 == 0).sum()) == 819


def test_small_tensors():
    w = synth.workload(0)
    x = synth.make_x(w)
    assert x.shape == (1, 16, 4, 5120) and x.dtype == np.uint16
    q, k = synth.make_qk(w)
    assert q.shape == (4, 5120) and not np.array_equal(q, k)
