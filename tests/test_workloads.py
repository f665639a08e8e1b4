"""Host logic of the seeded workloads: shapes, tables and slot mappings."""
import numpy as np

from mxfp4_sparse_paged_gb300 import workloads as W


def test_specs_match_the_five_workloads():
    s = W.SPECS
    assert (s[0].batch, s[0].q, s[0].lens, s[0].k) == (1, 1, ("fixed", 512), 128)
    assert (s[1].batch, s[1].lens, s[1].k, s[1].shuffle_pages) == (8, ("fixed", 8192), 2048, True)
    assert (s[2].batch, s[2].lens) == (64, ("uniform", 4096, 65536))
    assert (s[3].batch, s[3].q, s[3].lens) == (16, 4, ("fixed", 131072))
    assert (s[4].batch, s[4].lens[0], s[4].lens[1], s[4].lens[3]) == (256, "lognormal", 8192,
                                                                    131072)
    assert s[4].insert_in_step and s[4].outlier_scale == 20.0


def test_block_tables_are_a_partition_of_the_pool():
    for c in range(5):
        wl = W.make(c)
        pages = (wl.seq_lens.astype(np.int64) + 127) // 128
        used = np.concatenate([wl.block_table[s, :pages[s]] for s in range(wl.B)])
        assert len(np.unique(used)) == len(used)
        assert used.min() >= 0 and used.max() < wl.num_pages
        for s in range(wl.B):
            assert np.all(wl.block_table[s, pages[s]:] == -1)
        assert wl.block_table.dtype == np.int32 and wl.seq_lens.dtype == np.int32


def test_lengths_in_range():
    wl = W.make(2)
    assert wl.seq_lens.min() >= 4096 and wl.seq_lens.max() <= 65536
    wl = W.make(4)
    assert wl.seq_lens.min() >= 1 and wl.seq_lens.max() <= 131072
    assert 4000 < np.median(wl.seq_lens) < 16000
    assert W.make(3).seq_lens.tolist() == [131072] * 16


def test_slots_follow_the_block_table():
    wl = W.make(1)
    pos = np.array([0, 127, 128, 8191])
    sl = wl.slots(3, pos)
    assert np.array_equal(sl // 128, wl.block_table[3, pos // 128])
    assert np.array_equal(sl % 128, pos % 128)
    # decode-token slots and positions: q tokens at the end of each sequence
    wl = W.make(3)
    p = wl.positions().reshape(16, 4)
    assert np.array_equal(p[0], [131068, 131069, 131070, 131071])


def test_rows_are_deterministic_and_sliceable():
    wl = W.make(2)
    a = wl.rows(5, W.K_ROWS, 0, 10000)
    b = wl.rows(5, W.K_ROWS, 4000, 9000)
    assert np.array_equal(a[4000:9000], b)
    c = W.make(2).rows(5, W.K_ROWS, 4000, 9000)
    assert np.array_equal(b, c)
    assert not np.array_equal(wl.rows(5, W.V_ROWS, 0, 10), wl.rows(5, W.K_ROWS, 0, 10))


def test_outlier_channels_scaled():
    wl = W.make(4)
    assert len(wl.outlier_channels) == 3
    for kind in range(3):
        (ch,) = wl.outlier_channels[kind]
        r = wl.rows(0, kind, 0, 4096)
        assert r[:, ch].std() > 10 * np.delete(r, ch, axis=1).std()


def test_algorithmic_bytes():
    wl = W.make(3)
    ab = W.algorithmic_bytes(wl)
    assert ab["index_score"] == 68 * 16 * 131072
    assert ab["sparse_paged_decode"] == 136 * 64 * 2048
    assert W.algorithmic_bytes(W.make(0))["sparse_paged_decode"] == 136 * 128
