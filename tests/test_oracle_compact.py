"""Pins of the oracle's KV compaction (Medusa Heads glossary page, "Tree attention
and acceptance": the longest accepted branch is kept and its last hidden state
feeds the next round)."""
import numpy as np

from oracle import oracle as O


def test_compaction_moves_accepted_rows_including_overlaps():
    rng = np.random.default_rng(30)
    B, Hkv, D, N, Dmax, H = 5, 3, 8, 9, 4, 6
    Lmax = 40
    k = rng.integers(0, 2**16, size=(B, Hkv, Lmax, D), dtype=np.uint16)
    v = rng.integers(0, 2**16, size=(B, Hkv, Lmax, D), dtype=np.uint16)
    kv_len = np.array([0, 3, 10, 20, Lmax - N], np.int32)
    # paths with overlapping moves: destination L+i is the source of a later row
    paths = np.full((B, Dmax + 1), -1, np.int32)
    paths[0, :3] = [0, 2, 1]        # slot L+1 <- L+2 while L+2 <- L+1
    paths[1, :5] = [0, 4, 2, 8, 3]
    paths[2, :1] = [0]
    paths[3, :4] = [0, 3, 1, 2]
    paths[4, :2] = [0, 8]
    alen = np.array([2, 4, 0, 3, 1], np.int32)
    best = np.array([paths[b, alen[b]] for b in range(B)], np.int32)
    ht = rng.integers(0, 2**16, size=(B, N, H), dtype=np.uint16)
    k2, v2, kl2, h_next, src = O.kv_compact(k, v, kv_len, paths, alen, best, ht, N, Dmax)
    for b in range(B):
        L, a = kv_len[b], alen[b]
        assert kl2[b] == L + a + 1
        for c_old, c_new in ((k, k2), (v, v2)):
            assert np.array_equal(c_new[b, :, :L], c_old[b, :, :L])            # prefix untouched
            assert np.array_equal(c_new[b, :, L + a + 1:], c_old[b, :, L + a + 1:])
            for i in range(a + 1):
                assert np.array_equal(c_new[b, :, L + i], c_old[b, :, L + paths[b, i]])
        assert np.array_equal(h_next[b], ht[b, best[b]])
        assert src[b, : a + 1].tolist() == [L + n for n in paths[b, : a + 1]]
        assert (src[b, a + 1:] == -1).all()


def test_compaction_fp32_rows():
    rng = np.random.default_rng(31)
    B, Hkv, D, N, Dmax, Lmax = 1, 2, 4, 5, 2, 12
    k = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32)
    paths = np.array([[0, 3, 4]], np.int32)
    k2, v2, kl2, _, _ = O.kv_compact(k, v, np.array([6], np.int32), paths, np.array([2], np.int32),
                                     np.array([4], np.int32), None, N, Dmax)
    assert kl2[0] == 9
    assert np.array_equal(k2[0, :, 6:9], k[0, :, [6, 9, 10]].transpose(1, 0, 2))
