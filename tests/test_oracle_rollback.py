"""Pins of the oracle's paged KV-cache rollback ("LLM Inference & Speculative
Decoding: From Roofline Physics to Lossless Acceleration", s.1,
PagedKVCacheManager.rollback_to)."""
import numpy as np

import oracle
from conftest import read_golden


def test_page_example():
    """The page's own check: 10 positions in blocks of 4, rolled back to 6."""
    g = read_golden("rollback_page_example.txt")
    bs = int(g["block_size"][0])
    before = [int(v) for v in g["table_before"]]
    free = np.full(16, -7, np.int32)
    fb = [int(v) for v in g["free_before"]]
    free[: len(fb)] = fb
    table = np.full((1, 8), -1, np.int32)
    table[0, : len(before)] = before
    # 10 positions held, the last 4 of them drafts, none accepted: 10 - 4 = 6
    r = oracle.rollback([0], 4, [int(g["appended"][0])], table, [len(before)], bs, free, len(fb))
    after = [int(v) for v in g["table_after"]]
    assert r["seq_lens"][0] == int(g["seq_len_after"][0]) == int(g["target_len"][0])
    assert r["num_blocks"][0] == len(after)
    assert r["block_tables"][0, : len(after)].tolist() == after
    assert np.all(r["block_tables"][0, len(after):] == -1)
    fa = [int(v) for v in g["free_after"]]
    assert r["free_count"] == len(fa)
    assert r["free_list"][: len(fa)].tolist() == fa
    assert r["row_status"][0] == 0


def _random_batch(rng, B, k, bs, mb):
    nb = rng.integers(0, mb + 1, size=B).astype(np.int32)
    # seq_len consistent with the block count: (nb-1)*bs < len <= nb*bs, len >= k for most rows
    lens = np.where(nb > 0, (nb - 1) * bs + rng.integers(1, bs + 1, size=B), 0).astype(np.int32)
    tables = np.full((B, mb), -1, np.int32)
    perm = rng.permutation(B * mb).astype(np.int32)
    for b in range(B):
        tables[b, : nb[b]] = perm[b * mb: b * mb + nb[b]]
    na = rng.integers(0, k + 1, size=B).astype(np.int32)
    return na, lens, tables, nb


def test_invariants_random_batches():
    """Block conservation, table lengths ceil(len / block_size), untouched
    prefixes, and the free-list order of popping rows in batch order."""
    rng = np.random.default_rng(3)
    for trial in range(30):
        B, k, bs, mb = int(rng.integers(1, 60)), int(rng.integers(1, 9)), int(rng.integers(1, 17)), 12
        na, lens, tables, nb = _random_batch(rng, B, k, bs, mb)
        cap = B * mb + 5
        free = np.full(cap, -9, np.int32)
        pre = int(rng.integers(0, 4))
        free[:pre] = 10_000 + np.arange(pre)
        r = oracle.rollback(na, k, lens, tables, nb, bs, free, pre)
        valid = lens - (k - na) >= 0
        assert np.all(r["row_status"][valid] == 0) and np.all(r["row_status"][~valid] == 128)
        expect_free = list(free[:pre])
        for b in range(B):
            if not valid[b]:
                assert r["seq_lens"][b] == lens[b] and r["num_blocks"][b] == nb[b]
                assert np.array_equal(r["block_tables"][b], tables[b])
                continue
            new = lens[b] - (k - na[b])
            need = -(-new // bs) if new > 0 else 0
            keep = min(nb[b], need)
            assert r["seq_lens"][b] == new and r["num_blocks"][b] == keep
            assert np.array_equal(r["block_tables"][b, :keep], tables[b, :keep])
            assert np.all(r["block_tables"][b, keep:] == -1)
            expect_free += list(tables[b, keep: nb[b]][::-1])
        assert r["free_count"] == len(expect_free)
        assert r["free_list"][: len(expect_free)].tolist() == [int(v) for v in expect_free]
        # conservation: every block is in exactly one table or the free list
        held = np.concatenate([r["block_tables"][b, : r["num_blocks"][b]] for b in range(B)] +
                              [r["free_list"][pre: r["free_count"]]])
        orig = np.concatenate([tables[b, : nb[b]] for b in range(B)])
        assert sorted(held.tolist()) == sorted(orig.tolist())


def test_all_accepted_and_empty():
    """num_accepted = k keeps every position; a row rolled back to length 0
    gives back all its blocks."""
    tables = np.array([[5, 6, 7, -1], [8, 9, -1, -1]], np.int32)
    r = oracle.rollback([3, 0], 3, [9, 3], tables, [3, 1], 4, np.zeros(8, np.int32), 0)
    assert r["seq_lens"].tolist() == [9, 0]
    assert r["num_blocks"].tolist() == [3, 0]
    assert r["free_list"][: r["free_count"]].tolist() == [8]


def test_no_room_changes_nothing():
    tables = np.array([[1, 2, 3, 4]], np.int32)
    r = oracle.rollback([0], 8, [16], tables, [4], 4, np.zeros(1, np.int32), 0)  # 2 blocks, room for 1
    assert r["row_status"].tolist() == [256]
    assert r["seq_lens"].tolist() == [16] and r["num_blocks"].tolist() == [4] and r["free_count"] == 0
