"""Index preparation of the oracle against the pages' worked examples and
against a brute-force per-position reading of the slot layout."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _seqs(rows):
    return [oracle.SeqState(**r) for r in rows]


def test_worked_example_prefill():
    g = _load("worked_example_bs256.json")
    p = g["prefill"]
    m = oracle.prepare_prefill(_seqs(p["seqs"]), g["block_size"])
    assert m["cu_seqlens_q"].tolist() == p["cu_seqlens_q"]
    assert m["cu_seqlens_k"].tolist() == p["cu_seqlens_k"]
    assert m["max_seqlen_q"] == p["max_seqlen_q"] and m["max_seqlen_k"] == p["max_seqlen_k"]
    assert m["slot_mapping"].tolist() == p["slot_mapping"]
    assert m["positions"].tolist() == p["positions"]
    assert m["block_tables"] is None and p["block_tables"] is None


def test_worked_example_decode():
    g = _load("worked_example_bs256.json")
    d = g["decode"]
    m = oracle.prepare_decode(_seqs(d["seqs"]), g["block_size"])
    assert m["slot_mapping"].tolist() == d["slot_mapping"]
    assert m["context_lens"].tolist() == d["context_lens"]
    assert m["block_tables"].tolist() == d["block_tables"]
    assert m["positions"].tolist() == d["positions"]


def test_block_size4_walkthrough():
    g = _load("block_size4_walkthrough.json")
    bs = g["block_size"]
    for i, n in enumerate(g["lengths"]):
        assert oracle.num_blocks(n, bs) == g["num_blocks"][i]
        assert oracle.last_block_num_tokens(n, bs) == g["last_block_num_tokens"][i]
        prev = oracle.num_blocks(n - 1, bs) if n > 1 else 0
        assert (oracle.num_blocks(n, bs) - prev == 1) == g["opens_new_block"][i]
        assert (oracle.last_block_num_tokens(n, bs) == bs) == g["last_block_full"][i]
    ex = g["decode_example"]
    m = oracle.prepare_decode([oracle.SeqState(num_tokens=ex["num_tokens"],
                                               block_table=ex["block_table"])], bs)
    assert m["slot_mapping"].tolist() == [ex["slot"]]


@pytest.mark.parametrize("n", [1, 255, 256, 257, 511, 512, 513, 4096])
def test_block_counts_brute_force(n):
    bs = 256
    k = 0
    while k * bs < n:           # smallest k with k*bs >= n
        k += 1
    assert oracle.num_blocks(n, bs) == k
    assert oracle.last_block_num_tokens(n, bs) == n - (k - 1) * bs
    assert 1 <= oracle.last_block_num_tokens(n, bs) <= bs


def _slot_of(table, t, bs):
    return table[t // bs] * bs + t % bs


def test_chunked_prefill_mid_block_hand_values():
    """A chunk starting mid-block (positions 300..699, block_size 256, table
    [5, 9, 2]): offsets start at 300 % 256 = 44 inside block 9."""
    s = oracle.SeqState(num_tokens=700, block_table=[5, 9, 2], num_cached_tokens=300,
                        num_scheduled_tokens=400)
    m = oracle.prepare_prefill([s], 256)
    want = list(range(9 * 256 + 44, 9 * 256 + 256)) + list(range(2 * 256, 2 * 256 + 188))
    assert m["slot_mapping"].tolist() == want
    assert m["cu_seqlens_q"].tolist() == [0, 400] and m["cu_seqlens_k"].tolist() == [0, 700]
    assert m["positions"].tolist() == list(range(300, 700))
    assert m["block_tables"].tolist() == [[5, 9, 2]]     # keys partly cached -> tables passed


@pytest.mark.parametrize("bs", [4, 16, 256])
def test_prefill_slots_brute_force(bs):
    rng = np.random.default_rng(bs)
    seqs = []
    used = rng.permutation(10_000)
    cur = 0
    for _ in range(12):
        n = int(rng.integers(1, 5 * bs))
        cached = int(rng.integers(0, n))          # any start, block-aligned or not
        nb = oracle.num_blocks(n, bs)
        table = [int(x) for x in used[cur:cur + nb]]
        cur += nb
        seqs.append(oracle.SeqState(num_tokens=n, block_table=table, num_cached_tokens=cached,
                                    num_scheduled_tokens=n - cached))
    m = oracle.prepare_prefill(seqs, bs)
    want = [_slot_of(s.block_table, t, bs) for s in seqs
            for t in range(s.num_cached_tokens, s.num_cached_tokens + s.num_scheduled_tokens)]
    assert m["slot_mapping"].tolist() == want
    assert len(set(want)) == len(want)
    pad = m["block_tables"]
    for r, s in enumerate(seqs):
        assert pad[r, :len(s.block_table)].tolist() == s.block_table
        assert np.all(pad[r, len(s.block_table):] == -1)


def test_decode_slot_is_last_position():
    rng = np.random.default_rng(7)
    bs = 256
    seqs = []
    for n in [1, 2, 255, 256, 257, 511, 512, 513, 4096]:
        nb = oracle.num_blocks(n, bs)
        seqs.append(oracle.SeqState(num_tokens=n, block_table=[int(x) for x in rng.permutation(64)[:nb]]))
    m = oracle.prepare_decode(seqs, bs)
    for i, s in enumerate(seqs):
        assert m["slot_mapping"][i] == _slot_of(s.block_table, s.num_tokens - 1, bs)
        assert m["context_lens"][i] == s.num_tokens
        assert m["positions"][i] == s.num_tokens - 1


def test_no_block_tables_without_prefix_hit():
    seqs = [oracle.SeqState(num_tokens=10, block_table=[3], num_scheduled_tokens=10)]
    assert oracle.prepare_prefill(seqs, 256)["block_tables"] is None
