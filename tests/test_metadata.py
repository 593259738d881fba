"""Host index preparation of the package: bit-exact against the oracle's
(loop) version, the pages' worked example, and the workload generators."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def meta():
    from paged_kv_cache_kvh_gb300 import metadata
    return metadata


def _o(s):
    return oracle.SeqState(s.num_tokens, list(s.block_table), s.num_cached_tokens, s.num_scheduled_tokens)


def test_worked_example(meta):
    g = json.load(open(os.path.join(GOLDEN, "worked_example_bs256.json")))
    p = meta.prepare_prefill([W.SeqSpec(**r) for r in g["prefill"]["seqs"]], 256)
    assert p["slot_mapping"].tolist() == g["prefill"]["slot_mapping"]
    assert p["cu_seqlens_q"].tolist() == g["prefill"]["cu_seqlens_q"]
    assert p["cu_seqlens_k"].tolist() == g["prefill"]["cu_seqlens_k"]
    assert p["block_tables"] is None
    d = meta.prepare_decode([W.SeqSpec(**r) for r in g["decode"]["seqs"]], 256)
    assert d["slot_mapping"].tolist() == g["decode"]["slot_mapping"]
    assert d["context_lens"].tolist() == g["decode"]["context_lens"]
    assert d["block_tables"].tolist() == g["decode"]["block_tables"]


@pytest.mark.parametrize("factory", [W.tiny_decode, W.batched_decode, W.sweep_decode])
def test_decode_metadata_matches_oracle(meta, factory):
    wl = factory()
    a = meta.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    b = oracle.prepare_decode([_o(s) for s in wl.seqs], W.BLOCK_SIZE)
    for k in ("slot_mapping", "context_lens", "block_tables", "positions"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("factory", [W.varlen_prefill, W.prefix_prefill])
def test_prefill_metadata_matches_oracle(meta, factory):
    wl = factory()
    for call in wl.seqs:
        a = meta.prepare_prefill(call, W.BLOCK_SIZE)
        b = oracle.prepare_prefill([_o(s) for s in call], W.BLOCK_SIZE)
        for k in ("slot_mapping", "cu_seqlens_q", "cu_seqlens_k", "positions"):
            assert np.array_equal(a[k], b[k]), k
        assert a["max_seqlen_q"] == b["max_seqlen_q"] and a["max_seqlen_k"] == b["max_seqlen_k"]
        assert (a["block_tables"] is None) == (b["block_tables"] is None)
        if a["block_tables"] is not None:
            assert np.array_equal(a["block_tables"], b["block_tables"])


def test_workloads_shapes():
    t = W.tiny_decode()
    assert [s.num_tokens for s in t.seqs] == [37, 256, 300, 511] and t.num_blocks == 16
    b = W.batched_decode()
    ctx = np.array([s.num_tokens for s in b.seqs])
    assert len(ctx) == 256 and ctx.min() >= 512 and ctx.max() <= 4096 and b.num_blocks == 8192
    used = [x for s in b.seqs for x in s.block_table]
    assert len(used) == len(set(used))                      # no block handed out twice
    v = W.varlen_prefill()
    assert sum(len(c) for c in v.seqs) == 64
    assert all(sum(s.num_scheduled_tokens for s in c) <= W.MAX_NUM_BATCHED_TOKENS for c in v.seqs)
    p = W.prefix_prefill()
    seqs = p.seqs[0]
    assert len(seqs) == 128 and all(s.block_table[:4] == seqs[0].block_table[:4] for s in seqs)
    assert all(s.num_cached_tokens == 1024 and 64 <= s.num_scheduled_tokens <= 512 for s in seqs)
    used = [x for s in seqs for x in s.block_table[4:]] + seqs[0].block_table[:4]
    assert len(used) == len(set(used))
    w = W.sweep_decode()
    ctx = np.array([s.num_tokens for s in w.seqs])
    assert len(ctx) == 512 and ctx.min() >= 1 and ctx.max() <= 4096 and 500 < ctx.mean() < 1100


def test_admission_rule():
    assert W.split_by_token_budget([10, 10, 10], 20) == [[10, 10], [10]]
    assert W.split_by_token_budget([30, 5], 20) == [[30], [5]]
    assert W.split_by_token_budget([], 20) == []
