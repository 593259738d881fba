"""Device-built index preparation (pkv_build_prefill_metadata,
pkv_build_decode_metadata): bit-exact against the oracle's host version."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def _random_seqs(rng, n, bs=256, max_len=5000):
    seqs, cur = [], 0
    perm = rng.permutation(100000)
    for _ in range(n):
        total = int(rng.integers(1, max_len))
        cached = int(rng.integers(0, total))
        nb = oracle.num_blocks(total, bs)
        seqs.append(oracle.SeqState(total, [int(x) for x in perm[cur:cur + nb]], cached, total - cached))
        cur += nb
    return seqs


def _prefill_dev(pkv, seqs, capacity=None, num_blocks=100000):
    dev = "cuda"
    bt = oracle.pad_block_tables(seqs)
    T = sum(s.num_scheduled_tokens for s in seqs)
    out = pkv.pkv_build_prefill_metadata(
        to_dev(np.array([s.num_cached_tokens for s in seqs], np.int32), dev),
        to_dev(np.array([s.num_scheduled_tokens for s in seqs], np.int32), dev), to_dev(bt, dev), num_blocks,
        T if capacity is None else capacity)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, T


def test_worked_example(pkv):
    g = json.load(open(os.path.join(GOLDEN, "worked_example_bs256.json")))
    seqs = [oracle.SeqState(**r) for r in g["prefill"]["seqs"]]
    got, T = _prefill_dev(pkv, seqs)
    assert got["slot_mapping"][:T].tolist() == g["prefill"]["slot_mapping"]
    assert got["cu_seqlens_q"].tolist() == g["prefill"]["cu_seqlens_q"]
    assert got["cu_seqlens_k"].tolist() == g["prefill"]["cu_seqlens_k"]
    assert got["positions"][:T].tolist() == g["prefill"]["positions"]
    assert got["max_seqlens"].tolist() == [g["prefill"]["max_seqlen_q"], g["prefill"]["max_seqlen_k"]]
    d = g["decode"]
    ds = [oracle.SeqState(**r) for r in d["seqs"]]
    out = pkv.pkv_build_decode_metadata(to_dev(np.array([s.num_tokens for s in ds], np.int32), "cuda"),
                                        to_dev(oracle.pad_block_tables(ds), "cuda"), 16)
    assert out["slot_mapping"].tolist() == d["slot_mapping"]
    assert out["context_lens"].tolist() == d["context_lens"]
    assert out["positions"].tolist() == d["positions"]
    assert pkv.pkv_device_error() == 0


@pytest.mark.parametrize("n", [1, 7, 300, 1500])
def test_prefill_metadata_bit_exact(pkv, n):
    seqs = _random_seqs(np.random.default_rng(n), n)
    got, T = _prefill_dev(pkv, seqs)
    ref = oracle.prepare_prefill(seqs, 256)
    assert np.array_equal(got["slot_mapping"][:T], ref["slot_mapping"])
    assert np.array_equal(got["positions"][:T], ref["positions"])
    assert np.array_equal(got["cu_seqlens_q"], ref["cu_seqlens_q"])
    assert np.array_equal(got["cu_seqlens_k"], ref["cu_seqlens_k"])
    assert got["max_seqlens"].tolist() == [ref["max_seqlen_q"], ref["max_seqlen_k"]]
    assert pkv.pkv_device_error() == 0


@pytest.mark.parametrize("n", [1, 256, 4000])
def test_decode_metadata_bit_exact(pkv, n):
    rng = np.random.default_rng(n + 1)
    seqs = _random_seqs(rng, n, max_len=4097)
    seqs = [oracle.SeqState(s.num_tokens, s.block_table) for s in seqs]
    ref = oracle.prepare_decode(seqs, 256)
    out = pkv.pkv_build_decode_metadata(to_dev(np.array([s.num_tokens for s in seqs], np.int32), "cuda"),
                                        to_dev(ref["block_tables"], "cuda"), 100000)
    torch.cuda.synchronize()
    assert np.array_equal(out["slot_mapping"].cpu().numpy(), ref["slot_mapping"])
    assert np.array_equal(out["context_lens"].cpu().numpy(), ref["context_lens"])
    assert np.array_equal(out["positions"].cpu().numpy(), ref["positions"])
    assert pkv.pkv_device_error() == 0


def test_padding_rows_capacity_and_bad_blocks(pkv):
    dev = "cuda"
    # decode padding rows: len 0 -> slot -1, context 0
    out = pkv.pkv_build_decode_metadata(torch.tensor([5, 0, 0], dtype=torch.int32, device=dev),
                                        torch.tensor([[3], [0], [0]], dtype=torch.int32, device=dev), 8)
    assert out["slot_mapping"].tolist() == [3 * 256 + 4, -1, -1] and out["context_lens"].tolist() == [5, 0, 0]
    assert pkv.pkv_device_error() == 0
    # capacity smaller than the tokens: flagged, nothing written past it
    seqs = [oracle.SeqState(100, [0], 0, 100)]
    got, _ = _prefill_dev(pkv, seqs, capacity=60)
    assert pkv.pkv_device_error() & pkv.PKV_DEVERR_BAD_SEQLEN
    assert got["slot_mapping"][:60].tolist() == list(range(60))
    # block id outside the pool: slot -1 and flagged
    got, _ = _prefill_dev(pkv, [oracle.SeqState(10, [7], 0, 10)], num_blocks=4)
    assert pkv.pkv_device_error() & pkv.PKV_DEVERR_BAD_BLOCK
    assert np.all(got["slot_mapping"][:10] == -1)
