"""Seeded random shapes against the oracle, every output row compared.

Prefill: 1..6 sequences per call with random scheduled lengths, each either
without cached keys, with a cached prefix of whole 256-token blocks (a
prefix-cache hit) or continuing a chunk that ended mid-block; poisoned dead
slots on some seeds; the contiguous-keys mode cross-checked when nothing is
cached. Decode: random batches whose contexts include the block and split
edges (1, 255..257, 511..513, 4096). Odd seeds run the fp16 entry points.
PKV_STRESS=1 adds 80 prefill and 60 decode cases (seeds 100+) with wider
ranges: up to 8 sequences of up to 599 new tokens and 1499 cached ones; decode
batches up to 95 with contexts up to 4096 and the 32/64/128-token split edges."""
import os

import numpy as np
import pytest
import torch

import workloads as W
from test_gpu_decode import _decode_step
from test_gpu_prefill import _run, _seqs_with_tables

pytestmark = pytest.mark.gpu

_STRESS = os.environ.get("PKV_STRESS") == "1"
PREFILL_SEEDS = list(range(10)) + (list(range(100, 180)) if _STRESS else [])
DECODE_SEEDS = list(range(8)) + (list(range(100, 160)) if _STRESS else [])


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def _dtype(seed):
    return torch.float16 if seed % 2 else torch.bfloat16


@pytest.mark.parametrize("seed", PREFILL_SEEDS)
def test_random_prefill(pkv, seed):
    rng = np.random.default_rng(9000 + seed)
    wide = seed >= 100
    no_prefix = seed % 4 == 0
    specs = []
    for _ in range(int(rng.integers(1, 9 if wide else 7))):
        kind = 0 if no_prefix else int(rng.integers(0, 3))
        if kind == 0:
            cached = 0
        elif kind == 1:
            cached = W.BLOCK_SIZE * int(rng.integers(1, 5))       # whole cached blocks
        else:
            cached = int(rng.integers(1, 1500 if wide else 1200))  # chunk continuation, mid-block
        specs.append((cached, int(rng.integers(1, 600 if wide else 400))))
    seqs, nb = _seqs_with_tables(specs, rng)
    _run(pkv, seqs, nb, 9100 + seed, poison=seed % 3 == 0, check_contiguous=no_prefix, dtype=_dtype(seed))


@pytest.mark.parametrize("seed", DECODE_SEEDS)
def test_random_decode(pkv, seed):
    rng = np.random.default_rng(9500 + seed)
    wide = seed >= 100
    B = int(rng.integers(1, 96 if wide else 48))
    edges = [1, 255, 256, 257, 511, 512, 513, 4096]
    if wide:
        edges = [1, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 4095, 4096]
    p_edge, top = (0.4, 4097) if wide else (0.3, 3000)
    ctxs = [int(rng.choice(edges)) if rng.random() < p_edge else int(rng.integers(1, top)) for _ in range(B)]
    nb = sum(W.blocks_for(c) for c in ctxs) + 4
    wl = W.Workload(f"random_decode_{seed}", 9600 + seed, W._decode_seqs(ctxs, nb, rng), nb, "decode")
    _decode_step(pkv, wl, "cuda", poison=seed % 2 == 0, fused=seed % 3 != 0, table_pad=int(rng.integers(0, 3)),
                 dtype=_dtype(seed))
