"""Seeded random shapes against the oracle, every output row compared.

Prefill: 1..6 sequences per call with random scheduled lengths, each either
without cached keys, with a cached prefix of whole 256-token blocks (a
prefix-cache hit) or continuing a chunk that ended mid-block; poisoned dead
slots on some seeds; the contiguous-keys mode cross-checked when nothing is
cached. Decode: random batches whose contexts include the block and split
edges (1, 255..257, 511..513, 4096). Odd seeds run the fp16 entry points."""
import numpy as np
import pytest
import torch

import workloads as W
from test_gpu_decode import _decode_step
from test_gpu_prefill import _run, _seqs_with_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def _dtype(seed):
    return torch.float16 if seed % 2 else torch.bfloat16


@pytest.mark.parametrize("seed", range(10))
def test_random_prefill(pkv, seed):
    rng = np.random.default_rng(9000 + seed)
    no_prefix = seed % 4 == 0
    specs = []
    for _ in range(int(rng.integers(1, 7))):
        kind = 0 if no_prefix else int(rng.integers(0, 3))
        if kind == 0:
            cached = 0
        elif kind == 1:
            cached = W.BLOCK_SIZE * int(rng.integers(1, 5))       # whole cached blocks
        else:
            cached = int(rng.integers(1, 1200))                    # chunk continuation, mid-block
        specs.append((cached, int(rng.integers(1, 400))))
    seqs, nb = _seqs_with_tables(specs, rng)
    _run(pkv, seqs, nb, 9100 + seed, poison=seed % 3 == 0, check_contiguous=no_prefix, dtype=_dtype(seed))


@pytest.mark.parametrize("seed", range(8))
def test_random_decode(pkv, seed):
    rng = np.random.default_rng(9500 + seed)
    B = int(rng.integers(1, 48))
    edges = [1, 255, 256, 257, 511, 512, 513, 4096]
    ctxs = [int(rng.choice(edges)) if rng.random() < 0.3 else int(rng.integers(1, 3000)) for _ in range(B)]
    nb = sum(W.blocks_for(c) for c in ctxs) + 4
    wl = W.Workload(f"random_decode_{seed}", 9600 + seed, W._decode_seqs(ctxs, nb, rng), nb, "decode")
    _decode_step(pkv, wl, "cuda", poison=seed % 2 == 0, fused=seed % 3 != 0, table_pad=int(rng.integers(0, 3)),
                 dtype=_dtype(seed))
