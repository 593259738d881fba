"""Helpers for the GPU parity tests: build seeded cases, hand the oracle its
own copy of the inputs, compare outputs.

Nothing the CUDA path computes ever feeds the oracle: the oracle receives the
generated inputs (copied to the host BEFORE any kernel of the library runs)
and derives its own metadata and stored cache from them.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

TOL_MAX = 2e-2    # max abs error on bf16 / fp16 attention outputs (against the fp64 oracle)
TOL_MEAN = 2e-3   # mean abs error

# torch element type -> the oracle's name for it
ORACLE_DTYPE = {torch.bfloat16: "bf16", torch.float16: "f16"}


def bits(t: torch.Tensor) -> np.ndarray:
    """16-bit tensor (any device) -> host uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= TOL_MAX and mean <= TOL_MEAN, f"{what}: max abs err {mx:.3e}, mean {mean:.3e}"
    return mx, mean


def oracle_seq(s, table=None):
    return oracle.SeqState(num_tokens=s.num_tokens, block_table=list(s.block_table if table is None else table),
                           num_cached_tokens=s.num_cached_tokens, num_scheduled_tokens=s.num_scheduled_tokens)


class HostPool:
    """Host copy of the blocks some sequences use, with compact block ids."""

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, seqs):
        used = sorted({int(x) for s in seqs for x in s.block_table})
        self.remap = {old: new for new, old in enumerate(used)}
        idx = torch.tensor(used, dtype=torch.long, device=k_cache.device)
        self.k = bits(k_cache.index_select(0, idx))
        self.v = bits(v_cache.index_select(0, idx))
        self.seqs = [oracle_seq(s, [self.remap[int(x)] for x in s.block_table]) for s in seqs]

    def slots(self):
        return self.k.reshape(-1, *self.k.shape[2:]), self.v.reshape(-1, *self.v.shape[2:])


def pool_tensors(num_blocks: int, gen, device, dtype=torch.bfloat16):
    shape = (num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    return W.normal(shape, gen, device, dtype), W.normal(shape, gen, device, dtype)


def poison_dead_slots(k_cache: torch.Tensor, v_cache: torch.Tensor, seqs, live_tokens):
    """Fill every slot that holds no live token of any sequence with NaN.

    live_tokens(s) is how many leading positions of sequence s are live."""
    nb = k_cache.shape[0]
    live = torch.zeros(nb, W.BLOCK_SIZE, dtype=torch.bool)
    for s in seqs:
        n = live_tokens(s)
        for j, blk in enumerate(s.block_table):
            cnt = min(W.BLOCK_SIZE, n - j * W.BLOCK_SIZE)
            if cnt > 0:
                live[int(blk), :cnt] = True
    dead = (~live).to(k_cache.device)
    nan = torch.tensor(float("nan"), dtype=k_cache.dtype, device=k_cache.device)
    k_cache[dead] = nan
    v_cache[dead] = nan


def to_dev(a, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)
