"""Seeded synthetic workloads for paged-KV attention (Qwen3-0.6B attention shape).

This module only draws random numbers and hands out physical block ids, the
job the scheduler and block manager do in the pages. It holds none of the
method's arithmetic (no slot mapping, no gather, no attention): the oracle
and the CUDA path each derive those from what is generated here.

Recipe (the same for every consumer):
* integer draws (lengths, block permutations) use NumPy PCG64 seeded with the
  workload's seed;
* 16-bit tensors are fp32 N(0,1) from a seeded ``torch.Generator`` on the
  target device, rounded to nearest-even bf16 (the default) or fp16 (torch's
  conversions); the fp16 cases draw the same fp32 stream as the bf16 ones;
* physical block ids are a seeded permutation of the pool, so consecutive
  logical blocks of a sequence land on scattered physical blocks;
* every pool slot, used or not, starts as N(0,1) (tests may poison unused
  slots with NaN to prove they are never read);
* shapes: 16 query heads, 8 kv heads, head_dim 128, block_size 256.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HQ, HKV, HEAD_DIM, BLOCK_SIZE = 16, 8, 128, 256
SCALE = 1.0 / math.sqrt(HEAD_DIM)
MAX_NUM_BATCHED_TOKENS = 16384
MAX_MODEL_LEN = 4096


@dataclass
class SeqSpec:
    """One sequence as the scheduler hands it over (attribute names follow
    nano-vLLM's Sequence): ``num_tokens`` = len(seq) including any new
    token, ``num_cached_tokens`` prefix-cache hits, ``num_scheduled_tokens``
    tokens computed this prefill step, ``block_table`` physical block ids."""
    num_tokens: int
    block_table: list = field(default_factory=list)
    num_cached_tokens: int = 0
    num_scheduled_tokens: int = 0


def blocks_for(num_tokens: int, block_size: int = BLOCK_SIZE) -> int:
    """How many blocks the allocator hands a sequence of this length."""
    return -(-num_tokens // block_size)


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal(shape, gen: torch.Generator, device, dtype=torch.bfloat16, chunk_elems: int = 1 << 27) -> torch.Tensor:
    """N(0,1) tensor of a 16-bit type, generated in fp32 chunks to bound temporary memory."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(s + chunk_elems, flat.numel())
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


def normal_bf16(shape, gen: torch.Generator, device, chunk_elems: int = 1 << 27) -> torch.Tensor:
    return normal(shape, gen, device, torch.bfloat16, chunk_elems)


def fused_qkv(num_tokens: int, gen: torch.Generator, device, hq=HQ, hkv=HKV, d=HEAD_DIM, dtype=torch.bfloat16):
    """q, k, v as views of one fused projection output [N, (hq+2*hkv)*d], the
    layout nano-vLLM's attention receives (q/k/v rows strided by the fused width)."""
    qkv = normal((num_tokens, (hq + 2 * hkv) * d), gen, device, dtype)
    q = qkv[:, : hq * d].view(num_tokens, hq, d)
    k = qkv[:, hq * d: (hq + hkv) * d].view(num_tokens, hkv, d)
    v = qkv[:, (hq + hkv) * d:].view(num_tokens, hkv, d)
    return qkv, q, k, v


@dataclass
class Workload:
    name: str
    seed: int
    seqs: list                      # list[SeqSpec] per call; list of lists for multi-call prefill
    num_blocks: int                 # physical blocks in the pool
    kind: str                       # "decode" | "prefill"
    num_layers: int = 1
    hq: int = HQ
    hkv: int = HKV
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    scale: float = SCALE
    graph_batch: int = 0            # decode replayed through a graph of this many rows (0: eager)
    notes: str = ""


def _take_blocks(perm: np.ndarray, cursor: int, n: int):
    return [int(x) for x in perm[cursor:cursor + n]], cursor + n


def _decode_seqs(ctx_lens, num_blocks: int, rng: np.random.Generator, reserved: int = 0):
    """Give each sequence the blocks it needs from a shuffled pool."""
    perm = rng.permutation(num_blocks)
    cursor = reserved
    seqs = []
    for n in ctx_lens:
        table, cursor = _take_blocks(perm, cursor, blocks_for(int(n)))
        seqs.append(SeqSpec(num_tokens=int(n), block_table=table))
    assert cursor <= num_blocks, "pool too small"
    return seqs


def tiny_decode(seed: int = 1) -> Workload:
    """4 sequences with context_lens 37/256/300/511 in a 16-block pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = [37, 256, 300, 511]
    return Workload("tiny_decode_b4", seed, _decode_seqs(ctx, 16, rng), 16, "decode")


def batched_decode(seed: int = 2, num_seqs: int = 256, num_blocks: int = 8192,
                   lo: int = 512, hi: int = 4096) -> Workload:
    """256 sequences, context_lens uniform in [512, 4096], 8192-block pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(lo, hi + 1, size=num_seqs)
    return Workload(f"batched_decode_b{num_seqs}_ctx{lo}-{hi}", seed,
                    _decode_seqs(ctx, num_blocks, rng), num_blocks, "decode")


def sweep_decode(seed: int = 5, num_seqs: int = 512, num_layers: int = 28, mean: float = 800.0,
                 spare_blocks: int = 64) -> Workload:
    """512 sequences, context_lens geometric (mean 800) clipped to [1, 4096],
    a pool of the blocks they need plus 64 spare, 28 layers."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.clip(rng.geometric(1.0 / mean, size=num_seqs), 1, MAX_MODEL_LEN)
    need = sum(blocks_for(int(n)) for n in ctx)
    nb = need + spare_blocks
    return Workload(f"decode_sweep_{num_layers}l_b{num_seqs}", seed, _decode_seqs(ctx, nb, rng), nb,
                    "decode", num_layers=num_layers)


def split_by_token_budget(lengths, budget: int = MAX_NUM_BATCHED_TOKENS):
    """The scheduler's admission rule: admit prompts in order while the running
    token count stays within the budget; a prompt that does not fit opens the
    next call."""
    calls, cur, tot = [], [], 0
    for n in lengths:
        if cur and tot + n > budget:
            calls.append(cur)
            cur, tot = [], 0
        cur.append(int(n))
        tot += int(n)
    if cur:
        calls.append(cur)
    return calls


def varlen_prefill(seed: int = 3, num_prompts: int = 64, lo: int = 100, hi: int = 1024,
                   budget: int = MAX_NUM_BATCHED_TOKENS) -> Workload:
    """64 prompts, lengths uniform in [100, 1024], no prefix hits, split into
    calls of at most 16384 tokens; the pool has twice the blocks needed."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = rng.integers(lo, hi + 1, size=num_prompts)
    need = sum(blocks_for(int(n)) for n in lengths)
    nb = 2 * need
    perm = rng.permutation(nb)
    cursor = 0
    calls = []
    for call in split_by_token_budget(lengths, budget):
        seqs = []
        for n in call:
            table, cursor = _take_blocks(perm, cursor, blocks_for(n))
            seqs.append(SeqSpec(num_tokens=n, block_table=table, num_cached_tokens=0,
                                num_scheduled_tokens=n))
        calls.append(seqs)
    return Workload(f"varlen_prefill_{num_prompts}p_len{lo}-{hi}", seed, calls, nb, "prefill")


def prefix_prefill(seed: int = 4, num_seqs: int = 128, prefix_len: int = 1024, lo: int = 64,
                   hi: int = 512) -> Workload:
    """128 sequences sharing one 1024-token prefix held in 4 physical blocks
    (logical blocks 0..3 of every table, reference count 128), each with its
    own suffix of length uniform in [64, 512] in fresh blocks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    suffix = rng.integers(lo, hi + 1, size=num_seqs)
    n_prefix_blocks = blocks_for(prefix_len)
    need = n_prefix_blocks + sum(blocks_for(prefix_len + int(s)) - n_prefix_blocks for s in suffix)
    nb = 2 * need
    perm = rng.permutation(nb)
    prefix_table, cursor = _take_blocks(perm, 0, n_prefix_blocks)
    seqs = []
    for s in suffix:
        n = prefix_len + int(s)
        extra, cursor = _take_blocks(perm, cursor, blocks_for(n) - n_prefix_blocks)
        seqs.append(SeqSpec(num_tokens=n, block_table=list(prefix_table) + extra,
                            num_cached_tokens=prefix_len, num_scheduled_tokens=int(s)))
    return Workload(f"prefix_prefill_{num_seqs}s_prefix{prefix_len}_suffix{lo}-{hi}", seed, [seqs],
                    nb, "prefill")


def schedule_prefill_chunks(lengths, budget: int):
    """The prefill half of the scheduler in the newest listing ("vLLM 学习笔记 02：nano-vllm
    源码逐段精读", engine/scheduler.py ``schedule``), without prefix-cache hits:
    prompts wait in order; a call admits the prompt at the head of the queue
    while token budget is left; a prompt that does not fit is cut only when it
    is the first of its call (it gets what is left and stays at the head, its
    computed tokens counting as cached next time); otherwise the call closes.

    Returns a list of calls, each a list of (prompt index, start, count)."""
    lengths = [int(n) for n in lengths]
    done = [0] * len(lengths)
    head, calls = 0, []
    while head < len(lengths):
        call, used = [], 0
        while head < len(lengths) and used < budget:
            need = lengths[head] - done[head]
            left = budget - used
            if left < need and call:
                break
            take = min(need, left)
            call.append((head, done[head], take))
            used += take
            done[head] += take
            if done[head] == lengths[head]:
                head += 1
        calls.append(call)
    return calls


def chunked_prefill(seed: int = 6, num_prompts: int = 16, lo: int = 4096, hi: int = 12288,
                    budget: int = 5000) -> Workload:
    """16 prompts of 4096..12288 tokens under a 5000-token budget: every
    prompt longer than the budget is computed in chunks over several calls.
    5000 is not a multiple of the 256-token block, so continued chunks start
    in the middle of a block. Each
    prompt's blocks are allocated for its whole length when it is first
    admitted (engine/block_manager.py ``allocate``), from a shuffled pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = rng.integers(lo, hi + 1, size=num_prompts)
    need = sum(blocks_for(int(n)) for n in lengths)
    nb = need + 64
    perm = rng.permutation(nb)
    tables, cursor = [], 0
    for n in lengths:
        t, cursor = _take_blocks(perm, cursor, blocks_for(int(n)))
        tables.append(t)
    calls = [[SeqSpec(num_tokens=int(lengths[i]), block_table=list(tables[i]), num_cached_tokens=start,
                      num_scheduled_tokens=cnt) for i, start, cnt in call]
             for call in schedule_prefill_chunks(lengths, budget)]
    return Workload(f"chunked_prefill_{num_prompts}p_len{lo}-{hi}_budget{budget}", seed, calls, nb, "prefill",
                    notes=f"token budget {budget}")


def padded_decode(seed: int = 7, num_seqs: int = 200, graph_batch: int = 256, num_blocks: int = 8192,
                  lo: int = 512, hi: int = 4096) -> Workload:
    """A decode step replayed through a CUDA graph captured for a larger batch
    (engine/model_runner.py ``run_model``: the graph for the next captured
    size >= the batch is replayed after ``slot_mapping.fill_(-1)``,
    ``context_lens.zero_()`` and an overwrite of only the live part of the
    block-table buffer). 200 live sequences (context 512..4096) in a graph of
    256 rows; rows 200..255 are padding, and table entries past a row's live
    blocks keep whatever an earlier step left there."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(lo, hi + 1, size=num_seqs)
    seqs = _decode_seqs(ctx, num_blocks, rng)
    return Workload(f"padded_decode_b{num_seqs}_graph{graph_batch}", seed, seqs, num_blocks, "decode",
                    graph_batch=graph_batch)


CONFIGS = {
    1: tiny_decode,
    2: batched_decode,
    3: varlen_prefill,
    4: prefix_prefill,
    5: sweep_decode,
    6: chunked_prefill,
    7: padded_decode,
}
