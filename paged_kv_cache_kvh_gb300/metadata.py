"""Host-side index preparation for the paged-KV kernels.

Builds the arrays the kernels consume from per-sequence scheduler state
(objects with ``num_tokens``, ``num_cached_tokens``, ``num_scheduled_tokens``
and ``block_table``), as engine/model_runner.py's prepare_prefill and
prepare_decode do in "vLLM 学习笔记 02：nano-vllm 源码逐段精读":

* a token at absolute position t of a sequence lives in slot
  block_table[t // block_size] * block_size + t % block_size;
* prefill queries cover positions [num_cached_tokens, num_cached_tokens +
  num_scheduled_tokens) and keys cover [0, that end);
* decode stores the sequence's last token and attends over all num_tokens.

Vectorised NumPy; returns int32 arrays ready to copy to the device (pinned
when asked, so the host-to-device copy can be asynchronous).
"""
from __future__ import annotations

import numpy as np


def _tables(seqs, width=None, fill=-1):
    w = max((len(s.block_table) for s in seqs), default=0) if width is None else width
    bt = np.full((len(seqs), max(w, 1)), fill, dtype=np.int32)
    for r, s in enumerate(seqs):
        n = len(s.block_table)
        if n:
            bt[r, :n] = np.asarray(s.block_table, dtype=np.int32)
    return bt


def slots_for_positions(block_table, positions, block_size: int) -> np.ndarray:
    table = np.asarray(block_table, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    return (table[pos // block_size] * block_size + pos % block_size).astype(np.int32)


def prepare_prefill(seqs, block_size: int = 256, force_block_tables: bool = False, table_width=None):
    starts = np.array([s.num_cached_tokens for s in seqs], dtype=np.int64)
    lq = np.array([s.num_scheduled_tokens for s in seqs], dtype=np.int64)
    ends = starts + lq
    cu_q = np.zeros(len(seqs) + 1, dtype=np.int32)
    cu_k = np.zeros(len(seqs) + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(lq)
    cu_k[1:] = np.cumsum(ends)
    slot_parts, pos_parts = [], []
    for s, a, e in zip(seqs, starts, ends):
        pos = np.arange(a, e, dtype=np.int64)
        pos_parts.append(pos)
        if len(s.block_table):
            slot_parts.append(slots_for_positions(s.block_table, pos, block_size))
    has_prefix = bool(cu_k[-1] > cu_q[-1])
    return dict(
        positions=np.concatenate(pos_parts) if pos_parts else np.zeros(0, np.int64),
        cu_seqlens_q=cu_q,
        cu_seqlens_k=cu_k,
        max_seqlen_q=int(lq.max()) if len(seqs) else 0,
        max_seqlen_k=int(ends.max()) if len(seqs) else 0,
        slot_mapping=np.concatenate(slot_parts).astype(np.int32) if slot_parts else np.zeros(0, np.int32),
        block_tables=_tables(seqs, table_width) if (has_prefix or force_block_tables) else None,
    )


def prepare_decode(seqs, block_size: int = 256, table_width=None):
    n = np.array([s.num_tokens for s in seqs], dtype=np.int64)
    last = n - 1
    bt = _tables(seqs, table_width)
    rows = np.arange(len(seqs))
    slots = bt[rows, last // block_size].astype(np.int64) * block_size + last % block_size
    return dict(positions=last, slot_mapping=slots.astype(np.int32), context_lens=n.astype(np.int32),
                block_tables=bt)
