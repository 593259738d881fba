"""The persistent decode (2 CTAs per SM taking the live (sequence, chunk)
items from a workspace counter) on edge cases. A call takes it when its chunks
are whole 256-token blocks (num_seqs * ceil(max_context_len / 256) >= 608) and
it has at most 512 sequences; these batches are sized to take it.

Every sampled row is compared with the oracle, which receives its own host
copy of the inputs taken before any kernel of the library ran and applies its
own store.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import HostPool, assert_close, bits, poison_dead_slots, pool_tensors, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def _takes_persistent(num_seqs, max_ctx):
    return num_seqs * (-(-max_ctx // W.BLOCK_SIZE)) >= 608 and num_seqs <= 512


def _run(pkv, ctxs, seed, *, fused=False, pad=0, sample=None, dtype=torch.bfloat16, max_ctx=W.MAX_MODEL_LEN):
    """Decode (optionally with the store fused in) over live rows with the
    given contexts plus `pad` padding rows; compare sampled live rows with the
    oracle and check padding rows are zeros."""
    dev = "cuda"
    rng = np.random.default_rng(seed)
    B = len(ctxs)
    G = B + pad
    nb = sum(W.blocks_for(c) for c in ctxs) + 3
    seqs = W._decode_seqs(ctxs, nb, rng)
    gen = W.make_generator(seed, dev)
    kc, vc = pool_tensors(nb, gen, dev, dtype)
    poison_dead_slots(kc, vc, seqs, lambda s: s.num_tokens)
    _, q, k, v = W.fused_qkv(G, gen, dev, dtype=dtype)
    width = -(-max_ctx // W.BLOCK_SIZE)
    meta = pkv.metadata.prepare_decode(seqs, W.BLOCK_SIZE, table_width=width)
    sample = list(range(B)) if sample is None else sample
    host = HostPool(kc, vc, [seqs[i] for i in sample])       # before any kernel of the library
    qb, kb, vb = bits(q), bits(k), bits(v)
    slot = torch.full((G,), -1, dtype=torch.int32, device=dev)
    slot[:B] = to_dev(meta["slot_mapping"], dev)
    ctx = torch.zeros(G, dtype=torch.int32, device=dev)
    ctx[:B] = to_dev(meta["context_lens"], dev)
    bt = torch.full((G, width), 7777, dtype=torch.int32, device=dev)   # stale tails must never be read
    bt[:B, :meta["block_tables"].shape[1]] = to_dev(np.where(meta["block_tables"] < 0, 7777, meta["block_tables"]),
                                                     dev)
    ws = pkv.decode_workspace(G, max_ctx, dev)
    f16 = dtype == torch.float16
    if fused:
        fn = pkv.pkv_store_decode_f16 if f16 else pkv.pkv_store_decode
        out = fn(q, k, v, slot, kc, vc, bt, ctx, max_ctx, W.SCALE, ws)
    else:
        pkv.pkv_store_kvcache(k, v, kc, vc, slot)
        fn = pkv.pkv_decode_f16 if f16 else pkv.pkv_decode
        out = fn(q, kc, vc, bt, ctx, max_ctx, W.SCALE, ws)
    again = fn(q, kc, vc, bt, ctx, max_ctx, W.SCALE, ws) if not fused else None
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    if again is not None:
        assert torch.equal(out, again)          # the workspace counters and tickets were left zero
    om = oracle.prepare_decode(host.seqs, W.BLOCK_SIZE)
    ks, vs = host.slots()
    orc = oracle.default()
    orc.store_kvcache(kb[sample], vb[sample], ks, vs, om["slot_mapping"])
    ref = orc.decode(qb[sample], host.k, host.v, om["block_tables"], om["context_lens"], W.SCALE,
                     num_kv_heads=W.HKV, dtype="f16" if f16 else "bf16")
    assert_close(out[torch.tensor(sample, device=dev)], ref, f"persistent decode seed {seed}")
    if pad:
        assert torch.all(out[B:] == 0)
    return out


EDGES = [1, 2, 31, 32, 255, 256, 257, 511, 512, 513, 767, 768, 1000, 2048, 4095, 4096]


def test_edge_contexts(pkv):
    """Block and class edges of every kind, three times over (48 sequences)."""
    ctxs = EDGES * 3
    assert _takes_persistent(len(ctxs), W.MAX_MODEL_LEN)
    _run(pkv, ctxs, 601)


def test_edge_contexts_fused_store_and_padding(pkv):
    """The same with the store fused in and 16 padding rows (slot -1, context 0)."""
    ctxs = EDGES * 3
    _run(pkv, ctxs, 602, fused=True, pad=16)


def test_edge_contexts_f16(pkv):
    ctxs = EDGES * 3
    _run(pkv, ctxs, 603, dtype=torch.float16, fused=True)


def test_all_contexts_block_aligned(pkv):
    """Contexts that are whole blocks only (no partial chunks in the list)."""
    rng = np.random.default_rng(604)
    ctxs = [256 * int(x) for x in rng.integers(1, 17, size=64)]
    _run(pkv, ctxs, 604)


def test_all_contexts_short(pkv):
    """Contexts below one block only (no whole chunks, every row one item)."""
    rng = np.random.default_rng(605)
    ctxs = [int(x) for x in rng.integers(1, 256, size=200)]
    _run(pkv, ctxs, 605, sample=list(range(0, 200, 7)))


def test_largest_batch_and_the_grid_beyond_it(pkv):
    """512 sequences take the persistent form, 513 the grid form; both
    match the oracle on sampled rows, the first and last rows included."""
    rng = np.random.default_rng(606)
    ctxs = [int(x) for x in np.clip(rng.geometric(1 / 500, size=513), 1, 4096)]
    assert _takes_persistent(512, W.MAX_MODEL_LEN) and not _takes_persistent(513, W.MAX_MODEL_LEN)
    _run(pkv, ctxs[:512], 606, sample=[0, 1, 255, 510, 511])
    _run(pkv, ctxs, 607, sample=[0, 1, 255, 511, 512])
