"""Parity of store + decode (pkv_store_kvcache, pkv_decode) with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import ORACLE_DTYPE, HostPool, assert_close, bits, poison_dead_slots, pool_tensors, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def _decode_step(pkv, wl, device, *, sample=None, poison=False, max_ctx=W.MAX_MODEL_LEN, fused=True,
                 table_pad=0, stale_fill=None, dtype=torch.bfloat16):
    """Store the new token of every sequence, then decode; check against the oracle."""
    gen = W.make_generator(wl.seed, device)
    kc, vc = pool_tensors(wl.num_blocks, gen, device, dtype)
    seqs = wl.seqs
    B = len(seqs)
    if fused:
        _, q, k, v = W.fused_qkv(B, gen, device, dtype=dtype)
    else:
        q = W.normal((B, W.HQ, W.HEAD_DIM), gen, device, dtype)
        k = W.normal((B, W.HKV, W.HEAD_DIM), gen, device, dtype)
        v = W.normal((B, W.HKV, W.HEAD_DIM), gen, device, dtype)
    if poison:
        poison_dead_slots(kc, vc, seqs, lambda s: s.num_tokens)
    width = max(len(s.block_table) for s in seqs) + table_pad
    meta = pkv.metadata.prepare_decode(seqs, W.BLOCK_SIZE, table_width=width)
    ometa = oracle.prepare_decode([oracle.SeqState(s.num_tokens, list(s.block_table)) for s in seqs], W.BLOCK_SIZE)
    assert np.array_equal(meta["slot_mapping"], ometa["slot_mapping"])      # index work: bit-exact
    assert np.array_equal(meta["context_lens"], ometa["context_lens"])
    bt = meta["block_tables"]
    if stale_fill is not None:  # entries past ceil(ctx/256) must never be read
        for r, s in enumerate(seqs):
            bt[r, len(s.block_table):] = stale_fill
    sample = list(range(B)) if sample is None else sample
    host = HostPool(kc, vc, [seqs[i] for i in sample])       # pre-store copy for the oracle
    kb, vb, qb = bits(k), bits(v), bits(q)

    slot = to_dev(meta["slot_mapping"], device)
    ctx = to_dev(meta["context_lens"], device)
    btd = to_dev(bt, device)
    ws = pkv.decode_workspace(B, max_ctx, device)
    pkv.pkv_store_kvcache(k, v, kc, vc, slot)
    decode = pkv.pkv_decode_f16 if dtype == torch.float16 else pkv.pkv_decode
    out = decode(q, kc, vc, btd, ctx, max_ctx, W.SCALE, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    assert out.dtype == dtype

    # oracle: its own store into its own copy, then its own decode
    om = oracle.prepare_decode(host.seqs, W.BLOCK_SIZE)
    ks, vs = host.slots()
    orc = oracle.default()
    orc.store_kvcache(kb[sample], vb[sample], ks, vs, om["slot_mapping"])
    ref = orc.decode(qb[sample], host.k, host.v, om["block_tables"], om["context_lens"], W.SCALE,
                     num_kv_heads=W.HKV, dtype=ORACLE_DTYPE[dtype])
    got = out[torch.tensor(sample, device=device)]
    assert_close(got, ref, wl.name)
    return out, (kc, vc, k, v, q, slot, ctx, btd, ws)


def test_tiny_decode(pkv):
    """4 sequences, context 37/256/300/511, 16-block pool (the whole case)."""
    _decode_step(pkv, W.tiny_decode(), "cuda")


def test_tiny_decode_poisoned_and_stale_tables(pkv):
    """Dead slots hold NaN and table entries past ceil(ctx/256) are garbage:
    neither may reach the output."""
    _decode_step(pkv, W.tiny_decode(seed=11), "cuda", poison=True, table_pad=3, stale_fill=123456)


@pytest.mark.parametrize("ctxs", [[1, 2, 255, 256, 257, 511, 512, 513, 1000, 4096],
                                  [4096] * 3 + [1] * 3, [300]])
def test_ragged_contexts(pkv, ctxs):
    rng = np.random.default_rng(len(ctxs))
    nb = sum(W.blocks_for(c) for c in ctxs) + 5
    wl = W.Workload("ragged", 77, W._decode_seqs(ctxs, nb, rng), nb, "decode")
    _decode_step(pkv, wl, "cuda", poison=True, fused=False)


@pytest.mark.parametrize("num_seqs", [1, 5, 20, 40])
def test_split_sizes_for_small_batches(pkv, num_seqs):
    """Small batches split each 256-token block over several CTAs (32, 64,
    128 or 256 tokens each, picked from num_seqs and max_context_len); every
    split size gives the oracle's result, including a 4096-token context
    merged from 128 partials."""
    rng = np.random.default_rng(100 + num_seqs)
    ctxs = [4096] + [int(x) for x in rng.integers(1, 4097, size=num_seqs - 1)]
    nb = sum(W.blocks_for(c) for c in ctxs) + 3
    wl = W.Workload(f"split_{num_seqs}", 200 + num_seqs, W._decode_seqs(ctxs, nb, rng), nb, "decode")
    sample = list(range(min(num_seqs, 6)))
    _decode_step(pkv, wl, "cuda", sample=sample, poison=True)


def test_batched_decode_full_size(pkv):
    """256 sequences, context 512..4096, 8192-block pool: sampled sequences
    (shortest, longest and a random spread) against the oracle."""
    wl = W.batched_decode()
    ctx = np.array([s.num_tokens for s in wl.seqs])
    rng = np.random.default_rng(0)
    sample = sorted({int(ctx.argmin()), int(ctx.argmax()), *rng.choice(len(ctx), 10, replace=False).tolist()})
    _decode_step(pkv, wl, "cuda", sample=sample)


def test_sweep_shape_one_layer(pkv):
    """512 sequences with long-tailed contexts (1..4096): one layer, sampled."""
    wl = W.sweep_decode(num_layers=1)
    ctx = np.array([s.num_tokens for s in wl.seqs])
    order = np.argsort(ctx)
    sample = sorted({int(order[0]), int(order[1]), int(order[-1]), int(order[len(order) // 2]),
                     *np.random.default_rng(1).choice(len(ctx), 8, replace=False).tolist()})
    _decode_step(pkv, wl, "cuda", sample=sample)


def test_padding_rows_and_repeat_calls(pkv):
    """Graph-padding rows (slot -1, context 0) give zeros and write nothing;
    a second call with the same workspace gives bit-identical output
    (the split-KV tickets reset themselves)."""
    dev = "cuda"
    wl = W.tiny_decode(seed=5)
    gen = W.make_generator(5, dev)
    kc, vc = pool_tensors(wl.num_blocks, gen, dev)
    meta = __import__("paged_kv_cache_kvh_gb300").metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    B, pad = len(wl.seqs), 4
    q = W.normal_bf16((B + pad, W.HQ, W.HEAD_DIM), gen, dev)
    k = W.normal_bf16((B + pad, W.HKV, W.HEAD_DIM), gen, dev)
    v = W.normal_bf16((B + pad, W.HKV, W.HEAD_DIM), gen, dev)
    slot = torch.full((B + pad,), -1, dtype=torch.int32, device=dev)
    slot[:B] = to_dev(meta["slot_mapping"], dev)
    ctx = torch.zeros(B + pad, dtype=torch.int32, device=dev)
    ctx[:B] = to_dev(meta["context_lens"], dev)
    bt = torch.zeros(B + pad, 16, dtype=torch.int32, device=dev)
    bt[:B, :meta["block_tables"].shape[1]] = to_dev(meta["block_tables"], dev)
    before_k = kc.clone()
    ws = pkv.decode_workspace(B + pad, W.MAX_MODEL_LEN, dev)
    pkv.pkv_store_kvcache(k, v, kc, vc, slot)
    changed = (kc != before_k).flatten(1).any(dim=1).nonzero().flatten().tolist()
    assert set(changed) <= {int(s) // (W.BLOCK_SIZE) for s in meta["slot_mapping"]}
    o1 = pkv.pkv_decode(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
    o2 = pkv.pkv_decode(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert torch.all(o1[B:] == 0)
    assert pkv.pkv_device_error() == 0


def test_context_beyond_declared_max_is_flagged(pkv):
    dev = "cuda"
    wl = W.tiny_decode(seed=6)
    gen = W.make_generator(6, dev)
    kc, vc = pool_tensors(wl.num_blocks, gen, dev)
    meta = __import__("paged_kv_cache_kvh_gb300").metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    q = W.normal_bf16((4, W.HQ, W.HEAD_DIM), gen, dev)
    ws = pkv.decode_workspace(4, 256, dev)
    out = pkv.pkv_decode(q, kc, vc, to_dev(meta["block_tables"], dev), to_dev(meta["context_lens"], dev), 256,
                         W.SCALE, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() & pkv.PKV_DEVERR_BAD_SEQLEN
    assert torch.all(out[2:] == 0)          # contexts 300 and 511 exceed 256: zeros
    assert torch.all(torch.isfinite(out[:2].float()))


def test_bad_block_and_slot_are_flagged_not_dereferenced(pkv):
    dev = "cuda"
    gen = W.make_generator(9, dev)
    kc, vc = pool_tensors(4, gen, dev)
    q = W.normal_bf16((2, W.HQ, W.HEAD_DIM), gen, dev)
    k = W.normal_bf16((2, W.HKV, W.HEAD_DIM), gen, dev)
    bt = torch.tensor([[0, 1 << 20], [-5, 0]], dtype=torch.int32, device=dev)
    ctx = torch.tensor([300, 10], dtype=torch.int32, device=dev)
    ws = pkv.decode_workspace(2, 512, dev)
    pkv.pkv_decode(q, kc, vc, bt, ctx, 512, W.SCALE, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() & pkv.PKV_DEVERR_BAD_BLOCK
    pkv.pkv_store_kvcache(k, k, kc, vc, torch.tensor([5, 4 * 256], dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() & pkv.PKV_DEVERR_BAD_SLOT
    # the device is still healthy
    out = pkv.pkv_decode(q, kc, vc, torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device=dev), ctx, 512,
                         W.SCALE, ws)
    torch.cuda.synchronize()
    assert torch.all(torch.isfinite(out.float())) and pkv.pkv_device_error() == 0


@pytest.mark.parametrize("factory,dtype", [(W.tiny_decode, torch.bfloat16), (W.batched_decode, torch.bfloat16),
                                           (lambda: W.sweep_decode(num_layers=1), torch.bfloat16),
                                           (W.tiny_decode, torch.float16), (W.batched_decode, torch.float16)])
def test_store_decode_fused_matches_separate(pkv, factory, dtype):
    """pkv_store_decode == pkv_store_kvcache then pkv_decode: same output and
    the same cache, bit for bit (padding rows included); likewise for the
    fp16 entry points."""
    dev = "cuda"
    wl = factory()
    gen = W.make_generator(wl.seed + 1000, dev)
    kc, vc = pool_tensors(wl.num_blocks, gen, dev, dtype)
    B, pad = len(wl.seqs), 3
    _, q, k, v = W.fused_qkv(B + pad, gen, dev, dtype=dtype)
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE, table_width=16)
    slot = torch.full((B + pad,), -1, dtype=torch.int32, device=dev)
    slot[:B] = to_dev(meta["slot_mapping"], dev)
    ctx = torch.zeros(B + pad, dtype=torch.int32, device=dev)
    ctx[:B] = to_dev(meta["context_lens"], dev)
    bt = torch.zeros(B + pad, 16, dtype=torch.int32, device=dev)
    bt[:B] = to_dev(meta["block_tables"], dev)
    kc2, vc2 = kc.clone(), vc.clone()
    ws = pkv.decode_workspace(B + pad, W.MAX_MODEL_LEN, dev)
    f16 = dtype == torch.float16
    decode = pkv.pkv_decode_f16 if f16 else pkv.pkv_decode
    store_decode = pkv.pkv_store_decode_f16 if f16 else pkv.pkv_store_decode
    pkv.pkv_store_kvcache(k, v, kc, vc, slot)
    ref = decode(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
    got = store_decode(q, k, v, slot, kc2, vc2, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    assert torch.equal(got, ref)
    assert torch.equal(kc2, kc) and torch.equal(vc2, vc)


def test_store_decode_rejects_foreign_slot(pkv):
    """A slot that is not the sequence's newest position is flagged, not stored."""
    dev = "cuda"
    wl = W.tiny_decode(seed=8)
    gen = W.make_generator(8, dev)
    kc, vc = pool_tensors(wl.num_blocks, gen, dev)
    _, q, k, v = W.fused_qkv(4, gen, dev)
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    slot = to_dev(meta["slot_mapping"], dev)
    slot[1] = slot[1] - 1                         # one position too early
    before = kc.clone()
    ws = pkv.decode_workspace(4, W.MAX_MODEL_LEN, dev)
    pkv.pkv_store_decode(q, k, v, slot, kc, vc, to_dev(meta["block_tables"], dev),
                         to_dev(meta["context_lens"], dev), W.MAX_MODEL_LEN, W.SCALE, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() & pkv.PKV_DEVERR_BAD_SLOT
    bad = int(meta["slot_mapping"][1]) - 1
    assert torch.equal(kc.view(-1, 8, 128)[bad], before.view(-1, 8, 128)[bad])


# ---- fp16 element type (pkv_decode_f16) ------------------------------------

def test_f16_tiny_decode_poisoned_and_stale_tables(pkv):
    _decode_step(pkv, W.tiny_decode(seed=12), "cuda", poison=True, table_pad=3, stale_fill=123456,
                 dtype=torch.float16)


def test_f16_ragged_contexts(pkv):
    ctxs = [1, 2, 255, 256, 257, 511, 512, 513, 1000, 4096]
    rng = np.random.default_rng(40)
    nb = sum(W.blocks_for(c) for c in ctxs) + 5
    wl = W.Workload("ragged_f16", 78, W._decode_seqs(ctxs, nb, rng), nb, "decode")
    _decode_step(pkv, wl, "cuda", poison=True, fused=False, dtype=torch.float16)


def test_f16_batched_decode_full_size(pkv):
    """256 sequences, context 512..4096, fp16: sampled sequences against the oracle."""
    wl = W.batched_decode()
    ctx = np.array([s.num_tokens for s in wl.seqs])
    rng = np.random.default_rng(2)
    sample = sorted({int(ctx.argmin()), int(ctx.argmax()), *rng.choice(len(ctx), 8, replace=False).tolist()})
    _decode_step(pkv, wl, "cuda", sample=sample, dtype=torch.float16)


def test_f16_and_bf16_see_the_same_values(pkv):
    """Values exact in both types (small integers times powers of two): the
    bf16 and fp16 kernels read the same numbers and must agree to within
    one rounding of the output."""
    dev = "cuda"
    wl = W.tiny_decode(seed=13)
    rng = np.random.default_rng(13)
    shape = (wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    kc32 = torch.from_numpy(rng.integers(-8, 9, size=shape) / 8.0).float()
    vc32 = torch.from_numpy(rng.integers(-8, 9, size=shape) / 4.0).float()
    q32 = torch.from_numpy(rng.integers(-8, 9, size=(4, W.HQ, W.HEAD_DIM)) / 8.0).float()
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    bt, ctx = to_dev(meta["block_tables"], dev), to_dev(meta["context_lens"], dev)
    ws = pkv.decode_workspace(4, W.MAX_MODEL_LEN, dev)
    outs = {}
    for dt, fn in ((torch.bfloat16, pkv.pkv_decode), (torch.float16, pkv.pkv_decode_f16)):
        outs[dt] = fn(q32.to(dev, dt), kc32.to(dev, dt), vc32.to(dev, dt), bt, ctx, W.MAX_MODEL_LEN, W.SCALE,
                      ws).float()
    torch.cuda.synchronize()
    diff = (outs[torch.bfloat16] - outs[torch.float16]).abs()
    assert float(diff.max()) <= 2.0 ** -8 * 2.0 + 1e-6       # one bf16 ulp of |o| <= 2, plus fp16 rounding
    assert pkv.pkv_device_error() == 0


def test_many_sequences_grid_rows(pkv):
    """3,000 sequences of 1..600 tokens (grid form, 3,000 rows of CTAs along
    the second grid dimension, two to three splits each): sampled rows from the
    first, last and middle sequences against the oracle."""
    rng = np.random.default_rng(99)
    ctxs = [int(x) for x in rng.integers(1, 601, size=3000)]
    nb = sum(W.blocks_for(c) for c in ctxs) + 4
    wl = W.Workload("many_seqs", 99, W._decode_seqs(ctxs, nb, rng), nb, "decode")
    sample = sorted({0, 1, 1499, 1500, 2998, 2999, *rng.choice(3000, 6, replace=False).tolist()})
    _decode_step(pkv, wl, "cuda", sample=sample, poison=True)
