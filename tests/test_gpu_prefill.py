"""Parity of store + varlen prefill (pkv_store_kvcache, pkv_prefill_varlen) with the oracle."""
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


def _seqs_with_tables(specs, rng, spare=3):
    """specs: list of (num_cached, num_scheduled). Blocks from a shuffled pool."""
    need = sum(W.blocks_for(c + s) for c, s in specs)
    nb = need + spare
    perm = rng.permutation(nb)
    cur, seqs = 0, []
    for c, s in specs:
        n = c + s
        t = [int(x) for x in perm[cur:cur + W.blocks_for(n)]]
        cur += len(t)
        seqs.append(W.SeqSpec(num_tokens=n, block_table=t, num_cached_tokens=c, num_scheduled_tokens=s))
    return seqs, nb


def _rows_sample(cu_q, rng, per_seq=6):
    rows = []
    for b in range(len(cu_q) - 1):
        lq = int(cu_q[b + 1] - cu_q[b])
        if lq == 0:
            continue
        picks = {0, lq - 1, *rng.integers(0, lq, size=min(per_seq, lq)).tolist()}
        for i in picks:
            rows.append((int(cu_q[b]) + i, int(rng.integers(0, W.HQ))))
    return np.array(rows, dtype=np.int64)


def _run(pkv, seqs, nb, seed, *, poison=False, sample_rows=None, check_contiguous=False, dtype=torch.bfloat16):
    """Store the scheduled tokens of every sequence, run paged prefill, compare
    with the oracle (all rows, or sampled rows) and optionally with the
    contiguous-keys mode of the same kernel."""
    dev = "cuda"
    gen = W.make_generator(seed, dev)
    kc, vc = pool_tensors(nb, gen, dev, dtype)
    T = sum(s.num_scheduled_tokens for s in seqs)
    _, q, k, v = W.fused_qkv(T, gen, dev, dtype=dtype)
    prefill = pkv.pkv_prefill_varlen_f16 if dtype == torch.float16 else pkv.pkv_prefill_varlen
    if poison:
        poison_dead_slots(kc, vc, seqs, lambda s: s.num_tokens)
    meta = pkv.metadata.prepare_prefill(seqs, W.BLOCK_SIZE, force_block_tables=True)
    ometa = oracle.prepare_prefill([oracle.SeqState(s.num_tokens, list(s.block_table), s.num_cached_tokens,
                                                    s.num_scheduled_tokens) for s in seqs], W.BLOCK_SIZE)
    for key in ("slot_mapping", "cu_seqlens_q", "cu_seqlens_k", "positions"):
        assert np.array_equal(meta[key], ometa[key]), key
    host = HostPool(kc, vc, seqs)
    qb, kb, vb = bits(q), bits(k), bits(v)

    slot = to_dev(meta["slot_mapping"], dev)
    cu_q = to_dev(meta["cu_seqlens_q"], dev)
    cu_k = to_dev(meta["cu_seqlens_k"], dev)
    bt = to_dev(meta["block_tables"], dev)
    pkv.pkv_store_kvcache(k, v, kc, vc, slot)
    out = prefill(q, cu_q, cu_k, meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE,
                  k_cache=kc, v_cache=vc, block_tables=bt)
    # the same call through a host tile plan launches only the tiles with rows: identical bits
    plan = pkv.pkv_prefill_plan(meta["cu_seqlens_q"], meta["cu_seqlens_k"], dev)
    out_planned = prefill(q, cu_q, cu_k, meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE,
                          k_cache=kc, v_cache=vc, block_tables=bt, plan=plan)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    assert out.dtype == dtype
    assert torch.equal(out, out_planned)

    om = oracle.prepare_prefill(host.seqs, W.BLOCK_SIZE)
    ks, vs = host.slots()
    orc = oracle.default()
    orc.store_kvcache(kb, vb, ks, vs, om["slot_mapping"])
    bt_o = oracle.pad_block_tables(host.seqs)
    ref = orc.prefill_varlen(qb, om["cu_seqlens_q"], om["cu_seqlens_k"], W.SCALE, k_cache=host.k, v_cache=host.v,
                             block_tables=bt_o, num_kv_heads=W.HKV, rows=sample_rows, dtype=ORACLE_DTYPE[dtype])
    if sample_rows is None:
        assert_close(out, ref, "prefill")
    else:
        got = out[torch.from_numpy(sample_rows[:, 0]).to(dev), torch.from_numpy(sample_rows[:, 1]).to(dev)]
        assert_close(got, ref, "prefill (sampled rows)")
    if check_contiguous:
        # no prefix: the same keys from contiguous k/v must give the identical result
        out2 = prefill(q, cu_q, cu_k, meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE, k=k, v=v)
        torch.cuda.synchronize()
        assert torch.equal(out, out2)
    return out


@pytest.mark.parametrize("lens", [[1], [5, 2], [127, 128, 129], [1, 255, 256, 257, 300, 513], [1024, 77]])
def test_prefill_no_prefix(pkv, lens):
    rng = np.random.default_rng(sum(lens))
    seqs, nb = _seqs_with_tables([(0, n) for n in lens], rng)
    _run(pkv, seqs, nb, seed=len(lens), poison=True, check_contiguous=True)


@pytest.mark.parametrize("specs", [
    [(256, 10)],                       # prefix of one whole block
    [(1024, 64), (1024, 512)],         # prefix of 4 blocks
    [(1, 1), (300, 129), (44, 300)],   # chunked prefill starting mid-block
    [(511, 1), (257, 255), (128, 128)],
    [(3000, 1000)],                    # long context
])
def test_prefill_with_cached_prefix(pkv, specs):
    rng = np.random.default_rng(len(specs) + sum(c for c, _ in specs))
    seqs, nb = _seqs_with_tables(specs, rng)
    _run(pkv, seqs, nb, seed=sum(s for _, s in specs), poison=True)


def test_varlen_prefill_full_size(pkv):
    """64 prompts of 100..1024 tokens in <=16384-token calls, paged, sampled rows."""
    wl = W.varlen_prefill()
    rng = np.random.default_rng(3)
    for i, call in enumerate(wl.seqs):
        cu = np.concatenate([[0], np.cumsum([s.num_scheduled_tokens for s in call])])
        _run(pkv, call, wl.num_blocks, seed=100 + i, sample_rows=_rows_sample(cu, rng, 4), check_contiguous=True)


def test_prefix_prefill_full_size(pkv):
    """128 sequences sharing a 1024-token prefix in 4 blocks, suffixes 64..512, sampled rows."""
    wl = W.prefix_prefill()
    call = wl.seqs[0]
    cu = np.concatenate([[0], np.cumsum([s.num_scheduled_tokens for s in call])])
    _run(pkv, call, wl.num_blocks, seed=4, sample_rows=_rows_sample(cu, np.random.default_rng(4), 3))


def test_identical_sequences_identical_outputs(pkv):
    """Two sequences sharing the same prefix blocks, with identical suffix
    tokens, produce bit-identical outputs (prefix-cache reuse is exact)."""
    dev = "cuda"
    gen = W.make_generator(21, dev)
    kc, vc = pool_tensors(8, gen, dev)
    s = 200
    _, q1, k1, v1 = W.fused_qkv(s, gen, dev)
    q = torch.cat([q1, q1]).contiguous()
    k = torch.cat([k1, k1]).contiguous()
    v = torch.cat([v1, v1]).contiguous()
    seqs = [W.SeqSpec(1024 + s, [0, 1, 2, 3, 4], 1024, s), W.SeqSpec(1024 + s, [0, 1, 2, 3, 5], 1024, s)]
    meta = pkv.metadata.prepare_prefill(seqs, W.BLOCK_SIZE)
    pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(meta["slot_mapping"], dev))
    out = pkv.pkv_prefill_varlen(q, to_dev(meta["cu_seqlens_q"], dev), to_dev(meta["cu_seqlens_k"], dev),
                                 meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE, k_cache=kc, v_cache=vc,
                                 block_tables=to_dev(meta["block_tables"], dev))
    torch.cuda.synchronize()
    assert torch.equal(out[:s], out[s:])


def test_bad_seqlens_flagged(pkv):
    dev = "cuda"
    gen = W.make_generator(22, dev)
    q = W.normal_bf16((10, W.HQ, W.HEAD_DIM), gen, dev)
    k = W.normal_bf16((10, W.HKV, W.HEAD_DIM), gen, dev)
    cu_q = torch.tensor([0, 6, 10], dtype=torch.int32, device=dev)
    cu_k = torch.tensor([0, 4, 10], dtype=torch.int32, device=dev)   # first sequence: Lk < Lq
    pkv.pkv_prefill_varlen(q, cu_q, cu_k, 6, 6, W.SCALE, k=k, v=k)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() & pkv.PKV_DEVERR_BAD_SEQLEN


def test_many_items_per_cta_with_tail_tiles(pkv):
    """Hundreds of short sequences (thousands of query tiles, most of them
    ending in a partial, zeroed V tile), with and without cached prefixes."""
    rng = np.random.default_rng(99)
    specs = [(int(c), int(s)) for c, s in zip(rng.integers(0, 300, 400), rng.integers(1, 200, 400))]
    seqs, nb = _seqs_with_tables(specs, rng)
    cu = np.concatenate([[0], np.cumsum([s.num_scheduled_tokens for s in seqs])])
    _run(pkv, seqs, nb, seed=99, poison=True, sample_rows=_rows_sample(cu, np.random.default_rng(5), 3))


# ---- fp16 element type (pkv_prefill_varlen_f16) ----------------------------

@pytest.mark.parametrize("lens", [[1, 255, 256, 257, 300, 513], [1024, 77]])
def test_f16_prefill_no_prefix(pkv, lens):
    rng = np.random.default_rng(500 + sum(lens))
    seqs, nb = _seqs_with_tables([(0, n) for n in lens], rng)
    _run(pkv, seqs, nb, seed=500 + len(lens), poison=True, check_contiguous=True, dtype=torch.float16)


@pytest.mark.parametrize("specs", [[(1, 1), (300, 129), (44, 300)], [(1024, 64), (1024, 512)], [(3000, 1000)]])
def test_f16_prefill_with_cached_prefix(pkv, specs):
    rng = np.random.default_rng(600 + len(specs))
    seqs, nb = _seqs_with_tables(specs, rng)
    _run(pkv, seqs, nb, seed=600 + sum(s for _, s in specs), poison=True, dtype=torch.float16)


def test_f16_varlen_prefill_full_size_first_call(pkv):
    """The first <=16384-token call of the 64-prompt workload, fp16, sampled rows."""
    wl = W.varlen_prefill()
    call = wl.seqs[0]
    cu = np.concatenate([[0], np.cumsum([s.num_scheduled_tokens for s in call])])
    _run(pkv, call, wl.num_blocks, seed=700, sample_rows=_rows_sample(cu, np.random.default_rng(7), 3),
         check_contiguous=True, dtype=torch.float16)


def test_f16_prefix_prefill_full_size(pkv):
    """128 sequences sharing a 1024-token prefix, fp16, sampled rows."""
    wl = W.prefix_prefill()
    call = wl.seqs[0]
    cu = np.concatenate([[0], np.cumsum([s.num_scheduled_tokens for s in call])])
    _run(pkv, call, wl.num_blocks, seed=704, sample_rows=_rows_sample(cu, np.random.default_rng(8), 2),
         dtype=torch.float16)


# ---- chunked prefill: calls in order, the cache carried from call to call ----

def _run_calls(pkv, calls, nb, seed, rng, *, per_seq=None, poison=False):
    """Run a sequence of prefill calls (each: store its new tokens, then paged
    prefill) on one pool, as consecutive scheduler steps do; the oracle keeps
    its own copy of the pool and applies the same stores in the same order.
    per_seq=None compares every row, else that many sampled rows per sequence."""
    dev = "cuda"
    gen = W.make_generator(seed, dev)
    kc, vc = pool_tensors(nb, gen, dev)
    if poison:   # slots past each prompt's end are never read
        poison_dead_slots(kc, vc, [s for call in calls for s in call], lambda s: s.num_tokens)
    host = HostPool(kc, vc, [s for call in calls for s in call])
    ks, vs = host.slots()
    orc = oracle.default()
    for ci, call in enumerate(calls):
        T = sum(s.num_scheduled_tokens for s in call)
        _, q, k, v = W.fused_qkv(T, gen, dev)
        qb, kb, vb = bits(q), bits(k), bits(v)
        meta = pkv.metadata.prepare_prefill(call, W.BLOCK_SIZE, force_block_tables=True)
        pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(meta["slot_mapping"], dev))
        out = pkv.pkv_prefill_varlen(q, to_dev(meta["cu_seqlens_q"], dev), to_dev(meta["cu_seqlens_k"], dev),
                                     meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE, k_cache=kc, v_cache=vc,
                                     block_tables=to_dev(meta["block_tables"], dev))
        torch.cuda.synchronize()
        assert pkv.pkv_device_error() == 0
        oseqs = [oracle.SeqState(s.num_tokens, [host.remap[int(x)] for x in s.block_table], s.num_cached_tokens,
                                 s.num_scheduled_tokens) for s in call]
        om = oracle.prepare_prefill(oseqs, W.BLOCK_SIZE)
        assert np.array_equal(om["cu_seqlens_k"], meta["cu_seqlens_k"])
        orc.store_kvcache(kb, vb, ks, vs, om["slot_mapping"])
        rows = None if per_seq is None else _rows_sample(om["cu_seqlens_q"], rng, per_seq)
        ref = orc.prefill_varlen(qb, om["cu_seqlens_q"], om["cu_seqlens_k"], W.SCALE, k_cache=host.k,
                                 v_cache=host.v, block_tables=oracle.pad_block_tables(oseqs), num_kv_heads=W.HKV,
                                 rows=rows)
        if rows is None:
            assert_close(out, ref, f"call {ci}")
        else:
            got = out[torch.from_numpy(rows[:, 0]).to(dev), torch.from_numpy(rows[:, 1]).to(dev)]
            assert_close(got, ref, f"call {ci} (sampled rows)")


def test_chunked_prefill_small_all_rows(pkv):
    """Prompts of 700/300/900/1300 tokens under a 500-token budget: chunks
    continue at positions 500, 1000 (mid-block), a tail shares its call with
    a whole prompt; every row of every call against the oracle."""
    lengths = [700, 300, 900, 1300]
    plan = W.schedule_prefill_chunks(lengths, 500)
    assert any(start % W.BLOCK_SIZE for call in plan for _, start, _ in call)
    rng = np.random.default_rng(31)
    nb = sum(W.blocks_for(n) for n in lengths) + 4
    perm = rng.permutation(nb)
    tables, cur = [], 0
    for n in lengths:
        tables.append([int(x) for x in perm[cur:cur + W.blocks_for(n)]])
        cur += W.blocks_for(n)
    calls = [[W.SeqSpec(lengths[i], tables[i], start, cnt) for i, start, cnt in call] for call in plan]
    _run_calls(pkv, calls, nb, seed=31, rng=rng, poison=True)


def test_chunked_prefill_full_size(pkv):
    """16 prompts of 4096..12288 tokens under a 5000-token budget (35 calls,
    19 chunks starting mid-block): every call in order, sampled rows."""
    wl = W.chunked_prefill()
    _run_calls(pkv, wl.seqs, wl.num_blocks, seed=wl.seed, rng=np.random.default_rng(6), per_seq=3)


@pytest.mark.parametrize("specs", [[(0, 300), (0, 77), (0, 1000)], [(1024, 64), (256, 500), (0, 129)],
                                   [(5000, 300), (37, 900)], [(0, 1)]])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_plan_gives_identical_output(pkv, specs, dtype):
    """A host tile plan (pkv_prefill_plan) launches only the query tiles that
    hold rows, longest first; the output is bit-identical to the plain grid's."""
    dev = "cuda"
    rng = np.random.default_rng(len(specs))
    seqs, nb = _seqs_with_tables(specs, rng)
    gen = W.make_generator(31, dev)
    kc, vc = pool_tensors(nb, gen, dev, dtype)
    T = sum(s.num_scheduled_tokens for s in seqs)
    _, q, k, v = W.fused_qkv(T, gen, dev, dtype=dtype)
    meta = pkv.metadata.prepare_prefill(seqs, W.BLOCK_SIZE, force_block_tables=True)
    prefill = pkv.pkv_prefill_varlen_f16 if dtype == torch.float16 else pkv.pkv_prefill_varlen
    cu_q, cu_k, bt = to_dev(meta["cu_seqlens_q"], dev), to_dev(meta["cu_seqlens_k"], dev), to_dev(meta["block_tables"], dev)
    pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(meta["slot_mapping"], dev))
    plan = pkv.pkv_prefill_plan(meta["cu_seqlens_q"], meta["cu_seqlens_k"])
    assert plan.numel() == sum((s.num_scheduled_tokens + 127) // 128 for s in seqs)
    args = (q, cu_q, cu_k, meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE)
    a = prefill(*args, k_cache=kc, v_cache=vc, block_tables=bt)
    b = prefill(*args, k_cache=kc, v_cache=vc, block_tables=bt, plan=plan)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    assert torch.equal(a, b)


def test_plan_naming_missing_sequences_is_flagged(pkv):
    """A plan built for more sequences than the call has is skipped where it
    names a missing sequence (flagged), never dereferenced."""
    dev = "cuda"
    rng = np.random.default_rng(3)
    seqs, nb = _seqs_with_tables([(0, 200)], rng)
    gen = W.make_generator(32, dev)
    kc, vc = pool_tensors(nb, gen, dev)
    _, q, k, v = W.fused_qkv(200, gen, dev)
    meta = pkv.metadata.prepare_prefill(seqs, W.BLOCK_SIZE, force_block_tables=True)
    pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(meta["slot_mapping"], dev))
    plan = pkv.pkv_prefill_plan([0, 200, 400], [0, 200, 400])   # two sequences
    out = pkv.pkv_prefill_varlen(q, to_dev(meta["cu_seqlens_q"], dev), to_dev(meta["cu_seqlens_k"], dev),
                                 meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE, k_cache=kc, v_cache=vc,
                                 block_tables=to_dev(meta["block_tables"], dev), plan=plan)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error(clear=True) & pkv.PKV_DEVERR_BAD_SEQLEN
    ref = pkv.pkv_prefill_varlen(q, to_dev(meta["cu_seqlens_q"], dev), to_dev(meta["cu_seqlens_k"], dev),
                                 meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE, k_cache=kc, v_cache=vc,
                                 block_tables=to_dev(meta["block_tables"], dev))
    torch.cuda.synchronize()
    assert torch.equal(out, ref)          # the one real sequence is complete


def test_longest_prompt_and_context(pkv):
    """A single prompt at max_model_len (4096 tokens, 32 query tiles of up to 32
    key tiles, poisoned pool, keys also from contiguous k/v), then 96 new tokens
    at the end of a 4096-token context; sampled rows, the last rows included."""
    rng = np.random.default_rng(71)
    seqs, nb = _seqs_with_tables([(0, W.MAX_MODEL_LEN)], rng)
    meta_q = np.array([0, W.MAX_MODEL_LEN])
    _run(pkv, seqs, nb, 71, poison=True, sample_rows=_rows_sample(meta_q, rng, per_seq=24), check_contiguous=True)
    seqs, nb = _seqs_with_tables([(W.MAX_MODEL_LEN - 96, 96)], rng)
    _run(pkv, seqs, nb, 72, poison=True)


def test_sequence_without_new_tokens(pkv):
    """A sequence whose tokens are all cached (no query rows this call) between
    two that have some: it gets no rows, and the others are unaffected."""
    rng = np.random.default_rng(73)
    seqs, nb = _seqs_with_tables([(300, 5), (256, 0), (0, 77), (0, 0), (513, 140)], rng)
    _run(pkv, seqs, nb, 73, poison=True)
