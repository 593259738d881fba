"""The persistent prefill (one CTA per SM walking the tile plan's work units).
A planned call runs it when it has at least two units (query tile, sequence,
kv head) per SM and key ranges of at most 4096 tokens; these cases have many
more units than SMs, so every CTA runs several units back to back and the
hand-overs between units (Q reload, K/V ring running on, O handed back after
the epilogue, V tails on every ring slot) are exercised.

Each case compares every output row with the plain one-CTA-per-unit grid bit
for bit (the per-unit arithmetic is the same), and sampled rows with the
oracle, which gets its own host copy of the inputs taken before any kernel of
the library ran.
"""
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


def _seqs(specs, rng, spare=5):
    need = sum(W.blocks_for(c + s) for c, s in specs)
    nb = need + spare
    perm = rng.permutation(nb)
    cur, seqs = 0, []
    for c, s in specs:
        t = [int(x) for x in perm[cur:cur + W.blocks_for(c + s)]]
        cur += len(t)
        seqs.append(W.SeqSpec(num_tokens=c + s, block_table=t, num_cached_tokens=c, num_scheduled_tokens=s))
    return seqs, nb


def _sample_rows(cu_q, rng, per_seq=2):
    rows = []
    for b in range(len(cu_q) - 1):
        lq = int(cu_q[b + 1] - cu_q[b])
        for i in {lq - 1, *rng.integers(0, lq, size=per_seq).tolist()}:
            rows.append((int(cu_q[b]) + i, int(rng.integers(0, W.HQ))))
    return np.array(rows, dtype=np.int64)


def _case(pkv, specs, seed, dtype=torch.bfloat16, contiguous=False):
    dev = "cuda"
    rng = np.random.default_rng(seed)
    seqs, nb = _seqs(specs, rng)
    gen = W.make_generator(seed, dev)
    kc, vc = pool_tensors(nb, gen, dev, dtype)
    poison_dead_slots(kc, vc, seqs, lambda s: s.num_tokens)
    T = sum(s.num_scheduled_tokens for s in seqs)
    _, q, k, v = W.fused_qkv(T, gen, dev, dtype=dtype)
    meta = pkv.metadata.prepare_prefill(seqs, W.BLOCK_SIZE, force_block_tables=True)
    host = HostPool(kc, vc, seqs)                       # before any kernel of the library
    qb, kb, vb = bits(q), bits(k), bits(v)
    prefill = pkv.pkv_prefill_varlen_f16 if dtype == torch.float16 else pkv.pkv_prefill_varlen
    cu_q, cu_k = to_dev(meta["cu_seqlens_q"], dev), to_dev(meta["cu_seqlens_k"], dev)
    bt = to_dev(meta["block_tables"], dev)
    pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(meta["slot_mapping"], dev))
    plan = pkv.pkv_prefill_plan(meta["cu_seqlens_q"], meta["cu_seqlens_k"], dev)
    units = 8 * plan.numel()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert units >= 3 * sms, "the case should give every CTA several units"
    assert meta["max_seqlen_k"] <= 4096, "the case should take the persistent kernel"
    args = (q, cu_q, cu_k, meta["max_seqlen_q"], meta["max_seqlen_k"], W.SCALE)
    if contiguous:
        kw = dict(k=k, v=v)
    else:
        kw = dict(k_cache=kc, v_cache=vc, block_tables=bt)
    plain = prefill(*args, **kw)
    planned = prefill(*args, **kw, plan=plan)
    again = prefill(*args, **kw, plan=plan)             # the plan is reusable: same bits
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    assert torch.equal(planned, plain)
    assert torch.equal(again, planned)

    om = oracle.prepare_prefill(host.seqs, W.BLOCK_SIZE)
    ks, vs = host.slots()
    orc = oracle.default()
    orc.store_kvcache(kb, vb, ks, vs, om["slot_mapping"])
    rows = _sample_rows(om["cu_seqlens_q"], rng)
    ref = orc.prefill_varlen(qb, om["cu_seqlens_q"], om["cu_seqlens_k"], W.SCALE, k_cache=host.k, v_cache=host.v,
                             block_tables=oracle.pad_block_tables(host.seqs), num_kv_heads=W.HKV, rows=rows,
                             dtype=ORACLE_DTYPE[dtype])
    got = planned[torch.from_numpy(rows[:, 0]).to(dev), torch.from_numpy(rows[:, 1]).to(dev)]
    assert_close(got, ref, "planned prefill (sampled rows)")


def test_many_short_prompts(pkv):
    """72 prompts of 1..700 tokens, no cached keys (about 2,000 units)."""
    rng = np.random.default_rng(501)
    specs = [(0, int(n)) for n in rng.integers(1, 701, size=72)]
    _case(pkv, specs, 501)


def test_many_short_prompts_contiguous_keys(pkv):
    """The same kind of call with keys from contiguous k/v."""
    rng = np.random.default_rng(502)
    specs = [(0, int(n)) for n in rng.integers(1, 701, size=60)]
    _case(pkv, specs, 502, contiguous=True)


def test_cached_prefixes_and_mid_block_starts(pkv):
    """Cached prefixes of 0..1500 tokens (block-aligned or not) with 1..400
    new tokens each."""
    rng = np.random.default_rng(503)
    specs = [(int(c), int(s)) for c, s in zip(rng.integers(0, 1501, size=90), rng.integers(1, 401, size=90))]
    _case(pkv, specs, 503)


def test_many_short_prompts_f16(pkv):
    rng = np.random.default_rng(504)
    specs = [(int(c), int(s)) for c, s in zip(rng.integers(0, 300, size=64), rng.integers(1, 600, size=64))]
    _case(pkv, specs, 504, dtype=torch.float16)


def test_units_of_one_tile_each(pkv):
    """Prompts of 1..128 tokens: every unit is one key tile with a V tail, so
    consecutive units reuse the ring slots with fresh tails each time."""
    rng = np.random.default_rng(505)
    specs = [(0, int(n)) for n in rng.integers(1, 129, size=200)]
    _case(pkv, specs, 505)
