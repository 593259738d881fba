"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
(or an oracle error) when the oracle disagrees with:
* a library routine (torch's scaled_dot_product_attention in float64 on CPU,
  with its documented GQA and mask semantics),
* a closed form (uniform weights, one-hot weights, a single key),
* an invariant the pages fix (a paged cache through block tables gives the
  same result as a contiguous copy; the physical placement of blocks does not
  matter; keys after a query's position are never read; decode equals the last
  row of prefill; the store leaves untouched slots untouched).

``tests/test_oracle_attention.py`` runs them on the oracle as built;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and expects at least one to fail.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

BS = 256


# ---- input helpers (plain draws; no attention arithmetic) ------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float array -> bf16 bit patterns (round to nearest even via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


def randn_bits(rng, shape, scale=1.0):
    return bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


def f16_bits(x: np.ndarray) -> np.ndarray:
    """float array -> IEEE fp16 bit patterns (numpy's round to nearest even)."""
    return np.ascontiguousarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def f16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.float16)
    return t.double().numpy()


def randn_f16_bits(rng, shape, scale=1.0):
    return f16_bits(rng.standard_normal(shape) * scale)


def paged_from_contiguous(k, v, cu_k, rng, num_blocks, bs=BS, fill=None):
    """Scatter contiguous per-sequence K/V into a shuffled paged pool.

    Returns (k_cache, v_cache, block_tables). Slot of logical position t of
    sequence b is table[b][t // bs] * bs + t % bs -- the layout definition,
    written here as a brute-force per-token placement."""
    hkv, d = k.shape[1], k.shape[2]
    nseq = len(cu_k) - 1
    lens = [int(cu_k[i + 1] - cu_k[i]) for i in range(nseq)]
    nb_per = [-(-n // bs) for n in lens]
    width = max(max(nb_per), 1)
    perm = rng.permutation(num_blocks)
    assert sum(nb_per) <= num_blocks
    kc = np.empty((num_blocks * bs, hkv, d), dtype=np.uint16)
    vc = np.empty_like(kc)
    if fill is None:
        kc[:] = randn_bits(rng, kc.shape)
        vc[:] = randn_bits(rng, vc.shape)
    else:
        kc[:] = fill
        vc[:] = fill
    bt = np.full((nseq, width), -1, dtype=np.int32)
    cur = 0
    for b in range(nseq):
        for j in range(nb_per[b]):
            bt[b, j] = perm[cur]
            cur += 1
        for t in range(lens[b]):
            slot = bt[b, t // bs] * bs + t % bs
            kc[slot] = k[cu_k[b] + t]
            vc[slot] = v[cu_k[b] + t]
    return kc.reshape(num_blocks, bs, hkv, d), vc.reshape(num_blocks, bs, hkv, d), bt


def sdpa_reference(q, k, v, cu_q, cu_k, scale, widen=None):
    """torch SDPA (float64, CPU) per sequence, bottom-right causal mask given
    as an explicit boolean matrix, GQA through enable_gqa. ``widen`` turns bit
    patterns into float64 (bf16 by default)."""
    widen = bits_to_f64 if widen is None else widen
    outs = []
    for b in range(len(cu_q) - 1):
        qb = torch.from_numpy(widen(q[cu_q[b]:cu_q[b + 1]])).transpose(0, 1)   # [Hq, Lq, d]
        kb = torch.from_numpy(widen(k[cu_k[b]:cu_k[b + 1]])).transpose(0, 1)   # [Hkv, Lk, d]
        vb = torch.from_numpy(widen(v[cu_k[b]:cu_k[b + 1]])).transpose(0, 1)
        lq, lk = qb.shape[1], kb.shape[1]
        mask = torch.ones(lq, lk, dtype=torch.bool).tril(diagonal=lk - lq)
        o = F.scaled_dot_product_attention(qb[None], kb[None], vb[None], attn_mask=mask, scale=scale,
                                           enable_gqa=True)[0]
        outs.append(o.transpose(0, 1).numpy())
    return np.concatenate(outs, axis=0)


def _varlen_case(rng, lq_list, lk_list, hq, hkv, d):
    cu_q = np.concatenate([[0], np.cumsum(lq_list)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk_list)]).astype(np.int32)
    q = randn_bits(rng, (int(cu_q[-1]), hq, d))
    k = randn_bits(rng, (int(cu_k[-1]), hkv, d))
    v = randn_bits(rng, (int(cu_k[-1]), hkv, d))
    return q, k, v, cu_q, cu_k


# ---- pins -------------------------------------------------------------------

def pin_sdpa_equal_lengths(orc):
    """Lq == Lk (plain causal prefill), GQA 4 q heads / 2 kv heads, d=128."""
    rng = np.random.default_rng(11)
    q, k, v, cu_q, cu_k = _varlen_case(rng, [1, 7, 33], [1, 7, 33], 4, 2, 128)
    scale = 1 / math.sqrt(128)
    got = orc.prefill_varlen(q, cu_q, cu_k, scale, k=k, v=v, num_kv_heads=2)
    ref = sdpa_reference(q, k, v, cu_q, cu_k, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def pin_sdpa_prefix(orc):
    """Lk > Lq (prefix hit / chunked prefill): bottom-right causal alignment,
    paged keys through a shuffled block table, block_size 256, 4 q / 2 kv heads."""
    rng = np.random.default_rng(12)
    lq, lk = [5, 40, 3], [300, 40, 513]
    q, k, v, cu_q, cu_k = _varlen_case(rng, lq, lk, 4, 2, 128)
    kc, vc, bt = paged_from_contiguous(k, v, cu_k, rng, num_blocks=9)
    scale = 0.125
    got = orc.prefill_varlen(q, cu_q, cu_k, scale, k_cache=kc, v_cache=vc, block_tables=bt,
                             num_kv_heads=2)
    ref = sdpa_reference(q, k, v, cu_q, cu_k, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def pin_gqa_head_map(orc):
    """Query head h reads kv head h // (Hq/Hkv): with 8 q heads over 2 kv
    heads whose values differ by a constant offset, heads 0..3 see kv head 0
    and heads 4..7 see kv head 1 (constant keys make the weights uniform, so
    each output is the mean of its kv head's values)."""
    rng = np.random.default_rng(13)
    L = 9
    q = randn_bits(rng, (L, 8, 128))
    k = np.full((L, 2, 128), bf16_bits(np.array([0.5]))[0], dtype=np.uint16)
    v = np.empty((L, 2, 128), dtype=np.uint16)
    v[:, 0, :] = bf16_bits(np.full((L, 128), -3.0))
    v[:, 1, :] = bf16_bits(np.full((L, 128), 5.0))
    cu = np.array([0, L], dtype=np.int32)
    got = orc.prefill_varlen(q, cu, cu, 0.1, k=k, v=v, num_kv_heads=2)
    assert np.all(got[:, :4, :] == -3.0) and np.all(got[:, 4:, :] == 5.0)


def pin_uniform_keys_mean(orc):
    """Identical keys give equal weights: row i's output is the mean of
    v[0..i] (bottom-right causal with Lk = Lq)."""
    rng = np.random.default_rng(14)
    L = 20
    q = randn_bits(rng, (L, 2, 128))
    krow = randn_bits(rng, (1, 1, 128))
    k = np.repeat(krow, L, axis=0)
    v = randn_bits(rng, (L, 1, 128))
    cu = np.array([0, L], dtype=np.int32)
    got = orc.prefill_varlen(q, cu, cu, 0.2, k=k, v=v, num_kv_heads=1)
    vf = bits_to_f64(v)[:, 0, :]
    for i in range(L):
        mean = vf[: i + 1].mean(axis=0)
        np.testing.assert_allclose(got[i, 0], mean, rtol=0, atol=1e-12)
        np.testing.assert_allclose(got[i, 1], mean, rtol=0, atol=1e-12)


def pin_one_hot(orc):
    """One key far above the others: softmax is one-hot, output = that value row."""
    L, d = 6, 128
    q = bf16_bits(np.ones((L, 1, d)))
    k = bf16_bits(np.zeros((L, 1, d)))
    k[3] = bf16_bits(np.full((1, d), 8.0))       # score 8*128*scale vs 0
    rng = np.random.default_rng(15)
    v = randn_bits(rng, (L, 1, d))
    cu = np.array([0, L], dtype=np.int32)
    got = orc.prefill_varlen(q, cu, cu, 1.0, k=k, v=v, num_kv_heads=1)
    vf = bits_to_f64(v)[:, 0, :]
    for i in range(3, L):
        np.testing.assert_allclose(got[i, 0], vf[3], rtol=0, atol=1e-300)
    # rows before the hot key average uniformly over v[0..i] (all scores 0)
    for i in range(3):
        np.testing.assert_allclose(got[i, 0], vf[: i + 1].mean(axis=0), rtol=0, atol=1e-12)


def pin_single_key(orc):
    """Lq = Lk = 1: the output is v[0] exactly, whatever q and k are."""
    rng = np.random.default_rng(16)
    q = randn_bits(rng, (1, 2, 128))
    k = randn_bits(rng, (1, 1, 128))
    v = randn_bits(rng, (1, 1, 128))
    cu = np.array([0, 1], dtype=np.int32)
    got = orc.prefill_varlen(q, cu, cu, 0.3, k=k, v=v, num_kv_heads=1)
    assert np.array_equal(got[0, 0], bits_to_f64(v)[0, 0])
    assert np.array_equal(got[0, 1], bits_to_f64(v)[0, 0])


def pin_two_keys_logistic(orc):
    """d=4 hand check: two keys with score gap g give weights 1/(1+e^g) and
    e^g/(1+e^g) (the logistic form of a two-way softmax)."""
    q = bf16_bits(np.array([[[1.0, 0.0, 0.0, 0.0]]]))
    k = bf16_bits(np.array([[[0.0, 1.0, 0.0, 0.0]], [[2.0, 0.0, 0.0, 0.0]]]))
    v = bf16_bits(np.array([[[1.0, 2.0, 3.0, 4.0]], [[-4.0, 0.0, 8.0, 0.5]]]))
    cu_q = np.array([0, 1], dtype=np.int32)
    cu_k = np.array([0, 2], dtype=np.int32)
    got = orc.prefill_varlen(q, cu_q, cu_k, 0.5, k=k, v=v, num_kv_heads=1)[0, 0]
    g = 1.0                                   # 0.5 * (2 - 0)
    w1 = math.exp(g) / (1 + math.exp(g))
    w0 = 1 / (1 + math.exp(g))
    want = w0 * np.array([1, 2, 3, 4.0]) + w1 * np.array([-4, 0, 8, 0.5])
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


def pin_paged_equals_contiguous(orc):
    """Same keys through a shuffled paged pool or a contiguous buffer: identical."""
    rng = np.random.default_rng(17)
    lq = lk = [100, 257, 31]
    q, k, v, cu_q, cu_k = _varlen_case(rng, lq, lk, 4, 2, 128)
    kc, vc, bt = paged_from_contiguous(k, v, cu_k, rng, num_blocks=8)
    a = orc.prefill_varlen(q, cu_q, cu_k, 0.09, k=k, v=v, num_kv_heads=2)
    b = orc.prefill_varlen(q, cu_q, cu_k, 0.09, k_cache=kc, v_cache=vc, block_tables=bt,
                           num_kv_heads=2)
    assert np.array_equal(a, b)


def pin_causal_poison(orc):
    """Keys and values after a query's position are never read: NaN there
    changes nothing for rows at or before it."""
    rng = np.random.default_rng(18)
    L = 50
    q, k, v, cu_q, cu_k = _varlen_case(rng, [L], [L], 2, 1, 128)
    clean = orc.prefill_varlen(q, cu_q, cu_k, 0.1, k=k, v=v, num_kv_heads=1)
    p0 = 29
    kp, vp = k.copy(), v.copy()
    kp[p0 + 1:] = 0x7FC0      # bf16 NaN
    vp[p0 + 1:] = 0x7FC0
    pois = orc.prefill_varlen(q, cu_q, cu_k, 0.1, k=kp, v=vp, num_kv_heads=1)
    assert np.array_equal(clean[: p0 + 1], pois[: p0 + 1])
    assert np.all(np.isnan(pois[p0 + 1:]))


def pin_block_permutation(orc):
    """Moving a sequence's blocks to other physical blocks (and its table
    with them) leaves decode outputs bit-identical."""
    rng = np.random.default_rng(19)
    ctx = np.array([1, 255, 256, 257, 700], dtype=np.int32)
    k = randn_bits(rng, (int(ctx.sum()), 2, 128))
    v = randn_bits(rng, (int(ctx.sum()), 2, 128))
    cu = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    q = randn_bits(rng, (len(ctx), 4, 128))
    kc1, vc1, bt1 = paged_from_contiguous(k, v, cu, np.random.default_rng(1), num_blocks=12)
    kc2, vc2, bt2 = paged_from_contiguous(k, v, cu, np.random.default_rng(2), num_blocks=12)
    assert not np.array_equal(bt1, bt2)
    a = orc.decode(q, kc1, vc1, bt1, ctx, 0.1, num_kv_heads=2)
    b = orc.decode(q, kc2, vc2, bt2, ctx, 0.1, num_kv_heads=2)
    assert np.array_equal(a, b)


def pin_decode_is_last_prefill_row(orc):
    """Decode with context n equals the last row of a causal prefill of length n."""
    rng = np.random.default_rng(20)
    ctx = np.array([1, 37, 256, 300, 511], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    qall = randn_bits(rng, (int(ctx.sum()), 4, 128))
    k = randn_bits(rng, (int(ctx.sum()), 2, 128))
    v = randn_bits(rng, (int(ctx.sum()), 2, 128))
    kc, vc, bt = paged_from_contiguous(k, v, cu, rng, num_blocks=8)
    pre = orc.prefill_varlen(qall, cu, cu, 0.0884, k_cache=kc, v_cache=vc, block_tables=bt,
                             num_kv_heads=2)
    qdec = np.ascontiguousarray(qall[cu[1:] - 1])
    dec = orc.decode(qdec, kc, vc, bt, ctx, 0.0884, num_kv_heads=2)
    assert np.array_equal(dec, pre[cu[1:] - 1])


def pin_decode_sdpa(orc):
    """Decode against torch SDPA on the contiguous keys (one query at the end)."""
    rng = np.random.default_rng(21)
    ctx = np.array([3, 260, 513], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    k = randn_bits(rng, (int(ctx.sum()), 2, 128))
    v = randn_bits(rng, (int(ctx.sum()), 2, 128))
    q = randn_bits(rng, (len(ctx), 4, 128))
    kc, vc, bt = paged_from_contiguous(k, v, cu, rng, num_blocks=7)
    got = orc.decode(q, kc, vc, bt, ctx, 0.0884, num_kv_heads=2)
    cuq = np.arange(len(ctx) + 1, dtype=np.int32)
    ref = sdpa_reference(q, k, v, cuq, cu, 0.0884)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def pin_decode_empty_context(orc):
    """A graph-padding row (context_len 0) gives zeros, never NaN."""
    rng = np.random.default_rng(22)
    kc = randn_bits(rng, (2, BS, 1, 128))
    vc = randn_bits(rng, (2, BS, 1, 128))
    q = randn_bits(rng, (2, 2, 128))
    bt = np.array([[0], [1]], dtype=np.int32)
    got = orc.decode(q, kc, vc, bt, np.array([0, 5], dtype=np.int32), 0.1, num_kv_heads=1)
    assert np.all(got[0] == 0.0) and np.all(np.isfinite(got[1]))


def pin_shared_prefix(orc):
    """Two sequences with the same prefix blocks (shared physical blocks) and
    the same suffix values give identical outputs."""
    rng = np.random.default_rng(23)
    hkv, d = 2, 128
    pool = 6
    kc = randn_bits(rng, (pool, BS, hkv, d))
    vc = randn_bits(rng, (pool, BS, hkv, d))
    kc[4] = kc[2]
    vc[4] = vc[2]
    kc[5] = kc[3]
    vc[5] = vc[3]
    bt = np.array([[0, 1, 2], [0, 1, 4]], dtype=np.int32)   # blocks 0,1 shared; 2 and 4 equal copies
    s = 100
    q1 = randn_bits(rng, (s, 4, d))
    q = np.concatenate([q1, q1], axis=0)
    cu_q = np.array([0, s, 2 * s], dtype=np.int32)
    cu_k = np.array([0, 2 * BS + s, 4 * BS + 2 * s], dtype=np.int32)
    got = orc.prefill_varlen(q, cu_q, cu_k, 0.1, k_cache=kc, v_cache=vc, block_tables=bt,
                             num_kv_heads=hkv)
    assert np.array_equal(got[:s], got[s:])
    # and a copy that differs in a suffix block must differ
    kc[4, 0, 0, 0] ^= 0x0040
    got2 = orc.prefill_varlen(q, cu_q, cu_k, 0.1, k_cache=kc, v_cache=vc, block_tables=bt,
                              num_kv_heads=hkv)
    assert not np.array_equal(got2[:s], got2[s:])


def pin_store_layout(orc):
    """Store: the pages' worked example puts the 8 prefill tokens at slots
    0..5, 256, 257 (block_size 256); rows land exactly there, strided k/v rows
    (views of a fused qkv buffer) are read with their stride, slot -1 is
    skipped, and every other slot keeps its previous bytes."""
    rng = np.random.default_rng(24)
    hkv, d = 8, 128
    fused = randn_bits(rng, (9, (16 + 2 * hkv) * d))
    k = fused[:, 16 * d:(16 + hkv) * d].reshape(9, hkv, d)
    v = fused[:, (16 + hkv) * d:].reshape(9, hkv, d)
    slots = np.array([0, 1, 2, 3, 4, 5, 256, 257, -1], dtype=np.int32)
    kc = np.full((2 * BS, hkv, d), 0x7FC0, dtype=np.uint16)
    vc = np.full((2 * BS, hkv, d), 0x7FC0, dtype=np.uint16)
    orc.store_kvcache(k, v, kc, vc, slots)
    for i, s in enumerate(slots[:8]):
        assert np.array_equal(kc[s], k[i]) and np.array_equal(vc[s], v[i])
    written = set(int(s) for s in slots[:8])
    for s in range(2 * BS):
        if s not in written:
            assert np.all(kc[s] == 0x7FC0) and np.all(vc[s] == 0x7FC0)


def pin_element_widening(orc):
    """Every one of the 65536 bit patterns widens exactly as numpy reads it:
    bf16 as the top half of an IEEE float32, fp16 as IEEE binary16 (zeros
    with their sign, subnormals, infinities, NaNs)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):     # signalling-NaN patterns widen to quiet NaNs
        want_bf16 = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        want_f16 = bits.view(np.float16).astype(np.float64)
    for dtype, want in (("bf16", want_bf16), ("f16", want_f16)):
        got = orc.elements_to_f64(bits, dtype)
        np.testing.assert_array_equal(got, want)
        fin = np.isfinite(want)
        assert np.array_equal(np.signbit(got[fin]), np.signbit(want[fin]))


def pin_sdpa_f16_prefix(orc):
    """fp16 inputs: prefix-cache prefill against float64 SDPA on the same
    fp16 values read by torch. One sequence's keys are tiny (fp16
    subnormals) and another's values large (|v| up to thousands), so both
    ends of the fp16 range are decoded."""
    rng = np.random.default_rng(25)
    lq, lk = [6, 30, 2], [270, 30, 520]
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q = randn_f16_bits(rng, (int(cu_q[-1]), 4, 128))
    kf = rng.standard_normal((int(cu_k[-1]), 2, 128))
    kf[cu_k[1]:cu_k[2]] *= 3e-6                    # fp16 subnormal range (< 6.1e-5)
    vf = rng.standard_normal((int(cu_k[-1]), 2, 128))
    vf[cu_k[2]:] *= 2000.0
    k, v = f16_bits(kf), f16_bits(vf)
    kc, vc, bt = paged_from_contiguous(k, v, cu_k, rng, num_blocks=9)
    scale = 1 / math.sqrt(128)
    got = orc.prefill_varlen(q, cu_q, cu_k, scale, k_cache=kc, v_cache=vc, block_tables=bt,
                             num_kv_heads=2, dtype="f16")
    ref = sdpa_reference(q, k, v, cu_q, cu_k, scale, widen=f16_bits_to_f64)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def pin_decode_sdpa_f16(orc):
    """fp16 decode against float64 SDPA on the contiguous keys."""
    rng = np.random.default_rng(26)
    ctx = np.array([2, 257, 600], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    k = randn_f16_bits(rng, (int(ctx.sum()), 2, 128))
    v = randn_f16_bits(rng, (int(ctx.sum()), 2, 128), scale=10.0)
    q = randn_f16_bits(rng, (len(ctx), 4, 128))
    kc, vc, bt = paged_from_contiguous(k, v, cu, rng, num_blocks=7)
    got = orc.decode(q, kc, vc, bt, ctx, 0.0884, num_kv_heads=2, dtype="f16")
    cuq = np.arange(len(ctx) + 1, dtype=np.int32)
    ref = sdpa_reference(q, k, v, cuq, cu, 0.0884, widen=f16_bits_to_f64)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


ALL_PINS = [
    pin_sdpa_equal_lengths,
    pin_sdpa_prefix,
    pin_gqa_head_map,
    pin_uniform_keys_mean,
    pin_one_hot,
    pin_single_key,
    pin_two_keys_logistic,
    pin_paged_equals_contiguous,
    pin_causal_poison,
    pin_block_permutation,
    pin_decode_is_last_prefill_row,
    pin_decode_sdpa,
    pin_decode_empty_context,
    pin_shared_prefix,
    pin_store_layout,
    pin_element_widening,
    pin_sdpa_f16_prefix,
    pin_decode_sdpa_f16,
]
