"""Oracle parity of the decode paths that run inside CUDA graphs or fuse the
store: graph-padded replay, the bf16 store fused into the decode launch, and
the full 28-layer x 512-sequence sweep captured in one graph.

In every case the oracle receives host copies of the generated inputs taken
before any kernel of the library runs, applies its own store and runs its own
decode; the GPU's output (and, where stated, its cache bytes) are compared
with that.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import HostPool, assert_close, bits, pool_tensors, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def _graph_of(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                    # eager warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _oracle_decode(host, q_rows, k_rows, v_rows, dtype="bf16", tables=None):
    """Store the sampled sequences' new rows into the oracle's own copy of
    their blocks, then decode them. tables: optional block tables to hand the
    oracle instead of the compact ones (same live entries, other tails)."""
    om = oracle.prepare_decode(host.seqs, W.BLOCK_SIZE)
    ks, vs = host.slots()
    orc = oracle.default()
    orc.store_kvcache(k_rows, v_rows, ks, vs, om["slot_mapping"])
    bt = om["block_tables"] if tables is None else tables
    return orc.decode(q_rows, host.k, host.v, bt, om["context_lens"], W.SCALE, num_kv_heads=W.HKV, dtype=dtype)


@pytest.mark.parametrize("hi", [4096, 2000])
def test_padded_graph_replay_matches_oracle(pkv, hi):
    """engine/model_runner.py run_model ("vLLM 学习笔记 02：nano-vllm 源码逐段精读"):
    a 200-sequence decode step replayed through the graph captured for 256
    rows, after slot_mapping.fill_(-1), context_lens.zero_() and an overwrite
    of only the live part of each buffer. Sampled live rows (shortest and
    longest contexts, rows whose block-table tails hold an earlier step's
    entries) against the oracle, which is handed the same stale tails and
    must not read them either; the padding rows against the oracle's
    context-0 result (zeros); the stored rows against the oracle's store.
    With contexts up to 4096 the live part of the table buffer is its whole
    width (16 blocks) and the tails of shorter rows are -1; with contexts up
    to 2000 it is 8 blocks wide and columns 8..15 keep the earlier step's ids."""
    dev = "cuda"
    wl = W.padded_decode(hi=hi)
    B, G = len(wl.seqs), wl.graph_batch
    width = W.MAX_MODEL_LEN // W.BLOCK_SIZE
    gen = W.make_generator(wl.seed, dev)
    kc, vc = pool_tensors(wl.num_blocks, gen, dev)
    _, q_new, k_new, v_new = W.fused_qkv(B, gen, dev)
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    rng = np.random.default_rng(17)
    # the static graph buffers, first holding an "earlier step" of 256 live rows
    _, q_s, k_s, v_s = W.fused_qkv(G, gen, dev)
    slot_s = to_dev(rng.permutation(wl.num_blocks * W.BLOCK_SIZE)[:G].astype(np.int32), dev)
    ctx_s = to_dev(rng.integers(1, W.MAX_MODEL_LEN + 1, size=G).astype(np.int32), dev)
    bt_s = to_dev(rng.integers(0, wl.num_blocks, size=(G, width)).astype(np.int32), dev)
    out_s = torch.empty(G, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    ws = pkv.decode_workspace(G, W.MAX_MODEL_LEN, dev)

    ctx = np.array([s.num_tokens for s in wl.seqs])
    nblk = np.array([len(s.block_table) for s in wl.seqs])
    w_live = int(nblk.max())
    short_tables = np.flatnonzero(nblk < w_live)          # -1 padding, then the earlier step's entries
    sample = sorted({int(ctx.argmin()), int(ctx.argmax()), *short_tables[:3].tolist(),
                     *rng.choice(B, 6, replace=False).tolist()})
    kc0, vc0 = kc.clone(), vc.clone()
    host = HostPool(kc, vc, [wl.seqs[i] for i in sample])   # before any kernel of the library
    kb, vb, qb = bits(k_new)[sample], bits(v_new)[sample], bits(q_new)[sample]

    def step():
        pkv.pkv_store_kvcache(k_s, v_s, kc, vc, slot_s)
        pkv.pkv_decode(q_s, kc, vc, bt_s, ctx_s, W.MAX_MODEL_LEN, W.SCALE, ws, out=out_s)

    g = _graph_of(step)
    kc.copy_(kc0)
    vc.copy_(vc0)
    del kc0, vc0
    # the refresh before a replay, as run_model does it
    slot_s.fill_(-1)
    ctx_s.zero_()
    bt_s[:B, :w_live] = to_dev(meta["block_tables"], dev)
    slot_s[:B] = to_dev(meta["slot_mapping"], dev)
    ctx_s[:B] = to_dev(meta["context_lens"], dev)
    q_s[:B], k_s[:B], v_s[:B] = q_new, k_new, v_new
    bt_after = bt_s.cpu().numpy()          # what the replay reads: live part, -1 padding, stale tails
    g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0

    # the oracle's tables: live entries remapped to its compact pool, the rest
    # exactly as the replay saw them (-1 or stale ids it must never read)
    tables = bt_after[sample].copy()
    for r, i in enumerate(sample):
        n = len(wl.seqs[i].block_table)
        tables[r, :n] = host.seqs[r].block_table
    stale = any((tables[r, len(wl.seqs[i].block_table):] >= 0).any() for r, i in enumerate(sample))
    assert stale == (w_live < width)
    ref = _oracle_decode(host, qb, kb, vb, tables=tables)
    assert_close(out_s[torch.tensor(sample, device=dev)], ref, "graph-padded live rows")

    # padding rows: the oracle, given context 0 and the stale table rows the
    # replay saw, reads nothing and gives zeros; so must the GPU
    pad_rows = [B, (B + G) // 2, G - 1]
    ref_pad = oracle.default().decode(bits(q_s)[pad_rows], host.k, host.v, bt_after[pad_rows],
                                      np.zeros(len(pad_rows), np.int32), W.SCALE, num_kv_heads=W.HKV)
    assert np.all(ref_pad == 0)
    assert torch.equal(out_s[pad_rows].float().cpu(), torch.from_numpy(ref_pad).float())

    # the GPU cache at the sampled sequences' blocks equals the oracle's store
    idx = torch.tensor(sorted(host.remap, key=host.remap.get), dtype=torch.long, device=dev)
    assert np.array_equal(bits(kc.index_select(0, idx)), host.k)
    assert np.array_equal(bits(vc.index_select(0, idx)), host.v)


@pytest.mark.parametrize("factory", [W.tiny_decode, W.batched_decode])
def test_store_decode_fused_bf16_matches_oracle(pkv, factory):
    """pkv_store_decode (bf16) on the 4-sequence and the 256-sequence
    workloads against the oracle's own store and decode: the output rows and
    the stored cache bytes; padding rows (slot -1, context 0) give zeros and
    store nothing."""
    dev = "cuda"
    wl = factory()
    B, pad = len(wl.seqs), 2
    gen = W.make_generator(wl.seed + 2000, dev)
    kc, vc = pool_tensors(wl.num_blocks, gen, dev)
    _, q, k, v = W.fused_qkv(B + pad, gen, dev)
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE, table_width=16)
    ctxs = np.array([s.num_tokens for s in wl.seqs])
    if B <= 8:
        sample = list(range(B))
    else:
        rng = np.random.default_rng(3)
        sample = sorted({int(ctxs.argmin()), int(ctxs.argmax()), *rng.choice(B, 10, replace=False).tolist()})
    host = HostPool(kc, vc, [wl.seqs[i] for i in sample])   # before any kernel of the library
    qb, kb, vb = bits(q), bits(k), bits(v)
    whole = wl.num_blocks <= 64            # small pool: the oracle also gets a copy of all of it
    if whole:
        kc_h = bits(kc).reshape(-1, W.HKV, W.HEAD_DIM)
        vc_h = bits(vc).reshape(-1, W.HKV, W.HEAD_DIM)

    slot = torch.full((B + pad,), -1, dtype=torch.int32, device=dev)
    slot[:B] = to_dev(meta["slot_mapping"], dev)
    ctx = torch.zeros(B + pad, dtype=torch.int32, device=dev)
    ctx[:B] = to_dev(meta["context_lens"], dev)
    bt = torch.full((B + pad, 16), -1, dtype=torch.int32, device=dev)
    bt[:B] = to_dev(meta["block_tables"], dev)
    ws = pkv.decode_workspace(B + pad, W.MAX_MODEL_LEN, dev)
    out = pkv.pkv_store_decode(q, k, v, slot, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0

    ref = _oracle_decode(host, qb[sample], kb[sample], vb[sample])
    assert_close(out[torch.tensor(sample, device=dev)], ref, f"{wl.name} fused store + decode")
    assert torch.all(out[B:] == 0)
    idx = torch.tensor(sorted(host.remap, key=host.remap.get), dtype=torch.long, device=dev)
    assert np.array_equal(bits(kc.index_select(0, idx)), host.k)
    assert np.array_equal(bits(vc.index_select(0, idx)), host.v)
    if whole:
        # the whole pool: the oracle stores every sequence's new row into its
        # copy; the GPU's pool must match it byte for byte (padding stored nothing)
        om = oracle.prepare_decode([oracle.SeqState(s.num_tokens, list(s.block_table)) for s in wl.seqs],
                                   W.BLOCK_SIZE)
        oracle.default().store_kvcache(kb[:B], vb[:B], kc_h, vc_h, om["slot_mapping"])
        assert np.array_equal(bits(kc).reshape(-1, W.HKV, W.HEAD_DIM), kc_h)
        assert np.array_equal(bits(vc).reshape(-1, W.HKV, W.HEAD_DIM), vc_h)


def test_sweep_28_layers_full_graph_matches_oracle(pkv):
    """The full 28-layer sweep (512 sequences, contexts geometric with mean
    800 clipped to [1, 4096], a [2, 28, blocks, 256, 8, 128] cache): store +
    decode per layer captured in one CUDA graph and replayed once, with two
    launches per layer and with the store fused into the decode launch.
    Eight sampled sequences (shortest, longest, median, block edges, random)
    on the first, a middle and the last layer against the oracle, and the
    stored rows of those layers against the oracle's store."""
    dev = "cuda"
    wl = W.sweep_decode()
    L, B = wl.num_layers, len(wl.seqs)
    gen = W.make_generator(wl.seed, dev)
    kv = W.normal_bf16((2, L, wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM), gen, dev)
    qkv = [W.fused_qkv(B, gen, dev) for _ in range(L)]
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE, table_width=W.MAX_MODEL_LEN // W.BLOCK_SIZE)
    ctx_h = meta["context_lens"]
    order = np.argsort(ctx_h, kind="stable")
    edges = [i for i in range(B) if ctx_h[i] % W.BLOCK_SIZE in (0, 1)][:2]
    rng = np.random.default_rng(5)
    sample = sorted({int(order[0]), int(order[-1]), int(order[B // 2]), *edges,
                     *rng.choice(B, 8, replace=False).tolist()})[:10]
    layers = [0, L // 2, L - 1]
    hosts = {l: HostPool(kv[0, l], kv[1, l], [wl.seqs[i] for i in sample]) for l in layers}
    new_rows = {l: tuple(bits(t)[sample] for t in qkv[l][1:]) for l in layers}   # q, k, v of the sample

    slot = to_dev(meta["slot_mapping"], dev)
    ctx = to_dev(ctx_h, dev)
    bt = to_dev(meta["block_tables"], dev)
    ws = pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev)
    outs = torch.empty(L, B, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    outs_fused = torch.empty_like(outs)

    def sweep():
        for l in range(L):
            _, q, k, v = qkv[l]
            pkv.pkv_store_kvcache(k, v, kv[0, l], kv[1, l], slot)
            pkv.pkv_decode(q, kv[0, l], kv[1, l], bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws, out=outs[l])

    def sweep_fused():
        for l in range(L):
            _, q, k, v = qkv[l]
            pkv.pkv_store_decode(q, k, v, slot, kv[0, l], kv[1, l], bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws,
                                 out=outs_fused[l])

    # the store writes the same rows to the same slots every time, so both
    # graphs (and their warm-up passes) leave the cache in one state
    g, gf = _graph_of(sweep), _graph_of(sweep_fused)
    outs.zero_()
    outs_fused.zero_()
    g.replay()
    gf.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0

    sel = torch.tensor(sample, device=dev)
    for l in layers:
        host = hosts[l]
        qb, kb, vb = new_rows[l]
        ref = _oracle_decode(host, qb, kb, vb)
        assert_close(outs[l, sel], ref, f"sweep layer {l}")
        assert_close(outs_fused[l, sel], ref, f"sweep layer {l} (fused store)")
        idx = torch.tensor(sorted(host.remap, key=host.remap.get), dtype=torch.long, device=dev)
        assert np.array_equal(bits(kv[0, l].index_select(0, idx)), host.k)
        assert np.array_equal(bits(kv[1, l].index_select(0, idx)), host.v)
    del kv, g, gf
    torch.cuda.empty_cache()
