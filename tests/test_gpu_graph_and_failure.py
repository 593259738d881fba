"""Store + decode for several layers captured in one CUDA graph (the decode
path nano-vLLM replays), plus the bounded-wait failure path."""
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


def test_layers_in_one_graph_match_eager_and_oracle(pkv):
    dev = "cuda"
    L = 4
    wl = W.sweep_decode(seed=15, num_seqs=96, num_layers=L)
    B = len(wl.seqs)
    gen = W.make_generator(15, dev)
    shape = (2, L, wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    kv = W.normal_bf16(shape, gen, dev)
    kv0 = kv.clone()
    qkv = [W.fused_qkv(B, gen, dev) for _ in range(L)]
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE, table_width=16)
    slot = to_dev(meta["slot_mapping"], dev)
    ctx = to_dev(meta["context_lens"], dev)
    bt = to_dev(meta["block_tables"], dev)
    ws = pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev)
    outs = torch.empty(L, B, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)

    def step():
        for l in range(L):
            _, q, k, v = qkv[l]
            pkv.pkv_store_kvcache(k, v, kv[0, l], kv[1, l], slot)
            pkv.pkv_decode(q, kv[0, l], kv[1, l], bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws, out=outs[l])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                  # eager warm-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = outs.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    kv.copy_(kv0)
    outs.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs, eager)
    assert pkv.pkv_device_error() == 0

    # oracle on layer L-1 for a few sequences
    sample = [0, 1, B // 2, B - 1]
    host = HostPool(kv0[0, L - 1], kv0[1, L - 1], [wl.seqs[i] for i in sample])
    om = oracle.prepare_decode(host.seqs, W.BLOCK_SIZE)
    ks, vs = host.slots()
    _, q, k, v = qkv[L - 1]
    orc = oracle.default()
    orc.store_kvcache(bits(k)[sample], bits(v)[sample], ks, vs, om["slot_mapping"])
    ref = orc.decode(bits(q)[sample], host.k, host.v, om["block_tables"], om["context_lens"], W.SCALE,
                     num_kv_heads=W.HKV)
    assert_close(outs[L - 1, torch.tensor(sample, device=dev)], ref, "graph layer")

    # replay with new contents of the static buffers: padded rows (slot -1, ctx 0)
    slot[B // 2:] = -1
    ctx[B // 2:] = 0
    g.replay()
    torch.cuda.synchronize()
    assert torch.all(outs[:, B // 2:] == 0)
    assert pkv.pkv_device_error() == 0


def test_padded_graph_replay_matches_unpadded(pkv):
    """A 200-sequence decode step replayed through a graph captured for 256
    rows, with the buffer refresh the pages do before a replay
    (slot_mapping.fill_(-1), context_lens.zero_(), then only the live part of
    each buffer overwritten, so padding rows and table tails keep an earlier
    step's contents). The live rows must equal an eager, unpadded store +
    decode bit for bit, padding rows are zeros, and the caches end identical
    (padding stores nothing)."""
    dev = "cuda"
    wl = W.padded_decode()
    B, G = len(wl.seqs), wl.graph_batch
    width = W.MAX_MODEL_LEN // W.BLOCK_SIZE
    gen = W.make_generator(wl.seed, dev)
    kc, vc = pool_tensors(wl.num_blocks, gen, dev)
    _, q_new, k_new, v_new = W.fused_qkv(B, gen, dev)
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    rng = np.random.default_rng(7)
    # static graph buffers, first filled by an "earlier step" of 256 live rows
    _, q_s, k_s, v_s = W.fused_qkv(G, gen, dev)
    slot_s = to_dev(rng.permutation(wl.num_blocks * W.BLOCK_SIZE)[:G].astype(np.int32), dev)
    ctx_s = to_dev(rng.integers(1, W.MAX_MODEL_LEN + 1, size=G).astype(np.int32), dev)
    bt_s = to_dev(rng.integers(0, wl.num_blocks, size=(G, width)).astype(np.int32), dev)
    out_s = torch.empty(G, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    ws = pkv.decode_workspace(G, W.MAX_MODEL_LEN, dev)
    kc_eager, vc_eager = kc.clone(), vc.clone()
    kc0, vc0 = kc.clone(), vc.clone()

    def step():
        pkv.pkv_store_kvcache(k_s, v_s, kc, vc, slot_s)
        pkv.pkv_decode(q_s, kc, vc, bt_s, ctx_s, W.MAX_MODEL_LEN, W.SCALE, ws, out=out_s)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    kc.copy_(kc0)
    vc.copy_(vc0)
    # the refresh before a replay, as the pages' run_model does it
    slot_s.fill_(-1)
    ctx_s.zero_()
    w = meta["block_tables"].shape[1]
    bt_s[:B, :w] = to_dev(meta["block_tables"], dev)
    slot_s[:B] = to_dev(meta["slot_mapping"], dev)
    ctx_s[:B] = to_dev(meta["context_lens"], dev)
    q_s[:B], k_s[:B], v_s[:B] = q_new, k_new, v_new
    g.replay()
    # eager, unpadded
    ws2 = pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev)
    pkv.pkv_store_kvcache(k_new, v_new, kc_eager, vc_eager, to_dev(meta["slot_mapping"], dev))
    ref = pkv.pkv_decode(q_new, kc_eager, vc_eager, to_dev(meta["block_tables"], dev),
                         to_dev(meta["context_lens"], dev), W.MAX_MODEL_LEN, W.SCALE, ws2)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    assert torch.equal(out_s[:B], ref)
    assert torch.all(out_s[B:] == 0)
    assert torch.equal(kc, kc_eager) and torch.equal(vc, vc_eager)


def test_bounded_wait_times_out_and_gpu_stays_usable(pkv):
    pkv.pkv_device_error(clear=True)
    pkv.pkv_selftest_wait_timeout(2_000_000)     # 2 ms on a barrier nobody completes
    assert pkv.pkv_device_error(clear=True) & pkv.PKV_DEVERR_TIMEOUT
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0
