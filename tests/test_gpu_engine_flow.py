"""An engine-like run of several steps, all on the GPU and in fp16.

Prefill: device-built metadata (pkv_build_prefill_metadata) -> store -> paged
prefill with cached prefixes. Decode: every step builds its metadata on the
device (pkv_build_decode_metadata) and stores the new token inside the decode
launch (pkv_store_decode_f16); the step is captured once in a CUDA graph and
replayed with new inputs, as the pages' model runner replays its graphs. Each
step is compared with the oracle, which runs the same steps on its own copy
of the inputs (taken before any kernel of the library ran)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, bits, pool_tensors, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def test_prefill_then_graph_replayed_decode_f16(pkv):
    dev, dt = "cuda", torch.float16
    rng = np.random.default_rng(77)
    prompt = [700, 300, 530, 257, 64, 1024]
    cached = [0, 0, 256, 0, 0, 512]           # prefix-cache hits are whole blocks
    steps = 4
    B = len(prompt)
    need = [W.blocks_for(n + steps) for n in prompt]
    nb = sum(need) + 4
    perm = rng.permutation(nb)
    tables, cur = [], 0
    for n in need:
        tables.append([int(x) for x in perm[cur:cur + n]])
        cur += n
    gen = W.make_generator(77, dev)
    kc, vc = pool_tensors(nb, gen, dev, dt)
    kc_h = bits(kc).reshape(-1, W.HKV, W.HEAD_DIM)      # the oracle's pool, before any kernel runs
    vc_h = bits(vc).reshape(-1, W.HKV, W.HEAD_DIM)
    orc = oracle.default()
    width = max(len(t) for t in tables)
    bt_h = oracle.pad_block_tables([oracle.SeqState(1, t) for t in tables], width)
    bt = to_dev(bt_h, dev)

    # ---- prefill step ----
    sched = [p - c for p, c in zip(prompt, cached)]
    T = sum(sched)
    meta = pkv.pkv_build_prefill_metadata(to_dev(np.array(cached, np.int32), dev),
                                          to_dev(np.array(sched, np.int32), dev), bt, nb, T)
    _, q, k, v = W.fused_qkv(T, gen, dev, dtype=dt)
    pkv.pkv_store_kvcache(k, v, kc, vc, meta["slot_mapping"][:T])
    out = pkv.pkv_prefill_varlen_f16(q, meta["cu_seqlens_q"], meta["cu_seqlens_k"], max(sched), max(prompt),
                                     W.SCALE, k_cache=kc, v_cache=vc, block_tables=bt)
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    oseqs = [oracle.SeqState(p, t, c, s) for p, t, c, s in zip(prompt, tables, cached, sched)]
    om = oracle.prepare_prefill(oseqs, W.BLOCK_SIZE)
    assert np.array_equal(meta["slot_mapping"][:T].cpu().numpy(), om["slot_mapping"])
    assert meta["max_seqlens"].tolist() == [om["max_seqlen_q"], om["max_seqlen_k"]]
    orc.store_kvcache(bits(k), bits(v), kc_h, vc_h, om["slot_mapping"])
    ref = orc.prefill_varlen(bits(q), om["cu_seqlens_q"], om["cu_seqlens_k"], W.SCALE,
                             k_cache=kc_h.reshape(nb, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM),
                             v_cache=vc_h.reshape(nb, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM),
                             block_tables=bt_h, num_kv_heads=W.HKV, dtype="f16")
    assert_close(out, ref, "prefill")

    # ---- decode steps: one captured graph, replayed ----
    max_ctx = W.MAX_MODEL_LEN
    qkv_s = torch.zeros(B, (W.HQ + 2 * W.HKV) * W.HEAD_DIM, dtype=dt, device=dev)
    q_s = qkv_s[:, :W.HQ * W.HEAD_DIM].view(B, W.HQ, W.HEAD_DIM)
    k_s = qkv_s[:, W.HQ * W.HEAD_DIM:(W.HQ + W.HKV) * W.HEAD_DIM].view(B, W.HKV, W.HEAD_DIM)
    v_s = qkv_s[:, (W.HQ + W.HKV) * W.HEAD_DIM:].view(B, W.HKV, W.HEAD_DIM)
    ntok_s = torch.zeros(B, dtype=torch.int32, device=dev)   # 0 = padding row while capturing
    out_s = torch.empty(B, W.HQ, W.HEAD_DIM, dtype=dt, device=dev)
    ws = pkv.decode_workspace(B, max_ctx, dev)
    built = {}

    def step():
        m = pkv.pkv_build_decode_metadata(ntok_s, bt, nb)
        built.update(m)
        pkv.pkv_store_decode_f16(q_s, k_s, v_s, m["slot_mapping"], kc, vc, bt, m["context_lens"], max_ctx, W.SCALE,
                                 ws, out=out_s)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                  # all rows are padding: stores nothing
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0

    for s in range(steps):
        _, q, k, v = W.fused_qkv(B, gen, dev, dtype=dt)
        ntok = [p + s + 1 for p in prompt]
        q_s.copy_(q)
        k_s.copy_(k)
        v_s.copy_(v)
        ntok_s.copy_(torch.tensor(ntok, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        assert pkv.pkv_device_error() == 0
        dseqs = [oracle.SeqState(n, t) for n, t in zip(ntok, tables)]
        dm = oracle.prepare_decode(dseqs, W.BLOCK_SIZE)
        assert np.array_equal(built["slot_mapping"].cpu().numpy(), dm["slot_mapping"])
        assert np.array_equal(built["context_lens"].cpu().numpy(), dm["context_lens"])
        orc.store_kvcache(bits(k), bits(v), kc_h, vc_h, dm["slot_mapping"])
        ref = orc.decode(bits(q), kc_h.reshape(nb, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM),
                         vc_h.reshape(nb, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM), bt_h, dm["context_lens"], W.SCALE,
                         num_kv_heads=W.HKV, dtype="f16")
        assert_close(out_s, ref, f"decode step {s}")
    # the caches the graph wrote equal the oracle's, bit for bit
    assert np.array_equal(bits(kc).reshape(-1, W.HKV, W.HEAD_DIM), kc_h)
    assert np.array_equal(bits(vc).reshape(-1, W.HKV, W.HEAD_DIM), vc_h)
