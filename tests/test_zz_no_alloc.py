"""pkv_decode_noalloc: decode attention for callers that cannot allocate.

Callers such as an engine whose KV-cache pool already took all free device
memory, a plug-in whose host owns the only allocator, or a loop that must not
risk cudaMalloc's synchronisation cannot pass pkv_decode a workspace. This
entry point keeps its scratch in a fixed array inside the library instead.
The test calls it through the C ABI twice in a row and checks each result
against pkv_decode's on the same inputs, within the attention tolerance used
everywhere else. It lives in a file of its own, collected last, and needs no
state from other tests: it passes alone in a fresh process or after them.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import TOL_MAX, TOL_MEAN, pool_tensors, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


def _case(pkv, seed, ctxs, dev):
    rng = np.random.default_rng(seed)
    nb = sum(W.blocks_for(c) for c in ctxs) + 4
    seqs = W._decode_seqs(ctxs, nb, rng)
    gen = W.make_generator(seed, dev)
    kc, vc = pool_tensors(nb, gen, dev)
    _, q, k, v = W.fused_qkv(len(seqs), gen, dev)
    meta = pkv.metadata.prepare_decode(seqs, W.BLOCK_SIZE, table_width=W.MAX_MODEL_LEN // W.BLOCK_SIZE)
    pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(meta["slot_mapping"], dev))
    return q, kc, vc, to_dev(meta["block_tables"], dev), to_dev(meta["context_lens"], dev)


def _close(a, b):
    err = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all() and torch.isfinite(b.float()).all()
    assert float(err.max()) <= TOL_MAX and float(err.mean()) <= TOL_MEAN, (float(err.max()), float(err.mean()))


def test_noalloc_matches_decode_twice_in_a_row(pkv):
    dev = "cuda"
    ctxs = [1, 2, 255, 256, 257, 511, 700, 1024, 2049, 3333, 4096, 4096] * 4
    q, kc, vc, bt, ctx = _case(pkv, 31, ctxs, dev)
    B = q.shape[0]
    ws = pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev)
    ref = pkv.pkv_decode(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
    outs = []
    for _ in range(2):                         # two calls in a row share the one scratch array
        out = torch.full_like(ref, float("nan"))
        pkv.pkv_decode_noalloc(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, out)
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        _close(out, ref)
    assert pkv.pkv_device_error() == 0

    # a different, smaller batch afterwards: leftovers of the previous calls do not matter
    q2, kc2, vc2, bt2, ctx2 = _case(pkv, 32, [4096, 300, 1], dev)
    ws2 = pkv.decode_workspace(3, W.MAX_MODEL_LEN, dev)
    ref2 = pkv.pkv_decode(q2, kc2, vc2, bt2, ctx2, W.MAX_MODEL_LEN, W.SCALE, ws2)
    out2 = torch.empty_like(ref2)
    pkv.pkv_decode_noalloc(q2, kc2, vc2, bt2, ctx2, W.MAX_MODEL_LEN, W.SCALE, out2)
    torch.cuda.synchronize()
    _close(out2, ref2)


def test_noalloc_rejects_sizes_beyond_its_scratch(pkv):
    dev = "cuda"
    B = 1024                                   # 1024 sequences x 4096 context needs ~136 MB of scratch
    need = pkv.pkv_decode_workspace_bytes(B, W.MAX_MODEL_LEN)
    assert need > pkv.PKV_DECODE_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(1, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(B, 16, dtype=torch.int32, device=dev)
    ctx = torch.ones(B, dtype=torch.int32, device=dev)
    out = torch.zeros_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_noalloc(q, kc, kc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, out)
    assert e.value.status == pkv.PKV_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(out == 0)                 # nothing was launched


def test_noalloc_zero_sizes_and_rejections_match_decode(pkv):
    """Empty and all-padding calls, and argument errors: the same outcome as
    pkv_decode, and a refused call leaves the output untouched."""
    dev = "cuda"
    lib = pkv._lib
    # no sequences: nothing to do
    assert lib.pkv_decode_noalloc(None, 2048, None, None, 0, None, 16, None, 0, 16, 8, 128, 256, 4096, 0.1,
                                  None, None) == 0
    # every row a padding row and max_context_len 0: zeros, no device error
    q, kc, vc, bt, _ = _case(pkv, 33, [5, 9], dev)
    ctx0 = torch.zeros(2, dtype=torch.int32, device=dev)
    out = torch.full_like(q, float("nan"))
    pkv.pkv_decode_noalloc(q, kc, vc, bt, ctx0, 0, W.SCALE, out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
    assert pkv.pkv_device_error() == 0
    # argument errors: pkv_decode's status, and nothing written
    ws = pkv.decode_workspace(2, W.MAX_MODEL_LEN, dev)
    out = torch.full_like(q, 7.0)
    common = [q.data_ptr(), q.stride(0), kc.data_ptr(), vc.data_ptr(), kc.shape[0], bt.data_ptr(), bt.shape[1],
              ctx0.data_ptr(), 2]
    for heads, scale, out_ptr in ((32, W.SCALE, out.data_ptr()), (16, -1.0, out.data_ptr()),
                                  (16, W.SCALE, out.data_ptr() + 2), (16, W.SCALE, None)):
        tail = [heads, 8, 128, 256, W.MAX_MODEL_LEN, scale, out_ptr]
        want = lib.pkv_decode(*common, *tail, ws.data_ptr(), ws.numel(), None)
        got = lib.pkv_decode_noalloc(*common, *tail, None)
        assert want < 0 and got == want, (heads, scale, want, got)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
