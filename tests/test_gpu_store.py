"""store_kvcache is a copy: bit-exact against the oracle's store."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvh_gb300 as m
    m.pkv_device_error(clear=True)
    return m


@pytest.mark.parametrize("n_tokens,num_blocks,fused,hkv,dtype", [
    (1, 1, True, 8, torch.bfloat16), (4, 16, True, 8, torch.bfloat16), (256, 64, True, 8, torch.bfloat16),
    (16384, 160, True, 8, torch.bfloat16), (1000, 8, False, 8, torch.bfloat16), (333, 4, False, 2, torch.bfloat16),
    (77, 2, False, 3, torch.bfloat16), (512, 32, True, 8, torch.float16), (77, 2, False, 3, torch.float16)])
def test_store_bit_exact(pkv, n_tokens, num_blocks, fused, hkv, dtype):
    dev = "cuda"
    gen = W.make_generator(n_tokens, dev)
    rng = np.random.default_rng(n_tokens)
    kc = W.normal((num_blocks * W.BLOCK_SIZE, hkv, W.HEAD_DIM), gen, dev, dtype)
    vc = W.normal((num_blocks * W.BLOCK_SIZE, hkv, W.HEAD_DIM), gen, dev, dtype)
    if fused:
        _, _, k, v = W.fused_qkv(n_tokens, gen, dev, hkv=hkv, dtype=dtype)
    else:
        k = W.normal((n_tokens, hkv, W.HEAD_DIM), gen, dev, dtype)
        v = W.normal((n_tokens, hkv, W.HEAD_DIM), gen, dev, dtype)
    slots = rng.permutation(num_blocks * W.BLOCK_SIZE)[:n_tokens].astype(np.int32)
    slots[rng.random(n_tokens) < 0.1] = -1                      # padding tokens
    kc_h, vc_h, kb, vb = bits(kc), bits(vc), bits(k), bits(v)
    pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(slots, dev))
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    oracle.default().store_kvcache(kb, vb, kc_h, vc_h, slots)
    assert np.array_equal(bits(kc), kc_h) and np.array_equal(bits(vc), vc_h)


def test_store_unaligned_stride_path(pkv):
    """Row strides that are not a multiple of 8 elements take the 2-byte path."""
    dev = "cuda"
    gen = W.make_generator(3, dev)
    base = W.normal_bf16((50, 8 * 128 + 3), gen, dev)
    k = base[:, 3:].unflatten(1, (8, 128))
    v = base[:, :-3].unflatten(1, (8, 128))
    kc = torch.zeros(256, 8, 128, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    slots = np.arange(50, dtype=np.int32)[::-1].copy()
    kc_h, vc_h = bits(kc), bits(vc)
    pkv.pkv_store_kvcache(k, v, kc, vc, to_dev(slots, dev))
    torch.cuda.synchronize()
    oracle.default().store_kvcache(bits(base)[:, 3:].reshape(50, 8, 128), bits(base)[:, :-3].reshape(50, 8, 128),
                                   kc_h, vc_h, slots)
    assert np.array_equal(bits(kc), kc_h) and np.array_equal(bits(vc), vc_h)
