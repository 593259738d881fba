"""Store: argument errors the oracle rejects (what the pages never produce)."""
import numpy as np
import pytest

import oracle
from oracle_pins import randn_bits


def _bufs(n=4, slots=8):
    rng = np.random.default_rng(0)
    k = randn_bits(rng, (n, 2, 128))
    v = randn_bits(rng, (n, 2, 128))
    kc = np.zeros((slots, 2, 128), dtype=np.uint16)
    vc = np.zeros_like(kc)
    return k, v, kc, vc


def test_rejects_out_of_range_slot(orc):
    k, v, kc, vc = _bufs()
    with pytest.raises(oracle.OracleError):
        orc.store_kvcache(k, v, kc, vc, np.array([0, 1, 8, 2], dtype=np.int32))
    with pytest.raises(oracle.OracleError):
        orc.store_kvcache(k, v, kc, vc, np.array([0, -2, 3, 2], dtype=np.int32))


def test_rejects_duplicate_slot(orc):
    k, v, kc, vc = _bufs()
    with pytest.raises(oracle.OracleError):
        orc.store_kvcache(k, v, kc, vc, np.array([0, 5, 5, -1], dtype=np.int32))


def test_all_skipped_is_noop(orc):
    k, v, kc, vc = _bufs()
    orc.store_kvcache(k, v, kc, vc, np.full(4, -1, dtype=np.int32))
    assert not kc.any() and not vc.any()


def test_decode_rejects_bad_block(orc):
    rng = np.random.default_rng(1)
    kc = randn_bits(rng, (2, 256, 1, 128))
    q = randn_bits(rng, (1, 1, 128))
    with pytest.raises(oracle.OracleError):
        orc.decode(q, kc, kc, np.array([[2]], dtype=np.int32), np.array([3], dtype=np.int32), 0.1,
                   num_kv_heads=1)
    with pytest.raises(oracle.OracleError):
        orc.decode(q, kc, kc, np.array([[-1]], dtype=np.int32), np.array([3], dtype=np.int32), 0.1,
                   num_kv_heads=1)
