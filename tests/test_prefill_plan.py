"""pkv_prefill_plan (host logic): the tile plan lists exactly the (query tile,
sequence) pairs that hold rows, ordered by the number of 128-key tiles each
attends to, most first, ties by lower sequence then higher query tile."""
import numpy as np
import pytest

import paged_kv_cache_kvh_gb300 as pkv


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _expected(lq, lk):
    items = []
    for b, (q, k) in enumerate(zip(lq, lk)):
        for qt in range((q + 127) // 128):
            last = k - q + min(q - 1, qt * 128 + 127)
            items.append((-(last // 128 + 1), b, -qt))
    return [(-nq << 16) | b for _, b, nq in sorted(items)]


@pytest.mark.parametrize("seed", range(6))
def test_plan_items_and_order(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    lq = rng.integers(0, 1500, size=n)
    lk = lq + np.where(rng.random(n) < 0.5, 0, rng.integers(0, 3000, size=n))
    got = pkv.pkv_prefill_plan(_cu(lq), _cu(lk), device=None)
    assert got.dtype == np.int32
    assert got.tolist() == _expected(lq.tolist(), lk.tolist())
    assert len(got) == sum((q + 127) // 128 for q in lq.tolist())


def test_plan_worked_example():
    # two prompts: 300 new tokens (3 query tiles, no cache) and 64 new tokens after 1024 cached
    got = pkv.pkv_prefill_plan([0, 300, 364], [0, 300, 1388], device=None).tolist()
    # key tiles: seq 1's tile attends to 1088 keys -> 9 tiles; seq 0's tiles to 128, 256, 300 keys -> 1, 2, 3
    assert got == [(0 << 16) | 1, (2 << 16) | 0, (1 << 16) | 0, (0 << 16) | 0]


def test_plan_errors():
    with pytest.raises(pkv.PkvError):
        pkv.pkv_prefill_plan([0, 10], [0, 5], device=None)        # fewer keys than queries
    with pytest.raises(pkv.PkvError):
        pkv.pkv_prefill_plan([0, 10, 5], [0, 10, 20], device=None)  # cu_seqlens_q not monotone
    assert pkv.pkv_prefill_plan([0], [0], device=None).size == 0
