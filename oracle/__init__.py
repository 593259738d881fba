"""CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package. The product path (the
``paged_kv_cache_kvh_gb300`` package and its CUDA library) never imports,
links or executes it, and this package imports nothing from the product.

Contents
--------
* ``pkv_oracle.c`` (built by :func:`build` with gcc into ``_build/``): the
  store copy, the block-table gather and fp64 softmax attention, one pass with
  no tiling. Its header states what each function follows.
* Index preparation, written here in plain Python loops, following
  "vLLM 学习笔记 02：nano-vllm 源码逐段精读", engine/sequence.py listing
  (``num_blocks``, ``last_block_num_tokens``) and engine/model_runner.py
  listing (``prepare_prefill``, ``prepare_decode``, ``prepare_block_tables``);
  the same steps are walked through with a worked example in
  "Nano-vLLM代码手撕笔记", section "请求执行 – 输入序列预处理与context构建".

Every function here is pinned by ``tests/test_oracle_*.py`` to values the pages
print, closed forms, invariants or a library routine; none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")

ORACLE_ERRORS = {
    0: "ok",
    -1: "slot outside the pool",
    -2: "two tokens write the same slot",
    -3: "block table entry outside the pool",
    -4: "bad shape",
    -5: "out of memory",
}


# Element types of q, k, v and the caches (the store copies bits and has none).
ELEM_CODES = {"bf16": 0, "f16": 1}


class OracleError(RuntimeError):
    pass


def _elem(dtype: str) -> int:
    try:
        return ELEM_CODES[dtype]
    except KeyError:
        raise OracleError(f"unknown element type {dtype!r}") from None


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP over independent output rows)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, src, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: str):
        self.lib = ctypes.CDLL(lib_path)
        L = self.lib
        i64, vp, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_store_kvcache.restype = ctypes.c_int
        L.oracle_store_kvcache.argtypes = [vp, i64, vp, i64, vp, vp, vp, i64, i64, i64]
        L.oracle_prefill_varlen.restype = ctypes.c_int
        ci = ctypes.c_int
        L.oracle_prefill_varlen.argtypes = [vp, i64, vp, vp, i64, vp, vp, i64, vp, vp, vp, i64,
                                            i64, i64, i64, i64, i64, dbl, vp, i64, ci, vp]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_decode.argtypes = [vp, vp, vp, i64, vp, i64, vp, i64, i64, i64, i64, i64, dbl,
                                    vp, i64, ci, vp]
        L.oracle_elements_to_double.restype = ctypes.c_int
        L.oracle_elements_to_double.argtypes = [vp, i64, ci, vp]

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    @staticmethod
    def _check(status: int):
        if status != 0:
            raise OracleError(ORACLE_ERRORS.get(status, f"status {status}"))

    def elements_to_f64(self, bits, dtype: str = "bf16") -> np.ndarray:
        """Widen 16-bit patterns of element type ``dtype`` to float64, exactly."""
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(b.shape, dtype=np.float64)
        self._check(self.lib.oracle_elements_to_double(_ptr(b), b.size, _elem(dtype), _ptr(out)))
        return out

    def store_kvcache(self, k, v, k_cache, v_cache, slot_mapping):
        """In place on ``k_cache``/``v_cache`` (uint16 bit patterns of any 16-bit
        element type, [slots, Hkv, d]).

        ``k``/``v`` are [N, Hkv, d] uint16 arrays whose last two axes are
        contiguous; their first-axis stride may exceed Hkv*d (views into a
        fused qkv buffer)."""
        N, Hkv, d = k.shape
        D = Hkv * d
        for a in (k, v):
            assert a.dtype == np.uint16 and a.strides[2] == 2 and a.strides[1] == 2 * d
        for c in (k_cache, v_cache):
            assert c.dtype == np.uint16 and c.flags.c_contiguous
        slot = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        assert slot.shape == (N,)
        num_slots = k_cache.size // D
        self._check(self.lib.oracle_store_kvcache(
            _ptr(k), k.strides[0] // 2, _ptr(v), v.strides[0] // 2, _ptr(k_cache), _ptr(v_cache),
            _ptr(slot), N, D, num_slots))

    def prefill_varlen(self, q, cu_seqlens_q, cu_seqlens_k, scale, *, k_cache=None, v_cache=None,
                       block_tables=None, k=None, v=None, num_kv_heads, block_size=256, rows=None,
                       dtype="bf16"):
        """Causal varlen prefill. Paged when ``block_tables`` is given, else
        contiguous ``k``/``v``. Returns float64 [total_q, Hq, d], or [n, d]
        for ``rows`` = int64 array of (token, head) pairs. ``dtype`` ("bf16"
        or "f16") is the element type of the uint16 bit patterns passed in."""
        total_q, Hq, d = q.shape
        assert q.dtype == np.uint16 and q.strides[2] == 2 and q.strides[1] == 2 * d
        cu_q = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        cu_k = np.ascontiguousarray(cu_seqlens_k, dtype=np.int32)
        num_seqs = cu_q.size - 1
        if block_tables is not None:
            bt = np.ascontiguousarray(block_tables, dtype=np.int32)
            assert bt.ndim == 2 and bt.shape[0] == num_seqs
            kc = np.ascontiguousarray(k_cache)
            vc = np.ascontiguousarray(v_cache)
            num_blocks = kc.size // (block_size * num_kv_heads * d)
            kk = vv = None
            kv_stride = 0
            bt_stride = bt.shape[1]
        else:
            bt = kc = vc = None
            num_blocks = 0
            bt_stride = 0
            kk, vv = k, v
            assert kk.strides == vv.strides and kk.strides[2] == 2
            kv_stride = kk.strides[0] // 2
        if rows is None:
            out = np.zeros((total_q, Hq, d), dtype=np.float64)
            rows_arr, n_rows = None, 0
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
            n_rows = rows_arr.shape[0]
            out = np.zeros((n_rows, d), dtype=np.float64)
        self._check(self.lib.oracle_prefill_varlen(
            _ptr(q), q.strides[0] // 2, _ptr(kk), _ptr(vv), kv_stride, _ptr(kc), _ptr(vc), num_blocks,
            _ptr(cu_q), _ptr(cu_k), _ptr(bt), bt_stride, num_seqs, Hq, num_kv_heads, d, block_size,
            float(scale), _ptr(rows_arr), n_rows, _elem(dtype), _ptr(out)))
        return out

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale, *, num_kv_heads,
               block_size=256, seqs=None, dtype="bf16"):
        """Single-query paged decode. Returns float64 [B or len(seqs), Hq, d].
        ``dtype`` as for :meth:`prefill_varlen`."""
        q = np.ascontiguousarray(q)
        B, Hq, d = q.shape
        kc = np.ascontiguousarray(k_cache)
        vc = np.ascontiguousarray(v_cache)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_blocks = kc.size // (block_size * num_kv_heads * d)
        if seqs is None:
            seq_arr, n = None, 0
            out = np.zeros((B, Hq, d), dtype=np.float64)
        else:
            seq_arr = np.ascontiguousarray(seqs, dtype=np.int64)
            n = seq_arr.size
            out = np.zeros((n, Hq, d), dtype=np.float64)
        self._check(self.lib.oracle_decode(
            _ptr(q), _ptr(kc), _ptr(vc), num_blocks, _ptr(bt), bt.shape[1], _ptr(ctx), B, Hq,
            num_kv_heads, d, block_size, float(scale), _ptr(seq_arr), n, _elem(dtype), _ptr(out)))
        return out


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``pkv_oracle.c`` in this directory."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(build())
    return _DEFAULT


# ---------------------------------------------------------------------------
# Index preparation (host side of the method).
# ---------------------------------------------------------------------------

def num_blocks(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence of ``num_tokens`` occupies (engine/sequence.py listing)."""
    return (num_tokens + block_size - 1) // block_size


def last_block_num_tokens(num_tokens: int, block_size: int) -> int:
    """Tokens held by the sequence's last block (engine/sequence.py listing)."""
    return num_tokens - (num_blocks(num_tokens, block_size) - 1) * block_size


@dataclass
class SeqState:
    """What the scheduler hands the model runner for one sequence.

    ``num_tokens`` is len(seq); ``num_cached_tokens`` are prefix-cache hits;
    ``num_scheduled_tokens`` the tokens computed this step (prefill);
    ``block_table`` the physical block of each logical block."""
    num_tokens: int
    block_table: list = field(default_factory=list)
    num_cached_tokens: int = 0
    num_scheduled_tokens: int = 0


def pad_block_tables(seqs, width: int | None = None) -> np.ndarray:
    """Rows padded with -1 to the longest table (prepare_block_tables)."""
    w = max(len(s.block_table) for s in seqs) if width is None else width
    out = np.full((len(seqs), w), -1, dtype=np.int32)
    for r, s in enumerate(seqs):
        for c, blk in enumerate(s.block_table):
            out[r, c] = blk
    return out


def prepare_prefill(seqs, block_size: int):
    """Packed-prefill metadata (engine/model_runner.py, prepare_prefill).

    For each sequence, the query covers positions [num_cached_tokens,
    num_cached_tokens + num_scheduled_tokens) and the keys cover [0, end).
    The slot of every query position is written block by block: the first
    block touched starts at offset start % block_size, the last one stops at
    end. Block tables are returned only when some sequence has cached keys
    (cu_seqlens_k[-1] > cu_seqlens_q[-1])."""
    positions, slot_mapping = [], []
    cu_q, cu_k = [0], [0]
    max_q = max_k = 0
    for s in seqs:
        start = s.num_cached_tokens
        end = start + s.num_scheduled_tokens
        positions.extend(range(start, end))
        cu_q.append(cu_q[-1] + (end - start))
        cu_k.append(cu_k[-1] + end)
        max_q = max(max_q, end - start)
        max_k = max(max_k, end)
        if not s.block_table:
            continue
        first_block = start // block_size
        stop_block = (end + block_size - 1) // block_size
        for i in range(first_block, stop_block):
            lo = start % block_size if i == first_block else 0
            hi = end - i * block_size if i == stop_block - 1 else block_size
            base = s.block_table[i] * block_size
            slot_mapping.extend(range(base + lo, base + hi))
    block_tables = pad_block_tables(seqs) if cu_k[-1] > cu_q[-1] else None
    return dict(positions=np.array(positions, dtype=np.int64),
                cu_seqlens_q=np.array(cu_q, dtype=np.int32),
                cu_seqlens_k=np.array(cu_k, dtype=np.int32),
                max_seqlen_q=max_q, max_seqlen_k=max_k,
                slot_mapping=np.array(slot_mapping, dtype=np.int32),
                block_tables=block_tables)


def prepare_decode(seqs, block_size: int):
    """Decode metadata (engine/model_runner.py, prepare_decode): the new
    token is the sequence's last one, stored at its last block's last used
    offset; context_lens counts it."""
    positions, slot_mapping, context_lens = [], [], []
    for s in seqs:
        positions.append(s.num_tokens - 1)
        context_lens.append(s.num_tokens)
        slot_mapping.append(s.block_table[-1] * block_size
                            + last_block_num_tokens(s.num_tokens, block_size) - 1)
    return dict(positions=np.array(positions, dtype=np.int64),
                slot_mapping=np.array(slot_mapping, dtype=np.int32),
                context_lens=np.array(context_lens, dtype=np.int32),
                block_tables=pad_block_tables(seqs))
