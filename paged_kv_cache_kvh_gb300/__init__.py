"""paged_kv_cache_kvh_gb300 -- Python binding of libpkv.so (attention over a paged KV cache, GB300).

Argument marshalling only: every function here checks shapes, turns torch
tensors into pointers, sizes and the current CUDA stream, and calls the C
entry point of the same name (declared in ``include/pkv.h``). All work runs in
the library's CUDA kernels; there is no CPU fallback. Importing this package
fails loudly when ``libpkv.so`` has not been built
(``python paged_kv_cache_kvh_gb300/build_lib.py``).

Layouts (Qwen3-0.6B attention shape):
  q            [tokens, 16, 128] (row stride may exceed 2048, e.g. fused qkv)
  k, v         [tokens, 8, 128]
  k/v caches   [num_blocks, 256, 8, 128] contiguous
  slot_mapping, cu_seqlens_*, block_tables, context_lens  int32 on the GPU
Element type: bf16 for the plain names, fp16 for the ``*_f16`` names (one type
per call for q, k, v, caches and output); the store copies either.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import metadata  # noqa: F401  (host index preparation)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_DEVERR_BAD_SLOT = 0x1
PKV_DEVERR_BAD_BLOCK = 0x2
PKV_DEVERR_BAD_SEQLEN = 0x4
PKV_DEVERR_TIMEOUT = 0x8
PKV_ERR_SCRATCH_LIMIT = -9
PKV_DECODE_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
HEAD_DIM, BLOCK_SIZE, NUM_HEADS, NUM_KV_HEADS = 128, 256, 16, 8

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libpkv.so is not built ({LIB_PATH}); run python paged_kv_cache_kvh_gb300/build_lib.py")

_lib = ctypes.CDLL(LIB_PATH)
_i32, _i64, _u64, _vp, _f32, _sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p,
                                     ctypes.c_float, ctypes.c_size_t)
_SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_version": (ctypes.c_int, []),
    "pkv_store_kvcache": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _vp]),
    "pkv_prefill_varlen": (ctypes.c_int, [_vp, _i64, _i32, _vp, _vp, _i64, _i32, _vp, _vp, _i32, _vp, _vp, _i32,
                                          _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz,
                                          _vp]),
    "pkv_prefill_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "pkv_prefill_plan": (_i32, [_vp, _vp, _i32, _vp, _i32]),
    "pkv_decode": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                  _f32, _vp, _vp, _sz, _vp]),
    "pkv_decode_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "pkv_prefill_varlen_f16": (ctypes.c_int, [_vp, _i64, _i32, _vp, _vp, _i64, _i32, _vp, _vp, _i32, _vp, _vp, _i32,
                                              _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz,
                                              _vp]),
    "pkv_decode_f16": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                      _f32, _vp, _vp, _sz, _vp]),
    "pkv_store_decode_f16": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _vp,
                                            _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "pkv_store_decode": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _i32,
                                        _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "pkv_decode_noalloc": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                          _i32, _f32, _vp, _vp]),
    "pkv_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, _vp]),
    "pkv_build_prefill_metadata": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                                  _vp]),
    "pkv_build_decode_metadata": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "pkv_selftest_wait_timeout": (ctypes.c_int, [_u64, _vp]),
}
for _name, (_res, _args) in _SIGNATURES.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGNATURES)


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {pkv_status_string(status)} (status {status})")
        self.status = status


def pkv_status_string(status: int) -> str:
    return _lib.pkv_status_string(int(status)).decode()


def pkv_version() -> int:
    return int(_lib.pkv_version())


def _check(status: int, where: str):
    if status != PKV_OK:
        raise PkvError(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _dev_i32(t, name):
    _need(t.dtype == torch.int32 and t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous int32 CUDA tensor")


_TYPE_NAME = {torch.bfloat16: "bf16", torch.float16: "fp16"}


def _rows(t, name, heads, dtype=torch.bfloat16):
    _need(t.dtype == dtype and t.is_cuda, f"{name} must be a {_TYPE_NAME[dtype]} CUDA tensor")
    _need(t.dim() == 3 and t.shape[1] == heads and t.shape[2] == HEAD_DIM, f"{name} must be [N, {heads}, 128]")
    _need(t.stride(2) == 1 and t.stride(1) == HEAD_DIM, f"{name}: heads and dims must be contiguous within a row")


def _cache(t, name, dtype):
    _need(t is not None and t.dtype == dtype and t.is_cuda and t.is_contiguous()
          and tuple(t.shape[1:]) == (BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM),
          f"{name}: contiguous {_TYPE_NAME[dtype]} [blocks, 256, 8, 128]")


def pkv_store_kvcache(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """store_kvcache: k_cache[slot] = k[i], v_cache[slot] = v[i] for slot != -1.
    A bit-exact copy of 16-bit elements: bf16 or fp16, the same type throughout."""
    _need(k.dim() == 3 and v.shape == k.shape, "k, v must be [N, num_kv_heads, head_dim]")
    N, hkv, d = k.shape
    _need(k.dtype in _TYPE_NAME, "k, v, caches must be bf16 or fp16")
    for t, n in ((k, "k"), (v, "v")):
        _need(t.dtype == k.dtype and t.is_cuda and t.stride(2) == 1 and t.stride(1) == d,
              f"{n}: CUDA, same type as k, heads and dims contiguous")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t.dtype == k.dtype and t.is_contiguous() and t.shape[-2:] == (hkv, d),
              f"{n}: contiguous, same type as k, [..., {hkv}, {d}]")
    _dev_i32(slot_mapping, "slot_mapping")
    _need(slot_mapping.numel() == N, "slot_mapping must have one entry per token")
    num_slots = k_cache.numel() // (hkv * d)
    _check(_lib.pkv_store_kvcache(_ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(slot_mapping), N, hkv, d, num_slots, _stream(stream)), "pkv_store_kvcache")


def pkv_prefill_workspace_bytes(num_seqs: int, max_seqlen_q: int, num_heads: int = NUM_HEADS) -> int:
    return int(_lib.pkv_prefill_workspace_bytes(num_seqs, max_seqlen_q, num_heads))


def _prefill(entry, dtype, q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, softmax_scale, k, v,
             k_cache, v_cache, block_tables, out, workspace, stream):
    _rows(q, "q", NUM_HEADS, dtype)
    _dev_i32(cu_seqlens_q, "cu_seqlens_q")
    _dev_i32(cu_seqlens_k, "cu_seqlens_k")
    num_seqs = cu_seqlens_q.numel() - 1
    _need(cu_seqlens_k.numel() == num_seqs + 1, "cu_seqlens_k size")
    total_q = q.shape[0]
    if out is None:
        out = torch.empty((total_q, NUM_HEADS, HEAD_DIM), dtype=dtype, device=q.device)
    _need(out.is_contiguous() and out.shape == (total_q, NUM_HEADS, HEAD_DIM) and out.dtype == dtype,
          f"out must be contiguous {_TYPE_NAME[dtype]} [total_q, 16, 128]")
    if block_tables is not None:
        _dev_i32(block_tables, "block_tables")
        _cache(k_cache, "k_cache", dtype)
        _cache(v_cache, "v_cache", dtype)
        num_blocks, bt_stride = k_cache.shape[0], block_tables.shape[1]
        kk = vv = None
        kv_stride, total_k = 0, 0
    else:
        _rows(k, "k", NUM_KV_HEADS, dtype)
        _rows(v, "v", NUM_KV_HEADS, dtype)
        _need(k.stride(0) == v.stride(0) and k.shape == v.shape, "k and v must share shape and row stride")
        kk, vv = k, v
        kv_stride, total_k = k.stride(0), k.shape[0]
        num_blocks, bt_stride = 0, 0
    fn = getattr(_lib, entry)
    _check(fn(
        _ptr(q), q.stride(0), total_q, _ptr(kk), _ptr(vv), kv_stride, total_k,
        _ptr(k_cache) if block_tables is not None else None, _ptr(v_cache) if block_tables is not None else None,
        num_blocks, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_seqlen_q), int(max_seqlen_k),
        _ptr(block_tables), bt_stride, num_seqs, NUM_HEADS, NUM_KV_HEADS, HEAD_DIM, BLOCK_SIZE,
        float(softmax_scale), _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream)), entry)
    return out


def pkv_prefill_plan(cu_seqlens_q, cu_seqlens_k, device="cuda"):
    """Tile plan for pkv_prefill_varlen(_f16) from host cu_seqlens (numpy,
    lists or CPU tensors): the (query tile, sequence) items that hold rows,
    longest key range first, as an int32 tensor on `device` (numpy if None).
    Built once per step and passed as plan= to every layer's prefill."""
    cq = np.ascontiguousarray(np.asarray(cu_seqlens_q.cpu() if torch.is_tensor(cu_seqlens_q) else cu_seqlens_q,
                                         dtype=np.int32))
    ck = np.ascontiguousarray(np.asarray(cu_seqlens_k.cpu() if torch.is_tensor(cu_seqlens_k) else cu_seqlens_k,
                                         dtype=np.int32))
    num_seqs = cq.size - 1
    _need(num_seqs >= 0 and ck.size == num_seqs + 1, "cu_seqlens sizes")
    cap = int(cq[-1] - cq[0]) // 128 + num_seqs + 1 if num_seqs > 0 else 1
    items = np.empty(cap, dtype=np.int32)
    n = int(_lib.pkv_prefill_plan(cq.ctypes.data, ck.ctypes.data, num_seqs, items.ctypes.data, cap))
    if n < 0:
        raise PkvError(n, "pkv_prefill_plan")
    items = items[:n].copy()
    return items if device is None else torch.from_numpy(items).to(device)


def _plan_arg(plan, workspace):
    if plan is None:
        return workspace
    _need(workspace is None, "pass either plan or workspace")
    _need(torch.is_tensor(plan) and plan.is_cuda and plan.dtype == torch.int32 and plan.is_contiguous(),
          "plan must be a contiguous int32 CUDA tensor (pkv_prefill_plan)")
    return plan if plan.numel() > 0 else None


def pkv_prefill_varlen(q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, softmax_scale, *, k=None, v=None,
                       k_cache=None, v_cache=None, block_tables=None, out=None, workspace=None, plan=None,
                       stream=None):
    """flash_attn_varlen_func(q, k, v, ..., causal=True, block_table=block_tables).

    Paged keys (k_cache/v_cache through block_tables) when block_tables is
    given, else contiguous k/v. plan: optional tile plan (pkv_prefill_plan of
    the same cu_seqlens). Returns out [total_q, 16, 128] bf16."""
    workspace = _plan_arg(plan, workspace)
    return _prefill("pkv_prefill_varlen", torch.bfloat16, q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    softmax_scale, k, v, k_cache, v_cache, block_tables, out, workspace, stream)


def pkv_prefill_varlen_f16(q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, softmax_scale, *, k=None,
                           v=None, k_cache=None, v_cache=None, block_tables=None, out=None, workspace=None,
                           plan=None, stream=None):
    """pkv_prefill_varlen on fp16 tensors; returns fp16."""
    workspace = _plan_arg(plan, workspace)
    return _prefill("pkv_prefill_varlen_f16", torch.float16, q, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                    max_seqlen_k, softmax_scale, k, v, k_cache, v_cache, block_tables, out, workspace, stream)


def pkv_decode_workspace_bytes(num_seqs: int, max_context_len: int, num_heads: int = NUM_HEADS) -> int:
    return int(_lib.pkv_decode_workspace_bytes(num_seqs, num_heads, max_context_len))


def decode_workspace(num_seqs: int, max_context_len: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for pkv_decode (allocated by torch, outside the library)."""
    n = pkv_decode_workspace_bytes(num_seqs, max_context_len)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def _decode(entry, dtype, q, k_cache, v_cache, block_tables, context_lens, max_context_len, softmax_scale,
            workspace, out, stream):
    _rows(q, "q", NUM_HEADS, dtype)
    _cache(k_cache, "k_cache", dtype)
    _cache(v_cache, "v_cache", dtype)
    _dev_i32(block_tables, "block_tables")
    _dev_i32(context_lens, "context_lens")
    B = q.shape[0]
    _need(block_tables.dim() == 2 and block_tables.shape[0] >= B and context_lens.numel() >= B, "table sizes")
    if out is None:
        out = torch.empty((B, NUM_HEADS, HEAD_DIM), dtype=dtype, device=q.device)
    _need(out.is_contiguous() and out.shape == (B, NUM_HEADS, HEAD_DIM) and out.dtype == dtype,
          f"out must be contiguous {_TYPE_NAME[dtype]} [B, 16, 128]")
    _need(workspace.dtype == torch.uint8 and workspace.is_cuda, "workspace must be a uint8 CUDA tensor")
    _check(getattr(_lib, entry)(_ptr(q), q.stride(0), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, NUM_HEADS,
                                NUM_KV_HEADS, HEAD_DIM, BLOCK_SIZE, int(max_context_len), float(softmax_scale),
                                _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)), entry)
    return out


def pkv_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len, softmax_scale, workspace, *,
               out=None, stream=None):
    """flash_attn_with_kvcache(q.unsqueeze(1), k_cache, v_cache, cache_seqlens=context_lens,
    block_table=block_tables, causal=True). Returns out [num_seqs, 16, 128] bf16."""
    return _decode("pkv_decode", torch.bfloat16, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                   softmax_scale, workspace, out, stream)


def pkv_decode_f16(q, k_cache, v_cache, block_tables, context_lens, max_context_len, softmax_scale, workspace, *,
                   out=None, stream=None):
    """pkv_decode on fp16 tensors; returns fp16."""
    return _decode("pkv_decode_f16", torch.float16, q, k_cache, v_cache, block_tables, context_lens,
                   max_context_len, softmax_scale, workspace, out, stream)


def pkv_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, max_context_len, softmax_scale, out, *,
                       stream=None):
    """pkv_decode without a workspace, for callers that cannot allocate device
    memory (a KV pool that already took all free memory, a host that owns the
    only allocator, a loop that must not synchronise on cudaMalloc). Scratch
    comes from a fixed array inside the library, so the caller passes the
    output buffer too and nothing is allocated. Sizes beyond that array
    (PKV_DECODE_NOALLOC_SCRATCH_BYTES) raise PkvError(PKV_ERR_SCRATCH_LIMIT).
    Calls must not overlap on the GPU: they share the array."""
    _rows(q, "q", NUM_HEADS)
    _cache(k_cache, "k_cache", torch.bfloat16)
    _cache(v_cache, "v_cache", torch.bfloat16)
    _dev_i32(block_tables, "block_tables")
    _dev_i32(context_lens, "context_lens")
    B = q.shape[0]
    _need(block_tables.dim() == 2 and block_tables.shape[0] >= B and context_lens.numel() >= B, "table sizes")
    _need(out is not None and out.is_contiguous() and out.shape == (B, NUM_HEADS, HEAD_DIM)
          and out.dtype == torch.bfloat16, "out must be a caller-owned contiguous bf16 [B, 16, 128]")
    _check(_lib.pkv_decode_noalloc(_ptr(q), q.stride(0), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                   _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, NUM_HEADS,
                                   NUM_KV_HEADS, HEAD_DIM, BLOCK_SIZE, int(max_context_len), float(softmax_scale),
                                   _ptr(out), _stream(stream)), "pkv_decode_noalloc")
    return out


def _store_decode(entry, dtype, q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens,
                  max_context_len, softmax_scale, workspace, out, stream):
    _rows(q, "q", NUM_HEADS, dtype)
    _rows(k, "k", NUM_KV_HEADS, dtype)
    _rows(v, "v", NUM_KV_HEADS, dtype)
    _cache(k_cache, "k_cache", dtype)
    _cache(v_cache, "v_cache", dtype)
    _dev_i32(slot_mapping, "slot_mapping")
    _dev_i32(block_tables, "block_tables")
    _dev_i32(context_lens, "context_lens")
    B = q.shape[0]
    _need(k.shape[0] >= B and v.shape[0] >= B and slot_mapping.numel() >= B, "one new row per sequence")
    _need(block_tables.dim() == 2 and block_tables.shape[0] >= B and context_lens.numel() >= B, "table sizes")
    if out is None:
        out = torch.empty((B, NUM_HEADS, HEAD_DIM), dtype=dtype, device=q.device)
    _need(out.is_contiguous() and out.shape == (B, NUM_HEADS, HEAD_DIM) and out.dtype == dtype,
          f"out must be contiguous {_TYPE_NAME[dtype]} [B, 16, 128]")
    _need(workspace.dtype == torch.uint8 and workspace.is_cuda, "workspace must be a uint8 CUDA tensor")
    _check(getattr(_lib, entry)(_ptr(q), q.stride(0), _ptr(k), k.stride(0), _ptr(v), v.stride(0),
                                _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, NUM_HEADS,
                                NUM_KV_HEADS, HEAD_DIM, BLOCK_SIZE, int(max_context_len), float(softmax_scale),
                                _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)), entry)
    return out


def pkv_store_decode(q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens, max_context_len,
                     softmax_scale, workspace, *, out=None, stream=None):
    """store_kvcache of the step's new K/V rows fused into the decode launch.
    slot_mapping[b] must be -1 or the slot of position context_lens[b]-1."""
    return _store_decode("pkv_store_decode", torch.bfloat16, q, k, v, slot_mapping, k_cache, v_cache, block_tables,
                         context_lens, max_context_len, softmax_scale, workspace, out, stream)


def pkv_store_decode_f16(q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens, max_context_len,
                         softmax_scale, workspace, *, out=None, stream=None):
    """pkv_store_decode on fp16 tensors; returns fp16."""
    return _store_decode("pkv_store_decode_f16", torch.float16, q, k, v, slot_mapping, k_cache, v_cache,
                         block_tables, context_lens, max_context_len, softmax_scale, workspace, out, stream)


def pkv_build_prefill_metadata(num_cached_tokens, num_scheduled_tokens, block_tables, num_blocks, capacity,
                               stream=None):
    """prepare_prefill on the GPU. Inputs int32 CUDA tensors ([B], [B], [B, W]).
    Returns dict of device tensors: cu_seqlens_q, cu_seqlens_k, max_seqlens (2),
    slot_mapping [capacity], positions [capacity] (int64)."""
    for t, n in ((num_cached_tokens, "num_cached_tokens"), (num_scheduled_tokens, "num_scheduled_tokens"),
                 (block_tables, "block_tables")):
        _dev_i32(t, n)
    B = num_cached_tokens.numel()
    _need(num_scheduled_tokens.numel() == B and block_tables.dim() == 2 and block_tables.shape[0] == B, "sizes")
    dev = num_cached_tokens.device
    out = dict(cu_seqlens_q=torch.empty(B + 1, dtype=torch.int32, device=dev),
               cu_seqlens_k=torch.empty(B + 1, dtype=torch.int32, device=dev),
               max_seqlens=torch.empty(2, dtype=torch.int32, device=dev),
               slot_mapping=torch.empty(max(capacity, 1), dtype=torch.int32, device=dev),
               positions=torch.empty(max(capacity, 1), dtype=torch.int64, device=dev))
    _check(_lib.pkv_build_prefill_metadata(
        _ptr(num_cached_tokens), _ptr(num_scheduled_tokens), _ptr(block_tables), block_tables.shape[1], int(num_blocks),
        B, int(capacity), _ptr(out["cu_seqlens_q"]), _ptr(out["cu_seqlens_k"]), _ptr(out["max_seqlens"]),
        _ptr(out["slot_mapping"]), _ptr(out["positions"]), _stream(stream)), "pkv_build_prefill_metadata")
    return out


def pkv_build_decode_metadata(num_tokens, block_tables, num_blocks, stream=None):
    """prepare_decode on the GPU: slot_mapping, context_lens, positions (int64)."""
    _dev_i32(num_tokens, "num_tokens")
    _dev_i32(block_tables, "block_tables")
    B = num_tokens.numel()
    _need(block_tables.dim() == 2 and block_tables.shape[0] >= B, "block_tables [B, W]")
    dev = num_tokens.device
    out = dict(slot_mapping=torch.empty(B, dtype=torch.int32, device=dev),
               context_lens=torch.empty(B, dtype=torch.int32, device=dev),
               positions=torch.empty(B, dtype=torch.int64, device=dev))
    _check(_lib.pkv_build_decode_metadata(_ptr(num_tokens), _ptr(block_tables), block_tables.shape[1],
                                          int(num_blocks), B, _ptr(out["slot_mapping"]), _ptr(out["context_lens"]),
                                          _ptr(out["positions"]), _stream(stream)), "pkv_build_decode_metadata")
    return out


def pkv_device_error(clear: bool = True, stream=None) -> int:
    """Read (and by default clear) the device error word; synchronises the stream."""
    bits = ctypes.c_uint32(0)
    _check(_lib.pkv_device_error(ctypes.byref(bits), int(bool(clear)), _stream(stream)), "pkv_device_error")
    return int(bits.value)


def pkv_selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None):
    _check(_lib.pkv_selftest_wait_timeout(int(limit_ns), _stream(stream)), "pkv_selftest_wait_timeout")
