// pkv_abi.cu -- extern "C" entry points of libpkv.so (declared in include/pkv.h).
//
// Host-side argument checks mirror the asserts of store_kvcache in
// layers/attention.py ("vLLM 学习笔记 02：nano-vllm 源码逐段精读": unit
// element stride, heads contiguous, cache rows of num_kv_heads*head_dim,
// one slot per token) plus the limits of these kernels; a failed check
// returns an error code before anything is launched.
#include <cuda.h>  // driver types for the context-id query (resolved at run time, no libcuda link)

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <vector>

#include "pkv_common.cuh"

namespace pkv {
cudaError_t launch_store_kvcache(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                                 void* k_cache, void* v_cache, const int32_t* slot_mapping, int32_t num_tokens,
                                 int32_t D, int64_t num_slots, unsigned int* err, cudaStream_t stream);
struct FusedStore {
  const void* k;
  int64_t k_row_stride;
  const void* v;
  int64_t v_row_stride;
  const int32_t* slot_mapping;
};
cudaError_t launch_decode(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
                          int32_t num_blocks, const int32_t* block_tables, int32_t bt_stride,
                          const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len, float scale,
                          void* out, void* workspace, unsigned int* err, cudaStream_t stream,
                          const FusedStore* fused, Elem elem);
size_t decode_workspace_bytes(int32_t num_seqs, int32_t max_context_len);
cudaError_t launch_prefill(const void* q, int64_t q_row_stride, int32_t total_q, const void* k, const void* v,
                           int64_t kv_row_stride, int32_t total_k, const void* k_cache, const void* v_cache,
                           int32_t num_blocks, const int32_t* cu_q, const int32_t* cu_k, int32_t max_seqlen_q,
                           int32_t max_seqlen_k, const int32_t* block_tables, int32_t bt_stride, int32_t num_seqs,
                           float scale, const int32_t* items, int32_t num_items, void* out, unsigned int* err,
                           cudaStream_t stream, Elem elem);
size_t prefill_workspace_bytes(int32_t num_seqs, int32_t max_seqlen_q, int32_t num_heads);
cudaError_t launch_prefill_metadata(const int32_t* num_cached, const int32_t* num_scheduled,
                                    const int32_t* block_tables, int32_t bt_stride, int32_t num_blocks,
                                    int32_t num_seqs, int32_t capacity, int32_t* cu_q, int32_t* cu_k,
                                    int32_t* max_q_k, int32_t* slot_mapping, int64_t* positions, unsigned int* err,
                                    cudaStream_t stream);
cudaError_t launch_decode_metadata(const int32_t* num_tokens, const int32_t* block_tables, int32_t bt_stride,
                                   int32_t num_blocks, int32_t num_seqs, int32_t* slot_mapping, int32_t* context_lens,
                                   int64_t* positions, unsigned int* err, cudaStream_t stream);
}  // namespace pkv

namespace {

constexpr int kMaxDevices = 64;

// Per-device error word: OR of PKV_DEVERR_* bits raised by any kernel.
__device__ unsigned int g_pkv_error_word;

// Cached device addresses of the library's __device__ variables, keyed by the
// id of the context they were looked up in. Host threads share it under a lock.
constexpr int kNumSymbols = 2;
struct SymbolSlot {
  bool valid = false;
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
std::mutex g_symbol_lock;
SymbolSlot g_symbols[kMaxDevices][kNumSymbols];
std::once_flag g_cc_once[kMaxDevices];
int g_cc_ok[kMaxDevices] = {0};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (cuCtxGetId; ids are never
// reused), through driver entry points the runtime hands out. False when
// there is no current context yet or the driver lacks the query.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    (void)cudaGetLastError();
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned int* err) {
  __shared__ __align__(8) uint64_t never;
  const uint32_t bar = pkv::smem_u32(&never);
  if (threadIdx.x == 0) {
    pkv::mbar_init(bar, 1);  // one arrival expected, none will come
    pkv::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) pkv::mbar_wait(bar, 0, err, limit_ns);
}

int error_word(unsigned int** out) { return pkv::device_error_word(out); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int launched(cudaError_t e) {
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// The attention kernels are built for one head layout.
int check_attention_shape(int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size) {
  if (head_dim != pkv::kHeadDim || block_size != pkv::kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (num_kv_heads != 8 || num_heads != 16) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

}  // namespace

namespace pkv {

int symbol_address(const void* symbol, int slot, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kNumSymbols) {
    (void)cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  if (have_id) {
    std::lock_guard<std::mutex> lock(g_symbol_lock);
    const SymbolSlot& s = g_symbols[dev][slot];
    if (s.valid && s.ctx_id == id) {
      *out = s.addr;
      return PKV_OK;
    }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (!have_id) have_id = current_context_id(&id);  // the lookup made the context current
  if (have_id) {
    std::lock_guard<std::mutex> lock(g_symbol_lock);
    g_symbols[dev][slot] = SymbolSlot{true, id, p};
  }
  *out = p;
  return PKV_OK;
}

int device_error_word(unsigned int** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  std::call_once(g_cc_once[dev], [dev] {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    (void)cudaGetLastError();
    g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  });
  if (g_cc_ok[dev] != 1) return PKV_ERR_DEVICE;
  void* p = nullptr;
  const int st = symbol_address(&g_pkv_error_word, kSymbolErrorWord, &p);
  if (st != PKV_OK) return st;
  *out = static_cast<unsigned int*>(p);
  return PKV_OK;
}

int check_decode_args(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
                      int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                      const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale,
                      const void* out, const void* workspace, size_t workspace_bytes) {
  int st = check_attention_shape(num_heads, num_kv_heads, head_dim, block_size);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || num_blocks < 0 || block_table_stride < 0 || max_context_len < 0 ||
      max_context_len > (1 << 24))
    return PKV_ERR_BAD_SIZE;
  if (num_seqs == 0) return PKV_OK;
  if (!(softmax_scale > 0.f)) return PKV_ERR_BAD_SIZE;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_ERR_NULL_POINTER;
  if (q_row_stride < static_cast<int64_t>(num_heads) * head_dim) return PKV_ERR_BAD_STRIDE;
  if (!aligned16(q) || (q_row_stride % 8) != 0 || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PKV_ERR_ALIGNMENT;
  if (max_context_len > 0) {
    const size_t need = decode_workspace_bytes(num_seqs, max_context_len);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PKV_ERR_ALIGNMENT;
  }
  return PKV_OK;
}

}  // namespace pkv

extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL_POINTER: return "a required pointer is NULL";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape (head_dim 128, block_size 256, 16 q / 8 kv heads)";
    case PKV_ERR_BAD_STRIDE: return "row stride smaller than the row";
    case PKV_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_BAD_SIZE: return "negative count or size beyond the library's limits";
    case PKV_ERR_CUDA: return "CUDA call or kernel launch failed";
    case PKV_ERR_DEVICE: return "current device is not compute capability 10.3";
    case PKV_ERR_SCRATCH_LIMIT: return "sizes need more scratch than pkv_decode_noalloc's built-in array";
    default: return "unknown status";
  }
}

int pkv_version(void) { return 100; }

int pkv_store_kvcache(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride, void* k_cache,
                      void* v_cache, const int32_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                      int32_t head_dim, int64_t num_slots, cudaStream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_slots < 0) return PKV_ERR_BAD_SIZE;
  const int64_t D = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (D > (1 << 20)) return PKV_ERR_BAD_SIZE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_NULL_POINTER;
  if (k_row_stride < D || v_row_stride < D) return PKV_ERR_BAD_STRIDE;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 1u)
    return PKV_ERR_ALIGNMENT;
  unsigned int* err = nullptr;
  int st = error_word(&err);
  if (st != PKV_OK) return st;
  return launched(pkv::launch_store_kvcache(k, k_row_stride, v, v_row_stride, k_cache, v_cache, slot_mapping,
                                            num_tokens, static_cast<int32_t>(D), num_slots, err, stream));
}

size_t pkv_prefill_workspace_bytes(int32_t num_seqs, int32_t max_seqlen_q, int32_t num_heads) {
  return pkv::prefill_workspace_bytes(num_seqs, max_seqlen_q, num_heads);
}

int32_t pkv_prefill_plan(const int32_t* h_cu_seqlens_q, const int32_t* h_cu_seqlens_k, int32_t num_seqs,
                         int32_t* h_items, int32_t capacity) {
  if (!h_cu_seqlens_q || !h_cu_seqlens_k || (!h_items && capacity > 0)) return PKV_ERR_NULL_POINTER;
  if (num_seqs < 0 || num_seqs > 65535 || capacity < 0) return PKV_ERR_BAD_SIZE;
  struct Item {
    int32_t code;     // (qt << 16) | b
    int32_t n_tiles;  // 128-key tiles the query tile attends to
  };
  std::vector<Item> v;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int64_t lq = static_cast<int64_t>(h_cu_seqlens_q[b + 1]) - h_cu_seqlens_q[b];
    const int64_t lk = static_cast<int64_t>(h_cu_seqlens_k[b + 1]) - h_cu_seqlens_k[b];
    if (lq < 0 || lk < lq || lq >= (int64_t{1} << 22)) return PKV_ERR_BAD_SIZE;
    for (int64_t qt = (lq + 127) / 128 - 1; qt >= 0; --qt) {
      const int64_t last_pos = lk - lq + std::min<int64_t>(lq - 1, qt * 128 + 127);
      v.push_back({static_cast<int32_t>((qt << 16) | b), static_cast<int32_t>(last_pos / 128 + 1)});
    }
  }
  if (v.size() > static_cast<size_t>(capacity)) return PKV_ERR_BAD_SIZE;
  // most key tiles first; ties by lower sequence, then higher query tile (the build order)
  std::stable_sort(v.begin(), v.end(), [](const Item& x, const Item& y) { return x.n_tiles > y.n_tiles; });
  for (size_t i = 0; i < v.size(); ++i) h_items[i] = v[i].code;
  return static_cast<int32_t>(v.size());
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t max_context_len) {
  (void)num_heads;
  if (num_seqs <= 0 || max_context_len <= 0) return 0;
  return pkv::decode_workspace_bytes(num_seqs, max_context_len);
}

}  // extern "C"

namespace {
int prefill_common(const void* q, int64_t q_row_stride, int32_t total_q, const void* k, const void* v,
                   int64_t kv_row_stride, int32_t total_k, const void* k_cache, const void* v_cache,
                   int32_t num_blocks, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t max_seqlen_q,
                   int32_t max_seqlen_k, const int32_t* block_tables, int32_t block_table_stride, int32_t num_seqs,
                   int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                   float softmax_scale, void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                   pkv::Elem elem) {
  int st = check_attention_shape(num_heads, num_kv_heads, head_dim, block_size);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || num_blocks < 0 ||
      block_table_stride < 0)
    return PKV_ERR_BAD_SIZE;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PKV_OK;
  if (!(softmax_scale > 0.f)) return PKV_ERR_BAD_SIZE;
  if (!q || !out || !cu_seqlens_q || !cu_seqlens_k) return PKV_ERR_NULL_POINTER;
  const int64_t row = static_cast<int64_t>(num_heads) * head_dim;
  const int64_t kvrow = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (q_row_stride < row) return PKV_ERR_BAD_STRIDE;
  if (!aligned16(q) || (q_row_stride % 8) != 0 || !aligned16(out)) return PKV_ERR_ALIGNMENT;
  if (block_tables) {
    if (!k_cache || !v_cache) return PKV_ERR_NULL_POINTER;
    if (num_blocks == 0 || block_table_stride == 0) return PKV_ERR_BAD_SIZE;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGNMENT;
  } else {
    if (!k || !v) return PKV_ERR_NULL_POINTER;
    if (total_k == 0) return PKV_ERR_BAD_SIZE;
    if (kv_row_stride < kvrow) return PKV_ERR_BAD_STRIDE;
    if (!aligned16(k) || !aligned16(v) || (kv_row_stride % 8) != 0) return PKV_ERR_ALIGNMENT;
  }
  // The prefill needs no workspace; one passed is a tile plan (pkv_prefill_plan).
  const int32_t* items = nullptr;
  int32_t num_items = 0;
  if (workspace && workspace_bytes > 0) {
    if (workspace_bytes % 4 != 0 || workspace_bytes / 4 > (size_t{1} << 28)) return PKV_ERR_BAD_SIZE;
    if (reinterpret_cast<uintptr_t>(workspace) % 4 != 0) return PKV_ERR_ALIGNMENT;
    items = static_cast<const int32_t*>(workspace);
    num_items = static_cast<int32_t>(workspace_bytes / 4);
  }
  unsigned int* err = nullptr;
  st = error_word(&err);
  if (st != PKV_OK) return st;
  return launched(pkv::launch_prefill(q, q_row_stride, total_q, k, v, kv_row_stride, total_k, k_cache, v_cache,
                                      num_blocks, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                                      block_tables, block_table_stride, num_seqs, softmax_scale, items, num_items,
                                      out, err, stream, elem));
}

int decode_common(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache, int32_t num_blocks,
                  const int32_t* block_tables, int32_t block_table_stride, const int32_t* context_lens,
                  int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                  int32_t max_context_len, float softmax_scale, void* out, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream, const pkv::FusedStore* fused, pkv::Elem elem) {
  int st = pkv::check_decode_args(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables, block_table_stride,
                                  context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                  max_context_len, softmax_scale, out, workspace, workspace_bytes);
  if (st != PKV_OK || num_seqs == 0) return st;
  unsigned int* err = nullptr;
  st = error_word(&err);
  if (st != PKV_OK) return st;
  return launched(pkv::launch_decode(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                                     block_table_stride, context_lens, num_seqs, max_context_len, softmax_scale,
                                     out, workspace, err, stream, fused, elem));
}

int store_decode_common(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                        int64_t v_row_stride, const int32_t* slot_mapping, void* k_cache, void* v_cache,
                        int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale,
                        void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream, pkv::Elem elem) {
  if (num_seqs > 0) {
    if (!k || !v || !slot_mapping) return PKV_ERR_NULL_POINTER;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (k_row_stride < row || v_row_stride < row) return PKV_ERR_BAD_STRIDE;
    if (!aligned16(k) || !aligned16(v) || (k_row_stride % 8) != 0 || (v_row_stride % 8) != 0)
      return PKV_ERR_ALIGNMENT;
  }
  const pkv::FusedStore fused{k, k_row_stride, v, v_row_stride, slot_mapping};
  return decode_common(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables, block_table_stride,
                       context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                       softmax_scale, out, workspace, workspace_bytes, stream, &fused, elem);
}
}  // namespace

extern "C" {

// The bf16 and fp16 entry points share one body each; only the element type differs.

int pkv_prefill_varlen(const void* q, int64_t q_row_stride, int32_t total_q, const void* k, const void* v,
                       int64_t kv_row_stride, int32_t total_k, const void* k_cache, const void* v_cache,
                       int32_t num_blocks, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                       int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t* block_tables,
                       int32_t block_table_stride, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, float softmax_scale, void* out, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  return prefill_common(q, q_row_stride, total_q, k, v, kv_row_stride, total_k, k_cache, v_cache, num_blocks,
                        cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, block_tables, block_table_stride,
                        num_seqs, num_heads, num_kv_heads, head_dim, block_size, softmax_scale, out, workspace,
                        workspace_bytes, stream, pkv::Elem::kBF16);
}

int pkv_prefill_varlen_f16(const void* q, int64_t q_row_stride, int32_t total_q, const void* k, const void* v,
                           int64_t kv_row_stride, int32_t total_k, const void* k_cache, const void* v_cache,
                           int32_t num_blocks, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t* block_tables,
                           int32_t block_table_stride, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, float softmax_scale, void* out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  return prefill_common(q, q_row_stride, total_q, k, v, kv_row_stride, total_k, k_cache, v_cache, num_blocks,
                        cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, block_tables, block_table_stride,
                        num_seqs, num_heads, num_kv_heads, head_dim, block_size, softmax_scale, out, workspace,
                        workspace_bytes, stream, pkv::Elem::kF16);
}

int pkv_decode(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache, int32_t num_blocks,
               const int32_t* block_tables, int32_t block_table_stride, const int32_t* context_lens,
               int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
               int32_t max_context_len, float softmax_scale, void* out, void* workspace, size_t workspace_bytes,
               cudaStream_t stream) {
  return decode_common(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables, block_table_stride,
                       context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                       softmax_scale, out, workspace, workspace_bytes, stream, nullptr, pkv::Elem::kBF16);
}

int pkv_decode_f16(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
                   int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                   const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                   int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale, void* out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return decode_common(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables, block_table_stride,
                       context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                       softmax_scale, out, workspace, workspace_bytes, stream, nullptr, pkv::Elem::kF16);
}

int pkv_store_decode(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                     int64_t v_row_stride, const int32_t* slot_mapping, void* k_cache, void* v_cache,
                     int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                     const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale, void* out,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return store_decode_common(q, q_row_stride, k, k_row_stride, v, v_row_stride, slot_mapping, k_cache, v_cache,
                             num_blocks, block_tables, block_table_stride, context_lens, num_seqs, num_heads,
                             num_kv_heads, head_dim, block_size, max_context_len, softmax_scale, out, workspace,
                             workspace_bytes, stream, pkv::Elem::kBF16);
}

int pkv_store_decode_f16(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                         int64_t v_row_stride, const int32_t* slot_mapping, void* k_cache, void* v_cache,
                         int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale,
                         void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return store_decode_common(q, q_row_stride, k, k_row_stride, v, v_row_stride, slot_mapping, k_cache, v_cache,
                             num_blocks, block_tables, block_table_stride, context_lens, num_seqs, num_heads,
                             num_kv_heads, head_dim, block_size, max_context_len, softmax_scale, out, workspace,
                             workspace_bytes, stream, pkv::Elem::kF16);
}

int pkv_build_prefill_metadata(const int32_t* num_cached_tokens, const int32_t* num_scheduled_tokens,
                               const int32_t* block_tables, int32_t block_table_stride, int32_t num_blocks,
                               int32_t num_seqs, int32_t capacity, int32_t* cu_seqlens_q, int32_t* cu_seqlens_k,
                               int32_t* max_seqlens, int32_t* slot_mapping, int64_t* positions, cudaStream_t stream) {
  if (num_seqs < 0 || num_seqs > 65535 || capacity < 0 || block_table_stride < 0 || num_blocks < 0)
    return PKV_ERR_BAD_SIZE;
  if (!cu_seqlens_q || !cu_seqlens_k || !max_seqlens) return PKV_ERR_NULL_POINTER;
  if (num_seqs > 0 && (!num_cached_tokens || !num_scheduled_tokens || !block_tables || !slot_mapping || !positions))
    return PKV_ERR_NULL_POINTER;
  unsigned int* err = nullptr;
  int st = error_word(&err);
  if (st != PKV_OK) return st;
  return launched(pkv::launch_prefill_metadata(num_cached_tokens, num_scheduled_tokens, block_tables,
                                               block_table_stride, num_blocks, num_seqs, capacity, cu_seqlens_q,
                                               cu_seqlens_k, max_seqlens, slot_mapping, positions, err, stream));
}

int pkv_build_decode_metadata(const int32_t* num_tokens, const int32_t* block_tables, int32_t block_table_stride,
                              int32_t num_blocks, int32_t num_seqs, int32_t* slot_mapping, int32_t* context_lens,
                              int64_t* positions, cudaStream_t stream) {
  if (num_seqs < 0 || block_table_stride < 0 || num_blocks < 0) return PKV_ERR_BAD_SIZE;
  if (num_seqs == 0) return PKV_OK;
  if (!num_tokens || !block_tables || !slot_mapping || !context_lens || !positions) return PKV_ERR_NULL_POINTER;
  unsigned int* err = nullptr;
  int st = error_word(&err);
  if (st != PKV_OK) return st;
  return launched(pkv::launch_decode_metadata(num_tokens, block_tables, block_table_stride, num_blocks, num_seqs,
                                              slot_mapping, context_lens, positions, err, stream));
}

int pkv_device_error(uint32_t* bits, int clear, cudaStream_t stream) {
  unsigned int* err = nullptr;
  int st = error_word(&err);
  if (st != PKV_OK) return st;
  unsigned int h = 0;
  if (cudaMemcpyAsync(&h, err, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return PKV_ERR_CUDA;
  if (clear && cudaMemsetAsync(err, 0, sizeof(unsigned int), stream) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ERR_CUDA;
  if (bits) *bits = h;
  return PKV_OK;
}

int pkv_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  unsigned int* err = nullptr;
  int st = error_word(&err);
  if (st != PKV_OK) return st;
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 100000000ull) limit_ns = 100000000ull;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return launched(cudaGetLastError());
}

}  // extern "C"
