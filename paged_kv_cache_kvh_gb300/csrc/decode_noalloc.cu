// decode_noalloc.cu -- pkv_decode_noalloc: decode attention for callers that
// cannot allocate device memory.
//
// pkv_decode needs a caller-provided workspace for its split-KV partial
// results. Some callers have no way to provide one: an engine that sized its
// KV-cache pool to take all device memory left after start-up, a plug-in whose
// host process owns the only device allocator, or a latency-critical loop
// that must not call cudaMalloc (it can synchronise the device). For them this
// entry point runs the same decode with its scratch in a fixed array that is
// part of the library's device image: it is reserved on every GPU that loads
// the library and held until the process exits, so nothing is allocated per
// call.
//
// The array has no device address known to host code until it is looked up:
// in host code its name only stands for a host-side shadow symbol, and handing
// that to a kernel would fault or, where the GPU can reach host memory,
// silently touch the wrong memory. So every call asks the runtime for the real
// address (cudaGetSymbolAddress, with the calling thread's device current),
// checks the result and passes that address on to the kernel. The address is
// cached per device and context and looked up again when the context changes
// (a cudaDeviceReset moves the array). The first call on a device is the one
// that makes the lookup, and it may load the library's device code there:
// make that first call before any stream capture.
#include "pkv_common.cuh"

namespace {

// The scratch itself: PKV_DECODE_NOALLOC_SCRATCH_BYTES bytes per device.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[PKV_DECODE_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" int pkv_decode_noalloc(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
                                  int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                                  const int32_t* context_lens, int32_t num_seqs, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t max_context_len, float softmax_scale, void* out, cudaStream_t stream) {
  if (num_seqs < 0 || max_context_len < 0) return PKV_ERR_BAD_SIZE;
  if (num_seqs == 0) return PKV_OK;
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_heads, max_context_len);
  if (need > static_cast<size_t>(PKV_DECODE_NOALLOC_SCRATCH_BYTES)) return PKV_ERR_SCRATCH_LIMIT;
  // Everything pkv_decode would reject is rejected here first, so a refused
  // call leaves nothing queued on the stream.
  unsigned int* err = nullptr;
  int st = pkv::device_error_word(&err);
  if (st != PKV_OK) return st;
  void* scratch = nullptr;
  st = pkv::symbol_address(&g_decode_noalloc_scratch, pkv::kSymbolDecodeScratch, &scratch);
  if (st != PKV_OK) return st;
  st = pkv::check_decode_args(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables, block_table_stride,
                              context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                              softmax_scale, out, scratch, static_cast<size_t>(PKV_DECODE_NOALLOC_SCRATCH_BYTES));
  if (st != PKV_OK) return st;
  // The split-KV tickets and the two work counters after them at the start
  // of the scratch must start at zero. The array keeps whatever the previous
  // call left, so clear them on the stream.
  if (need > 0) {
    const size_t tickets = (static_cast<size_t>(num_seqs) + 2) * sizeof(int32_t);
    if (cudaMemsetAsync(scratch, 0, tickets, stream) != cudaSuccess) {
      (void)cudaGetLastError();
      return PKV_ERR_CUDA;
    }
  }
  return pkv_decode(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables, block_table_stride, context_lens,
                    num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len, softmax_scale, out,
                    scratch, static_cast<size_t>(PKV_DECODE_NOALLOC_SCRATCH_BYTES), stream);
}
