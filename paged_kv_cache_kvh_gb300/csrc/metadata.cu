// metadata.cu -- the index preparation of a step, built on the GPU.
//
// engine/model_runner.py in "vLLM 学习笔记 02：nano-vllm 源码逐段精读" builds
// the attention metadata on the host with per-token Python loops
// (prepare_prefill, prepare_decode) and copies it over every step. Here the
// host only uploads what the scheduler already has per sequence (token
// counts and the padded block table) and these kernels derive the rest:
//   prefill  cu_seqlens_q/k (prefix sums of num_scheduled_tokens and of
//            num_cached + num_scheduled), max_seqlen_q/k, and for every new
//            token its position t = num_cached + i and its slot
//            block_table[t / 256] * 256 + t % 256;
//   decode   slot of position len-1, context_lens = len, positions = len-1.
// Integer work only; the results are bit-identical to the host versions.
#include "pkv_common.cuh"

namespace pkv {

namespace {

constexpr int kScanThreads = 1024;

// One CTA: exclusive prefix sums over the sequences in chunks of 1024, plus
// the maxima. cu_q/cu_k get num_seqs+1 entries.
__global__ void __launch_bounds__(kScanThreads) prefill_scan_kernel(const int32_t* __restrict__ num_cached,
                                                                    const int32_t* __restrict__ num_scheduled,
                                                                    int32_t num_seqs, int32_t* __restrict__ cu_q,
                                                                    int32_t* __restrict__ cu_k,
                                                                    int32_t* __restrict__ max_q_k,
                                                                    unsigned int* err) {
  __shared__ int32_t sq[kScanThreads], sk[kScanThreads];
  __shared__ int32_t carry_q, carry_k, mq, mk;
  if (threadIdx.x == 0) {
    carry_q = 0;
    carry_k = 0;
    mq = 0;
    mk = 0;
    cu_q[0] = 0;
    cu_k[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < num_seqs; base += kScanThreads) {
    const int b = base + threadIdx.x;
    int lq = 0, lk = 0;
    if (b < num_seqs) {
      const int c = num_cached[b], s = num_scheduled[b];
      if (c < 0 || s < 0) {
        flag_error(err, PKV_DEVERR_BAD_SEQLEN);
      } else {
        lq = s;
        lk = c + s;
      }
    }
    sq[threadIdx.x] = lq;
    sk[threadIdx.x] = lk;
    __syncthreads();
    // Hillis-Steele inclusive scan in shared memory
    for (int off = 1; off < kScanThreads; off <<= 1) {
      const int aq = threadIdx.x >= off ? sq[threadIdx.x - off] : 0;
      const int ak = threadIdx.x >= off ? sk[threadIdx.x - off] : 0;
      __syncthreads();
      sq[threadIdx.x] += aq;
      sk[threadIdx.x] += ak;
      __syncthreads();
    }
    if (b < num_seqs) {
      cu_q[b + 1] = carry_q + sq[threadIdx.x];
      cu_k[b + 1] = carry_k + sk[threadIdx.x];
      atomicMax(&mq, lq);
      atomicMax(&mk, lk);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_q += sq[kScanThreads - 1];
      carry_k += sk[kScanThreads - 1];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    max_q_k[0] = mq;
    max_q_k[1] = mk;
  }
}

// grid.y = sequence; threads stride over its scheduled tokens.
__global__ void prefill_fill_kernel(const int32_t* __restrict__ num_cached, const int32_t* __restrict__ num_scheduled,
                                    const int32_t* __restrict__ block_tables, int32_t bt_stride, int32_t num_blocks,
                                    const int32_t* __restrict__ cu_q, int32_t capacity,
                                    int32_t* __restrict__ slot_mapping, int64_t* __restrict__ positions,
                                    unsigned int* err) {
  const int b = blockIdx.y;
  const int c = num_cached[b], s = num_scheduled[b];
  if (c < 0 || s < 0) return;
  const int64_t out0 = cu_q[b];
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < s; i += gridDim.x * blockDim.x) {
    const int64_t o = out0 + i;
    if (o >= capacity) {
      flag_error(err, PKV_DEVERR_BAD_SEQLEN);
      return;
    }
    const int t = c + i;
    const int lb = t / kBlockSize;
    int32_t slot = -1;
    if (lb < bt_stride) {
      const int blk = block_tables[static_cast<int64_t>(b) * bt_stride + lb];
      if (blk >= 0 && blk < num_blocks) slot = blk * kBlockSize + t % kBlockSize;
    }
    if (slot < 0) flag_error(err, PKV_DEVERR_BAD_BLOCK);
    slot_mapping[o] = slot;
    positions[o] = t;
  }
}

__global__ void decode_meta_kernel(const int32_t* __restrict__ num_tokens, const int32_t* __restrict__ block_tables,
                                   int32_t bt_stride, int32_t num_blocks, int32_t num_seqs,
                                   int32_t* __restrict__ slot_mapping, int32_t* __restrict__ context_lens,
                                   int64_t* __restrict__ positions, unsigned int* err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= num_seqs) return;
  const int n = num_tokens[b];
  int32_t slot = -1;
  if (n > 0) {  // n == 0: a padding row (slot -1, context 0), as the graph replay fills them
    const int t = n - 1;
    const int lb = t / kBlockSize;
    if (lb < bt_stride) {
      const int blk = block_tables[static_cast<int64_t>(b) * bt_stride + lb];
      if (blk >= 0 && blk < num_blocks) slot = blk * kBlockSize + t % kBlockSize;
    }
    if (slot < 0) flag_error(err, PKV_DEVERR_BAD_BLOCK);
  } else if (n < 0) {
    flag_error(err, PKV_DEVERR_BAD_SEQLEN);
  }
  slot_mapping[b] = slot;
  context_lens[b] = n > 0 ? n : 0;
  positions[b] = n > 0 ? n - 1 : 0;
}

}  // namespace

cudaError_t launch_prefill_metadata(const int32_t* num_cached, const int32_t* num_scheduled,
                                    const int32_t* block_tables, int32_t bt_stride, int32_t num_blocks,
                                    int32_t num_seqs, int32_t capacity, int32_t* cu_q, int32_t* cu_k,
                                    int32_t* max_q_k, int32_t* slot_mapping, int64_t* positions, unsigned int* err,
                                    cudaStream_t stream) {
  prefill_scan_kernel<<<1, kScanThreads, 0, stream>>>(num_cached, num_scheduled, num_seqs, cu_q, cu_k, max_q_k, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || num_seqs == 0) return e;
  const dim3 grid(4, num_seqs);
  prefill_fill_kernel<<<grid, 256, 0, stream>>>(num_cached, num_scheduled, block_tables, bt_stride, num_blocks, cu_q,
                                                capacity, slot_mapping, positions, err);
  return cudaGetLastError();
}

cudaError_t launch_decode_metadata(const int32_t* num_tokens, const int32_t* block_tables, int32_t bt_stride,
                                   int32_t num_blocks, int32_t num_seqs, int32_t* slot_mapping, int32_t* context_lens,
                                   int64_t* positions, unsigned int* err, cudaStream_t stream) {
  if (num_seqs == 0) return cudaSuccess;
  decode_meta_kernel<<<(num_seqs + 255) / 256, 256, 0, stream>>>(num_tokens, block_tables, bt_stride, num_blocks,
                                                                  num_seqs, slot_mapping, context_lens, positions, err);
  return cudaGetLastError();
}

}  // namespace pkv
