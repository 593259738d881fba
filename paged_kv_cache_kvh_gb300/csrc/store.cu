// store.cu -- slot_mapping scatter of new K/V rows into the paged cache.
//
// The operation is store_kvcache of layers/attention.py in
// "vLLM 学习笔记 02：nano-vllm 源码逐段精读": token i's K and V rows go to
// row slot_mapping[i] of k_cache / v_cache, slot -1 means skip.
//
// GB300 design: the copy is HBM-bound (8 KB of traffic per token for the
// Qwen3-0.6B shape), so the kernel is about bytes in flight. One warp moves one
// token: each lane issues all of its 16-byte loads (K and V) before any store,
// so a 2 KB + 2 KB token row is eight independent 16-byte requests per lane.
// Loads are read-only and not kept in L1; stores use the default policy so the
// freshly written rows stay in L2 for the attention kernel that reads them next.
#include "pkv_common.cuh"

namespace pkv {

namespace {

constexpr int kStoreWarps = 8;  // tokens per 256-thread block

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Vector path: rows of D16 16-byte chunks (D = 8*D16 elements).
template <int kChunksPerLane>
__global__ void __launch_bounds__(kStoreWarps * 32) store_kvcache_v16_kernel(
    const uint4* __restrict__ k, int64_t k_stride16, const uint4* __restrict__ v, int64_t v_stride16,
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ slot_mapping,
    int32_t num_tokens, int32_t D16, int64_t num_slots, unsigned int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t token = static_cast<int64_t>(blockIdx.x) * kStoreWarps + (threadIdx.x >> 5);
  if (token >= num_tokens) return;
  const int64_t slot = slot_mapping[token];
  if (slot == -1) return;
  if (slot < 0 || slot >= num_slots) {
    if (lane == 0) flag_error(err, PKV_DEVERR_BAD_SLOT);
    return;
  }
  const uint4* ks = k + token * k_stride16;
  const uint4* vs = v + token * v_stride16;
  uint4* kd = k_cache + slot * D16;
  uint4* vd = v_cache + slot * D16;
  if (kChunksPerLane > 0 && D16 == kChunksPerLane * 32) {
    constexpr int kN = kChunksPerLane > 0 ? kChunksPerLane : 1;
    uint4 kr[kN], vr[kN];
#pragma unroll
    for (int i = 0; i < kChunksPerLane; ++i) kr[i] = ld_nc_v4(ks + lane + 32 * i);
#pragma unroll
    for (int i = 0; i < kChunksPerLane; ++i) vr[i] = ld_nc_v4(vs + lane + 32 * i);
#pragma unroll
    for (int i = 0; i < kChunksPerLane; ++i) kd[lane + 32 * i] = kr[i];
#pragma unroll
    for (int i = 0; i < kChunksPerLane; ++i) vd[lane + 32 * i] = vr[i];
  } else {
    for (int i = lane; i < D16; i += 32) {
      const uint4 a = ld_nc_v4(ks + i);
      const uint4 b = ld_nc_v4(vs + i);
      kd[i] = a;
      vd[i] = b;
    }
  }
}

// Fallback for unaligned strides or row lengths: 2-byte copies.
__global__ void __launch_bounds__(kStoreWarps * 32) store_kvcache_u16_kernel(
    const uint16_t* __restrict__ k, int64_t k_stride, const uint16_t* __restrict__ v, int64_t v_stride,
    uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache, const int32_t* __restrict__ slot_mapping,
    int32_t num_tokens, int32_t D, int64_t num_slots, unsigned int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t token = static_cast<int64_t>(blockIdx.x) * kStoreWarps + (threadIdx.x >> 5);
  if (token >= num_tokens) return;
  const int64_t slot = slot_mapping[token];
  if (slot == -1) return;
  if (slot < 0 || slot >= num_slots) {
    if (lane == 0) flag_error(err, PKV_DEVERR_BAD_SLOT);
    return;
  }
  for (int i = lane; i < D; i += 32) {
    k_cache[slot * D + i] = k[token * k_stride + i];
    v_cache[slot * D + i] = v[token * v_stride + i];
  }
}

}  // namespace

cudaError_t launch_store_kvcache(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                                 void* k_cache, void* v_cache, const int32_t* slot_mapping, int32_t num_tokens,
                                 int32_t D, int64_t num_slots, unsigned int* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const dim3 grid((num_tokens + kStoreWarps - 1) / kStoreWarps), block(kStoreWarps * 32);
  const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
                         reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) &
                        15) == 0 &&
                       (k_row_stride % 8) == 0 && (v_row_stride % 8) == 0 && (D % 8) == 0;
  if (aligned) {
    const int32_t D16 = D / 8;
    if (D16 == 128) {
      store_kvcache_v16_kernel<4><<<grid, block, 0, stream>>>(
          static_cast<const uint4*>(k), k_row_stride / 8, static_cast<const uint4*>(v), v_row_stride / 8,
          static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, num_tokens, D16, num_slots,
          err);
    } else {
      store_kvcache_v16_kernel<0><<<grid, block, 0, stream>>>(
          static_cast<const uint4*>(k), k_row_stride / 8, static_cast<const uint4*>(v), v_row_stride / 8,
          static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, num_tokens, D16, num_slots,
          err);
    }
  } else {
    store_kvcache_u16_kernel<<<grid, block, 0, stream>>>(
        static_cast<const uint16_t*>(k), k_row_stride, static_cast<const uint16_t*>(v), v_row_stride,
        static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache), slot_mapping, num_tokens, D, num_slots,
        err);
  }
  return cudaGetLastError();
}

}  // namespace pkv
