// decode.cu -- single-query GQA attention over the paged KV cache (split-KV).
//
// The operation is the flash_attn_with_kvcache call of layers/attention.py in
// "vLLM 学习笔记 02：nano-vllm 源码逐段精读": one query per sequence, keys
// 0..context_lens[b]-1 reached through block_tables, causal (a no-op for the
// last position), query head h on kv head h/2.
//
// GB300 design (HBM-bound: 4 KB of K+V per token for 8 kv heads x 128 dims):
//  * One CTA per (chunk c, sequence b), a chunk being `chunk` consecutive
//    tokens inside one 256-token block (chunk = 256, 128, 64 or 32, chosen on
//    the host so that small batches still give the GPU enough CTAs). A
//    chunk's tokens are one contiguous K region and one V region of the
//    cache, so the producer warp streams them with plain bulk copies
//    (cp.async.bulk, 1-D TMA), kT tokens x 2 KB per stage, through a
//    kStages-deep shared-memory ring guarded by mbarriers.
//  * Consumer warp w owns kv head w and both query heads 2w, 2w+1 that read
//    it, so each K/V byte is loaded once for the whole GQA group. Lane l holds
//    dims 4l..4l+3. Per stage every lane forms 2*kT partial dot products and a
//    transposed butterfly (2*kT-1 shuffles for 2*kT results) leaves lane l
//    with one complete logit; softmax statistics are half-warp reductions.
//  * Split-KV merge without a second launch: each CTA writes (m, l, o) for its
//    chunk to the workspace, and the CTA that finishes last for a sequence
//    (atomic ticket, no waiting) merges them and resets the ticket to zero.
//    Sequences with a single chunk write the output directly.
//  * Logits are kept in the log2 domain (q is pre-scaled by scale*log2(e))
//    and exponentials use ex2.approx.
//  * The element type (bf16 or fp16) is a template parameter: it only changes
//    how packed pairs are widened to fp32 and how the output is rounded.
#include "pkv_common.cuh"

#ifndef PKV_DECODE_TOKENS_PER_STAGE
#define PKV_DECODE_TOKENS_PER_STAGE 8
#endif
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 3
#endif

namespace pkv {

// New-token rows for pkv_store_decode (k/v row strides in elements).
struct FusedStore {
  const void* k;
  int64_t k_row_stride;
  const void* v;
  int64_t v_row_stride;
  const int32_t* slot_mapping;
};

namespace {

constexpr int kHkv = 8;
constexpr int kGroup = 2;
constexpr int kHq = kHkv * kGroup;
constexpr int kRowBytes = kHkv * kHeadDim * 2;  // one token's K (or V) row: 2048 B
constexpr int kConsumerWarps = kHkv;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

struct DecodeParams {
  const uint16_t* q;  // 16-bit elements of the call's type
  int64_t q_row_stride;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  int32_t num_blocks;
  const int32_t* block_tables;
  int32_t bt_stride;
  const int32_t* context_lens;
  int32_t max_ctx;
  int32_t num_seqs;
  int32_t nsplit;
  int32_t chunk;      // tokens per CTA: 256, 128, 64 or 32 (divides the block size)
  float scale_log2;
  uint16_t* out;
  int32_t* tickets;   // [num_seqs], then the persistent form's work counters {next item, CTAs done}
  float2* ml;         // [num_seqs, nsplit, 16] (running max in log2 units, sum)
  float* opart;       // [num_seqs, nsplit, 16, 128] unnormalised partial outputs
  // Fused store (pkv_store_decode); k_new == nullptr for plain decode.
  const uint4* k_new;
  const uint4* v_new;
  int64_t k_new_stride16;  // row strides in 16-byte units
  int64_t v_new_stride16;
  const int32_t* slot_mapping;
  uint4* k_cache_w;
  uint4* v_cache_w;
  unsigned int* err;
};

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr));
  return r;
}

// Transposed butterfly: lane l ends with the warp-wide sum of value index
// (l >> (5 - log2 N)); N values per lane, N a power of two <= 32.
template <int N>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane) {
  int n = N;
  int offset = 16;
#pragma unroll
  for (int r = 0; r < 5; ++r) {
    if (n > 1) {
      const int half = n >> 1;
      const bool upper = (lane & offset) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, offset);
        }
      }
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], offset);
    }
    offset >>= 1;
  }
  return v[0];
}

// Split-KV merge of sequence b's nch partials (m, l, o) for query head hq,
// dims d0..d0+7 (one thread), written to the output row:
//   o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c,  M = max_c m_c.
// The partials sit in L2 (other CTAs wrote them), so the merge is bound by
// round trips: it reads them four chunks at a time, every load of a group in
// flight together, and keeps a running maximum (rescaling what it has summed
// when the maximum grows), one pass over the chunks.
template <Elem E>
__device__ __forceinline__ void merge_partials(const DecodeParams& p, int b, int nch, int hq, int d0) {
  using Ops = ElemOps<E>;
  constexpr int kG = 4;
  const int64_t base = static_cast<int64_t>(b) * p.nsplit * kHq + hq;
  float M = -INFINITY, den = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int c0 = 0; c0 < nch; c0 += kG) {
    float2 ml[kG];
    float4 x[kG], y[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      if (c0 + j < nch) {
        const int64_t slot = base + static_cast<int64_t>(c0 + j) * kHq;
        ml[j] = __ldcg(p.ml + slot);
        x[j] = __ldcg(reinterpret_cast<const float4*>(p.opart + slot * kHeadDim + d0));
        y[j] = __ldcg(reinterpret_cast<const float4*>(p.opart + slot * kHeadDim + d0 + 4));
      } else {
        ml[j] = make_float2(-INFINITY, 0.f);
        x[j] = y[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mg = M;
#pragma unroll
    for (int j = 0; j < kG; ++j) Mg = fmaxf(Mg, ml[j].x);
    if (Mg > M) {
      const float sc = (M == -INFINITY) ? 0.f : ex2_approx(M - Mg);
      den *= sc;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= sc;
      M = Mg;
    }
    const float Mu = (M == -INFINITY) ? 0.f : M;
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      const float w = ex2_approx(ml[j].x - Mu);
      den = fmaf(w, ml[j].y, den);
      acc[0] = fmaf(w, x[j].x, acc[0]);
      acc[1] = fmaf(w, x[j].y, acc[1]);
      acc[2] = fmaf(w, x[j].z, acc[2]);
      acc[3] = fmaf(w, x[j].w, acc[3]);
      acc[4] = fmaf(w, y[j].x, acc[4]);
      acc[5] = fmaf(w, y[j].y, acc[5]);
      acc[6] = fmaf(w, y[j].z, acc[6]);
      acc[7] = fmaf(w, y[j].w, acc[7]);
    }
  }
  const float r = den > 0.f ? 1.f / den : 0.f;
  uint4 w;
  w.x = Ops::pack(acc[0] * r, acc[1] * r);
  w.y = Ops::pack(acc[2] * r, acc[3] * r);
  w.z = Ops::pack(acc[4] * r, acc[5] * r);
  w.w = Ops::pack(acc[6] * r, acc[7] * r);
  *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * kHq + hq) * kHeadDim + d0) = w;
}

template <Elem E, int kT, int kStages>
__global__ void __launch_bounds__(kThreads, (kStages * 2 * kT * kRowBytes <= 100 * 1024) ? 2 : 1)
    decode_split_kernel(const DecodeParams p) {
  using Ops = ElemOps<E>;
  static_assert(2 * kT <= 32 && (kT & (kT - 1)) == 0, "kT must be a power of two <= 16");
  constexpr int kStageBytes = 2 * kT * kRowBytes;
  constexpr int kN = 2 * kT;                 // logits per warp per stage
  constexpr int kLog2N = (kN == 32) ? 5 : (kN == 16) ? 4 : (kN == 8) ? 3 : (kN == 4) ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  float* pbuf = reinterpret_cast<float*>(smem + kStages * kStageBytes);   // [8 warps][kN]
  uint64_t* bars = reinterpret_cast<uint64_t*>(pbuf + kConsumerWarps * kN);
  int* s_last = reinterpret_cast<int*>(bars + 2 * kStages);

  const int c = blockIdx.x;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int ctx = p.context_lens[b];
  if (ctx < 0 || ctx > p.max_ctx || ctx > p.bt_stride * kBlockSize) {
    if (threadIdx.x == 0 && c == 0) flag_error(p.err, PKV_DEVERR_BAD_SEQLEN);
    ctx = 0;
  }
  if (ctx == 0) {  // graph padding row: zeros
    if (c == 0) {
      uint4* o = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(b) * kHq * kHeadDim);
      for (int i = threadIdx.x; i < kHq * kHeadDim / 8; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int nchunks = (ctx + p.chunk - 1) / p.chunk;
  if (c >= nchunks) return;
  const int tok0 = c * p.chunk;  // first position of this chunk; the chunk lies inside one block
  const int ntok = min(p.chunk, ctx - tok0);
  const int pb = p.block_tables[static_cast<int64_t>(b) * p.bt_stride + tok0 / kBlockSize];
  const bool bad_block = pb < 0 || pb >= p.num_blocks;
  const int niter = bad_block ? 0 : (ntok + kT - 1) / kT;

  const uint32_t smem0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  if (p.k_new != nullptr && c == nchunks - 1) {
    // Fused store: this CTA owns the sequence's newest position ctx-1, whose
    // slot the new token's K/V row must reach before the block is streamed.
    const int64_t slot = p.slot_mapping[b];
    if (slot != -1) {
      const int64_t expect = static_cast<int64_t>(pb) * kBlockSize + (ctx - 1) % kBlockSize;
      if (bad_block || slot != expect) {
        if (threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_BAD_SLOT);
      } else if (threadIdx.x < 2 * kRowBytes / 16) {
        const bool is_v = threadIdx.x >= kRowBytes / 16;
        const int i = threadIdx.x % (kRowBytes / 16);
        const uint4* src = is_v ? p.v_new + b * p.v_new_stride16 : p.k_new + b * p.k_new_stride16;
        uint4* dst = (is_v ? p.v_cache_w : p.k_cache_w) + slot * (kRowBytes / 16);
        dst[i] = src[i];
        // make the write visible to the bulk copies (async proxy) issued after the CTA barrier
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
    }
  }
  if (threadIdx.x == 0) {
    if (bad_block) flag_error(p.err, PKV_DEVERR_BAD_BLOCK);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncwarp();  // every warp reaches each CTA barrier converged
  __syncthreads();

  float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
  float m0 = -INFINITY, m1 = -INFINITY, lsum = 0.f;
  const int h = warp;

  if (warp == kConsumerWarps) {
    // ---------------- producer: one elected lane streams the block ----------------
    if (lane == 0 && niter > 0) {
      const int64_t base = (static_cast<int64_t>(pb) * kBlockSize + tok0 % kBlockSize) * kRowBytes;
      const uint8_t* ksrc = p.k_cache + base;
      const uint8_t* vsrc = p.v_cache + base;
      int issued = 0;
      for (int it = 0; it < niter; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(empty0 + 8 * s, ((it / kStages) - 1) & 1, p.err)) break;
        const int rows = min(kT, ntok - it * kT);
        const uint32_t bytes = static_cast<uint32_t>(rows) * kRowBytes;
        const uint32_t dst = smem0 + s * kStageBytes;
        mbar_arrive_expect_tx(full0 + 8 * s, 2 * bytes);
        bulk_g2s(dst, ksrc + static_cast<int64_t>(it) * kT * kRowBytes, bytes, full0 + 8 * s);
        bulk_g2s(dst + kT * kRowBytes, vsrc + static_cast<int64_t>(it) * kT * kRowBytes, bytes, full0 + 8 * s);
        ++issued;
      }
      // Never leave a copy in flight into this CTA's shared memory.
      for (int it = max(0, issued - kStages); it < issued; ++it)
        mbar_wait(full0 + 8 * (it % kStages), (it / kStages) & 1, p.err);
    }
  } else {
    // ---------------- consumers: warp h = kv head h, query heads 2h, 2h+1 ----------------
    float q0[4], q1[4];
    {
      const uint16_t* qrow = p.q + static_cast<int64_t>(b) * p.q_row_stride;
      const uint2 a = *reinterpret_cast<const uint2*>(qrow + (kGroup * h) * kHeadDim + lane * 4);
      const uint2 bq = *reinterpret_cast<const uint2*>(qrow + (kGroup * h + 1) * kHeadDim + lane * 4);
      q0[0] = Ops::lo(a.x) * p.scale_log2;
      q0[1] = Ops::hi(a.x) * p.scale_log2;
      q0[2] = Ops::lo(a.y) * p.scale_log2;
      q0[3] = Ops::hi(a.y) * p.scale_log2;
      q1[0] = Ops::lo(bq.x) * p.scale_log2;
      q1[1] = Ops::hi(bq.x) * p.scale_log2;
      q1[2] = Ops::lo(bq.y) * p.scale_log2;
      q1[3] = Ops::hi(bq.y) * p.scale_log2;
    }
    const int idx = lane >> (5 - kLog2N);         // logit index this lane ends up holding
    const int my_t = idx % kT;
    const bool owner = (lane & ((1 << (5 - kLog2N)) - 1)) == 0;
    const bool my_g1 = lane >= 16;
    float* wp = pbuf + warp * kN;
    const uint32_t wp_addr = smem_u32(wp);
    for (int it = 0; it < niter; ++it) {
      const int s = it % kStages;
      // all lanes wait (each needs the acquire) and agree before the full-warp shuffles
      if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (it / kStages) & 1, p.err))) break;
      const int rows = min(kT, ntok - it * kT);
      const uint32_t kaddr = smem0 + s * kStageBytes + h * (kHeadDim * 2) + lane * 8;
      const uint32_t vaddr = kaddr + kT * kRowBytes;
      float part[kN];
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        const uint2 kr = lds64(kaddr + t * kRowBytes);
        const float k0 = Ops::lo(kr.x), k1 = Ops::hi(kr.x);
        const float k2 = Ops::lo(kr.y), k3 = Ops::hi(kr.y);
        part[t] = fmaf(q0[0], k0, fmaf(q0[1], k1, fmaf(q0[2], k2, q0[3] * k3)));
        part[kT + t] = fmaf(q1[0], k0, fmaf(q1[1], k1, fmaf(q1[2], k2, q1[3] * k3)));
      }
      float sc = transpose_reduce<kN>(part, lane);
      if (my_t >= rows) sc = -INFINITY;
      float mx = sc;
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mx0 = __shfl_sync(0xffffffffu, mx, 0);
      const float mx1 = __shfl_sync(0xffffffffu, mx, 16);
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float a0 = ex2_approx(m0 - mu0), a1 = ex2_approx(m1 - mu1);
      const float pv = ex2_approx(sc - (my_g1 ? mu1 : mu0));
      lsum = lsum * (my_g1 ? a1 : a0) + (owner ? pv : 0.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o0[i] *= a0;
        o1[i] *= a1;
      }
      m0 = mn0;
      m1 = mn1;
      if (owner) wp[idx] = pv;
      __syncwarp();
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        if (t < rows) {
          float w0, w1;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(w0) : "r"(wp_addr + 4 * t));
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(w1) : "r"(wp_addr + 4 * (kT + t)));
          const uint2 vr = lds64(vaddr + t * kRowBytes);
          const float v0 = Ops::lo(vr.x), v1 = Ops::hi(vr.x);
          const float v2 = Ops::lo(vr.y), v3 = Ops::hi(vr.y);
          o0[0] = fmaf(w0, v0, o0[0]);
          o0[1] = fmaf(w0, v1, o0[1]);
          o0[2] = fmaf(w0, v2, o0[2]);
          o0[3] = fmaf(w0, v3, o0[3]);
          o1[0] = fmaf(w1, v0, o1[0]);
          o1[1] = fmaf(w1, v1, o1[1]);
          o1[2] = fmaf(w1, v2, o1[2]);
          o1[3] = fmaf(w1, v3, o1[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    // row sums: half-warp g holds the partial sums of query head 2h+g
    float l = lsum;
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const float l0 = __shfl_sync(0xffffffffu, l, 0);
    const float l1 = __shfl_sync(0xffffffffu, l, 16);
    if (nchunks == 1) {
      const float r0 = l0 > 0.f ? 1.f / l0 : 0.f, r1 = l1 > 0.f ? 1.f / l1 : 0.f;
      uint16_t* orow = p.out + static_cast<int64_t>(b) * kHq * kHeadDim;
      uint2 w;
      w.x = Ops::pack(o0[0] * r0, o0[1] * r0);
      w.y = Ops::pack(o0[2] * r0, o0[3] * r0);
      *reinterpret_cast<uint2*>(orow + (kGroup * h) * kHeadDim + lane * 4) = w;
      w.x = Ops::pack(o1[0] * r1, o1[1] * r1);
      w.y = Ops::pack(o1[2] * r1, o1[3] * r1);
      *reinterpret_cast<uint2*>(orow + (kGroup * h + 1) * kHeadDim + lane * 4) = w;
    } else {
      const int64_t slot = (static_cast<int64_t>(b) * p.nsplit + c) * kHq + kGroup * h;
      *reinterpret_cast<float4*>(p.opart + slot * kHeadDim + lane * 4) = make_float4(o0[0], o0[1], o0[2], o0[3]);
      *reinterpret_cast<float4*>(p.opart + (slot + 1) * kHeadDim + lane * 4) =
          make_float4(o1[0], o1[1], o1[2], o1[3]);
      if (lane == 0) {
        p.ml[slot] = make_float2(m0, l0);
        p.ml[slot + 1] = make_float2(m1, l1);
      }
    }
  }

  if (nchunks == 1) return;
  // ---------------- split-KV merge by the last CTA of this sequence ----------------
  __syncwarp();  // the producer warp's lane 0 streamed alone: reconverge first
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(p.tickets + b, 1);
    *s_last = (prev == nchunks - 1) ? 1 : 0;
  }
  __syncwarp();
  __syncthreads();
  if (*s_last == 0) return;
  __threadfence();
  if (threadIdx.x < kHq * 16) merge_partials<E>(p, b, nchunks, threadIdx.x >> 4, (threadIdx.x & 15) * 8);
  if (threadIdx.x == 0) p.tickets[b] = 0;  // ready for the next call
}

// ---------------------------------------------------------------------------
// Persistent form for whole-block chunks (large batches). The grid kernel
// launches one CTA per (chunk, sequence) pair up to max_context_len, so a
// batch of long-tailed contexts (most far below the declared maximum, as in a
// graph captured for max_model_len) launches mostly CTAs that find no live
// block, and every live CTA pays its own ramp-up. Here 2 CTAs per SM walk
// only the live items, the producer's ring running on from one item to the
// next. The item list is built by every CTA in shared memory from
// context_lens, the same way in each CTA: first every whole 256-token chunk
// (sequence order), then the partial last chunks bucketed by size, largest
// bucket first. CTAs take the next list position from a counter in the
// workspace as they go (longest-first, first come first served): a static
// split measured CTAs finishing up to 18% apart, as their shares of the
// memory bandwidth differ. Each item's q row (4 KB) arrives with its first
// stage; the split-KV partials and the last-CTA merge are the grid kernel's.
constexpr int kPersistMaxSeqs = 512;   // item tables in shared memory
constexpr int kQRowBytes = kHq * kHeadDim * 2;
constexpr int kBuckets = 8;            // size classes of the partial chunks

__device__ __forceinline__ void named_sync_consumers() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

template <Elem E, int kT, int kStages>
__global__ void __launch_bounds__(kThreads, 2) decode_persistent_kernel(const DecodeParams p) {
  using Ops = ElemOps<E>;
  static_assert(2 * kT <= 32 && (kT & (kT - 1)) == 0, "kT must be a power of two <= 16");
  constexpr int kStageBytes = 2 * kT * kRowBytes;
  constexpr int kN = 2 * kT;
  constexpr int kLog2N = (kN == 32) ? 5 : (kN == 16) ? 4 : (kN == 8) ? 3 : (kN == 4) ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* qbuf = smem + kStages * kStageBytes;                                  // 2 x 4 KB
  float* pbuf = reinterpret_cast<float*>(qbuf + 2 * kQRowBytes);                 // [8 warps][kN]
  int4* hdr = reinterpret_cast<int4*>(pbuf + kConsumerWarps * kN);               // one per stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(hdr + kStages);                   // full, empty, qfree[2]
  int* misc = reinterpret_cast<int*>(bars + 2 * kStages + 2);                    // 96 ints
  int* sF = misc + 96;                                                           // [B + 1]
  int* plist = sF + kPersistMaxSeqs + 1;                                         // [B]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const int B = p.num_seqs;
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  const uint32_t qfree0 = empty0 + 8 * kStages;

  // ---- item tables ----
  // Warps 0..7 each take a slice of 64 sequences (two rounds of 32 lanes),
  // the context lengths held in registers. Pass 1 counts whole chunks and
  // partial chunks per size class; pass 2 writes each sequence's whole-chunk
  // prefix into sF and each partial chunk's sequence into plist, at its
  // class's place. Rows with a bad length count as padding (no items); the
  // producer warp writes the zeros of padding rows (rows b with b % G == cta)
  // and initialises the barriers meanwhile.
  static_assert(kPersistMaxSeqs == kConsumerWarps * 64, "two 32-lane rounds per slice");
  int* cnt = misc + 32;  // [8 warps][8 classes]
  int ctxv[2] = {0, 0};
  auto size_class = [](int ctx) -> int {
    const int part = ctx & (kBlockSize - 1);
    return part ? (kBuckets - 1) - (part >> 5) : -1;
  };
  if (warp < kConsumerWarps) {
    int full = 0;
    int mycnt = 0;  // lane k < 8: partial chunks of class k in this slice
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int b = warp * 64 + r * 32 + lane;
      int ctx = b < B ? p.context_lens[b] : 0;
      if (ctx < 0 || ctx > p.max_ctx || ctx > p.bt_stride * kBlockSize) {
        if (b % G == cta) flag_error(p.err, PKV_DEVERR_BAD_SEQLEN);
        ctx = 0;
      }
      ctxv[r] = ctx;
      full += ctx >> 8;
      const int cl = size_class(ctx);
#pragma unroll
      for (int k = 0; k < kBuckets; ++k) {
        const int c = __popc(__ballot_sync(0xffffffffu, cl == k));
        if (lane == k) mycnt += c;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) full += __shfl_xor_sync(0xffffffffu, full, off);
    if (lane == 0) misc[16 + warp] = full;
    if (lane < kBuckets) cnt[warp * kBuckets + lane] = mycnt;
  } else {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(full0 + 8 * s, 1);
        mbar_init(empty0 + 8 * s, kConsumerWarps);
      }
      mbar_init(qfree0, kConsumerWarps);
      mbar_init(qfree0 + 8, kConsumerWarps);
      mbar_fence_init();
    }
    for (int b = cta; b < B; b += G) {
      const int ctx = p.context_lens[b];
      if (ctx <= 0 || ctx > p.max_ctx || ctx > p.bt_stride * kBlockSize) {
        uint4* o = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(b) * kHq * kHeadDim);
        for (int i = lane; i < kHq * kHeadDim / 8; i += 32) o[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  __syncthreads();
  if (warp < kConsumerWarps) {
    int run = 0, n_full_all = 0;
    for (int w = 0; w < kConsumerWarps; ++w) {
      const int f = misc[16 + w];
      if (w < warp) run += f;
      n_full_all += f;
    }
    // lane k < 8: where this slice's class-k partial chunks go in plist
    int cbase = 0, n_part_all = 0;
    for (int k = 0; k < kBuckets; ++k) {
      int tot = 0, before = 0;
      for (int w = 0; w < kConsumerWarps; ++w) {
        const int c = cnt[w * kBuckets + k];
        tot += c;
        if (w < warp) before += c;
      }
      if (k < lane) cbase += tot;
      if (k == lane) cbase += before;
      n_part_all += tot;
    }
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int b = warp * 64 + r * 32 + lane;
      const int nf = ctxv[r] >> 8;
      int x = nf;  // inclusive scan over the round
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (b < B) sF[b] = run + x - nf;
      run += __shfl_sync(0xffffffffu, x, 31);
      const int cl = size_class(ctxv[r]);
#pragma unroll
      for (int k = 0; k < kBuckets; ++k) {
        const uint32_t m = __ballot_sync(0xffffffffu, cl == k);
        const int base_k = __shfl_sync(0xffffffffu, cbase, k);
        if (cl == k) plist[base_k + __popc(m & below)] = b;
        if (lane == k) cbase += __popc(m);
      }
    }
    if (tid == 0) {
      sF[B] = n_full_all;
      misc[1] = n_full_all;               // whole chunks
      misc[2] = n_full_all + n_part_all;  // all items
    }
  }
  __syncthreads();
  const int n_full = misc[1];
  const int n_items = misc[2];

  if (warp == kConsumerWarps) {
    // ---------------- producer warp: lane 0 streams every item's chunk ----------------
    struct Item {
      int b, c, nch, ntok, pb;
      bool valid, bad;
    };
    // the next item of the list, first come first served (lane 0)
    int* work = p.tickets + B;
    auto fetch = [&]() -> Item {
      Item it{};
      const int idx = atomicAdd(work, 1);
      it.valid = idx < n_items;
      if (!it.valid) return it;
      if (idx < n_full) {
        int lo = 0, hi = B;  // largest b with sF[b] <= idx (sF non-decreasing)
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (sF[mid] <= idx) lo = mid; else hi = mid;
        }
        it.b = lo;
        it.c = idx - sF[lo];
      } else {
        it.b = plist[idx - n_full];
        it.c = sF[it.b + 1] - sF[it.b];  // the partial chunk follows the whole ones
      }
      const int ctx = p.context_lens[it.b];
      it.nch = (ctx + kBlockSize - 1) / kBlockSize;
      it.ntok = min(kBlockSize, ctx - it.c * kBlockSize);
      it.pb = p.block_tables[static_cast<int64_t>(it.b) * p.bt_stride + it.c];
      it.bad = it.pb < 0 || it.pb >= p.num_blocks;
      if (it.bad) flag_error(p.err, PKV_DEVERR_BAD_BLOCK);
      return it;
    };
    int st = 0;      // stages posted (lane 0)
    int nit = 0;     // items started
    bool ok = true;
    Item cur{};
    if (lane == 0) cur = fetch();
    while (true) {
      if (!__shfl_sync(0xffffffffu, static_cast<int>(cur.valid), 0)) {
        if (lane == 0) {
          // end of work: a header-only stage
          const int s = st % kStages;
          if (st < kStages || mbar_wait(empty0 + 8 * s, ((st / kStages) - 1) & 1, p.err)) {
            hdr[s] = make_int4(-1, 0, 4, 0);
            mbar_arrive(full0 + 8 * s);
            ++st;
          }
        }
        break;
      }
      const int qs = nit & 1;
      int64_t store_slot = -1;  // fused store: the new row's slot, or -1
      if (lane == 0) {
        if (nit >= 2) ok = mbar_wait(qfree0 + 8 * qs, ((nit >> 1) - 1) & 1, p.err);
        if (p.k_new != nullptr && cur.c == cur.nch - 1 && !cur.bad) {
          const int64_t slot = p.slot_mapping[cur.b];
          if (slot != -1) {
            const int ctx = p.context_lens[cur.b];
            if (slot != static_cast<int64_t>(cur.pb) * kBlockSize + (ctx - 1) % kBlockSize)
              flag_error(p.err, PKV_DEVERR_BAD_SLOT);
            else
              store_slot = slot;
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, static_cast<int>(ok), 0)) break;
      store_slot = __shfl_sync(0xffffffffu, store_slot, 0);
      if (store_slot >= 0) {
        // fused store: the new token's K/V row reaches its slot before the
        // block is streamed; the warp copies 128 bytes per lane, loads first
        const int b = __shfl_sync(0xffffffffu, cur.b, 0);
        const uint4* ks = p.k_new + b * p.k_new_stride16;
        const uint4* vs = p.v_new + b * p.v_new_stride16;
        uint4 kr[kRowBytes / 16 / 32], vr[kRowBytes / 16 / 32];
#pragma unroll
        for (int j = 0; j < kRowBytes / 16 / 32; ++j) {
          kr[j] = ks[lane + 32 * j];
          vr[j] = vs[lane + 32 * j];
        }
        uint4* kd = p.k_cache_w + store_slot * (kRowBytes / 16);
        uint4* vd = p.v_cache_w + store_slot * (kRowBytes / 16);
#pragma unroll
        for (int j = 0; j < kRowBytes / 16 / 32; ++j) {
          kd[lane + 32 * j] = kr[j];
          vd[lane + 32 * j] = vr[j];
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) {
        const int niter = cur.bad ? 1 : (cur.ntok + kT - 1) / kT;
        const int64_t base = (static_cast<int64_t>(cur.pb) * kBlockSize) * kRowBytes;
        Item nxt{};
        for (int it = 0; it < niter; ++it) {
          const int s = st % kStages;
          if (st >= kStages && !(ok = mbar_wait(empty0 + 8 * s, ((st / kStages) - 1) & 1, p.err))) break;
          const int rows = cur.bad ? 0 : min(kT, cur.ntok - it * kT);
          const int flags = (it == 0 ? 1 : 0) | (it == niter - 1 ? 2 : 0) | (qs << 4);
          hdr[s] = make_int4(cur.b, rows, flags, (cur.c << 16) | cur.nch);
          const uint32_t bytes = 2u * rows * kRowBytes + (it == 0 ? kQRowBytes : 0u);
          const uint32_t dst = smem0 + s * kStageBytes;
          mbar_arrive_expect_tx(full0 + 8 * s, bytes);
          if (it == 0)
            bulk_g2s(smem_u32(qbuf) + qs * kQRowBytes, p.q + static_cast<int64_t>(cur.b) * p.q_row_stride,
                     kQRowBytes, full0 + 8 * s);
          if (rows > 0) {
            const int64_t off = base + static_cast<int64_t>(it) * kT * kRowBytes;
            bulk_g2s(dst, p.k_cache + off, rows * kRowBytes, full0 + 8 * s);
            bulk_g2s(dst + kT * kRowBytes, p.v_cache + off, rows * kRowBytes, full0 + 8 * s);
          }
          ++st;
          if (it == 0) nxt = fetch();  // the next item's lookups overlap this item's copies
        }
        cur = nxt;
      }
      if (!__shfl_sync(0xffffffffu, static_cast<int>(ok), 0)) break;
      ++nit;
    }
    if (lane == 0) {
      // Never leave a copy in flight into this CTA's shared memory.
      for (int i = max(0, st - kStages); i < st; ++i) mbar_wait(full0 + 8 * (i % kStages), (i / kStages) & 1, p.err);
      // This CTA takes no more items; the last CTA to get here resets the
      // counters for the next call (every CTA's last fetch came before).
      __threadfence();
      if (atomicAdd(work + 1, 1) == G - 1) {
        work[0] = 0;
        work[1] = 0;
      }
    }
    return;
  }

  // ---------------- consumers: warp h = kv head h, query heads 2h, 2h+1 ----------------
  const int h = warp;
  const int idx = lane >> (5 - kLog2N);
  const int my_t = idx % kT;
  const bool owner = (lane & ((1 << (5 - kLog2N)) - 1)) == 0;
  const bool my_g1 = lane >= 16;
  float* wp = pbuf + warp * kN;
  const uint32_t wp_addr = smem_u32(wp);
  float q0[4], q1[4];
  float o0[4], o1[4];
  float m0 = -INFINITY, m1 = -INFINITY, lsum = 0.f;
  int* s_last = misc;
  for (int st = 0;; ++st) {
    const int s = st % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (st / kStages) & 1, p.err))) break;
    const int4 hd = hdr[s];
    if (hd.z & 4) break;
    const int b = hd.x, rows = hd.y;
    if (hd.z & 1) {
      // a new item: this warp's two query rows from the q buffer, scaled to log2 units
      const uint16_t* qrow = reinterpret_cast<const uint16_t*>(qbuf + ((hd.z >> 4) & 1) * kQRowBytes);
      const uint2 a = *reinterpret_cast<const uint2*>(qrow + (kGroup * h) * kHeadDim + lane * 4);
      const uint2 bq = *reinterpret_cast<const uint2*>(qrow + (kGroup * h + 1) * kHeadDim + lane * 4);
      q0[0] = Ops::lo(a.x) * p.scale_log2;
      q0[1] = Ops::hi(a.x) * p.scale_log2;
      q0[2] = Ops::lo(a.y) * p.scale_log2;
      q0[3] = Ops::hi(a.y) * p.scale_log2;
      q1[0] = Ops::lo(bq.x) * p.scale_log2;
      q1[1] = Ops::hi(bq.x) * p.scale_log2;
      q1[2] = Ops::lo(bq.y) * p.scale_log2;
      q1[3] = Ops::hi(bq.y) * p.scale_log2;
      __syncwarp();
      if (lane == 0) mbar_arrive(qfree0 + 8 * ((hd.z >> 4) & 1));
#pragma unroll
      for (int i = 0; i < 4; ++i) o0[i] = o1[i] = 0.f;
      m0 = m1 = -INFINITY;
      lsum = 0.f;
    }
    const uint32_t kaddr = smem0 + s * kStageBytes + h * (kHeadDim * 2) + lane * 8;
    const uint32_t vaddr = kaddr + kT * kRowBytes;
    if (rows > 0) {
      float part[kN];
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        const uint2 kr = lds64(kaddr + t * kRowBytes);
        const float k0 = Ops::lo(kr.x), k1 = Ops::hi(kr.x);
        const float k2 = Ops::lo(kr.y), k3 = Ops::hi(kr.y);
        part[t] = fmaf(q0[0], k0, fmaf(q0[1], k1, fmaf(q0[2], k2, q0[3] * k3)));
        part[kT + t] = fmaf(q1[0], k0, fmaf(q1[1], k1, fmaf(q1[2], k2, q1[3] * k3)));
      }
      float sc = transpose_reduce<kN>(part, lane);
      if (my_t >= rows) sc = -INFINITY;
      float mx = sc;
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mx0 = __shfl_sync(0xffffffffu, mx, 0);
      const float mx1 = __shfl_sync(0xffffffffu, mx, 16);
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float a0 = ex2_approx(m0 - mu0), a1 = ex2_approx(m1 - mu1);
      const float pv = ex2_approx(sc - (my_g1 ? mu1 : mu0));
      lsum = lsum * (my_g1 ? a1 : a0) + (owner ? pv : 0.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o0[i] *= a0;
        o1[i] *= a1;
      }
      m0 = mn0;
      m1 = mn1;
      if (owner) wp[idx] = pv;
      __syncwarp();
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        if (t < rows) {
          float w0, w1;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(w0) : "r"(wp_addr + 4 * t));
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(w1) : "r"(wp_addr + 4 * (kT + t)));
          const uint2 vr = lds64(vaddr + t * kRowBytes);
          const float v0 = Ops::lo(vr.x), v1 = Ops::hi(vr.x);
          const float v2 = Ops::lo(vr.y), v3 = Ops::hi(vr.y);
          o0[0] = fmaf(w0, v0, o0[0]);
          o0[1] = fmaf(w0, v1, o0[1]);
          o0[2] = fmaf(w0, v2, o0[2]);
          o0[3] = fmaf(w0, v3, o0[3]);
          o1[0] = fmaf(w1, v0, o1[0]);
          o1[1] = fmaf(w1, v1, o1[1]);
          o1[2] = fmaf(w1, v2, o1[2]);
          o1[3] = fmaf(w1, v3, o1[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (!(hd.z & 2)) continue;
    // ---- the item's last stage: its (m, l, o) ----
    const int c = hd.w >> 16, nch = hd.w & 0xffff;
    float l = lsum;
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const float l0 = __shfl_sync(0xffffffffu, l, 0);
    const float l1 = __shfl_sync(0xffffffffu, l, 16);
    if (nch == 1) {
      const float r0 = l0 > 0.f ? 1.f / l0 : 0.f, r1 = l1 > 0.f ? 1.f / l1 : 0.f;
      uint16_t* orow = p.out + static_cast<int64_t>(b) * kHq * kHeadDim;
      uint2 w;
      w.x = Ops::pack(o0[0] * r0, o0[1] * r0);
      w.y = Ops::pack(o0[2] * r0, o0[3] * r0);
      *reinterpret_cast<uint2*>(orow + (kGroup * h) * kHeadDim + lane * 4) = w;
      w.x = Ops::pack(o1[0] * r1, o1[1] * r1);
      w.y = Ops::pack(o1[2] * r1, o1[3] * r1);
      *reinterpret_cast<uint2*>(orow + (kGroup * h + 1) * kHeadDim + lane * 4) = w;
      continue;
    }
    const int64_t pslot = (static_cast<int64_t>(b) * p.nsplit + c) * kHq + kGroup * h;
    *reinterpret_cast<float4*>(p.opart + pslot * kHeadDim + lane * 4) = make_float4(o0[0], o0[1], o0[2], o0[3]);
    *reinterpret_cast<float4*>(p.opart + (pslot + 1) * kHeadDim + lane * 4) = make_float4(o1[0], o1[1], o1[2], o1[3]);
    if (lane == 0) {
      p.ml[pslot] = make_float2(m0, l0);
      p.ml[pslot + 1] = make_float2(m1, l1);
    }
    // split-KV merge by whichever CTA finishes the sequence's last chunk
    named_sync_consumers();
    if (tid == 0) {
      __threadfence();
      const int prev = atomicAdd(p.tickets + b, 1);
      *s_last = (prev == nch - 1) ? 1 : 0;
    }
    named_sync_consumers();
    if (*s_last == 0) continue;
    __threadfence();
    merge_partials<E>(p, b, nch, tid >> 4, (tid & 15) * 8);
    if (tid == 0) p.tickets[b] = 0;  // ready for the next call
  }
}

constexpr int kDecT = PKV_DECODE_TOKENS_PER_STAGE;
constexpr int kDecStages = PKV_DECODE_STAGES;

constexpr size_t decode_smem_bytes() {
  return static_cast<size_t>(kDecStages) * 2 * kDecT * kRowBytes + kConsumerWarps * 2 * kDecT * sizeof(float) +
         2 * kDecStages * sizeof(uint64_t) + 16;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t persistent_smem_bytes() {
  return static_cast<size_t>(kDecStages) * 2 * kDecT * kRowBytes + 2 * kQRowBytes +
         kConsumerWarps * 2 * kDecT * sizeof(float) + kDecStages * sizeof(int4) + (2 * kDecStages + 2) * sizeof(uint64_t) +
         96 * sizeof(int) + (2 * kPersistMaxSeqs + 1) * sizeof(int);
}
static_assert(2 * (persistent_smem_bytes() + 1024) <= 228 * 1024, "two persistent decode CTAs must fit an SM");

template <Elem E>
cudaError_t launch_typed(const DecodeParams& p, int32_t num_seqs, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<E, kDecT, kDecStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(decode_smem_bytes()));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_persistent_kernel<E, kDecT, kDecStages>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(persistent_smem_bytes()));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  if (p.chunk == kBlockSize && num_seqs <= kPersistMaxSeqs) {
    // whole-block chunks: two CTAs per SM walk the live items
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    decode_persistent_kernel<E, kDecT, kDecStages><<<2 * sms, kThreads, persistent_smem_bytes(), stream>>>(p);
    return cudaGetLastError();
  }
  const dim3 grid(p.nsplit, num_seqs);
  decode_split_kernel<E, kDecT, kDecStages><<<grid, kThreads, decode_smem_bytes(), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Tokens per CTA for these sizes: the largest of 256, 128, 64, 32 that still
// gives at least kMinCtas CTAs (two resident per SM, about two waves on a
// 152-SM GB300), else 32. A function of the call's sizes only, so the
// workspace query and the launch always agree.
constexpr int kMinCtas = 608;
int decode_chunk(int32_t num_seqs, int32_t max_context_len) {
  int chunk = kBlockSize;
  while (chunk > 32 && static_cast<int64_t>(num_seqs) * ((max_context_len + chunk - 1) / chunk) < kMinCtas) chunk >>= 1;
  return chunk;
}

int decode_num_splits(int32_t num_seqs, int32_t max_context_len) {
  const int chunk = decode_chunk(num_seqs, max_context_len);
  return (max_context_len + chunk - 1) / chunk;
}

// Workspace: per-sequence tickets and two work counters (zero between calls),
// then the split-KV partials.
size_t decode_counter_bytes(int32_t num_seqs) {
  return align_up((static_cast<size_t>(num_seqs) + 2) * sizeof(int32_t), 256);
}

size_t decode_workspace_bytes(int32_t num_seqs, int32_t max_context_len) {
  const size_t ns = static_cast<size_t>(num_seqs);
  const size_t nsplit = static_cast<size_t>(decode_num_splits(num_seqs, max_context_len));
  return decode_counter_bytes(num_seqs) + align_up(ns * nsplit * kHq * sizeof(float2), 256) +
         ns * nsplit * kHq * kHeadDim * sizeof(float);
}

cudaError_t launch_decode(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
                          int32_t num_blocks, const int32_t* block_tables, int32_t bt_stride,
                          const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len, float scale,
                          void* out, void* workspace, unsigned int* err, cudaStream_t stream,
                          const FusedStore* fused, Elem elem) {
  if (num_seqs == 0) return cudaSuccess;
  DecodeParams p;
  p.k_new = fused ? static_cast<const uint4*>(fused->k) : nullptr;
  p.v_new = fused ? static_cast<const uint4*>(fused->v) : nullptr;
  p.k_new_stride16 = fused ? fused->k_row_stride / 8 : 0;
  p.v_new_stride16 = fused ? fused->v_row_stride / 8 : 0;
  p.slot_mapping = fused ? fused->slot_mapping : nullptr;
  p.k_cache_w = static_cast<uint4*>(const_cast<void*>(k_cache));
  p.v_cache_w = static_cast<uint4*>(const_cast<void*>(v_cache));
  p.q = static_cast<const uint16_t*>(q);
  p.q_row_stride = q_row_stride;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.num_blocks = num_blocks;
  p.block_tables = block_tables;
  p.bt_stride = bt_stride;
  p.context_lens = context_lens;
  p.max_ctx = max_context_len;
  p.num_seqs = num_seqs;
  p.chunk = decode_chunk(num_seqs, max_context_len);
  p.nsplit = decode_num_splits(num_seqs, max_context_len);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = static_cast<uint16_t*>(out);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t ns = static_cast<size_t>(num_seqs);
  p.tickets = reinterpret_cast<int32_t*>(ws);
  ws += decode_counter_bytes(num_seqs);
  p.ml = reinterpret_cast<float2*>(ws);
  ws += align_up(ns * p.nsplit * kHq * sizeof(float2), 256);
  p.opart = reinterpret_cast<float*>(ws);
  p.err = err;
  if (p.nsplit == 0) p.nsplit = 1;
  return elem == Elem::kF16 ? launch_typed<Elem::kF16>(p, num_seqs, stream)
                            : launch_typed<Elem::kBF16>(p, num_seqs, stream);
}

}  // namespace pkv
