// prefill.cu -- causal variable-length prefill attention on tcgen05 tensor cores.
//
// The operation is the flash_attn_varlen_func(..., causal=True, block_table)
// call of layers/attention.py in "vLLM 学习笔记 02：nano-vllm 源码逐段精读":
// query row i of sequence b sits at position Lk_b - Lq_b + i and attends to
// keys 0..that position, keys taken either from contiguous k/v or, on a
// prefix-cache hit, from the paged cache through block_tables.
//
// GB300 design. One CTA computes a 128-row query tile of one sequence for the
// two query heads that share kv head hk (GQA group of 2), so every K/V tile
// it loads feeds two 128x128x128 products of each kind:
//   warp 0      TMA producer: Q tiles once, then K_n, V_n (128 keys x 128
//               dims, two 64-dim boxes with 128-byte swizzle) into a 3-slot
//               ring. In paged mode tile n's row coordinate is
//               block_tables[b][n/2]*256 + (n%2)*128 -- a 128-key tile never
//               straddles a 256-token block, so one tensor map covers the pool.
//   warp 1      allocates 512 TMEM columns and one lane issues every
//               tcgen05.mma: S_g = Q_g K_n^T into TMEM, then O_g += P_g V_n.
//   warps 2-5   softmax for query head 2hk   (thread = TMEM lane = query row)
//   warps 6-9   softmax for query head 2hk+1
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
// Issue order per key tile n:  PV_0(n), S_0(n+1), PV_1(n), S_1(n+1), so
// while one softmax group works the tensor core runs the other group's
// products. Each tcgen05.commit covers every earlier product of the issuing
// thread, so "S_g(n+1) complete" also means PV_g(n) is complete: the softmax
// group may then rescale O_g in TMEM and overwrite its P_g buffer.
// Softmax keeps a per-row running max in log2 units and only moves it when it
// grows by more than 8 (2^8 headroom in fp32/bf16), so O is rescaled rarely.
// The last V tile's rows beyond the sequence are zeroed in shared memory
// before use, so stale or NaN cache contents never reach the product.
// The producer also warms L2 with the Q tiles of the CTA one wave ahead.
// Epilogue: O is staged in the (then free) P buffers and leaves as whole
// 512-byte rows (both heads of a query row); warp 1 releases TMEM once every
// softmax warp has staged its rows. There is no CTA-wide barrier at the end,
// so no role ever waits at one with lanes still busy in their role.
// The element type (bf16 or fp16) is a template parameter: it sets the
// tensor-core operand format, the tensor maps' element type and how P and
// the output are rounded; P <= 2^8 fits either type.
#include <cuda.h>

#include "pkv_common.cuh"

namespace pkv {

namespace {

constexpr int kHkv = 8;
constexpr int kGroup = 2;
constexpr int kHq = kHkv * kGroup;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kTileBytes = 128 * kHeadDim * 2;  // 32 KB
constexpr int kHalfBytes = kTileBytes / 2;      // 16 KB: 128 rows x 64 dims
constexpr int kKvSlots = 3;
constexpr int kThreads = 320;

constexpr int kOffQ = 0;                                // 2 tiles
constexpr int kOffP = 2 * kTileBytes;                   // 2 tiles
constexpr int kOffKV = 4 * kTileBytes;                  // kKvSlots tiles
constexpr int kOffBar = kOffKV + kKvSlots * kTileBytes;  // barriers
// barrier indices
constexpr int kBarQ = 0;
constexpr int kBarKvFull = 1;                   // +slot
constexpr int kBarKvFree = kBarKvFull + kKvSlots;
constexpr int kBarSFull = kBarKvFree + kKvSlots;  // +g
constexpr int kBarPReady = kBarSFull + 2;         // +g
constexpr int kBarOFinal = kBarPReady + 2;
constexpr int kBarVTail = kBarOFinal + 1;
constexpr int kBarDrain = kBarVTail + 1;
constexpr int kBarStaged = kBarDrain + 1;          // the 8 softmax warps have staged their O rows
constexpr int kNumBars = kBarStaged + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem address, abort flag
constexpr size_t kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory above the 227 KB a CTA can opt into");

struct PrefillParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_tables;
  int32_t bt_stride;
  int32_t num_blocks;
  int32_t num_seqs;
  int32_t max_q_tiles;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  int32_t total_q;
  int32_t total_k;  // rows of contiguous k/v (ignored when paged)
  int32_t paged;
  float scale_log2;
  int32_t ahead;  // block index distance to the CTA likely to run next on this SM (the SM count)
  const int32_t* items;  // optional tile plan: (qt << 16) | b per item, CTA = 8 * item + hk; NULL: all pairs
  uint16_t* out;  // 16-bit elements of the call's type
  unsigned int* err;
};

// Bounded wait that also gives up as soon as another role of the CTA has
// aborted (so one lost arrival costs one time-out, not one per wait).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      flag_error(err, PKV_DEVERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// 8-column TMEM load / store (32 lanes x 8 x 32 bit), for the rare O rescale
// while the tile's 128 probabilities are still held in registers.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
// keeps uses of a tmem_ld8 result after the tcgen05.wait::ld that completes it
__device__ __forceinline__ void tmem_reg_fence8(uint32_t (&r)[8]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <Elem E>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using Ops = ElemOps<E>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzle atoms.
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (query tile, sequence, kv head), longest tiles first ----
  // Without a plan the grid covers every (query tile, sequence) pair, query
  // tiles in descending order; with one, CTA 8i + hk takes the plan's item i.
  const int per_tile = p.num_seqs * kHkv;
  auto item_of = [&](int cta, int& qt_, int& b_, int& hk_) {
    hk_ = cta % kHkv;
    if (p.items) {
      const int code = p.items[cta / kHkv];
      qt_ = code >> 16;
      b_ = code & 0xffff;
    } else {
      qt_ = p.max_q_tiles - 1 - cta / per_tile;
      b_ = (cta % per_tile) / kHkv;
    }
  };
  int qt, b, hk;
  item_of(static_cast<int>(blockIdx.x), qt, b, hk);
  if (b >= p.num_seqs || qt < 0) {  // a plan for other cu_seqlens: skip the item
    if (threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_BAD_SEQLEN);
    return;
  }

  const int cq0 = p.cu_q[b], cq1 = p.cu_q[b + 1];
  const int ck0 = p.cu_k[b], ck1 = p.cu_k[b + 1];
  const int Lq = cq1 - cq0, Lk = ck1 - ck0;
  const bool bad = Lq < 0 || Lk < Lq || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k || cq0 < 0 ||
                   cq1 > p.total_q || (p.paged ? (Lk > p.bt_stride * kBlockSize) : (ck0 < 0 || ck1 > p.total_k));
  if (bad) {
    if (threadIdx.x == 0 && qt == 0 && hk == 0) flag_error(p.err, PKV_DEVERR_BAD_SEQLEN);
    return;
  }
  const int r0 = qt * kBM;
  if (r0 >= Lq) return;
  const int rows_valid = min(kBM, Lq - r0);
  const int pos0 = Lk - Lq + r0;                 // position of the tile's first query row
  const int last_pos = pos0 + rows_valid - 1;
  const int n_tiles = last_pos / kBN + 1;
  const int tail_keys = Lk - (n_tiles - 1) * kBN;  // valid keys in the last tile (1..128)
  const bool v_tail = tail_keys < kBN;

  auto k_row = [&](int n) -> int {
    if (!p.paged) return ck0 + n * kBN;
    int blk = p.block_tables[static_cast<int64_t>(b) * p.bt_stride + (n * kBN) / kBlockSize];
    if (blk < 0 || blk >= p.num_blocks) {
      flag_error(p.err, PKV_DEVERR_BAD_BLOCK);
      blk = 0;
    }
    return blk * kBlockSize + (n * kBN) % kBlockSize;
  };
  // ring item i: K_{i/2} (even i) or V_{i/2} (odd i), into slot i % kKvSlots
  auto load_kv = [&](int i) {
    const int slot = i % kKvSlots;
    const CUtensorMap* tm = (i & 1) ? &tm_v : &tm_k;
    const int row = k_row(i >> 1);
    const uint32_t dst = sbase + kOffKV + slot * kTileBytes;
    mbar_arrive_expect_tx(bar(kBarKvFull + slot), kTileBytes);
    tma_load_3d(dst, tm, 0, hk, row, bar(kBarKvFull + slot));
    tma_load_3d(dst + kHalfBytes, tm, 64, hk, row, bar(kBarKvFull + slot));
  };

  // Thread 0 is the producer's issuing lane: right after initialising the
  // barriers it starts the Q loads and fills the K/V ring, before the TMEM
  // allocation and the CTA barrier, so the copies are in flight sooner.
  int early = 0;  // ring items issued here (thread 0 only)
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), (i == kBarPReady || i == kBarPReady + 1) ? 4 : (i == kBarStaged ? 8 : 1));
    *s_abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    mbar_arrive_expect_tx(bar(kBarQ), 2 * kTileBytes);
    for (int g = 0; g < kGroup; ++g) {
      const uint32_t dst = sbase + kOffQ + g * kTileBytes;
      tma_load_3d(dst, &tm_q, 0, kGroup * hk + g, cq0 + r0, bar(kBarQ));
      tma_load_3d(dst + kHalfBytes, &tm_q, 64, kGroup * hk + g, cq0 + r0, bar(kBarQ));
    }
    for (; early < kKvSlots && early < 2 * n_tiles; ++early) load_kv(early);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();  // warp 0 arrives converged, after thread 0 has initialised the barriers
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // =========================== TMA producer ===========================
    int issued = early;
    if (lane == 0) {
      for (int i = early; i < 2 * n_tiles; ++i) {
        const int slot = i % kKvSlots;
        if (i >= kKvSlots && !wait_or_abort(bar(kBarKvFree + slot), ((i / kKvSlots) - 1) & 1, s_abort, p.err))
          break;
        load_kv(i);
        ++issued;
      }
    }
    if (lane == 0) {
      // Warm L2 with the Q tiles of the CTA launched a wave after this one:
      // Q is read once, so its first load would otherwise come from HBM (its
      // K/V tiles are shared with the sequence's other query tiles and are
      // usually in L2 already).
      const int nb = static_cast<int>(blockIdx.x) + p.ahead;
      if (nb < static_cast<int>(gridDim.x)) {
        int qt2, b2, hk2;
        item_of(nb, qt2, b2, hk2);
        const int q0 = b2 < p.num_seqs ? p.cu_q[b2] : 0, q1 = b2 < p.num_seqs ? p.cu_q[b2 + 1] : 0;
        if (qt2 * kBM < q1 - q0) {
          for (int g = 0; g < kGroup; ++g) {
            tma_prefetch_l2_3d(&tm_q, 0, kGroup * hk2 + g, q0 + qt2 * kBM);
            tma_prefetch_l2_3d(&tm_q, 64, kGroup * hk2 + g, q0 + qt2 * kBM);
          }
        }
      }
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);
    if (v_tail && issued == 2 * n_tiles) {
      // Zero the rows of the last V tile that lie past the sequence end.
      const int i = 2 * n_tiles - 1;
      const int slot = i % kKvSlots;
      const bool ok = wait_or_abort(bar(kBarKvFull + slot), (i / kKvSlots) & 1, s_abort, p.err);
      if (ok) {
        const uint32_t base = sbase + kOffKV + slot * kTileBytes;
        // rows tail_keys..127 of both 64-dim halves: 128-byte rows, swizzle
        // only permutes 16-byte chunks within a row.
        const int nz = (kBN - tail_keys) * 2 * 8;  // 16-byte chunks
        for (int c = lane; c < nz; c += 32) {
          const int row = tail_keys + (c >> 4);
          const int half = (c >> 3) & 1;
          const int chunk = c & 7;
          sts128(base + half * kHalfBytes + row * 128 + chunk * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarVTail));
    }
    if (lane == 0) {
      // Never leave a copy in flight into this CTA's shared memory.
      mbar_wait(bar(kBarQ), 0, p.err);
      for (int i = max(0, issued - kKvSlots); i < issued; ++i)
        mbar_wait(bar(kBarKvFull + i % kKvSlots), (i / kKvSlots) & 1, p.err);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16kind_f32(kBM, kBN, false, false, Ops::kMmaFormat);
      constexpr uint32_t idesc_pv = idesc_f16kind_f32(kBM, kHeadDim, false, true, Ops::kMmaFormat);
      bool ok = wait_or_abort(bar(kBarQ), 0, s_abort, p.err);
      auto slot_of = [](int i) { return i % kKvSlots; };
      auto par_of = [](int i) { return static_cast<uint32_t>((i / kKvSlots) & 1); };
      // Descriptor low halves: each product below costs two 32-bit adds and
      // the tcgen05.mma (this one thread issues every product of the CTA).
      const uint32_t lo_kmaj = desc_lo(sbase, 16), lo_v = desc_lo(sbase, kHalfBytes);
      auto issue_s = [&](int g, int n) {
        const uint32_t qa = lo_kmaj + ((kOffQ + g * kTileBytes) >> 4);
        const uint32_t kbb = lo_kmaj + (kOffKV >> 4) + slot_of(2 * n) * (kTileBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
          mma_f16kind_lo(tmem + g * 128, qa + off, kbb + off, idesc_s, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int g, int n) {
        const uint32_t pa = lo_kmaj + ((kOffP + g * kTileBytes) >> 4);
        const uint32_t vbb = lo_v + (kOffKV >> 4) + slot_of(2 * n + 1) * (kTileBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint32_t aoff = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
          mma_f16kind_lo(tmem + 256 + g * 128, pa + aoff, vbb + ((ks * 16 * 128) >> 4), idesc_pv,
                         (n > 0 || ks > 0) ? 1u : 0u);
        }
      };
      if (ok) ok = wait_or_abort(bar(kBarKvFull + slot_of(0)), par_of(0), s_abort, p.err);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        mma_commit(bar(kBarSFull + 0));
        issue_s(1, 0);
        mma_commit(bar(kBarSFull + 1));
        mma_commit(bar(kBarKvFree + slot_of(0)));
      }
      for (int n = 0; ok && n < n_tiles; ++n) {
        const int iv = 2 * n + 1;
        if (n == n_tiles - 1 && v_tail)
          ok = wait_or_abort(bar(kBarVTail), 0, s_abort, p.err);
        else
          ok = wait_or_abort(bar(kBarKvFull + slot_of(iv)), par_of(iv), s_abort, p.err);
        if (!ok) break;
        if (!(ok = wait_or_abort(bar(kBarPReady + 0), n & 1, s_abort, p.err))) break;
        tc_fence_after();
        issue_pv(0, n);
        const bool more = n + 1 < n_tiles;
        if (more) {
          if (!(ok = wait_or_abort(bar(kBarKvFull + slot_of(2 * n + 2)), par_of(2 * n + 2), s_abort, p.err)))
            break;
          tc_fence_after();
          issue_s(0, n + 1);
          mma_commit(bar(kBarSFull + 0));
        }
        if (!(ok = wait_or_abort(bar(kBarPReady + 1), n & 1, s_abort, p.err))) break;
        tc_fence_after();
        issue_pv(1, n);
        mma_commit(bar(kBarKvFree + slot_of(iv)));
        if (more) {
          issue_s(1, n + 1);
          mma_commit(bar(kBarSFull + 1));
          mma_commit(bar(kBarKvFree + slot_of(2 * n + 2)));
        }
      }
      mma_commit(bar(kBarOFinal));
      if (!ok) {
        // make sure no product is still writing TMEM before it is released
        mma_commit(bar(kBarDrain));
        mbar_wait(bar(kBarDrain), 0, p.err);
      }
    }
  } else {
    // =========================== softmax groups ===========================
    const int g = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // query row within the tile == TMEM lane
    const int pos = pos0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + g * 128;
    const uint32_t tO = tmem + lane_base + 256 + g * 128;
    const uint32_t prow = sbase + kOffP + g * kTileBytes + row * 128;
    const int swz = row & 7;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max, log2 units (scaled)
    float l = 0.f;
    bool ok = true;
    for (int n = 0; n < n_tiles; ++n) {
      // every lane waits (each needs the acquire); the warp then agrees, so
      // the warp-collective tensor-memory loads below run on all 32 lanes
      ok = wait_or_abort(bar(kBarSFull + g), n & 1, s_abort, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_wait_ld();
        tmem_reg_fence(r0);
        tmem_reg_fence(r1);
        tmem_reg_fence(r2);
        tmem_reg_fence(r3);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          s[j] = __uint_as_float(r0[j]);
          s[32 + j] = __uint_as_float(r1[j]);
          s[64 + j] = __uint_as_float(r2[j]);
          s[96 + j] = __uint_as_float(r3[j]);
        }
      }
      const int key0 = n * kBN;
      if (key0 + kBN - 1 > pos0 || key0 + kBN > Lk) {
        const int lim = min(pos, Lk - 1) - key0;  // keys j <= lim are visible
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j > lim) s[j] = -INFINITY;
      }
      // Row max, row sum and the exponent arguments use the 3-input max and the
      // packed fp32x2 instructions: the softmax warps issue about a third fewer
      // instructions per tile, and the tile's softmax is issue-limited.
      float ma = s[0], mb = s[1];
#pragma unroll
      for (int j = 2; j < 126; j += 4) {
        ma = fmax3(ma, s[j], s[j + 1]);
        mb = fmax3(mb, s[j + 2], s[j + 3]);
      }
      float mx = fmaxf(fmax3(ma, s[126], s[127]), mb);
      mx *= sl2;
      float m_use = m;
      if (mx > m + 8.0f) m_use = mx;  // move the max only when it grows by > 2^8
      const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_use);
      l *= alpha;
      // P = 2^(s*sl2 - m_use), rounded to the element type, into the swizzled K-major A tile
      const uint64_t sl2x2 = f32x2_pack(sl2, sl2);
      const uint64_t negm2 = f32x2_pack(-m_use, -m_use);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
#pragma unroll
        for (int j = c * 8; j < c * 8 + 8; j += 2) {
          float a0, a1;
          f32x2_unpack(f32x2_fma(f32x2_pack(s[j], s[j + 1]), sl2x2, negm2), a0, a1);
          s[j] = ex2_approx(a0);
          s[j + 1] = ex2_approx(a1);
        }
        const int half = c >> 3;
        const uint32_t addr = prow + half * kHalfBytes + (((c & 7) ^ swz) << 4);
        const float* e = s + c * 8;
        sts128(addr, Ops::pack(e[0], e[1]), Ops::pack(e[2], e[3]), Ops::pack(e[4], e[5]), Ops::pack(e[6], e[7]));
      }
      m = m_use;
      // rescale the running output (PV_g(n-1) is complete: S_g(n) was issued after it)
      if (n > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
        for (int c = 0; c < 16; ++c) {
          uint32_t r[8];
          tmem_ld8(tO + c * 8, r);
          tmem_wait_ld();
          tmem_reg_fence8(r);
#pragma unroll
          for (int j = 0; j < 8; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          tmem_st8(tO + c * 8, r);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPReady + g));
      // The row sum is not needed for P: add it up after P is handed over.
      {
        uint64_t acc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = f32x2_pack(s[2 * a], s[2 * a + 1]);
#pragma unroll
        for (int j = 8; j < 128; j += 8)
#pragma unroll
          for (int a = 0; a < 4; ++a) acc[a] = f32x2_add(acc[a], f32x2_pack(s[j + 2 * a], s[j + 2 * a + 1]));
        float t0, t1, t2, t3, t4, t5, t6, t7;
        f32x2_unpack(acc[0], t0, t1);
        f32x2_unpack(acc[1], t2, t3);
        f32x2_unpack(acc[2], t4, t5);
        f32x2_unpack(acc[3], t6, t7);
        l += ((t0 + t1) + (t2 + t3)) + ((t4 + t5) + (t6 + t7));
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(bar(kBarOFinal), 0, s_abort, p.err));
    // Epilogue. Every product is complete, so the two P buffers (64 KB) are
    // free: each thread stages its normalised O row there (the two query heads
    // of a row side by side, 512 B, 16-byte chunks rotated by the row to spread
    // the banks), then each warp stores whole rows: the two heads of a query
    // row are adjacent in out, so one warp instruction writes 512 contiguous
    // bytes instead of touching 32 rows.
    const uint32_t stage = sbase + kOffP;
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + c * 32, r);
        tmem_wait_ld();
        tmem_reg_fence(r);
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          const int q = g * 16 + c * 4 + j / 8;  // 16-byte chunk of the 512-byte row
          sts128(stage + row * 512 + ((q ^ (row & 31)) << 4),
                 Ops::pack(__uint_as_float(r[j + 0]) * inv, __uint_as_float(r[j + 1]) * inv),
                 Ops::pack(__uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv),
                 Ops::pack(__uint_as_float(r[j + 4]) * inv, __uint_as_float(r[j + 5]) * inv),
                 Ops::pack(__uint_as_float(r[j + 6]) * inv, __uint_as_float(r[j + 7]) * inv));
        }
      }
    }
    // all 8 softmax warps arrive, whatever happened, so the wait below (and
    // warp 1's before releasing TMEM) always ends; every tensor-memory read of
    // this warp is complete here
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarStaged));
    const bool staged = __all_sync(0xffffffffu, wait_or_abort(bar(kBarStaged), 0, s_abort, p.err));
    if (ok && staged) {
      uint16_t* obase = p.out + (static_cast<int64_t>(cq0 + r0) * kHq + kGroup * hk) * kHeadDim + lane * 8;
      for (int rr = warp - 2; rr < rows_valid; rr += 8) {
        uint32_t a, b2, c2, d;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a), "=r"(b2), "=r"(c2), "=r"(d)
                     : "r"(stage + rr * 512 + ((lane ^ (rr & 31)) << 4)));
        *reinterpret_cast<uint4*>(obase + static_cast<int64_t>(rr) * kHq * kHeadDim) = make_uint4(a, b2, c2, d);
      }
    }
  }

  if (warp == 1) {
    // TMEM is released after every softmax warp's last tensor-memory read
    // (they all arrive on kBarStaged once O is staged); no CTA-wide barrier,
    // so no role waits at one with some of its lanes still busy. The wait is
    // time-bounded but ignores the abort flag: the softmax warps always arrive.
    __syncwarp();
    mbar_wait(bar(kBarStaged), 0, p.err);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [rows, heads, 128] view of 16-bit elements with rows row_stride_elems apart;
// box = 128 rows x 1 head x 64 dims.
bool encode_rows_heads_dims(CUtensorMap* tm, const void* base, int64_t rows, int heads, int64_t row_stride_elems,
                            Elem elem) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2),
                                 static_cast<cuuint64_t>(row_stride_elems * 2)};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = elem == Elem::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return enc(tm, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <Elem E>
cudaError_t launch_typed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                         unsigned nblocks, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  prefill_tc_kernel<E><<<nblocks, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_workspace_bytes(int32_t, int32_t, int32_t) { return 0; }

// prefill_persistent.cu: the same units walked by one CTA per SM (tile plan given).
cudaError_t launch_prefill_persistent(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                      const int32_t* cu_q, const int32_t* cu_k, const int32_t* block_tables,
                                      int32_t bt_stride, int32_t num_blocks, int32_t num_seqs, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, int32_t total_q, int32_t total_k, bool paged,
                                      float scale, const int32_t* items, int32_t num_items, void* out,
                                      unsigned int* err, cudaStream_t stream, Elem elem);

// Which kernel runs a planned call. The persistent kernel hides each unit's
// fixed costs (about 4 us: set-up, first loads, pipeline ramp, epilogue)
// behind its neighbours' tiles, but its steady key tile measured a few per
// cent slower on GB300, and with fewer units than two per SM there is little
// to overlap. So it takes calls with at least two units per SM whose key
// ranges are at most 4096 tokens (32 key tiles per unit at most): measured
// +7% on 16k-token calls of 100..1024-token prompts and +8% on 128 prompts
// behind a 1024-token cached prefix, while 5,000-token chunks on up to 7,000
// cached tokens ran 2-8% faster one CTA per unit.
bool use_persistent(int32_t num_items, int32_t max_seqlen_k, int sms) {
  return static_cast<int64_t>(num_items) * kHkv >= 2 * static_cast<int64_t>(sms) && max_seqlen_k <= 4096;
}

cudaError_t launch_prefill(const void* q, int64_t q_row_stride, int32_t total_q, const void* k, const void* v,
                           int64_t kv_row_stride, int32_t total_k, const void* k_cache, const void* v_cache,
                           int32_t num_blocks, const int32_t* cu_q, const int32_t* cu_k, int32_t max_seqlen_q,
                           int32_t max_seqlen_k, const int32_t* block_tables, int32_t bt_stride, int32_t num_seqs,
                           float scale, const int32_t* items, int32_t num_items, void* out, unsigned int* err,
                           cudaStream_t stream, Elem elem) {
  if (num_seqs == 0 || max_seqlen_q == 0 || total_q == 0) return cudaSuccess;
  CUtensorMap tq, tk, tv;
  const bool paged = block_tables != nullptr;
  if (!encode_rows_heads_dims(&tq, q, total_q, kHq, q_row_stride, elem)) return cudaErrorInvalidValue;
  if (paged) {
    const int64_t slots = static_cast<int64_t>(num_blocks) * kBlockSize;
    if (!encode_rows_heads_dims(&tk, k_cache, slots, kHkv, kHkv * kHeadDim, elem) ||
        !encode_rows_heads_dims(&tv, v_cache, slots, kHkv, kHkv * kHeadDim, elem))
      return cudaErrorInvalidValue;
  } else {
    if (total_k == 0) return cudaErrorInvalidValue;
    if (!encode_rows_heads_dims(&tk, k, total_k, kHkv, kv_row_stride, elem) ||
        !encode_rows_heads_dims(&tv, v, total_k, kHkv, kv_row_stride, elem))
      return cudaErrorInvalidValue;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
  if (items && num_items > 0 && use_persistent(num_items, max_seqlen_k, sms))
    return launch_prefill_persistent(tq, tk, tv, cu_q, cu_k, block_tables, bt_stride, num_blocks, num_seqs,
                                     max_seqlen_q, max_seqlen_k, total_q, total_k, paged, scale, items, num_items,
                                     out, err, stream, elem);
  PrefillParams p;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.block_tables = block_tables;
  p.bt_stride = bt_stride;
  p.num_blocks = num_blocks;
  p.num_seqs = num_seqs;
  p.max_q_tiles = (max_seqlen_q + kBM - 1) / kBM;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_k = max_seqlen_k;
  p.total_q = total_q;
  p.total_k = paged ? 0 : total_k;
  p.paged = paged ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.ahead = sms;
  p.items = num_items > 0 ? items : nullptr;
  p.out = static_cast<uint16_t*>(out);
  p.err = err;
  const int64_t nblocks = p.items ? static_cast<int64_t>(num_items) * kHkv
                                  : static_cast<int64_t>(p.max_q_tiles) * num_seqs * kHkv;
  if (nblocks > 0x7fffffff) return cudaErrorInvalidValue;
  const unsigned nb = static_cast<unsigned>(nblocks);
  return elem == Elem::kF16 ? launch_typed<Elem::kF16>(tq, tk, tv, p, nb, stream)
                            : launch_typed<Elem::kBF16>(tq, tk, tv, p, nb, stream);
}

}  // namespace pkv
