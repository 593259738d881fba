// prefill_persistent.cu -- causal varlen prefill attention, persistent form.
//
// Same operation and the same per-tile arithmetic as prefill_tc_kernel
// (prefill.cu): the flash_attn_varlen_func(..., causal=True, block_table) call
// of layers/attention.py in "vLLM 学习笔记 02：nano-vllm 源码逐段精读".
// A work unit is (128-row query tile, sequence, kv head) with the two query
// heads of the kv head; its output is bit-identical to the one-CTA-per-unit
// kernel's.
//
// Why persistent. On short prompts (100..1024 tokens) a unit has only 1..8
// key tiles, and a CTA that computes one unit spends about as long on its
// fixed costs (launch, barrier set-up, TMEM allocation, the first Q and K/V
// loads, the pipeline ramp, the epilogue) as on its tiles: shared memory
// (224 KB) allows one such CTA per SM, so nothing hides them. Here one CTA per
// SM walks a list of units and overlaps each unit's start with the previous
// unit's end:
//   * TMEM (512 columns) and the barriers are set up once per CTA;
//   * the K/V ring runs on across units (ring slot and phase counters never
//     reset), so the producer streams the next unit's tiles while the current
//     one finishes;
//   * the next unit's Q is loaded as soon as the last S products of the
//     current unit have read Q, after an L2 prefetch issued one unit ahead;
//   * the MMA thread issues the next unit's first S products right after the
//     current unit's last P.V products, while the softmax warps run the
//     epilogue; each softmax group hands its O columns back (o_free) as soon
//     as it has read them, and the next unit's first P.V product of that group
//     (which overwrites O) waits only for that.
// Units come from the host tile plan (pkv_prefill_plan: (query tile,
// sequence) items, most key tiles first), expanded into 8 kv heads each.
// CTA c takes units c, 2G-1-c, 2G+c, 4G-1-c, ... of the list (a snake over
// rounds of G = gridDim.x units), which on the plan's longest-first order
// balances the SMs as well as first-come dynamic scheduling would, with no
// shared counter to reset between calls.
// The producer warp decodes units (validity checks, lengths, tile counts) and
// posts them through a 4-slot descriptor ring to the MMA thread and the
// softmax warps; units that hold no rows are skipped there and never posted.
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
constexpr int kDescSlots = 4;
constexpr int kThreads = 320;

constexpr int kOffQ = 0;                                 // 2 tiles
constexpr int kOffP = 2 * kTileBytes;                    // 2 tiles (P, and O staging in the epilogue)
constexpr int kOffKV = 4 * kTileBytes;                   // kKvSlots tiles
constexpr int kOffBar = kOffKV + kKvSlots * kTileBytes;  // barriers
// barrier indices
constexpr int kBarQFull = 0;
constexpr int kBarQFree = 1;
constexpr int kBarKvFull = 2;                       // +slot
constexpr int kBarKvFree = kBarKvFull + kKvSlots;   // +slot
constexpr int kBarSFull = kBarKvFree + kKvSlots;    // +g
constexpr int kBarPReady = kBarSFull + 2;           // +g, 4 warps
constexpr int kBarOFinal = kBarPReady + 2;          // +g
constexpr int kBarOFree = kBarOFinal + 2;           // +g, 4 warps
constexpr int kBarVTail = kBarOFree + 2;           // +ring slot: that slot's V tile had its tail rows zeroed
constexpr int kBarDescFull = kBarVTail + kKvSlots;  // +slot
constexpr int kBarDescFree = kBarDescFull + kDescSlots;  // +slot, MMA lane + 8 softmax warps
constexpr int kBarDone = kBarDescFree + kDescSlots;      // 8 softmax warps: TMEM no longer read
constexpr int kBarDrain = kBarDone + 1;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kDescWords = 12;
constexpr int kOffDesc = kOffBar + kNumBars * 8;
constexpr int kOffMisc = kOffDesc + kDescSlots * kDescWords * 4;  // tmem address, abort flag
constexpr size_t kSmemBytes = kOffMisc + 16 + 1024;               // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory above the 227 KB a CTA can opt into");

// Descriptor words (int32), written by the producer lane, read by the others.
enum : int {
  kDValid = 0,  // 1: a unit, -1: no more units
  kDB,
  kDHk,
  kDCq0,
  kDR0,
  kDRows,
  kDPos0,
  kDLk,
  kDTiles,
  kDTail,
  kDCk0,
};

struct PersistParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_tables;
  int32_t bt_stride;
  int32_t num_blocks;
  int32_t num_seqs;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  int32_t total_q;
  int32_t total_k;  // rows of contiguous k/v (ignored when paged)
  int32_t paged;
  float scale_log2;
  const int32_t* items;  // tile plan: (qt << 16) | b per item
  int32_t num_units;     // 8 * number of plan items
  uint16_t* out;
  unsigned int* err;
};

struct Unit {
  int valid;  // 1 unit with rows, 0 skip, -1 end of list
  int b, hk, cq0, ck0, r0, rows, pos0, Lk, n_tiles, tail;
};

// Bounded wait that also gives up as soon as another role of the CTA has aborted.
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

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
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
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, int v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Unit k of this CTA in the snake order over rounds of G units.
__device__ __forceinline__ int unit_index(int k, int cta, int G) {
  return k * G + ((k & 1) ? (G - 1 - cta) : cta);
}

// Decode unit u of the list (one thread). Units without rows are skipped
// (valid 0); a plan entry naming a sequence the call lacks, or inconsistent
// lengths, flag PKV_DEVERR_BAD_SEQLEN and are skipped.
__device__ __forceinline__ Unit decode_unit(const PersistParams& p, int u) {
  Unit x{};
  if (u >= p.num_units) {
    x.valid = -1;
    return x;
  }
  x.valid = 0;
  x.hk = u % kHkv;
  const int code = p.items[u / kHkv];
  const int qt = code >> 16;
  x.b = code & 0xffff;
  if (x.b >= p.num_seqs || qt < 0) {
    if (x.hk == 0) flag_error(p.err, PKV_DEVERR_BAD_SEQLEN);
    return x;
  }
  const int cq0 = p.cu_q[x.b], cq1 = p.cu_q[x.b + 1];
  const int ck0 = p.cu_k[x.b], ck1 = p.cu_k[x.b + 1];
  const int Lq = cq1 - cq0, Lk = ck1 - ck0;
  const bool bad = Lq < 0 || Lk < Lq || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k || cq0 < 0 || cq1 > p.total_q ||
                   (p.paged ? (Lk > p.bt_stride * kBlockSize) : (ck0 < 0 || ck1 > p.total_k));
  if (bad) {
    if (qt == 0 && x.hk == 0) flag_error(p.err, PKV_DEVERR_BAD_SEQLEN);
    return x;
  }
  x.r0 = qt * kBM;
  if (x.r0 >= Lq) return x;
  x.valid = 1;
  x.cq0 = cq0;
  x.ck0 = ck0;
  x.Lk = Lk;
  x.rows = min(kBM, Lq - x.r0);
  x.pos0 = Lk - Lq + x.r0;
  x.n_tiles = (x.pos0 + x.rows - 1) / kBN + 1;
  x.tail = Lk - (x.n_tiles - 1) * kBN;  // valid keys in the last tile (1..128)
  return x;
}

// The producer lane decodes units until one holds rows (or the list ends).
__device__ __forceinline__ Unit next_unit(const PersistParams& p, int& k, int cta, int G) {
  while (true) {
    Unit x = decode_unit(p, unit_index(k, cta, G));
    ++k;
    if (x.valid != 0) return x;
  }
}

// Once-per-unit steps of the roles.

// Read posted descriptor d (every lane of the caller waits for it); valid =
// -2 when the CTA aborted while waiting. Plain loads from a warp-uniform
// address, so the values are known uniform.
__device__ __forceinline__ Unit read_unit(uint32_t full_bar, uint32_t parity, const int* w, volatile int* abort_flag,
                                       unsigned int* err) {
  Unit x{};
  if (!wait_or_abort(full_bar, parity, abort_flag, err)) {
    x.valid = -2;
    return x;
  }
  x.valid = w[kDValid];
  x.b = w[kDB];
  x.hk = w[kDHk];
  x.cq0 = w[kDCq0];
  x.r0 = w[kDR0];
  x.rows = w[kDRows];
  x.pos0 = w[kDPos0];
  x.Lk = w[kDLk];
  x.n_tiles = w[kDTiles];
  x.tail = w[kDTail];
  x.ck0 = w[kDCk0];
  return x;
}

// Post a descriptor into its slot (one thread), after the slot's previous
// occupant was released; false once the CTA aborts.
__device__ __forceinline__ bool post_unit(const Unit& x, int posted, uint32_t desc0, uint32_t full_bar0,
                                       uint32_t free_bar0, volatile int* abort_flag, unsigned int* err) {
  const int slot = posted % kDescSlots;
  if (posted >= kDescSlots &&
      !wait_or_abort(free_bar0 + 8u * slot, ((posted / kDescSlots) - 1) & 1, abort_flag, err))
    return false;
  const uint32_t a = desc0 + slot * kDescWords * 4;
  sts32(a + 4 * kDValid, x.valid);
  sts32(a + 4 * kDB, x.b);
  sts32(a + 4 * kDHk, x.hk);
  sts32(a + 4 * kDCq0, x.cq0);
  sts32(a + 4 * kDR0, x.r0);
  sts32(a + 4 * kDRows, x.rows);
  sts32(a + 4 * kDPos0, x.pos0);
  sts32(a + 4 * kDLk, x.Lk);
  sts32(a + 4 * kDTiles, x.n_tiles);
  sts32(a + 4 * kDTail, x.tail);
  sts32(a + 4 * kDCk0, x.ck0);
  mbar_arrive(full_bar0 + 8u * slot);
  return true;
}

// Softmax-warp epilogue of one unit (whole warp): read this thread's O row
// from TMEM 32 columns at a time, hand O_g back once its last columns are
// read, stage the normalised row in the thread's P row (P's swizzled layout:
// dims 0..63 in the first half, 64..127 in the second), then store the warp's
// 32 rows, two 256-byte rows per instruction.
template <Elem E>
__device__ __forceinline__ void store_unit_rows(uint32_t tO, uint32_t prow, uint32_t pbase, int quad, int lane, float l,
                                             uint32_t o_free_bar, uint16_t* obase, int rows) {
  using Ops = ElemOps<E>;
  const int swz = (quad * 32 + lane) & 7;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(tO + c * 32, r);
    tmem_wait_ld();
    tmem_reg_fence(r);
    if (c == 3) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free_bar);  // the next unit's first P.V may overwrite O_g
    }
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      const int chunk = c * 4 + j / 8;  // 16-byte chunk (8 dims) of the 256-byte row
      const uint32_t addr = prow + (chunk >> 3) * kHalfBytes + (((chunk & 7) ^ swz) << 4);
      sts128(addr, Ops::pack(__uint_as_float(r[j + 0]) * inv, __uint_as_float(r[j + 1]) * inv),
             Ops::pack(__uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv),
             Ops::pack(__uint_as_float(r[j + 4]) * inv, __uint_as_float(r[j + 5]) * inv),
             Ops::pack(__uint_as_float(r[j + 6]) * inv, __uint_as_float(r[j + 7]) * inv));
    }
  }
  __syncwarp();
  const int ch = lane & 15;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int rr = quad * 32 + 2 * i + (lane >> 4);
    const uint4 v = lds128(pbase + (ch >> 3) * kHalfBytes + rr * 128 + (((ch & 7) ^ (rr & 7)) << 4));
    if (rr < rows) *reinterpret_cast<uint4*>(obase + static_cast<int64_t>(rr) * kHq * kHeadDim + ch * 8) = v;
  }
  __syncwarp();
}

template <Elem E>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, const PersistParams p) {
  using Ops = ElemOps<E>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;  // 1024-byte alignment for the swizzle atoms
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x);
  const int G = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;
      if (i == kBarPReady || i == kBarPReady + 1 || i == kBarOFree || i == kBarOFree + 1) count = 4;
      if (i >= kBarDescFree && i < kBarDescFree + kDescSlots) count = 9;
      if (i == kBarDone) count = 8;
      mbar_init(bar(i), count);
    }
    *s_abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  const uint32_t desc0 = sbase + kOffDesc;
  auto issue_q = [&](const Unit& x) {
    mbar_arrive_expect_tx(bar(kBarQFull), 2 * kTileBytes);
    for (int g = 0; g < kGroup; ++g) {
      const uint32_t dst = sbase + kOffQ + g * kTileBytes;
      tma_load_3d(dst, &tm_q, 0, kGroup * x.hk + g, x.cq0 + x.r0, bar(kBarQFull));
      tma_load_3d(dst + kHalfBytes, &tm_q, 64, kGroup * x.hk + g, x.cq0 + x.r0, bar(kBarQFull));
    }
  };
  // ring item i of unit x (K_{i/2} for even i, V_{i/2} for odd i) into ring slot `slot`
  auto issue_kv = [&](const Unit& x, int i, int slot) {
    const int n = i >> 1;
    int row;
    if (p.paged) {
      int blk = p.block_tables[static_cast<int64_t>(x.b) * p.bt_stride + (n * kBN) / kBlockSize];
      if (blk < 0 || blk >= p.num_blocks) {
        flag_error(p.err, PKV_DEVERR_BAD_BLOCK);
        blk = 0;
      }
      row = blk * kBlockSize + (n * kBN) % kBlockSize;
    } else {
      row = x.ck0 + n * kBN;
    }
    const CUtensorMap* tm = (i & 1) ? &tm_v : &tm_k;
    const uint32_t dst = sbase + kOffKV + slot * kTileBytes;
    mbar_arrive_expect_tx(bar(kBarKvFull + slot), kTileBytes);
    tma_load_3d(dst, tm, 0, x.hk, row, bar(kBarKvFull + slot));
    tma_load_3d(dst + kHalfBytes, tm, 64, x.hk, row, bar(kBarKvFull + slot));
  };
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // Posted descriptor d lives in slot d % kDescSlots; every reader waits for
  // it, copies it and arrives on the slot's free barrier.
  auto read_desc = [&](int d) -> Unit {
    const int slot = d % kDescSlots;
    return read_unit(bar(kBarDescFull + slot), (d / kDescSlots) & 1,
                     reinterpret_cast<const int*>(smem + kOffDesc) + slot * kDescWords, s_abort, p.err);
  };

  if (warp == 0) {
    // =========================== TMA producer ===========================
    // Lane 0 decodes units, posts descriptors and issues every copy; the
    // whole warp zeroes the rows of a unit's last V tile past the sequence.
    int k = 0;        // next list position to decode (lane 0)
    int posted = 0;   // descriptors posted
    int ri = 0;       // K/V ring items issued (K_n, V_n alternate), across units
    int nq = 0;       // Q loads issued (one per posted unit)
    bool ok = true;
    Unit cur{};
    // post a descriptor (lane 0); false once the CTA aborts
    auto post = [&](const Unit& x) -> bool {
      return post_unit(x, posted++, desc0, bar(kBarDescFull), bar(kBarDescFree), s_abort, p.err);
    };
    if (lane == 0) {
      cur = next_unit(p, k, cta, G);
      ok = post(cur);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    while (ok && __shfl_sync(0xffffffffu, cur.valid, 0) > 0) {
      Unit nxt{};
      if (lane == 0) {
        // Q of this unit, both query heads, once the previous unit's last S
        // products have read the Q buffers
        if (nq > 0) ok = wait_or_abort(bar(kBarQFree), (nq - 1) & 1, s_abort, p.err);
        if (ok) {
          issue_q(cur);
          ++nq;
        }
        // The next unit is decoded (global loads), its Q warmed in L2 and its
        // descriptor posted (the MMA thread looks one unit ahead) at the first
        // point where the producer would otherwise block on a ring slot, or
        // after this unit's copies are all issued.
        bool have_nxt = false;
        auto take_next = [&]() {
          nxt = next_unit(p, k, cta, G);
          if (nxt.valid > 0) {
            for (int g = 0; g < kGroup; ++g) {
              tma_prefetch_l2_3d(&tm_q, 0, kGroup * nxt.hk + g, nxt.cq0 + nxt.r0);
              tma_prefetch_l2_3d(&tm_q, 64, kGroup * nxt.hk + g, nxt.cq0 + nxt.r0);
            }
          }
          have_nxt = true;
          return post(nxt);
        };
        // K_n, V_n of this unit through the ring
        for (int i = 0; ok && i < 2 * cur.n_tiles; ++i) {
          const int slot = ri % kKvSlots;
          if (ri >= kKvSlots) {
            const uint32_t par = ((ri / kKvSlots) - 1) & 1;
            if (!have_nxt && !mbar_try_wait(bar(kBarKvFree + slot), par) && !(ok = take_next())) break;
            if (!(ok = wait_or_abort(bar(kBarKvFree + slot), par, s_abort, p.err))) break;
          }
          issue_kv(cur, i, slot);
          ++ri;
        }
        if (ok && !have_nxt) ok = take_next();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ri = __shfl_sync(0xffffffffu, ri, 0);
      const int tail = __shfl_sync(0xffffffffu, cur.tail, 0);
      if (!ok) break;
      if (tail < kBN) {
        // Zero the rows of this unit's last V tile that lie past the sequence
        // end (stale or NaN cache rows must not meet the zero probabilities).
        const int i = ri - 1;  // ring item of V_{n_tiles-1}
        const int slot = i % kKvSlots;
        if (lane == 0) ok = wait_or_abort(bar(kBarKvFull + slot), (i / kKvSlots) & 1, s_abort, p.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t base = sbase + kOffKV + slot * kTileBytes;
        const int nz = (kBN - tail) * 2 * 8;  // 16-byte chunks in both 64-dim halves
        for (int c = lane; c < nz; c += 32) {
          const int row = tail + (c >> 4);
          const int half = (c >> 3) & 1;
          const int chunk = c & 7;
          sts128(base + half * kHalfBytes + row * 128 + chunk * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarVTail + slot));
      }
      if (lane == 0) cur = nxt;
    }
    if (lane == 0) {
      // Never leave a copy in flight into this CTA's shared memory.
      if (nq > 0) mbar_wait(bar(kBarQFull), (nq - 1) & 1, p.err);
      for (int i = max(0, ri - kKvSlots); i < ri; ++i)
        mbar_wait(bar(kBarKvFull + i % kKvSlots), (i / kKvSlots) & 1, p.err);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16kind_f32(kBM, kBN, false, false, Ops::kMmaFormat);
      constexpr uint32_t idesc_pv = idesc_f16kind_f32(kBM, kHeadDim, false, true, Ops::kMmaFormat);
      // Descriptor low halves: each product below costs two 32-bit adds and
      // the tcgen05.mma (this one thread issues every product of the CTA).
      const uint32_t lo_kmaj = desc_lo(sbase, 16), lo_v = desc_lo(sbase, kHalfBytes);
      auto issue_s = [&](int g, uint32_t kslot) {
        const uint32_t qa = lo_kmaj + ((kOffQ + g * kTileBytes) >> 4);
        const uint32_t kbb = lo_kmaj + (kOffKV >> 4) + kslot * (kTileBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
          mma_f16kind_lo(tmem + g * 128, qa + off, kbb + off, idesc_s, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int g, uint32_t vslot, bool first) {
        const uint32_t pa = lo_kmaj + ((kOffP + g * kTileBytes) >> 4);
        const uint32_t vbb = lo_v + (kOffKV >> 4) + vslot * (kTileBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint32_t aoff = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
          mma_f16kind_lo(tmem + 256 + g * 128, pa + aoff, vbb + ((ks * 16 * 128) >> 4), idesc_pv,
                         (!first || ks > 0) ? 1u : 0u);
        }
      };
      int d = 0;    // descriptors read
      int rc = 0;   // ring item of the current tile's K (V is rc + 1)
      int t = 0;    // tiles across units (S / P phases)
      int nu = 0;   // units started (Q, O phases)
      uint32_t vt_par = 0;  // bit s: parity of the next V-tail phase of ring slot s
      bool ok = true;
      Unit cur = read_desc(d++);
      ok = cur.valid != -2;
      if (ok) mbar_arrive(bar(kBarDescFree + (d - 1) % kDescSlots));
      if (ok && cur.valid > 0) {
        ok = wait_or_abort(bar(kBarQFull), 0, s_abort, p.err);
        if (ok) ok = wait_or_abort(bar(kBarKvFull + rc % kKvSlots), (rc / kKvSlots) & 1, s_abort, p.err);
        if (ok) {
          tc_fence_after();
          issue_s(0, rc % kKvSlots);
          mma_commit(bar(kBarSFull + 0));
          issue_s(1, rc % kKvSlots);
          mma_commit(bar(kBarSFull + 1));
          mma_commit(bar(kBarKvFree + rc % kKvSlots));
          if (cur.n_tiles == 1) mma_commit(bar(kBarQFree));
        }
        // Invariant at the top of each unit: its S_0(0), S_1(0) are issued.
        // Tiles 0..N-2 run the per-unit kernel's body unchanged; only the
        // last tile carries the hand-over to the next unit.
        int N = cur.n_tiles, tail = cur.tail;
        while (ok) {
          for (int n = 0; n < N - 1; ++n) {
            const int rv = rc + 1, rk = rc + 2;
            if (!(ok = wait_or_abort(bar(kBarKvFull + rv % kKvSlots), (rv / kKvSlots) & 1, s_abort, p.err))) break;
            if (!(ok = wait_or_abort(bar(kBarPReady + 0), t & 1, s_abort, p.err))) break;
            if (n == 0 && nu > 0 && !(ok = wait_or_abort(bar(kBarOFree + 0), (nu - 1) & 1, s_abort, p.err)))
              break;
            tc_fence_after();
            issue_pv(0, rv % kKvSlots, n == 0);
            if (!(ok = wait_or_abort(bar(kBarKvFull + rk % kKvSlots), (rk / kKvSlots) & 1, s_abort, p.err))) break;
            tc_fence_after();
            issue_s(0, rk % kKvSlots);
            mma_commit(bar(kBarSFull + 0));
            if (!(ok = wait_or_abort(bar(kBarPReady + 1), t & 1, s_abort, p.err))) break;
            if (n == 0 && nu > 0 && !(ok = wait_or_abort(bar(kBarOFree + 1), (nu - 1) & 1, s_abort, p.err)))
              break;
            tc_fence_after();
            issue_pv(1, rv % kKvSlots, n == 0);
            mma_commit(bar(kBarKvFree + rv % kKvSlots));
            issue_s(1, rk % kKvSlots);
            mma_commit(bar(kBarSFull + 1));
            mma_commit(bar(kBarKvFree + rk % kKvSlots));
            if (n + 1 == N - 1) mma_commit(bar(kBarQFree));  // the last S products reading this Q
            ++t;
            rc = rk;
          }
          if (!ok) break;
          // ---- the unit's last tile, then tile 0 of the next unit ----
          const int rv = rc + 1, rk = rc + 2;
          const bool first = N == 1;
          if (tail < kBN)
            ok = wait_or_abort(bar(kBarVTail + rv % kKvSlots), (vt_par >> (rv % kKvSlots)) & 1u, s_abort, p.err);
          else
            ok = wait_or_abort(bar(kBarKvFull + rv % kKvSlots), (rv / kKvSlots) & 1, s_abort, p.err);
          if (!ok) break;
          if (!(ok = wait_or_abort(bar(kBarPReady + 0), t & 1, s_abort, p.err))) break;
          if (first && nu > 0 && !(ok = wait_or_abort(bar(kBarOFree + 0), (nu - 1) & 1, s_abort, p.err))) break;
          tc_fence_after();
          issue_pv(0, rv % kKvSlots, first);
          mma_commit(bar(kBarOFinal + 0));
          // Both groups' last P.V go before the next unit's S products: the
          // epilogues start as early as possible, and the next unit's Q and
          // K_0, still in flight, hold up no product of this unit.
          if (!(ok = wait_or_abort(bar(kBarPReady + 1), t & 1, s_abort, p.err))) break;
          if (first && nu > 0 && !(ok = wait_or_abort(bar(kBarOFree + 1), (nu - 1) & 1, s_abort, p.err))) break;
          tc_fence_after();
          issue_pv(1, rv % kKvSlots, first);
          mma_commit(bar(kBarKvFree + rv % kKvSlots));
          mma_commit(bar(kBarOFinal + 1));
          const Unit nxt = read_desc(d++);
          if (!(ok = nxt.valid != -2)) break;
          mbar_arrive(bar(kBarDescFree + (d - 1) % kDescSlots));
          const bool more = nxt.valid > 0;
          if (more) {
            if (!(ok = wait_or_abort(bar(kBarQFull), (nu + 1) & 1, s_abort, p.err))) break;
            if (!(ok = wait_or_abort(bar(kBarKvFull + rk % kKvSlots), (rk / kKvSlots) & 1, s_abort, p.err))) break;
            tc_fence_after();
            issue_s(0, rk % kKvSlots);
            mma_commit(bar(kBarSFull + 0));
            issue_s(1, rk % kKvSlots);
            mma_commit(bar(kBarSFull + 1));
            mma_commit(bar(kBarKvFree + rk % kKvSlots));
            if (nxt.n_tiles == 1) mma_commit(bar(kBarQFree));
          }
          ++t;
          if (tail < kBN) vt_par ^= 1u << (rv % kKvSlots);
          if (!more) break;
          ++nu;
          N = nxt.n_tiles;
          tail = nxt.tail;
          rc = rk;
        }
      }
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
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + g * 128;
    const uint32_t tO = tmem + lane_base + 256 + g * 128;
    const uint32_t pbase = sbase + kOffP + g * kTileBytes;
    const uint32_t prow = pbase + row * 128;
    const int swz = row & 7;
    const float sl2 = p.scale_log2;
    int d = 0, t = 0, nu = 0;
    bool ok = true;
    while (true) {
      // Only what the tile loop needs is read now; the epilogue reads the
      // output placement from the same slot, which is released after it.
      const int dslot = d % kDescSlots;
      ok = __all_sync(0xffffffffu, wait_or_abort(bar(kBarDescFull + dslot), (d / kDescSlots) & 1, s_abort, p.err));
      ++d;
      if (!ok) break;
      const int* dw = reinterpret_cast<const int*>(smem + kOffDesc) + dslot * kDescWords;
      Unit u{};
      u.valid = dw[kDValid];
      if (u.valid < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarDescFree + dslot));
        break;
      }
      u.n_tiles = dw[kDTiles];
      u.pos0 = dw[kDPos0];
      u.Lk = dw[kDLk];
      const int pos = u.pos0 + row;
      float m = -INFINITY;  // running max, log2 units (scaled)
      float l = 0.f;
      for (int n = 0; n < u.n_tiles; ++n, ++t) {
        ok = wait_or_abort(bar(kBarSFull + g), t & 1, s_abort, p.err);
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
        if (key0 + kBN - 1 > u.pos0 || key0 + kBN > u.Lk) {
          const int lim = min(pos, u.Lk - 1) - key0;  // keys j <= lim are visible
#pragma unroll
          for (int j = 0; j < 128; ++j)
            if (j > lim) s[j] = -INFINITY;
        }
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
          sts128(addr, Ops::pack(e[0], e[1]), Ops::pack(e[2], e[3]), Ops::pack(e[4], e[5]),
                 Ops::pack(e[6], e[7]));
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
      if (!ok) break;
      // ---- epilogue: read O_g, hand its columns back, stage, store ----
      ok = __all_sync(0xffffffffu, wait_or_abort(bar(kBarOFinal + g), nu & 1, s_abort, p.err));
      if (!ok) break;
      tc_fence_after();
      {
        const int cq0 = dw[kDCq0], r0 = dw[kDR0], hk = dw[kDHk], rows = dw[kDRows];
        uint16_t* obase = p.out + (static_cast<int64_t>(cq0 + r0) * kHq + kGroup * hk + g) * kHeadDim;
        store_unit_rows<E>(tO, prow, pbase, quad, lane, l, bar(kBarOFree + g), obase, rows);
      }
      if (lane == 0) mbar_arrive(bar(kBarDescFree + dslot));
      ++nu;
    }
    // every softmax warp arrives, whatever happened, so warp 1's wait ends
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarDone));
  }

  if (warp == 1) {
    // TMEM is released after every softmax warp's last tensor-memory access.
    __syncwarp();
    mbar_wait(bar(kBarDone), 0, p.err);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <Elem E>
cudaError_t launch_typed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PersistParams& p,
                         unsigned nblocks, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_persistent_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  prefill_persistent_kernel<E><<<nblocks, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

// Launch over the units of a tile plan (num_items plan items, 8 units each),
// one CTA per SM at most. Tensor maps as prefill.cu encodes them.
cudaError_t launch_prefill_persistent(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                      const int32_t* cu_q, const int32_t* cu_k, const int32_t* block_tables,
                                      int32_t bt_stride, int32_t num_blocks, int32_t num_seqs, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, int32_t total_q, int32_t total_k, bool paged,
                                      float scale, const int32_t* items, int32_t num_items, void* out,
                                      unsigned int* err, cudaStream_t stream, Elem elem) {
  if (num_items <= 0) return cudaSuccess;
  if (static_cast<int64_t>(num_items) * kHkv > 0x7fffffff) return cudaErrorInvalidValue;
  PersistParams p;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.block_tables = block_tables;
  p.bt_stride = bt_stride;
  p.num_blocks = num_blocks;
  p.num_seqs = num_seqs;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_k = max_seqlen_k;
  p.total_q = total_q;
  p.total_k = paged ? 0 : total_k;
  p.paged = paged ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.items = items;
  p.num_units = num_items * kHkv;
  p.out = static_cast<uint16_t*>(out);
  p.err = err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
  const unsigned nb = static_cast<unsigned>(min(p.num_units, sms));
  return elem == Elem::kF16 ? launch_typed<Elem::kF16>(tq, tk, tv, p, nb, stream)
                            : launch_typed<Elem::kBF16>(tq, tk, tv, p, nb, stream);
}

}  // namespace pkv
