// gemm_simt.cu -- two-level tiled FP32 product on the CUDA cores (FFMA).
//
// Tiling ("Tiling Strategies" sections 2-4, "CMU DLSys Lecture 12" section 5):
//   * block tile: each block owns a BM x BN tile of C (64 x 256 with 1 x 4
//     warps in the default configuration; two blocks resident per SM);
//   * K-slices of BK flow through a ring of kStages shared-memory stages
//     filled by asynchronous copies (TMA and cp.async).  This generalises the
//     double buffer of "Tiling Strategies" section 3: the copies of the next
//     kStages - 1 slices are in flight while one slice is consumed, and no
//     register holds staged data;
//   * thread tile: each thread owns a TM x TN tile of C in registers and
//     performs one outer product per k (TM + TN operands, TM*TN FFMA), with
//     the operands of step k+2 (k+1 when A is copied by TMA) loaded from
//     shared memory while step k's FFMAs issue ("Tiling Hierarchy on GPUs",
//     "Register Tiling", "Register prefetching", "Reducing Overhead Slots").
//
// Shared-memory layout.  The A slab is stored transposed, a[k][m], so a
// thread's rows of A at one k are 16-byte vectors; from A stored M x K it is
// filled by 4-byte copies, each warp copying 4 rows x 8 consecutive k (four
// 32-byte global sectors) into 32 distinct banks (row length BM + 4 floats);
// from A stored K x M (the A^T B layouts) by one TMA copy per K-slice.  The B
// slab keeps the layout b[k][n] and is always filled by TMA, one copy of the
// whole slab per K-slice issued by one thread: B stored K x N with rows on
// 16-byte boundaries is read in place, any other B (stored N x K, or rows of
// a pitch that is not a multiple of 4 floats) is first restaged into that
// layout by a copy kernel (operand_stage.cu).  A stored K x M without
// 16-byte rows is restaged the same way.
//
// Warp tiling ("Tiling Hierarchy on GPUs", "Warp Tiling"): the 32 lanes of a
// warp form an LM x LN grid (4 x 8 or 8 x 4); lane (lm, ln) owns rows
// lm*4 + 4*LM*t + i and columns ln*4 + 4*LN*c + j of the warp's region.  A
// 128-bit shared load is served at most 16 lanes per wavefront, and the two
// quarter-warps of a half-warp share a wavefront only when they read disjoint
// words with lanes that share a word paired up.  With quarter q = lane / 8,
// the 4-valued coordinate is  lane % 2 + 2 (q % 2)  and the 8-valued one is
// (lane / 2) % 4 + 4 ((q % 2) xor (q / 2)),  so every fragment load, of A or
// of B, takes two wavefronts, the minimum.
//
// Tails ("CMU DLSys Lecture 12" section 5): copies outside M, N or K are
// zero-filled (source size 0), which adds nothing to the sums, and only
// entries inside M x N are stored.
//
// Scheduling.  Tiles are numbered along a grouped raster -- kGroupM tile-rows
// are walked column by column -- so blocks resident at the same time share
// the A row-panels and B column-panels they read through L2.  When the tile
// count leaves a partial last wave, the kernel runs persistent (one block per
// resident slot, launched cooperatively so that all are resident at once):
// all but the last full wave of tiles are processed whole ("data-parallel"),
// and the remaining tiles' K-slices are divided evenly among all blocks
// ("stream-K").  Every block then does the same amount of work.  Each block's
// share is at least one whole tile, so a split tile has exactly two
// contributors: the block holding slices [x, S) stores its partial sums into
// C and raises a flag; the block holding slices [0, x) -- which reaches the
// tile last -- waits for the flag, adds the partial to its own sums and
// stores the total.  With fewer tiles than slots, all tiles are split this way
// over more blocks than tiles, and a tile can have up to about five
// contributors: each block waits for the next block's flag, adds C (the sum
// of the slices after its own) to its sums, stores, and raises its own flag
// for the block before it.  With few tiles, or C without 16-byte rows, a
// kernel of its own (gemm_simt_reduce_kernel) gives every block an equal
// share instead; the blocks store their partial sums into scratch slots and
// then reduce each tile together, each a band of its rows.  The order of the
// additions is fixed, so results are deterministic.  Every wait is bounded:
// past the time limit the block records a timeout in the device status word
// and finishes.
#include <atomic>
#include <cstdint>

#include "bounds_check.cuh"
#include "tmm_internal.h"

namespace tmm {

// Flags of split tiles: kFlagRegions rings of kMaxPersistentBlocks words; a
// call uses region epoch % kFlagRegions and raises flags to its epoch, so no
// reset is needed between calls and calls in flight together use distinct
// regions (up to kFlagRegions of them).
constexpr int kFlagRegions = 16;
constexpr int kMaxPersistentBlocks = 4096;
__device__ unsigned int g_simt_flags[kFlagRegions * kMaxPersistentBlocks];
// Device status word (bit 0: a stream-K wait ran out of time; bit 1: a TMA
// wait did; bit 2: a range check of the bounds-checked build failed).
__device__ unsigned int g_simt_status;

namespace {

constexpr int kGroupM = 16;

// How the A slab reaches its k-major shared-memory layout:
//   kCopyTransposing  -- A stored M x K (k contiguous): each element is placed
//                        by a 4-byte copy (4 rows x 8 k per warp instruction,
//                        into 32 distinct banks);
//   kCopyTma          -- A stored K x M with 16-byte rows: one TMA copy of the
//                        whole slab per K-slice, issued by one thread and
//                        counted on the stage's mbarrier with B's copy.
// The B slab is always copied by TMA.
constexpr int kCopyTransposing = 0, kCopyTma = 3;

template <int TM_, int TN_, int kWarpsM_, int kWarpsN_, int BK_, int kStages_, int kMinBlocks_>
struct SimtConfig {
  static constexpr int TM = TM_, TN = TN_;
  static constexpr int kWarpsM = kWarpsM_, kWarpsN = kWarpsN_;
  static constexpr int LM = (TM >= TN) ? 4 : 8;     // lane grid rows
  static constexpr int LN = 32 / LM;                // lane grid columns
  static constexpr int BM = kWarpsM * LM * TM;
  static constexpr int BN = kWarpsN * LN * TN;
  static constexpr int BK = BK_;
  static constexpr int kStages = kStages_;
  static constexpr int kThreads = 32 * kWarpsM * kWarpsN;
  static constexpr int kWarps = kWarpsM * kWarpsN;
  static constexpr int kMinBlocks = kMinBlocks_;
  // Row pitch of the k-major A slab: 4 mod 32 floats when filled by
  // transposing copies, which spreads a warp's 4 rows x 8 k over 32 banks; a
  // TMA copy writes its box densely.
  template <int kACopy>
  __host__ __device__ static constexpr int as_ld() {
    return kACopy == kCopyTma ? BM : BM + 4;
  }
  // A TMA copy moves boxes of at most 256 columns; a wider B slab is held as
  // consecutive sub-slabs of kBBox columns (BK x BN floats either way).
  static constexpr int kBBox = BN < 256 ? BN : 256;
  static constexpr int kBsLd = kBBox;
  template <int kACopy>
  __host__ __device__ static constexpr int a_slab_floats() {
    return BK * as_ld<kACopy>();
  }
  static constexpr int kBSlabFloats = BK * BN;
  template <int kACopy>
  __host__ __device__ static constexpr int stage_floats() {
    return a_slab_floats<kACopy>() + kBSlabFloats;
  }
  // The ring starts on a 128-byte boundary (the TMA destination rule) and is
  // followed by one mbarrier per stage.
  template <int kACopy>
  __host__ __device__ static constexpr int smem_bytes() {
    return kStages * stage_floats<kACopy>() * 4 + 128 + 8 * kStages;
  }
  // A copies: groups of 4 rows x 8 k per warp instruction.
  static constexpr int kARowGroups = BM / 4;
  static constexpr int kARowGroupsPerWarp = kARowGroups / kWarps;
  static constexpr int kACopies = kARowGroupsPerWarp * (BK / 8);

  static_assert(TM % 4 == 0 && TN % 4 == 0, "thread tiles are made of 4 x 4 quadrants");
  static_assert(BK % 8 == 0, "slice depth");
  static_assert(kARowGroups % kWarps == 0, "A copy groups divide among warps");
  static_assert((BM + 4) % 32 == 4, "pitch for transposing copies");
  static_assert(BN % kBBox == 0, "whole TMA boxes of B");
  static_assert((BK * (BM + 4) * 4) % 128 == 0 && (BK * BM * 4) % 128 == 0 &&
                (BK * BN * 4) % 128 == 0 && (BK * kBBox * 4) % 128 == 0,
                "TMA destinations on 128-byte boundaries");
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Asynchronous global->shared copies; a false predicate copies zero bytes and
// zero-fills the destination.  The source is then not read, and is replaced by
// `safe` (an address inside the operand) all the same.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const float *src, bool pred,
                                           const float *safe) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst),
               "l"(pred ? src : safe), "r"(pred ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t dst, const float *src, bool pred,
                                            const float *safe) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(pred ? src : safe), "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Two FP32 values in one 64-bit register pair (lo = first).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// Two IEEE single-precision fused multiply-adds in one instruction: each half
// is rounded once, exactly as fmaf; the pair costs one issue slot.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned int load_acquire(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Wait until *flag == value, an acquire load every 128 ns (a chain's
// hand-over is on its critical path: a sleep doubling up to 1 us between
// relaxed polls measured slower, 1000 x 1000 x 2990 44.1 against 45.4
// TFLOP/s).  False when limit_ns passes first.
__device__ __forceinline__ bool wait_flag(const unsigned int *flag, unsigned int value,
                                          int64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (load_acquire(flag) != value) {
    if (int64_t(global_timer_ns() - t0) > limit_ns) return false;
    __nanosleep(128);
  }
  return true;
}
__device__ __forceinline__ void store_release(unsigned int *p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// mbarrier and bulk-tensor (TMA) primitives of the TMA copy kinds.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait for phase `parity` of the barrier to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (int64_t(global_timer_ns() - t0) > limit_ns) return false;
  return true;
}
// As mbar_wait; while waiting also gives up at once when `dead` is set (a
// register flag of the caller, read only after the first poll has failed).
__device__ __forceinline__ bool mbar_wait_unless(uint32_t bar, uint32_t parity, int64_t limit_ns,
                                                 const bool &dead) {
  if (mbar_try_wait(bar, parity)) return true;
  if (dead) return false;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (int64_t(global_timer_ns() - t0) > limit_ns) return false;
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int &tm,
                                            int &tn) {
  const int per_group = kGroupM * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * kGroupM;
  const int rows = min(tiles_m - first_m, kGroupM);
  const int in_group = tile - group * per_group;
  tm = first_m + in_group % rows;
  tn = in_group / rows;
}

struct SimtParams {
  int M, N, K;
  const float *A;
  int64_t lda;
  const float *B;
  int64_t ldb;
  float *C;
  int64_t ldc;
  int tiles_m, tiles_n;
  int slices;            // K-slices per tile
  int dp_tiles;          // tiles [0, dp_tiles) are processed whole, striding by gridDim.x
  int64_t sk_iters;      // (tiles - dp_tiles) * slices, divided evenly among the blocks
  unsigned int epoch;    // this call's flag value (never 0)
  int64_t wait_limit_ns; // bound on a stream-K wait
  int drop_signal_block; // testing hook: this block never raises its flag (-1: none)
  // Small problems (fewer tiles than resident blocks) chained through C:
  // with parts > 0, tile t's K-slices go to blocks t parts .. t parts +
  // parts - 1 in unequal parts, part q holding part_base + (parts - 1 - q)
  // part_step slices (part 0 also the remainder); with parts == 0, every
  // block an equal share of all tiles' K-slices, at least a quarter of a tile.
  int parts, part_base, part_step, part_rem;
};

// First K-slice of part q of a tile split per tile (q == parts: the tile's end).
__device__ __forceinline__ int part_begin(const SimtParams &p, int q) {
  if (q >= p.parts) return p.slices;
  return q * p.part_base + p.part_step * (q * (p.parts - 1) - q * (q - 1) / 2) +
         (q > 0 ? p.part_rem : 0);
}

// First K-slice unit (tile t, slice s is unit t S + s) of block b's equal
// share of T units over G blocks.
__device__ __forceinline__ int64_t share_begin(int64_t T, int64_t G, int64_t b) {
  return b * T / G;
}
// The block whose share holds unit u.
__device__ __forceinline__ int64_t share_owner(int64_t T, int64_t G, int64_t u) {
  int64_t c = u * G / T;
  while (c + 1 < G && share_begin(T, G, c + 1) <= u) ++c;
  while (c > 0 && share_begin(T, G, c) > u) --c;
  return c;
}

// One block's work on tile `tile`, K-slices [s_begin, s_end).  kACopy: how
// the A slab is copied (kCopyTransposing for A stored M x K, kCopyTma for A
// stored K x M).  kVecC: C takes 16-byte stores (C 16-byte aligned, ldc and N
// multiples of 4), decided per call; element-wise stores otherwise.
template <class Cf, int kACopy, bool kVecC>
struct SimtBlock {
  // Accumulators in pairs along N: acc[i][jp] holds columns 2 jp (lo), 2 jp + 1 (hi).
  uint64_t acc[Cf::TM][Cf::TN / 2];
  int lane, warp, tid;
  int a_off, b_off;   // this thread's first row and column of the tile
  int b_frag;         // offset of its first B column in the B slab

  __device__ __forceinline__ void init_lanes() {
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
    const int q = lane >> 3;
    const int four = (lane & 1) + 2 * (q & 1);
    const int eight = ((lane >> 1) & 3) + 4 * ((q & 1) ^ (q >> 1));
    const int lm = (Cf::LM == 4) ? four : eight;
    const int ln = (Cf::LM == 4) ? eight : four;
    const int wm = warp / Cf::kWarpsN, wn = warp % Cf::kWarpsN;
    a_off = wm * (Cf::LM * Cf::TM) + lm * 4;
    b_off = wn * (Cf::LN * Cf::TN) + ln * 4;
    // A warp's columns lie in one sub-slab (checked below).
    b_frag = (b_off / Cf::kBBox) * (Cf::BK * Cf::kBBox) + b_off % Cf::kBBox;
  }
  static_assert(Cf::kBBox % (Cf::LN * Cf::TN) == 0, "a warp's B columns in one TMA box");

  // Row of C (relative to the block tile's a_off) of accumulator row r.
  __device__ __forceinline__ static constexpr int row_of(int r) {
    return 4 * Cf::LM * (r / 4) + r % 4;
  }

  // With TMA copies, `bars` holds one mbarrier per stage and bit i of
  // `phases` the parity its next completion will have.  A wait that runs out
  // of time is handled off the fast path (tma_wait_failed): the thread sets
  // the status word and waits no more (its later waits give up at once), so
  // the kernel still runs to its end in bounded time, its results not valid;
  // thread 0, the only one issuing copies, first waits (bounded) for every
  // copy it has in flight and then issues no more (re-arming a stage whose
  // copy has not landed is unsafe), so no copy lands after the block is gone.
  __device__ __forceinline__ void mainloop(const SimtParams &p, float *smem, int m0, int n0,
                                           int s_begin, int s_end, const CUtensorMap *a_map,
                                           const CUtensorMap *b_map, uint32_t bars,
                                           uint32_t &phases) {
    constexpr int BK = Cf::BK, kAsLd = Cf::template as_ld<kACopy>();
    constexpr int kBsLd = Cf::kBsLd;
    constexpr int kASlab = Cf::template a_slab_floats<kACopy>();
    constexpr int kStageFloats = Cf::template stage_floats<kACopy>();
    constexpr int kStages = Cf::kStages;
    constexpr bool kTmaA = kACopy == kCopyTma;
    constexpr uint32_t kTmaBytes = (kTmaA ? kASlab * 4 : 0) + Cf::kBSlabFloats * 4;

    // Transposing copies of A (stored M x K): warp instruction (r, h) copies
    // rows 4 (warp + kWarps r) + lane/8 of the tile, k 8 h + lane % 8.
    const int t_row = (lane >> 3) + 4 * warp;
    const int t_k = lane & 7;
    const float *a_src = p.A;
    int64_t a_step = 0;        // between copy groups
    uint32_t a_rows_ok = 0;    // bit r: row t_row + 4 kWarps r inside M
    uint32_t a_dst0 = 0;
    if (!kTmaA) {
#pragma unroll
      for (int r = 0; r < Cf::kARowGroupsPerWarp; ++r)
        a_rows_ok |= uint32_t(m0 + t_row + 4 * Cf::kWarps * r < p.M) << r;
      a_src = p.A + int64_t(min(m0 + t_row, p.M - 1)) * p.lda + t_k;
      a_step = int64_t(4 * Cf::kWarps) * p.lda;
      a_dst0 = smem_addr(smem) + 4u * (t_k * kAsLd + t_row);
    }

    // extra_tx: bytes the stage's barrier expects beyond the copies (testing
    // hook: a barrier that never completes).
    auto issue_slice = [&](int s, int stage, uint32_t extra_tx) {
      const int k0 = s * BK;
      const uint32_t st_off = 4u * stage * kStageFloats;
      if (!kTmaA) {
        const int64_t st_base = int64_t(smem_addr(smem) + st_off);
        (void)st_base;
        const float *a = a_src + k0;
#pragma unroll
        for (int it = 0; it < Cf::kACopies; ++it) {
          const int r = it % Cf::kARowGroupsPerWarp, h = it / Cf::kARowGroupsPerWarp;
          const uint32_t dst = a_dst0 + st_off + 4u * (8 * h * kAsLd + 4 * Cf::kWarps * r);
          const float *src = a + r * a_step + 8 * h;
          const bool ok = ((a_rows_ok >> r) & 1u) && (k0 + t_k + 8 * h < p.K);
          // The copy stays inside A and the A slab (debug build only).
          cp_async_4(dst, src,
                     ok && TMM_IN_BOUNDS(in_matrix(src, p.A, p.M, p.K, p.lda) &&
                                             in_region(int64_t(dst) - st_base, kASlab),
                                         &g_simt_status),
                     p.A);
        }
      }
      if (tid == 0 && !tma_dead) {
        // The box origins lie inside the matrices (the copy fills the rest with zeros).
        (void)TMM_IN_BOUNDS(k0 < p.K && n0 < p.N && (!kTmaA || m0 < p.M), &g_simt_status);
        const uint32_t bar = bars + 8u * stage, st = smem_addr(smem) + st_off;
        mbar_arrive_expect_tx(bar, kTmaBytes + extra_tx);
        if (kTmaA) tma_load_2d(st, a_map, m0, k0, bar);
#pragma unroll
        for (int j = 0; j < Cf::BN / Cf::kBBox; ++j)
          tma_load_2d(st + 4u * (kASlab + j * BK * Cf::kBBox), b_map, n0 + j * Cf::kBBox, k0,
                      bar);
      }
    };

    zero_acc();

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s_begin + s < s_end)
        issue_slice(s_begin + s, s,
                    (s == 0 && int(blockIdx.x) == p.drop_signal_block) ? 16u : 0u);
      cp_async_commit();
    }

    int stage = 0;
    for (int s = s_begin; s < s_end; ++s) {
      cp_async_wait<kStages - 2>();   // slice s has landed (this thread's copies) ...
      // ... and its TMA copies ...
      if (!mbar_wait_unless(bars + 8u * stage, (phases >> stage) & 1u, p.wait_limit_ns,
                            tma_dead))
        tma_wait_failed(p, bars, phases, stage, s, s_end);
      phases ^= 1u << stage;
      __syncthreads();                // ... and everyone's; slice s-1's stage is free
      {
        const int sn = s + kStages - 1;
        int stage_n = stage + kStages - 1;
        if (stage_n >= kStages) stage_n -= kStages;
        if (sn < s_end) issue_slice(sn, stage_n, 0u);
        cp_async_commit();
      }
      const float *st = smem + stage * kStageFloats;
      slice_products<kAsLd, kBsLd>(st, st + kASlab);
      if (++stage == kStages) stage = 0;
    }
    cp_async_wait<0>();
    __syncthreads();   // the next tile's copies may overwrite any stage
  }

  // Set once one of this thread's TMA waits has run out of time.
  bool tma_dead = false;

  // The wait for slice s (in `stage`) ran out of time.  Thread 0 has copies in
  // flight for slices s .. min(s_end, s + kStages - 1) - 1, one per stage from
  // `stage` on, each at its stage's parity in `phases`.
  __device__ __forceinline__ void tma_wait_failed(const SimtParams &p, uint32_t bars,
                                                  uint32_t phases, int stage, int s, int s_end) {
    if (!tma_dead) {   // this thread's first failure
      atomicOr(&g_simt_status, 2u);
      if (tid == 0) {
        const int last = min(s_end, s + Cf::kStages - 1);
        for (int q = s, st = stage; q < last; ++q, st = (st + 1) % Cf::kStages)
          mbar_wait(bars + 8u * st, (phases >> st) & 1u, p.wait_limit_ns);
      }
    }
    tma_dead = true;
  }

  __device__ __forceinline__ void zero_acc() {
#pragma unroll
    for (int i = 0; i < Cf::TM; ++i)
#pragma unroll
      for (int j = 0; j < Cf::TN / 2; ++j) acc[i][j] = 0;   // +0.0f in both halves
  }

  // This thread's fragments at k of a staged slice: TM values of the k-major A
  // slab `as` (row pitch kAsLd) and TN values of the B slab `bs` (pitch kBsLd).
  template <int kAsLd, int kBsLd>
  __device__ __forceinline__ void load_frag(const float *as, const float *bs, int k,
                                            float (&af)[Cf::TM], uint64_t (&bf)[Cf::TN / 2]) {
    const float *a = as + k * kAsLd + a_off;
    const float *b = bs + k * kBsLd + b_frag;
#pragma unroll
    for (int t = 0; t < Cf::TM / 4; ++t) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (TMM_IN_BOUNDS(in_region(4 * (a + 4 * Cf::LM * t - as),
                                  Cf::template a_slab_floats<kACopy>(), 4),
                        &g_simt_status))
        v = *reinterpret_cast<const float4 *>(a + 4 * Cf::LM * t);
      af[4 * t + 0] = v.x; af[4 * t + 1] = v.y; af[4 * t + 2] = v.z; af[4 * t + 3] = v.w;
    }
#pragma unroll
    for (int c = 0; c < Cf::TN / 4; ++c) {
      ulonglong2 v = make_ulonglong2(0, 0);
      if (TMM_IN_BOUNDS(in_region(4 * (b + 4 * Cf::LN * c - bs),
                                  Cf::kBSlabFloats, 4),
                        &g_simt_status))
        v = *reinterpret_cast<const ulonglong2 *>(b + 4 * Cf::LN * c);
      bf[2 * c + 0] = v.x; bf[2 * c + 1] = v.y;
    }
  }

  // The BK outer products of one staged slice (the whole slice unrolled; the
  // packed code fits the instruction cache), the fragments of step k + kPrefetch
  // loaded while step k's packed FMAs issue.  Two steps ahead with A copied by
  // transposing copies (4096^3 66.1 against 64.8 TFLOP/s one step ahead;
  // 4000 x 3001 x 2047 58.8 against 57.6), one with A copied by TMA (4096^3
  // 66.7 against 65.8 two steps ahead).
  static constexpr int kPrefetch = kACopy == kCopyTma ? 1 : 2;
  template <int kAsLd, int kBsLd>
  __device__ __forceinline__ void slice_products(const float *as, const float *bs) {
    constexpr int BK = Cf::BK, D = kPrefetch, kBufs = kPrefetch + 1;
    float af[kBufs][Cf::TM];
    uint64_t bf[kBufs][Cf::TN / 2];
#pragma unroll
    for (int d = 0; d < D; ++d) load_frag<kAsLd, kBsLd>(as, bs, d, af[d], bf[d]);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      if (k + D < BK)
        load_frag<kAsLd, kBsLd>(as, bs, k + D, af[(k + D) % kBufs], bf[(k + D) % kBufs]);
      // Outer product: acc[i][j] += a[i] * b[j], two columns per instruction.
#pragma unroll
      for (int i = 0; i < Cf::TM; ++i) {
        const uint64_t ai = pack2(af[k % kBufs][i], af[k % kBufs][i]);
#pragma unroll
        for (int j = 0; j < Cf::TN / 2; ++j)
          acc[i][j] = ffma2(ai, bf[k % kBufs][j], acc[i][j]);
      }
    }
  }

  // This thread's partial sums into a BM x BN row-major slot (16-byte stores).
  __device__ __forceinline__ void store_partial(float *slot) {
#pragma unroll
    for (int r = 0; r < Cf::TM; ++r) {
      float *row = slot + (a_off + row_of(r)) * Cf::BN + b_off;
      float a[Cf::TN];
#pragma unroll
      for (int j = 0; j < Cf::TN / 2; ++j) unpack2(acc[r][j], a[2 * j], a[2 * j + 1]);
#pragma unroll
      for (int c = 0; c < Cf::TN / 4; ++c)
        if (TMM_IN_BOUNDS(in_region(4 * (row + 4 * Cf::LN * c - slot), Cf::BM * Cf::BN, 4),
                          &g_simt_status))
          *reinterpret_cast<float4 *>(row + 4 * Cf::LN * c) =
              make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
    }
  }

  // Tile t of a small problem split in equal shares over all G blocks: every
  // block whose share meets the tile has stored its partial sums into its
  // slot and raised the slot's flag.  Once all n flags are up (bounded
  // waits), contributor j (this block) adds rows [j BM / n, (j + 1) BM / n)
  // of the n partials, in contributor order, and stores them into C: the n
  // contributors reduce the tile together, each reading a 1/n-th of every
  // partial.  The first contributor's share may begin in the tile before,
  // which makes tile t its second segment.
  __device__ __forceinline__ void reduce_split_tile(const SimtParams &p, const float *partials,
                                                    int t, int64_t G, int64_t b,
                                                    const unsigned int *flags) {
    const int64_t T = p.sk_iters;
    const int64_t u0 = int64_t(t) * p.slices, u1 = u0 + p.slices;
    const int64_t c_lo = share_owner(T, G, u0), c_hi = share_owner(T, G, u1 - 1);
    const int64_t first_slot = 2 * c_lo + (share_begin(T, G, c_lo) < u0 ? 1 : 0);
    auto slot_of = [&](int64_t c) { return c == c_lo ? first_slot : 2 * c; };
    if (tid == 0) {
      for (int64_t c = c_lo; c <= c_hi; ++c)
        if (!wait_flag(&flags[slot_of(c)], p.epoch, p.wait_limit_ns))
          atomicOr(&g_simt_status, 1u);
    }
    __syncthreads();
    int tm, tn;
    tile_coords(t, p.tiles_m, p.tiles_n, tm, tn);
    const int m0 = tm * Cf::BM, n0 = tn * Cf::BN;
    const int n = int(c_hi - c_lo + 1), j = int(b - c_lo);
    const int r0 = j * Cf::BM / n, r1 = (j + 1) * Cf::BM / n;
    // 16 loads of 16 bytes in flight per thread: positions x contributors.
    if (n <= 2)
      reduce_rows<8, 2>(p, partials, m0, n0, r0, r1, c_lo, c_hi, first_slot, G);
    else if (n <= 4)
      reduce_rows<4, 4>(p, partials, m0, n0, r0, r1, c_lo, c_hi, first_slot, G);
    else
      reduce_rows<2, 8>(p, partials, m0, n0, r0, r1, c_lo, c_hi, first_slot, G);
  }

  // Rows [r0, r1) of a split tile: the partial sums of contributors c_lo ..
  // c_hi (slot first_slot for c_lo, 2 c for the others) added in contributor
  // order and stored into C.  Each thread takes P 16-byte positions at a time
  // and loads them from Q contributors at a time, all P Q loads in flight.
  template <int P, int Q>
  __device__ __forceinline__ void reduce_rows(const SimtParams &p, const float *partials, int m0,
                                              int n0, int r0, int r1, int64_t c_lo, int64_t c_hi,
                                              int64_t first_slot, int64_t G) {
    constexpr int kRowVecs = Cf::BN / 4;
    constexpr int64_t kSlotFloats = int64_t(Cf::BM) * Cf::BN;
    const int nvec = (r1 - r0) * kRowVecs;
    for (int base = tid; base < nvec; base += P * Cf::kThreads) {
      float4 v[P];
      for (int64_t cc = c_lo; cc <= c_hi; cc += Q) {
        float4 w[P][Q];
#pragma unroll
        for (int i = 0; i < P; ++i) {
          const int idx = base + i * Cf::kThreads;
          const int64_t off = int64_t(r0 + idx / kRowVecs) * Cf::BN + 4 * (idx % kRowVecs);
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            const int64_t c = cc + q;
            const int64_t slot = c == c_lo ? first_slot : 2 * c;
            w[i][q] = (idx < nvec && c <= c_hi &&
                       TMM_IN_BOUNDS(in_region(4 * (slot * kSlotFloats + off),
                                               2 * G * kSlotFloats, 4),
                                     &g_simt_status))
                          ? __ldcg(reinterpret_cast<const float4 *>(partials +
                                                                    slot * kSlotFloats + off))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int i = 0; i < P; ++i)
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            if (cc + q > c_hi) break;
            if (cc + q == c_lo) {
              v[i] = w[i][q];
            } else {
              v[i].x = v[i].x + w[i][q].x; v[i].y = v[i].y + w[i][q].y;
              v[i].z = v[i].z + w[i][q].z; v[i].w = v[i].w + w[i][q].w;
            }
          }
      }
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const int idx = base + i * Cf::kThreads;
        if (idx >= nvec) break;
        const int gr = m0 + r0 + idx / kRowVecs, gc = n0 + 4 * (idx % kRowVecs);
        if (gr >= p.M) continue;
        float *dst = p.C + int64_t(gr) * p.ldc + gc;
        if (kVecC) {
          if (gc < p.N && TMM_IN_BOUNDS(in_matrix(dst, p.C, p.M, p.N, p.ldc, 4), &g_simt_status))
            *reinterpret_cast<float4 *>(dst) = v[i];
        } else {
          const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (gc + e < p.N &&
                TMM_IN_BOUNDS(in_matrix(dst + e, p.C, p.M, p.N, p.ldc), &g_simt_status))
              dst[e] = vv[e];
        }
      }
    }
  }

  // Accumulator (r, 4c + j) is C[m0 + a_off + row_of(r)][n0 + b_off + 4 LN c + j].
  // Stores this thread's part of the tile; kAdd: the running sum of the later
  // K-slices, already in C, is added first (partial + own, in that order).
  template <bool kAdd>
  __device__ __forceinline__ void epilogue(const SimtParams &p, int m0, int n0, float *smem) {
    if (kAdd && kVecC)
      add_staged(p, m0, n0, smem);
    else if (kAdd)
      add_elementwise(p, m0, n0);
    else
      store(p, m0, n0);
  }

  __device__ __forceinline__ void store(const SimtParams &p, int m0, int n0) {
    const int row0 = m0 + a_off;
    const int col0 = n0 + b_off;
    float *c_base = p.C + int64_t(row0) * p.ldc + col0;
#pragma unroll
    for (int r = 0; r < Cf::TM; ++r) {
      const int dr = row_of(r);
      if (row0 + dr >= p.M) continue;
      float *c_row = c_base + int64_t(dr) * p.ldc;
      float a[Cf::TN];
#pragma unroll
      for (int j = 0; j < Cf::TN / 2; ++j) unpack2(acc[r][j], a[2 * j], a[2 * j + 1]);
#pragma unroll
      for (int c = 0; c < Cf::TN / 4; ++c) {
        const int dc = 4 * Cf::LN * c;
        if (kVecC) {
          if (col0 + dc < p.N &&
              TMM_IN_BOUNDS(in_matrix(c_row + dc, p.C, p.M, p.N, p.ldc, 4), &g_simt_status))
            *reinterpret_cast<float4 *>(c_row + dc) =
                make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (col0 + dc + j < p.N &&
                TMM_IN_BOUNDS(in_matrix(c_row + dc + j, p.C, p.M, p.N, p.ldc), &g_simt_status))
              c_row[dc + j] = a[4 * c + j];
        }
      }
    }
  }

  // The add when C takes 16-byte stores: this thread's part of the running
  // sum is copied by 16-byte cp.async (through L2) into the stage ring, free
  // once the mainloop has ended, every row in flight at once, then added and
  // stored -- one round trip to L2, where loads into registers (the
  // accumulators leave room for a few rows at a time) took one per row group.
  // Vector (i, c) of a round of kRows rows sits at float4 slot
  // (i TN/4 + c) kThreads + tid: a warp's copies and reads cover 512
  // contiguous bytes, and a thread reads back only what it copied (visible to
  // it once its own copies are waited for).
  __device__ __forceinline__ void add_staged(const SimtParams &p, int m0, int n0, float *smem) {
    constexpr int kRingFloats = Cf::kStages * Cf::template stage_floats<kACopy>();
    constexpr int kVecs = Cf::TN / 4;
    constexpr int kFit = kRingFloats / (Cf::kThreads * Cf::TN);
    constexpr int kRows = kFit >= Cf::TM ? Cf::TM : kFit >= 4 ? 4 : kFit >= 2 ? 2 : 1;
    static_assert(kFit >= 1 && Cf::TM % kRows == 0, "a round of rows fits the ring");
    const int row0 = m0 + a_off;
    const int col0 = n0 + b_off;
    float *c_base = p.C + int64_t(row0) * p.ldc + col0;
    const uint32_t ring = smem_addr(smem);
#pragma unroll
    for (int r0 = 0; r0 < Cf::TM; r0 += kRows) {
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const int dr = row_of(r0 + i);
        const bool row_ok = row0 + dr < p.M;
        const float *c_row = c_base + int64_t(dr) * p.ldc;
#pragma unroll
        for (int c = 0; c < kVecs; ++c) {
          const int slot = (i * kVecs + c) * Cf::kThreads + tid;
          const float *src = c_row + 4 * Cf::LN * c;
          const bool ok = row_ok && col0 + 4 * Cf::LN * c < p.N;
          cp_async_16(ring + 16u * slot, src,
                      ok && TMM_IN_BOUNDS(in_matrix(src, p.C, p.M, p.N, p.ldc, 4) &&
                                              in_region(16 * int64_t(slot), kRingFloats, 4),
                                          &g_simt_status),
                      p.C);
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const int r = r0 + i;
        const int dr = row_of(r);
        if (row0 + dr >= p.M) continue;
        float *c_row = c_base + int64_t(dr) * p.ldc;
        float a[Cf::TN];
#pragma unroll
        for (int j = 0; j < Cf::TN / 2; ++j) unpack2(acc[r][j], a[2 * j], a[2 * j + 1]);
#pragma unroll
        for (int c = 0; c < kVecs; ++c) {
          const int dc = 4 * Cf::LN * c;
          if (col0 + dc >= p.N) continue;
          const int slot = (i * kVecs + c) * Cf::kThreads + tid;
          const float4 w = *reinterpret_cast<const float4 *>(smem + 4 * slot);
          float4 v = make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
          v.x = w.x + v.x; v.y = w.y + v.y; v.z = w.z + v.z; v.w = w.w + v.w;
          if (TMM_IN_BOUNDS(in_matrix(c_row + dc, p.C, p.M, p.N, p.ldc, 4), &g_simt_status))
            *reinterpret_cast<float4 *>(c_row + dc) = v;
        }
      }
    }
    __syncthreads();   // the next tile's copies may overwrite the ring
  }

  // The add when C takes element-wise stores: the running sum is loaded
  // element by element through L2 (a 4-byte copy into shared memory would go
  // through L1, which may hold an older sum of the same lines), kAddRows rows
  // of it before the first store, so the loads are in flight together (a
  // store before a load of the same array would order them one after another).
  __device__ __forceinline__ void add_elementwise(const SimtParams &p, int m0, int n0) {
    constexpr int kAddRows = 4;
    static_assert(Cf::TM % kAddRows == 0, "whole row groups");
    const int row0 = m0 + a_off;
    const int col0 = n0 + b_off;
    float *c_base = p.C + int64_t(row0) * p.ldc + col0;
#pragma unroll
    for (int r0 = 0; r0 < Cf::TM; r0 += kAddRows) {
      float w[kAddRows][Cf::TN];
#pragma unroll
      for (int i = 0; i < kAddRows; ++i) {
        const int dr = row_of(r0 + i);
        const bool row_ok = row0 + dr < p.M;
        const float *c_row = c_base + int64_t(dr) * p.ldc;
#pragma unroll
        for (int c = 0; c < Cf::TN / 4; ++c)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int dc = 4 * Cf::LN * c + j;
            w[i][4 * c + j] =
                row_ok && col0 + dc < p.N &&
                        TMM_IN_BOUNDS(in_matrix(c_row + dc, p.C, p.M, p.N, p.ldc), &g_simt_status)
                    ? __ldcg(c_row + dc) : 0.f;
          }
      }
#pragma unroll
      for (int i = 0; i < kAddRows; ++i) {
        const int r = r0 + i;
        const int dr = row_of(r);
        if (row0 + dr >= p.M) continue;
        float *c_row = c_base + int64_t(dr) * p.ldc;
        float a[Cf::TN];
#pragma unroll
        for (int j = 0; j < Cf::TN / 2; ++j) unpack2(acc[r][j], a[2 * j], a[2 * j + 1]);
#pragma unroll
        for (int c = 0; c < Cf::TN / 4; ++c)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int dc = 4 * Cf::LN * c + j;
            if (col0 + dc < p.N &&
                TMM_IN_BOUNDS(in_matrix(c_row + dc, p.C, p.M, p.N, p.ldc), &g_simt_status))
              c_row[dc] = w[i][4 * c + j] + a[4 * c + j];
          }
      }
    }
  }
};

// a_map, b_map: the tensor maps of A and B for the TMA copy kinds, else unused.
// a_map, b_map: the tensor maps of A and B for the TMA copy kinds, else unused.
template <class Cf, int kACopy, bool kVecC>
__global__ void __launch_bounds__(Cf::kThreads, Cf::kMinBlocks)
gemm_simt_kernel(const __grid_constant__ CUtensorMap a_map,
                 const __grid_constant__ CUtensorMap b_map, const SimtParams p) {
  extern __shared__ __align__(16) float smem_raw[];
  constexpr int kRingFloats = Cf::kStages * Cf::template stage_floats<kACopy>();
  // The ring on a 128-byte boundary, then one mbarrier per stage.
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  float *smem = smem_raw + (base - raw) / 4;
  const uint32_t bars = base + uint32_t(kRingFloats * 4);
  uint32_t phases = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < Cf::kStages; ++i) mbar_init(bars + 8u * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  SimtBlock<Cf, kACopy, kVecC> blk;
  blk.init_lanes();

  // Whole tiles.
  for (int tile = blockIdx.x; tile < p.dp_tiles; tile += gridDim.x) {
    int tm, tn;
    tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
    blk.mainloop(p, smem, tm * Cf::BM, tn * Cf::BN, 0, p.slices, &a_map, &b_map, bars, phases);
    blk.template epilogue<false>(p, tm * Cf::BM, tn * Cf::BN, smem);
  }
  if (p.sk_iters == 0) return;

  // This block's share of the split tiles' K-slices: an even share of all of
  // them, or one part of one tile.
  const int64_t g = gridDim.x, b = blockIdx.x;
  int64_t it_start = b * p.sk_iters / g, it_end = (b + 1) * p.sk_iters / g;
  if (p.parts > 0) {
    const int64_t t = b / p.parts;
    const int q = int(b - t * p.parts);
    it_start = t * p.slices + part_begin(p, q);
    it_end = t * p.slices + part_begin(p, q + 1);
  }
  unsigned int *flags = g_simt_flags + (p.epoch % kFlagRegions) * kMaxPersistentBlocks;
  for (int64_t it = it_start; it < it_end;) {
    const int tile = p.dp_tiles + int(it / p.slices);
    const int s_begin = int(it % p.slices);
    const int64_t rest = it_end - it;
    const int s_end = rest < int64_t(p.slices - s_begin) ? s_begin + int(rest) : p.slices;
    int tm, tn;
    tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
    const int m0 = tm * Cf::BM, n0 = tn * Cf::BN;
    blk.mainloop(p, smem, m0, n0, s_begin, s_end, &a_map, &b_map, bars, phases);
    if (s_begin == 0 && s_end == p.slices) {
      blk.template epilogue<false>(p, m0, n0, smem);
    } else if (s_end == p.slices) {
      // Slices [s_begin, S): store the partial sums, then raise this block's flag.
      blk.template epilogue<false>(p, m0, n0, smem);
      __syncthreads();
      if (threadIdx.x == 0 && int(b) != p.drop_signal_block) {
        __threadfence();
        store_release(&flags[b], p.epoch);
      }
    } else {
      // Slices [s_begin, s_end) with s_end < S: the next block holds the slices
      // from s_end on and has stored their sum into C; wait for it, add.
      if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        while (load_acquire(&flags[b + 1]) != p.epoch) {
          if (int64_t(global_timer_ns() - t0) > p.wait_limit_ns) {
            atomicOr(&g_simt_status, 1u);
            break;
          }
          __nanosleep(128);
        }
      }
      __syncthreads();
      blk.template epilogue<true>(p, m0, n0, smem);
      if (s_begin > 0) {
        // A middle share (small problems only): C now holds the sum of slices
        // [s_begin, S), which the previous block waits for.
        __syncthreads();
        if (threadIdx.x == 0 && int(b) != p.drop_signal_block) {
          __threadfence();
          store_release(&flags[b], p.epoch);
        }
      }
    }
    it += s_end - s_begin;
  }
}

// The small-problem split whose blocks reduce the split tiles together: every
// block takes an equal share of all tiles' K-slices -- at most two segments,
// the end of one tile and the start of the next -- and stores the partial
// sums of a segment that is not a whole tile into its slot of `partials`
// (slot 2 b + segment, BM x BN floats, row-major); the blocks sharing a tile
// then reduce it together.  A kernel of its own, so that the code of the
// other kernels is compiled exactly as without it.
template <class Cf, int kACopy, bool kVecC>
__global__ void __launch_bounds__(Cf::kThreads, Cf::kMinBlocks)
gemm_simt_reduce_kernel(const __grid_constant__ CUtensorMap a_map,
                        const __grid_constant__ CUtensorMap b_map, const SimtParams p,
                        float *partials) {
  extern __shared__ __align__(16) float smem_raw[];
  constexpr int kRingFloats = Cf::kStages * Cf::template stage_floats<kACopy>();
  // The ring on a 128-byte boundary, then one mbarrier per stage.
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  float *smem = smem_raw + (base - raw) / 4;
  const uint32_t bars = base + uint32_t(kRingFloats * 4);
  uint32_t phases = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < Cf::kStages; ++i) mbar_init(bars + 8u * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  SimtBlock<Cf, kACopy, kVecC> blk;
  blk.init_lanes();

  // Small problems reduced together: this block's equal share of all
  // tiles' K-slices, at most two segments, each leaving its partial sums in
  // its slot and raising the slot's flag; only then does the block wait, to
  // reduce its split tiles with the other blocks sharing them, so every
  // flag is raised before any block waits.  One run-time loop keeps one
  // copy of the mainloop.
  const int64_t g = gridDim.x, b = blockIdx.x;
  unsigned int *flags = g_simt_flags + (p.epoch % kFlagRegions) * kMaxPersistentBlocks;
  constexpr int64_t kSlotFloats = int64_t(Cf::BM) * Cf::BN;
  const int64_t it_begin = share_begin(p.sk_iters, g, b);
  const int64_t it_end = share_begin(p.sk_iters, g, b + 1);
  for (int64_t it = it_begin; it < it_end;) {
    const int tile = int(it / p.slices), s_begin = int(it % p.slices);
    const int64_t rest = it_end - it;
    const int s_end = rest < int64_t(p.slices - s_begin) ? s_begin + int(rest) : p.slices;
    const int seg = it == it_begin ? 0 : 1;
    it += s_end - s_begin;
    int tm, tn;
    tile_coords(tile, p.tiles_m, p.tiles_n, tm, tn);
    const int m0 = tm * Cf::BM, n0 = tn * Cf::BN;
    blk.mainloop(p, smem, m0, n0, s_begin, s_end, &a_map, &b_map, bars, phases);
    if (s_begin == 0 && s_end == p.slices) {
      blk.template epilogue<false>(p, m0, n0, smem);
      continue;
    }
    blk.store_partial(partials + (2 * b + seg) * kSlotFloats);
    __syncthreads();
    if (threadIdx.x == 0 && int(b) != p.drop_signal_block) {
      __threadfence();
      store_release(&flags[2 * b + seg], p.epoch);
    }
  }
  for (int64_t u = it_begin; u < it_end;) {
    const int tile = int(u / p.slices), s_begin = int(u % p.slices);
    const int64_t rest = it_end - u;
    const int s_end = rest < int64_t(p.slices - s_begin) ? s_begin + int(rest) : p.slices;
    u += s_end - s_begin;
    if (s_begin == 0 && s_end == p.slices) continue;
    blk.reduce_split_tile(p, partials, tile, g, b, flags);
    __syncthreads();
  }
}

// ---- host side ------------------------------------------------------------------

using DefaultConfig = SimtConfig<8, 16, 1, 4, 16, 4, 2>;
// With B copied by TMA, A's transposing copies are the only per-thread ones;
// a 64 x 512 tile on 8 warps (one block per SM, B in two 256-column boxes)
// halves them per thread: 4096^3 64.5 against 63.9 TFLOP/s, 8192 x 8192 x 1024
// 63.3 against 63.1.  Used when its tiles fill two waves of SMs.  (A stored
// K x M, copied by TMA as well, measured no better on it: 4096^3 67.3 against
// 66.9 on the default tile, 8192 x 8192 x 1024 66.1 against 66.7.)
using WideNConfig = SimtConfig<8, 16, 1, 8, 16, 4, 1>;

struct LaunchState {
  std::atomic<uint64_t> configured{0};   // bit per device: smem opt-in done
  std::atomic<int> blocks_per_sm[64];
};

std::atomic<unsigned int> g_epoch{0};
std::atomic<int64_t> g_wait_limit_ns{int64_t(10) * 1000 * 1000 * 1000};
std::atomic<int> g_drop_signal_block{-1};

// Slices by which each part of a tile split per tile is longer than the next
// (measured, TFLOP/s for steps 0 / 1 / 2 / 3: 1024^3 34.6 / 35.8 / 35.8 / 32.4;
// 1000 x 1000 x 2990 44.0 / 44.7 / 42.7 / 42.7; the even split across tile
// boundaries before: 35.2 and 41.5).
constexpr int kChainStep = 1;

// Tiling and work split: fills prm and returns the grid size.
//   * When the tile count leaves the last wave of `slots` resident blocks
//     partly empty: one block per slot, the last full wave plus the remainder
//     split over K (stream-K, two blocks per split tile, one flag per block).
//   * With fewer tiles than slots, the blocks sharing a tile chain their sums
//     through C: each tile in up to four unequal parts when there is room for
//     two blocks per tile (the part holding the end of K -- the first of the
//     chain to store its sum -- the smallest, each earlier part kChainStep
//     slices longer, so the sum handed down the chain arrives while the part
//     receiving it still computes), else equal shares of all tiles' K-slices
//     of at least a quarter of a tile.
//   * Those chains hand a tile's sum over one contributor after another, and
//     element by element where C takes no 16-byte stores.  When C takes none,
//     or when the chains would keep fewer than 2/5 of the slots busy (few
//     tiles), every block instead takes an equal share (at least four slices)
//     and the blocks sharing a tile reduce it together from *partial_slots
//     slots of partial sums (two per block, two flags): 1024 x 1023 x 1024
//     21.5 -> 31.9 TFLOP/s, 512 x 512 x 4096 21.7 -> 39.1, 256^3 1.33 -> 1.67;
//     with most slots busy the unequal chains stay ahead (1024^3 37.0 against
//     32.9, 2048^3 61.9 against 57.9): two blocks sharing an SM progress
//     unequally, which the chains absorb and equal shares wait for.
// Every split needs the blocks co-resident (*cooperative).
int64_t plan_simt(SimtParams &prm, const GemmProblem &p, bool vec_c, bool may_reduce, int BM,
                  int BN, int BK, int64_t slots, bool *cooperative, int64_t *partial_slots) {
  const int64_t tiles_m = (p.M + BM - 1) / BM;
  const int64_t tiles_n = (p.N + BN - 1) / BN;
  const int64_t tiles = tiles_m * tiles_n;
  const int slices = int((p.K + BK - 1) / BK);
  prm.M = int(p.M); prm.N = int(p.N); prm.K = int(p.K);
  prm.A = p.A; prm.lda = p.lda; prm.B = p.B; prm.ldb = p.ldb; prm.C = p.C; prm.ldc = p.ldc;
  prm.tiles_m = int(tiles_m); prm.tiles_n = int(tiles_n);
  prm.slices = slices;
  prm.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  prm.drop_signal_block = g_drop_signal_block.load(std::memory_order_relaxed);
  prm.parts = 0;
  *partial_slots = 0;
  const bool flags_fit = slots > 0 && 2 * slots <= kMaxPersistentBlocks;
  const int64_t rem = slots > 0 ? tiles % slots : 0;
  const bool stream_k = flags_fit && tiles > slots && rem != 0 && rem * 10 < slots * 9 &&
                        slices >= 4;
  int64_t small_blocks = 0;
  bool reduce_split = false;
  if (!stream_k && flags_fit && tiles < slots) {
    const int64_t parts = std::min<int64_t>({4, slots / tiles, slices / 4});
    int64_t chain_blocks = 0;
    if (parts >= 2) {
      chain_blocks = tiles * parts;
    } else {
      const int64_t iters = tiles * slices;
      int64_t share = (iters + slots - 1) / slots;
      share = share > (slices + 3) / 4 ? share : (slices + 3) / 4;
      share = share > 4 ? share : 4;
      const int64_t g = (iters + share - 1) / share;
      if (g * 8 >= tiles * 9) chain_blocks = g;
    }
    if (may_reduce && (!vec_c || chain_blocks * 5 < slots * 2)) {
      const int64_t g = std::min<int64_t>(slots, tiles * slices / 4);
      if (g * 8 >= tiles * 9) {
        small_blocks = g;
        reduce_split = true;
      }
    }
    if (!reduce_split && chain_blocks > 0) {
      small_blocks = chain_blocks;
      if (parts >= 2) {
        int step = kChainStep;
        while (step > 0 && slices - step * parts * (parts - 1) / 2 < 4 * parts) --step;
        const int base = int((slices - step * parts * (parts - 1) / 2) / parts);
        prm.parts = int(parts);
        prm.part_step = step;
        prm.part_base = base;
        prm.part_rem = int(slices - step * parts * (parts - 1) / 2 - base * parts);
      }
    }
  }
  *cooperative = stream_k || small_blocks > 0;
  if (*cooperative) {
    const int64_t sk_tiles = stream_k ? rem + slots : tiles;
    prm.dp_tiles = int(tiles - sk_tiles);
    prm.sk_iters = sk_tiles * slices;
    unsigned int e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    if (e == 0) e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    prm.epoch = e;
    if (reduce_split) *partial_slots = 2 * small_blocks;
    return stream_k ? slots : small_blocks;
  }
  prm.dp_tiles = int(tiles);
  prm.sk_iters = 0;
  prm.epoch = 0;
  return tiles;
}

// Shared-memory opt-in and the resident blocks per SM of one kernel, once per device.
template <class Kernel>
cudaError_t configure(Kernel kernel, int threads, int smem_bytes, LaunchState &state,
                      const DeviceInfo &dev, int *blocks_per_sm) {
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(state.configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem_bytes);
    if (e != cudaSuccess) return e;
    state.blocks_per_sm[dev.id & 63].store(nb, std::memory_order_relaxed);
    state.configured.fetch_or(bit, std::memory_order_release);
  }
  *blocks_per_sm = state.blocks_per_sm[dev.id & 63].load(std::memory_order_relaxed);
  return cudaSuccess;
}

// kSmall: the tile configuration small problems use, which therefore has a
// kernel for the reduced split as well (the 64 x 512 tile serves products of
// at least two waves only).
template <class Cf, int kACopy, bool kVecC, bool kSmall>
cudaError_t launch_variant(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream) {
  static LaunchState state, state_reduce;
  auto kernel = gemm_simt_kernel<Cf, kACopy, kVecC>;
  constexpr int kSmemBytes = Cf::template smem_bytes<kACopy>();
  int blocks_per_sm = 0, blocks_per_sm_reduce = 0;
  cudaError_t e = configure(kernel, Cf::kThreads, kSmemBytes, state, dev, &blocks_per_sm);
  if (e != cudaSuccess) return e;
  blocks_per_sm_reduce = blocks_per_sm;
  if constexpr (kSmall) {   // the 64 x 512 tile never takes the reduced split
    e = configure(gemm_simt_reduce_kernel<Cf, kACopy, kVecC>, Cf::kThreads, kSmemBytes,
                  state_reduce, dev, &blocks_per_sm_reduce);
    if (e != cudaSuccess) return e;
  }
  const int64_t tiles = ((p.M + Cf::BM - 1) / Cf::BM) * ((p.N + Cf::BN - 1) / Cf::BN);
  if (tiles > 0x7fffffff) return cudaErrorInvalidConfiguration;

  CUtensorMap a_map = {}, b_map = {};
  if (kACopy == kCopyTma)       // A stored K x M: boxes of BM columns x BK rows, a[k][m]
    e = encode_f32_2d(&a_map, p.A, p.K, p.M, p.lda, Cf::BM, Cf::BK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  // B stored K x N: boxes of kBBox columns x BK rows, b[k][n]
  e = encode_f32_2d(&b_map, p.B, p.K, p.N, p.ldb, Cf::kBBox, Cf::BK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  SimtParams prm = {};
  bool coop = false;
  int64_t partial_slots = 0;
  // The slots of the reduced split are those its kernel keeps resident.
  const int64_t slots = int64_t(std::min(blocks_per_sm, blocks_per_sm_reduce)) * dev.sm_count;
  int64_t grid = plan_simt(prm, p, kVecC, kSmall, Cf::BM, Cf::BN, Cf::BK, slots, &coop,
                           &partial_slots);
  void *partials = nullptr;
  if (partial_slots > 0 &&
      scratch_alloc(&partials, size_t(partial_slots) * Cf::BM * Cf::BN * sizeof(float), dev,
                    stream) != cudaSuccess) {
    // No scratch for the partial sums: the chains through C need none.
    grid = plan_simt(prm, p, kVecC, false, Cf::BM, Cf::BN, Cf::BK, slots, &coop,
                     &partial_slots);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(Cf::kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  if (coop) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if constexpr (kSmall) {
    if (partials)
      e = cudaLaunchKernelEx(&cfg, gemm_simt_reduce_kernel<Cf, kACopy, kVecC>, a_map, b_map, prm,
                             static_cast<float *>(partials));
    else
      e = cudaLaunchKernelEx(&cfg, kernel, a_map, b_map, prm);
  } else {
    e = cudaLaunchKernelEx(&cfg, kernel, a_map, b_map, prm);
  }
  // Freed in stream order, after the kernel has read the partial sums.
  const cudaError_t f = scratch_free(partials, stream);
  return e != cudaSuccess ? e : f;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A (stored M x K, or K x M with 16-byte rows) and B (stored K x N with
// 16-byte rows) as the kernels read them.
template <bool kVecC>
cudaError_t launch_layout(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream) {
  if (p.transa) return launch_variant<DefaultConfig, kCopyTma, kVecC, true>(p, dev, stream);
  using W = WideNConfig;
  const int64_t wide_tiles = (p.M + W::BM - 1) / W::BM * ((p.N + W::BN - 1) / W::BN);
  return wide_tiles >= 2 * int64_t(dev.sm_count)
             ? launch_variant<W, kCopyTransposing, kVecC, false>(p, dev, stream)
             : launch_variant<DefaultConfig, kCopyTransposing, kVecC, true>(p, dev, stream);
}

}  // namespace

// The product in any layout: an operand the kernels cannot copy by TMA as it
// is stored -- B stored N x K, B stored K x N or A stored K x M with a row
// pitch that is not a multiple of 4 floats or a base off a 16-byte boundary --
// is first restaged into a K x N (K x M) copy with 16-byte rows, in scratch
// allocated and freed on `stream` (the restaging copies read and write the
// operand once).  A stored M x K is read as stored, by transposing copies.
cudaError_t launch_simt(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream) {
  // Rows on 16-byte boundaries: 16-byte aligned base, pitch a multiple of 4 floats.
  const bool tma_b = !p.transb && aligned16(p.B) && p.ldb % 4 == 0;
  const bool tma_a = !p.transa || (aligned16(p.A) && p.lda % 4 == 0);
  GemmProblem q = p;
  const int64_t ld_b = (p.N + 3) / 4 * 4, ld_a = (p.M + 3) / 4 * 4;
  // A restaged copy whose byte count does not fit in size_t cannot be allocated.
  const unsigned __int128 b_need = tma_b ? 0 : (unsigned __int128)p.K * ld_b * sizeof(float);
  const unsigned __int128 a_need = tma_a ? 0 : (unsigned __int128)p.K * ld_a * sizeof(float);
  if (b_need + a_need + 256 > SIZE_MAX) return cudaErrorMemoryAllocation;
  const size_t b_bytes = size_t(b_need);
  const size_t b_span = (b_bytes + 255) / 256 * 256;
  const size_t a_bytes = size_t(a_need);
  void *scratch = nullptr;
  cudaError_t e = cudaSuccess;
  if (b_bytes + a_bytes > 0) {
    e = scratch_alloc(&scratch, b_span + a_bytes, dev, stream);
    if (e != cudaSuccess) return e;
  }
  if (!tma_b) {
    float *b = static_cast<float *>(scratch);
    e = p.transb ? stage_transpose(p.B, p.ldb, p.N, p.K, b, ld_b, dev, stream)
                 : stage_rows(p.B, p.ldb, p.K, p.N, b, ld_b, dev, stream);
    q.B = b;
    q.ldb = ld_b;
    q.transb = 0;
  }
  if (e == cudaSuccess && !tma_a) {
    float *a = reinterpret_cast<float *>(static_cast<char *>(scratch) + b_span);
    e = stage_rows(p.A, p.lda, p.K, p.M, a, ld_a, dev, stream);
    q.A = a;
    q.lda = ld_a;
  }
  const bool vec_c = aligned16(p.C) && p.ldc % 4 == 0 && p.N % 4 == 0;
  if (e == cudaSuccess)
    e = vec_c ? launch_layout<true>(q, dev, stream) : launch_layout<false>(q, dev, stream);
  // Freed in stream order, after the product has read the staged copies.
  const cudaError_t f = scratch_free(scratch, stream);
  return e != cudaSuccess ? e : f;
}

cudaError_t simt_device_status(unsigned int *status, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_simt_status, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_simt_status, &zero, sizeof(unsigned int));
}

void simt_plan_for_testing(int64_t M, int64_t N, int64_t K, int wide, int vec_c, int may_reduce,
                           int64_t slots, int64_t out[9]) {
  GemmProblem p = {M, N, K, nullptr, K, nullptr, N, nullptr, N};
  SimtParams prm = {};
  bool coop = false;
  int64_t partial_slots = 0;
  const int BN = wide ? WideNConfig::BN : DefaultConfig::BN;
  const int64_t grid = plan_simt(prm, p, vec_c != 0, may_reduce != 0, DefaultConfig::BM, BN,
                                 DefaultConfig::BK, slots, &coop, &partial_slots);
  out[0] = grid;
  out[1] = coop ? 1 : 0;
  out[2] = partial_slots;
  out[3] = prm.dp_tiles;
  out[4] = prm.sk_iters;
  out[5] = prm.parts;
  out[6] = prm.part_base;
  out[7] = prm.part_step;
  out[8] = prm.part_rem;
}

void simt_set_test_hooks(int drop_signal_block, int64_t wait_limit_ns) {
  g_drop_signal_block.store(drop_signal_block, std::memory_order_relaxed);
  g_wait_limit_ns.store(wait_limit_ns > 0 ? wait_limit_ns : int64_t(10) * 1000 * 1000 * 1000,
                        std::memory_order_relaxed);
}

}  // namespace tmm
