// The BF16 tensor-core GEMM engine of the linear layer's backward pass, shared
// by the weight gradient (G = A^T dY, then the DGE factor) and the input
// gradient (dX = dY W^T).
//
// Both products are C[R x C] = sum over L of P[r, l] * Q[c, l] with BF16 P and Q
// and an fp32 result:
//   weight gradient: R = K features, C = N outputs, L = M tokens; P = A and Q = dY
//     are stored with the reduction (token) dimension strided, i.e. MN-major;
//   input gradient:  R = M tokens, C = K features, L = N outputs; P = dY and
//     Q = W are stored with the reduction dimension contiguous, i.e. K-major.
// TMA loads [64 x 64] BF16 boxes with 128-byte swizzle and tcgen05.mma
// kind::f16 reads them through MN-major or K-major descriptors, so no operand
// is ever transposed in memory.
//
// Accumulation precision: the tensor core's fp32 accumulation drifts by about
// 1e-9 x (number of accumulated products) relative (a biased, truncation-like
// error), which would exceed 1e-5 at 16k.  The reduction range of every tile is
// therefore split into chunks of 32 x 64 (16 x 64 where a split tail's halves
// come out more even that way); each chunk is accumulated in
// one of two TMEM buffers and the epilogue warps add it into fp32 registers
// (round to nearest), so the error stays at the chunk level (chunks of 2048
// products: about 2e-6 of the sum, against 1e-6 for 1024 and 4.4e-6 for 4096,
// measured on the 13B shapes, where 2048 was 1-5% faster than 1024).  While the
// epilogue drains one buffer the MMA warp fills the other.
//
// Roles (18 warps): warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer,
// warps 2-17 epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (one output row per
// thread) and columns (w-2)/4 * 64 .. +63 of the 256-wide tile, adding each
// chunk into fp32 registers.  After the last chunk of a tile the warp hands its
// sums, 16 rows x 32 columns at a time, through a swizzled staging tile to the
// epilogue functor, which sees coalesced row chunks (lane l: 4 columns, chunk
// l % 8, of rows l / 8 + 4 i), while the tensor core already fills both TMEM
// buffers with the next tile.  Sixteen epilogue warps (64 sums per thread, not
// 128) keep this final pass short enough to hide behind the two chunks the
// tensor core accumulates meanwhile; with eight, the DGE factor arithmetic
// (latency-bound at two warps per scheduler) stalled the MMAs at every tile.
// Every mbarrier wait is bounded; on expiry the
// CTA records FP4_FLAG_TIMEOUT, drains its TMA loads and MMAs, frees TMEM and
// exits.
//
// Split tail: when the last wave of tiles would occupy at most half of the CTA
// pairs, each of its tiles is computed as two halves of the reduction range on
// two pairs (work items after the whole tiles, one per pair).  Each half
// publishes its fp32 sums to the caller's workspace and counts itself in; the
// half that counts second adds the other's sums to its own (a + b, so the
// result does not depend on which half finishes first) and runs the epilogue.
// No CTA ever waits for another.
//
// PAIR: tiles of 256 x 256 per CTA pair (a cluster of two CTAs on two SMs): each
// CTA loads its 128 rows of P and 128 of the tile's 256 rows of Q per stage (32
// KB instead of 48 KB for the same MMA work), the leader issues M = 256
// tcgen05 MMAs (cta_group::2), and each CTA's TMEM holds its 128 rows x 256
// columns.  Short reduction loops run single-CTA 128 x 256 tiles.
//
// The epilogue functor provides
//   void prefetch(int row0, int col0, int lane) const;    called when a tile's last chunk starts:
//                                                          the warp's 32 rows x 64 columns follow
//   struct Pre;                                           values loaded before the block is staged
//   Pre load(int row0, int gcol, bool col_ok, int lane) const;   rows row0 + lane / 8 + 4 i (i < 4)
//   void store(const Pre&, int i, int grow, int gcol, float4 g) const;   4 results of row grow
#pragma once

#include "common.cuh"

namespace fp4 {
namespace bwd {

constexpr int kBM = 128;      // output rows per CTA tile
constexpr int kBN = 256;      // output columns per tile
constexpr int kBT = 64;       // reduction elements per stage
constexpr int kMmaT = 16;     // reduction elements per MMA (BF16 K = 16)
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + 32 * kEpiWarps;   // 576 (18 warps: up to 5 per scheduler, so 96 registers)
constexpr int kNAcc = 2;
constexpr int kChunkLong = 32;    // stages (of 64) per TMEM accumulation chunk: 2048 reduction elements,
constexpr int kChunkShort = 16;   // or 1024 when a split tail would halve an odd number of long chunks
constexpr int kEpiCols = kBN / (kEpiWarps / 4);  // columns per epilogue warp (64)
constexpr int kBlk = 32;                         // epilogue block: 32 rows x 32 columns per warp,
constexpr int kHalf = 16;                        // staged 16 rows at a time
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 64;                          // elements per TMA box side (128 bytes of BF16)
constexpr int kBoxBytes = kBox * kBT * 2;         // 8 KB
// epilogue staging per warp: 16 rows x 32 fp32 columns (128-byte swizzle), read
// back as coalesced row chunks (TMA stays free for the main loop's stages)
constexpr int kOutBytes = kHalf * kBlk * 4;       // 2 KB
constexpr int kEpiWarpBytes = kOutBytes;
constexpr int kGroupRows = 8;                     // tile raster: groups of 8 row blocks

template <bool KMAJOR, bool PAIR>
struct Cfg {
  static constexpr int kCtas = PAIR ? 2 : 1;
  static constexpr int kBCols = kBN / kCtas;                  // Q rows (output columns) per CTA
  static constexpr int kAStage = (kBM / kBox) * kBoxBytes;    // 16 KB
  static constexpr int kBStage = (kBCols / kBox) * kBoxBytes; // 16 or 32 KB
  static constexpr int kStageBytes = kAStage + kBStage;
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kDataBytes = kStages * kStageBytes + kEpiWarps * kEpiWarpBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kNAcc + 1;
  static constexpr int kSmemBytes = 1024 + kDataBytes + 8 * kNumBars + 16;
  // Instruction descriptor, kind::f16: fp32 accumulator (bit 4), A and B BF16
  // (bits 7, 10), A and B MN-major (bits 15, 16) unless K-major, N = 256,
  // M = 128 per CTA.
  static constexpr uint32_t kMajorBits = KMAJOR ? 0u : ((1u << 15) | (1u << 16));
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | kMajorBits |
                                     (uint32_t(kBN >> 3) << 17) | (uint32_t((kBM * kCtas) >> 4) << 24);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget exceeded");
};

struct Shape {
  int R, C, L;        // output rows, output columns, reduction length
  int chunk;          // stages per accumulation chunk (kChunkLong or kChunkShort; plan_split picks it)
  int q_wrap;         // > 0: Q's reduction index is taken modulo q_wrap (a multiple of kBT), so
                      // P's reduction may hold several parts that all meet the same Q; 0: none
  int whole, split;   // tiles computed whole, then `split` tiles computed as two halves
  float* part;        // split > 0: the halves' partial sums (SplitPlan layout)
  uint32_t* cnt;      // split > 0: one arrival counter per tile, warp and CTA, zeroed before launch
  uint32_t* status;
  uint64_t wait_ns;
};

// One unit of a pair's work: a whole tile (slot < 0) or one half of a split
// tile (slot = 2 x split index + half) over chunks [c0, c1).
struct Work {
  int tile, c0, c1, slot;
};

// Work items are dealt round robin: items [0, whole) are whole tiles and
// [whole, whole + 2 split) the halves.  whole is a multiple of the number of
// pairs whenever split > 0, so every half runs in the last round on its own pair.
__device__ __forceinline__ bool work_item(int k, int pair_id, int npairs, int nchunks, const Shape& p, Work& w) {
  const int item = pair_id + k * npairs;
  if (item < p.whole) {
    w.tile = item;
    w.c0 = 0;
    w.c1 = nchunks;
    w.slot = -1;
    return true;
  }
  const int s = item - p.whole;
  if (s >= 2 * p.split) return false;
  w.tile = p.whole + (s >> 1);
  w.c0 = (s & 1) ? nchunks / 2 : 0;
  w.c1 = (s & 1) ? nchunks : nchunks / 2;
  w.slot = s;
  return true;
}

// Tile t -> (row block, column block): groups of kGroupRows row blocks, row
// blocks fastest within a group, so the CTAs running at one time share few
// panels of P and Q in L2.
__device__ __forceinline__ void tile_coords(int t, int num_r, int num_n, int& rb, int& nb) {
  const int per_group = kGroupRows * num_n;
  const int g = t / per_group, in = t - g * per_group;
  const int r0 = g * kGroupRows;
  const int gsize = num_r - r0 < kGroupRows ? num_r - r0 : kGroupRows;
  rb = r0 + in % gsize;
  nb = in / gsize;
}

template <bool KMAJOR, bool PAIR, class Epi>
__device__ __forceinline__ void run(const CUtensorMap& tmA, const CUtensorMap& tmB, const Shape& p,
                                    const Epi& epi) {
  using C = Cfg<KMAJOR, PAIR>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * C::kAStage;
  uint8_t* sEpi = smem + kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kDataBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  const uint32_t accf0 = empty0 + 8 * kStages;
  const uint32_t acce0 = accf0 + 8 * kNAcc;
  const uint32_t done_bar = acce0 + 8 * kNAcc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // 0: the CTA that issues the MMAs

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < kNAcc; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, C::kCtas * kEpiWarps);
    }
    mbar_init(done_bar, 1);
    if constexpr (PAIR) fence_mbar_init_cluster();
    else fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_for<PAIR>(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  cta_sync<PAIR>();   // (pair) both CTAs' barriers exist before either CTA signals the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  constexpr int kTileR = kBM * C::kCtas;   // output rows per tile (per pair)
  const int num_r = (p.R + kTileR - 1) / kTileR;
  const int num_n = (p.C + kBN - 1) / kBN;
  const int lblocks = (p.L + kBT - 1) / kBT;
  const int chunk_stages = p.chunk;
  const int nchunks = (lblocks + chunk_stages - 1) / chunk_stages;
  const int pair_id = int(blockIdx.x) / C::kCtas, npairs = int(gridDim.x) / C::kCtas;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    Work w;
    for (int k = 0; ok && work_item(k, pair_id, npairs, nchunks, p, w); ++k) {
      int rb, nb;
      tile_coords(w.tile, num_r, num_n, rb, nb);
      const int arow = rb * kTileR + int(rank) * kBM;          // this CTA's 128 rows of P
      const int bcol = nb * kBN + int(rank) * C::kBCols;       // this CTA's rows of Q
      const int lb_end = w.c1 * chunk_stages < lblocks ? w.c1 * chunk_stages : lblocks;
      for (int lb = w.c0 * chunk_stages; lb < lb_end; ++lb) {
        if (!mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          // completion is counted on the MMA-issuing CTA's full barrier
          const uint32_t fb = full0 + 8 * stage;
          if (rank == 0) mbar_arrive_expect_tx(fb, C::kCtas * C::kStageBytes);
          const uint32_t a_dst = smem_u32(sA + stage * C::kAStage);
          const uint32_t b_dst = smem_u32(sB + stage * C::kBStage);
          // box coordinates (x = the contiguous dimension): K-major boxes hold
          // 64 reduction elements of 64 rows, MN-major boxes 64 rows of 64
          // reduction elements
#pragma unroll
          for (int h = 0; h < kBM / kBox; ++h) {
            const int r = arow + h * kBox, l = lb * kBT;
            tma_load_2d_to<PAIR>(a_dst + h * kBoxBytes, &tmA, fb, KMAJOR ? l : r, KMAJOR ? r : l);
          }
#pragma unroll
          for (int h = 0; h < C::kBCols / kBox; ++h) {
            const int r = bcol + h * kBox, l = p.q_wrap > 0 ? (lb * kBT) % p.q_wrap : lb * kBT;
            tma_load_2d_to<PAIR>(b_dst + h * kBoxBytes, &tmB, fb, KMAJOR ? l : r, KMAJOR ? r : l);
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    // every stage this CTA filled has been released by the MMAs (so its loads
    // have landed and no commit is still on its way) before the CTA may exit
    for (int s = 0; s < kStages; ++s) {
      const uint32_t n_s = issued / kStages + (uint32_t(s) < issued % kStages ? 1u : 0u);
      if (n_s > 0 && !mbar_wait_warp(empty0 + 8 * s, (n_s - 1) & 1u, p.wait_ns) && lane == 0)
        atomicOr(p.status, FP4_FLAG_TIMEOUT);
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------ MMA issuer (the pair's leader)
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
    Work w;
    for (int k = 0; ok && work_item(k, pair_id, npairs, nchunks, p, w); ++k) {
      for (int ch = w.c0; ch < w.c1 && ok; ++ch) {
        const int lb0 = ch * chunk_stages;
        const int lb1 = lb0 + chunk_stages < lblocks ? lb0 + chunk_stages : lblocks;
        if (!mbar_wait_warp(acce0 + 8 * acc, acc_phase ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + uint32_t(acc * kBN);
        for (int lb = lb0; lb < lb1; ++lb) {
          if (!mbar_wait_warp(full0 + 8 * stage, phase, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = a_base + stage * C::kAStage, b0 = b_base + stage * C::kBStage;
#pragma unroll
            for (int k = 0; k < kBT / kMmaT; ++k) {
              // K-major, 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024
              // bytes apart (SBO); 16 elements = 32 bytes further per MMA.
              // MN-major: 64-row atoms kBoxBytes apart (LBO), 8-element groups
              // 1024 bytes apart (SBO); 16 elements = 2048 bytes per MMA.
              const uint32_t koff = KMAJOR ? uint32_t(k * kMmaT * 2) : uint32_t(k * kMmaT * 128);
              const uint32_t lbo = KMAJOR ? 16u : uint32_t(kBoxBytes);
              const uint64_t ad = smem_desc_sw128(a0 + koff, lbo, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + koff, lbo, 1024);
              if constexpr (PAIR) mma_f16_pair(d_tmem, ad, bd, C::kIdesc, (lb != lb0 || k != 0) ? 1u : 0u);
              else mma_f16(d_tmem, ad, bd, C::kIdesc, (lb != lb0 || k != 0) ? 1u : 0u);
            }
            commit_to<PAIR>(empty0 + 8 * stage, 0x3);   // the stage is free (in both CTAs of a pair)
          }
          __syncwarp();
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) commit_to<PAIR>(accf0 + 8 * acc, 0x3);   // the chunk's accumulator(s) are ready
        __syncwarp();
        if (++acc == kNAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    if (lane == 0) commit_to<PAIR>(done_bar, 0x1);
    __syncwarp();
    if (!mbar_wait_warp(done_bar, 0, p.wait_ns) && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------ chunk promotion + epilogue (own 128 rows)
    const int ew = warp - 2;
    const int q = warp & 3;
    const int c_base = (ew / 4) * kEpiCols;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    uint8_t* out_s = sEpi + ew * kEpiWarpBytes;          // 16 x 32 fp32, 128-byte swizzle
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    constexpr int kNBlk = kEpiCols / kBlk;
    Work w;
    for (int k = 0; ok && work_item(k, pair_id, npairs, nchunks, p, w); ++k) {
      int rb, nb;
      tile_coords(w.tile, num_r, num_n, rb, nb);
      const int row0 = rb * kTileR + int(rank) * kBM + q * 32;  // first output row of this warp's 32-row slab
      float sum[kEpiCols];
#pragma unroll
      for (int c = 0; c < kEpiCols; ++c) sum[c] = 0.0f;
      for (int ch = w.c0; ch < w.c1; ++ch) {
        // what the final pass reads is fetched into L2 while the last chunk accumulates
        if (ch + 1 == w.c1) epi.prefetch(row0, nb * kBN + c_base, lane);
        // the warp leaves the wait converged and with one verdict (tcgen05.ld is warp-wide)
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(accf0 + 8 * acc, acc_phase, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kEpiCols; c += 32) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tmem + lane_base + uint32_t(acc * kBN + c_base + c), r0);
          tmem_ld16(tmem + lane_base + uint32_t(acc * kBN + c_base + c + 16), r1);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            sum[c + t] += __uint_as_float(r0[t]);
            sum[c + 16 + t] += __uint_as_float(r1[t]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_on_issuer<PAIR>(acce0 + 8 * acc);
        if (++acc == kNAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) break;
      if (row0 >= p.R) continue;
      if (w.slot >= 0) {
        // half of a split tile: publish this warp's sums (thread-major, coalesced),
        // count in, and finish the tile only if the other half is already in
        constexpr int kVec = kEpiCols / 4;
        const size_t wbase = ((size_t(w.slot) * C::kCtas + rank) * kEpiWarps + ew) * kVec * 32;
        float4* mine = reinterpret_cast<float4*>(p.part) + wbase;
#pragma unroll
        for (int v = 0; v < kVec; ++v)
          mine[v * 32 + lane] = make_float4(sum[4 * v], sum[4 * v + 1], sum[4 * v + 2], sum[4 * v + 3]);
        __threadfence();   // each lane's stores are visible before the count
        __syncwarp();
        uint32_t before = 0;
        if (lane == 0)
          before = atomicAdd(p.cnt + (size_t(w.slot >> 1) * C::kCtas + rank) * kEpiWarps + ew, 1u);
        before = __shfl_sync(0xFFFFFFFFu, before, 0);
        if (before == 0) continue;   // the other half finishes these rows
        __threadfence();
        const float4* other = reinterpret_cast<const float4*>(p.part) +
                              ((size_t(w.slot ^ 1) * C::kCtas + rank) * kEpiWarps + ew) * kVec * 32;
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
          const float4 o = __ldcg(other + v * 32 + lane);
          sum[4 * v] += o.x;
          sum[4 * v + 1] += o.y;
          sum[4 * v + 2] += o.z;
          sum[4 * v + 3] += o.w;
        }
      }
      // the sums go through the staging tile to the functor as coalesced row
      // chunks; this runs while the tensor core starts the next tile
#pragma unroll
      for (int j = 0; j < kNBlk; ++j) {
        const int col0 = nb * kBN + c_base + j * kBlk;
        if (col0 >= p.C) break;  // same for the whole warp
        const int c = lane & 7, gcol = col0 + 4 * c;
        const bool col_ok = gcol < p.C;   // C % 8 == 0: the 4 columns are all in or all out
#pragma unroll
        for (int h = 0; h < kBlk / kHalf; ++h) {
          const int hrow0 = row0 + h * kHalf;
          // the functor's loads first (one memory latency), then the staging
          const typename Epi::Pre pre = epi.load(hrow0, gcol, col_ok, lane);
          __syncwarp();  // the staging tile is free
          if ((lane >> 4) == h) {
            // lanes 16h..16h+15 hold rows 16h..16h+15: staged row lane % 16, chunk k at k ^ (lane & 7)
            uint8_t* orow = out_s + (lane & (kHalf - 1)) * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(orow + ((k ^ (lane & 7)) << 4)) =
                  make_float4(sum[j * kBlk + 4 * k], sum[j * kBlk + 4 * k + 1], sum[j * kBlk + 4 * k + 2],
                              sum[j * kBlk + 4 * k + 3]);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < kHalf / 4; ++i) {
            const int r = (lane >> 3) + 4 * i;
            const int grow = hrow0 + r;
            if (grow < p.R && col_ok) {
              const float4 g = *reinterpret_cast<const float4*>(out_s + r * 128 + ((c ^ (r & 7)) << 4));
              epi.store(pre, i, grow, gcol, g);
            }
          }
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  }

  // (pair) neither CTA leaves or frees TMEM while its partner may still signal it
  __syncwarp();
  tc_fence_before();
  cta_sync<PAIR>();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_for<PAIR>(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

// CTA pairs once the reduction loop is long (32 or more stages of 64); short
// loops keep single-CTA tiles.
inline bool use_pairs(int64_t red) { return red >= 2048; }

// Tile count, split tail and workspace layout of one backward GEMM on a device
// with `sms` SMs: [counters, 256-byte aligned][partial sums].
struct SplitPlan {
  int64_t tiles, units, whole, split;
  int chunk;   // stages per accumulation chunk when the split tail runs
  size_t cnt_bytes, part_bytes, total;
};

// Stages of the longer half when a tile of `stages` stages is split at the
// middle chunk boundary (chunks of `chunk` stages; as work_item splits them).
inline int64_t split_half_stages(int64_t stages, int chunk) {
  const int64_t nchunks = (stages + chunk - 1) / chunk;
  const int64_t h0 = (nchunks / 2) * chunk < stages ? (nchunks / 2) * chunk : stages;
  return h0 > stages - h0 ? h0 : stages - h0;
}

inline SplitPlan plan_split(int64_t rows, int64_t cols, int64_t red, int sms) {
  const int ctas = use_pairs(red) ? 2 : 1;
  SplitPlan sp{};
  sp.tiles = ((rows + kBM * ctas - 1) / (kBM * ctas)) * ((cols + kBN - 1) / kBN);
  sp.units = sms / ctas;
  const int64_t stages = (red + kBT - 1) / kBT;
  const int64_t rem = sp.tiles % sp.units;
  const bool tail = rem > 0 && 2 * rem <= sp.units;
  // long chunks, unless the split tail's halves would come out more even with
  // short ones (the tail's time is its longer half); the choice depends on the
  // shape only, so a call with and without a workspace sums the same chunks
  const int64_t nlong = (stages + kChunkLong - 1) / kChunkLong, nshort = (stages + kChunkShort - 1) / kChunkShort;
  sp.chunk = kChunkLong;
  if (tail && nshort >= 2 &&
      (nlong < 2 || split_half_stages(stages, kChunkShort) < split_half_stages(stages, kChunkLong)))
    sp.chunk = kChunkShort;
  const int64_t nchunks = (stages + sp.chunk - 1) / sp.chunk;
  sp.split = (tail && nchunks >= 2) ? rem : 0;
  sp.whole = sp.tiles - sp.split;
  sp.cnt_bytes = (size_t(sp.split) * ctas * kEpiWarps * 4 + 255) / 256 * 256;
  sp.part_bytes = size_t(2 * sp.split) * ctas * kEpiWarps * kEpiCols * 32 * 4;
  sp.total = sp.split ? sp.cnt_bytes + sp.part_bytes : 0;
  return sp;
}

inline fp4_status schedule(Shape& s, const SplitPlan& sp, void* workspace, size_t ws_bytes, cudaStream_t cs) {
  s.whole = int(sp.tiles);
  s.split = 0;
  s.part = nullptr;
  s.cnt = nullptr;
  s.chunk = sp.chunk;   // a function of the shape alone, with or without the split
  if (workspace == nullptr || sp.split == 0) return FP4_OK;
  if (ws_bytes < sp.total) return FP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FP4_ERR_ALIGNMENT;
  s.whole = int(sp.whole);
  s.split = int(sp.split);
  s.cnt = static_cast<uint32_t*>(workspace);
  s.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + sp.cnt_bytes);
  if (cudaMemsetAsync(s.cnt, 0, sp.cnt_bytes, cs) != cudaSuccess) return launch_status();
  return FP4_OK;
}

// Launches kernel<...> (a __global__ wrapper of run) with one CTA (pair) per
// work item up to one per SM (pair), in clusters of two when PAIR.
template <bool KMAJOR, bool PAIR, class Kern, class... Args>
fp4_status launch(Kern kern, const Shape& s, int sms, cudaStream_t cs, Args... args) {
  using C = Cfg<KMAJOR, PAIR>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t items = int64_t(s.whole) + 2 * int64_t(s.split);
  const int64_t units = sms / C::kCtas;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(unsigned(C::kCtas * (items < units ? items : units)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = cs;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(C::kCtas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return launch_status();
  return launch_status();
}

}  // namespace bwd
}  // namespace fp4
