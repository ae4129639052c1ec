// Forward FP4 GEMM of the quantized linear layer on sm_103a tensor cores.
//
// The page "首个 FP4 精度的大模型训练框架来了" (czzqal.com), GeMM passage,
// describes a custom FP4 GEMM kernel that stages FP4 A and B through FP16 in
// shared memory and emulates the FP4 tile multiply on FP8 tensor cores (no FP4
// hardware existed then).  sm_103a multiplies E2M1 natively, so this kernel
// instead feeds the packed codes by TMA straight into 128-byte-swizzled shared
// memory and runs tcgen05.mma kind::mxf4 with every UE8M0 block scale equal to
// 1.0, accumulating exactly in fp32 in tensor memory (every product is a
// multiple of 1/4 of magnitude <= 36, so sums stay exact for K <= 16384).
//
// The epilogue applies the per-row and per-column scales (they factor out of
// the K-sum: A is quantized per token and W per channel, granularity passage)
// and adds the sparse compensation dA*W (outlier passage), then stores Y.
//
// Structure: persistent CTAs (one per SM), 320 threads:
//   warp 0    TMA producer (one elected lane issues),
//   warp 1    TMEM allocator and MMA issuer (one lane issues, commits to mbarriers),
//   warps 2-9 epilogue: warp w owns TMEM lanes 32*(w%4)..+31 (one output row per
//             thread) and columns (w-2)/4 * BN/2 .. +BN/2 of the tile.
// Tiles are 128 x 240: two 240-column fp32 accumulators plus the 32 scale-factor
// columns fill the 512 TMEM columns exactly, so the epilogue of one tile
// overlaps the main loop of the next.  Each epilogue thread first forms its
// row's compensation sum over the dA entries (one row segment of W per entry,
// all its loads in flight at once) while the tile's main loop still runs, then
// reads the accumulator in groups of 8 columns, scales, adds and stores.
// Every mbarrier wait is bounded; on expiry the CTA records FP4_FLAG_TIMEOUT,
// drains its TMA loads and MMAs, frees TMEM and exits.
//
// Compensation on the tensor cores.  Outliers gather in a few channels, so dA
// has few distinct nonzero columns H.  When the caller passes a workspace and
// |H| <= kHotMax, small prep kernels build, for the columns in H,
//   P  = fl32(dA[:,H] * s_A)   (M x |H|)    and   Q^T = fl32(W[H,:] * s_W)^T  (N x |H|),
// each split exactly into two TF32 parts (x = hi + lo + O(2^-23 |x|)), and the
// GEMM kernel runs, after the FP4 K loop of a tile, three more pipeline stages
// per 32 columns of H: kind::tf32 MMAs of hi*hi, hi*lo and lo*hi into the same
// accumulator (the dropped lo*lo term is below 2^-22 relative).  The epilogue
// then scales acc + P Q^T by 1/(s_A s_W), which equals acc/(s_A s_W) + dA W up to
// fp32 rounding, and does no compensation work of its own.  Without a
// workspace, or with more distinct columns, the epilogue forms the sum itself.
#include <algorithm>

#include "common.cuh"

namespace fp4 {
namespace {

constexpr int kBM = 128;          // rows of A per tile (TMEM lanes)
constexpr int kBKBytes = 128;     // bytes of K per stage = 256 E2M1 values (one swizzle row)
constexpr int kMmaKBytes = 32;    // 64 E2M1 values per MMA
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;

// PAIR: tiles of 256 x BN per CTA pair (a cluster of two CTAs on two SMs): each
// CTA loads its 128 rows of A and half of the tile's BN rows of B per stage, the
// leader CTA issues M = 256 tcgen05 MMAs (cta_group::2), and each CTA's TMEM
// holds its 128 rows x BN columns of the accumulator.  Per SM a stage then
// carries 31 KB instead of 46 KB for the same MMA work, which pays once the K
// loop is long; short K loops run single-CTA 128 x BN tiles.
template <int BN, int NACC, bool PAIR>
struct FwdCfg {
  static constexpr int kCtas = PAIR ? 2 : 1;
  static constexpr int kBRows = BN / kCtas;             // rows of B per CTA
  static constexpr int kAStage = kBM * kBKBytes;
  static constexpr int kBStage = kBRows * kBKBytes;
  static constexpr int kStageBytes = kAStage + kBStage;  // per CTA; the leader's barrier counts the pair's
  static constexpr int kStages = PAIR ? 6 : 4;
  // scale-factor columns (all bytes 0x7F = 2^0) after the accumulators
  static constexpr uint32_t kSfaCol = ((NACC * BN + 15) / 16) * 16;
  static constexpr uint32_t kSfbCol = kSfaCol + 16;
  static constexpr int kBarBytes = 8 * (2 * kStages + 2 * NACC + 1) + 16;
  static constexpr int kInvSwBytes = kEpiWarps * (BN / 2) * 4;
  // per-warp output staging for the TMA store: 32 rows x 80 bytes (40 BF16 or 20 fp32 columns)
  static constexpr int kOutRowBytes = 80;
  static constexpr int kOutBytes = 32 * kOutRowBytes;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiWarps * kOutBytes + kBarBytes + kInvSwBytes;
  static constexpr int kEpiCols = BN / 2;  // columns per epilogue warp
  static_assert(kEpiCols % 8 == 0, "epilogue slices are groups of 8 columns");
  static_assert(kSfbCol + 16 <= kTmemCols, "accumulators and scale factors exceed TMEM");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "invalid N tile");
  static_assert(kStages >= 2, "too few pipeline stages");
  static_assert(kBRows % 8 == 0, "B tile rows must be whole 8-row swizzle atoms");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget exceeded");
};

// Instruction descriptor, kind::mxf4: A and B E2M1 (format 1), both K-major,
// UE8M0 scale type, M = 128 per CTA (256 for a pair), N = BN, dense K = 64, scale-factor ids 0.
template <int BN, bool PAIR>
__host__ __device__ constexpr uint32_t idesc_mxf4() {
  return (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (1u << 23) | (uint32_t((kBM * (PAIR ? 2 : 1)) >> 4) << 24);
}

constexpr int kHotMax = 128;    // distinct dA columns handled on the tensor cores
constexpr int kHotChunk = 32;   // TF32 values per 128-byte row: one pipeline stage of K

// Filled on the device by the prep kernels, read by every CTA of the GEMM.
struct HotInfo {
  int hc;     // distinct nonzero columns of dA
  int hp;     // hc rounded up to a multiple of kHotChunk
  int mode;   // 1: compensation on the tensor cores; 2: the same, packed (3 hc <= kHotChunk)
  int pad;
};

// Instruction descriptor, kind::tf32: fp32 accumulator, A and B TF32, both K-major, M as for mxf4.
template <int BN, bool PAIR>
__host__ __device__ constexpr uint32_t idesc_tf32() {
  return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t((kBM * (PAIR ? 2 : 1)) >> 4) << 24);
}

// Round an fp32 value to TF32 (10 explicit mantissa bits), nearest, ties to even.
__device__ __forceinline__ float round_tf32(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0xFFFu + ((u >> 13) & 1u);
  return __uint_as_float(u & 0xFFFFE000u);
}

// x = hi + lo + r with hi, lo TF32 values and |r| <= 2^-23 |x| (lo is the
// rounded remainder x - hi, which fp32 holds exactly).
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = round_tf32(x);
  lo = round_tf32(x - hi);
}

// Numbers the marked columns in ascending order (word prefix counts), lists
// them, and decides whether the tensor-core path applies.  Run by one CTA of
// 512 threads; reads the bitmap from L2.
__device__ void hot_scan(const uint32_t* bitmap, uint32_t* word_prefix, int32_t* hlist, HotInfo* info, int nwords,
                         uint32_t* wsum) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const uint32_t bits = t < nwords ? __ldcg(bitmap + t) : 0u;
  const uint32_t c = __popc(bits);
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  uint32_t base = 0, total = 0;
  for (int i = 0; i < 16; ++i) {
    total += wsum[i];
    if (i < w) base += wsum[i];
  }
  const uint32_t excl = base + incl - c;
  if (t < nwords) word_prefix[t] = excl;
  const bool on = total > 0 && total <= uint32_t(kHotMax);
  const bool packed = on && 3 * total <= uint32_t(kHotChunk);
  if (on) {
    uint32_t m = bits, h = excl;
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1u;
      hlist[h++] = t * 32 + b;
    }
  }
  if (t == 0) {
    HotInfo hi;
    hi.hc = int(total);
    hi.hp = int((total + kHotChunk - 1) / kHotChunk) * kHotChunk;
    hi.mode = packed ? 2 : (on ? 1 : 0);
    hi.pad = 0;
    *info = hi;
  }
}

// Marks the columns of every dA entry in a K-bit bitmap (cleared beforehand,
// together with `done`).  Outlier columns repeat across rows, so each CTA marks
// a bitmap of its own in shared memory and ORs only its nonzero words into the
// global one; the last CTA to finish numbers the columns (hot_scan) and resets
// `done` for the next call.  512 threads per CTA.
__global__ void __launch_bounds__(512) hot_mark_kernel(const int32_t* __restrict__ rp, const int32_t* __restrict__ ci,
                                                       int M, int K, uint32_t* bitmap, uint32_t* done,
                                                       uint32_t* word_prefix, int32_t* hlist, HotInfo* info,
                                                       uint32_t* status) {
  __shared__ uint32_t local[16384 / 32];
  __shared__ uint32_t wsum[16];
  __shared__ bool last;
  const int nwords = K >> 5;
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) local[w] = 0u;
  __syncthreads();
  const int nnz = __ldg(rp + M);
  bool bad = false;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += gridDim.x * blockDim.x) {
    const int k = __ldg(ci + e);
    if (uint32_t(k) < uint32_t(K)) atomicOr(local + (k >> 5), 1u << (k & 31));
    else bad = true;
  }
  if (bad) atomicOr(status, FP4_FLAG_INTERNAL);
  __syncthreads();
  for (int w = threadIdx.x; w < nwords; w += blockDim.x)
    if (local[w]) atomicOr(bitmap + w, local[w]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  hot_scan(bitmap, word_prefix, hlist, info, nwords, wsum);
  if (threadIdx.x == 0) *done = 0u;
}

// Builds both operands of the compensation product, 256 threads per CTA:
//   CTAs [0, p_ctas): one warp per row i: P[i, 0..hp) = 0, then the row's
//     entries, scaled by s_A[i] and split, at their column numbers (the row's
//     columns are distinct);
//   the rest: one thread per output column j and 4 columns h of H:
//     Q^T[j, h] = fl32(W[H[h], j] * s_W[j]), split; zero for h in [hc, hp).
// Packed mode (3 hc <= 32): the three products sit side by side in the first 32
// columns of the hi arrays, P_hi[i] = [P_hi | P_lo | P_hi | 0], Q_hi[j] =
// [Q_hi | Q_hi | Q_lo | 0], so that one TF32 stage computes all of them.
__global__ void __launch_bounds__(256) hot_build_kernel(
    const int32_t* __restrict__ rp, const int32_t* __restrict__ ci, const float* __restrict__ cv,
    const float* __restrict__ s_a, const uint16_t* __restrict__ W, int64_t ldw, const float* __restrict__ s_w,
    const uint32_t* __restrict__ bitmap, const uint32_t* __restrict__ word_prefix, const int32_t* __restrict__ hlist,
    const HotInfo* __restrict__ info, float* p_hi, float* p_lo, float* q_hi, float* q_lo, int M, int N, int K,
    int p_ctas) {
  const HotInfo hi = *info;
  if (!hi.mode) return;
  if (int(blockIdx.x) < p_ctas) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= M) return;
    float4* ph = reinterpret_cast<float4*>(p_hi + int64_t(row) * kHotMax);
    float4* pl = reinterpret_cast<float4*>(p_lo + int64_t(row) * kHotMax);
    for (int i = lane; i < hi.hp / 4; i += 32) {
      ph[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      pl[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();
    const int e0 = __ldg(rp + row), e1 = __ldg(rp + row + 1);
    const float sa = __ldg(s_a + row);
    for (int e = e0 + lane; e < e1; e += 32) {
      const int k = __ldg(ci + e);
      if (uint32_t(k) >= uint32_t(K)) continue;   // flagged by the marking pass
      const uint32_t wd = __ldg(bitmap + (k >> 5));
      const int h = int(__ldg(word_prefix + (k >> 5)) + __popc(wd & ((1u << (k & 31)) - 1u)));
      float a, b;
      split_tf32(__fmul_rn(__ldg(cv + e), sa), a, b);
      if (hi.mode == 2) {
        float* pr = p_hi + int64_t(row) * kHotMax;
        pr[h] = a;
        pr[hi.hc + h] = b;
        pr[2 * hi.hc + h] = a;
      } else {
        p_hi[int64_t(row) * kHotMax + h] = a;
        p_lo[int64_t(row) * kHotMax + h] = b;
      }
    }
    return;
  }
  const int nj = (N + 255) / 256;
  const int qb = int(blockIdx.x) - p_ctas;
  const int h0 = 4 * (qb / nj);
  if (h0 >= hi.hp) return;
  const int j = (qb % nj) * 256 + threadIdx.x;
  if (j >= N) return;
  const float sw = __ldg(s_w + j);
  if (hi.mode == 2) {
    // packed: row j of Q_hi is [Q_hi | Q_hi | Q_lo | 0] over its first 32 columns
    float* qr = q_hi + int64_t(j) * kHotMax;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int h = h0 + t;
      if (h < hi.hc) {
        float a, b;
        split_tf32(__fmul_rn(bf16_bits_to_float(__ldg(W + int64_t(__ldg(hlist + h)) * ldw + j)), sw), a, b);
        qr[h] = a;
        qr[hi.hc + h] = a;
        qr[2 * hi.hc + h] = b;
      }
    }
    if (h0 == 0)
      for (int x = 3 * hi.hc; x < kHotChunk; ++x) qr[x] = 0.0f;
    return;
  }
  float a[4], b[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int h = h0 + t;
    const float x = h < hi.hc ? __fmul_rn(bf16_bits_to_float(__ldg(W + int64_t(__ldg(hlist + h)) * ldw + j)), sw)
                              : 0.0f;
    split_tf32(x, a[t], b[t]);
  }
  reinterpret_cast<float4*>(q_hi + int64_t(j) * kHotMax)[h0 / 4] = make_float4(a[0], a[1], a[2], a[3]);
  reinterpret_cast<float4*>(q_lo + int64_t(j) * kHotMax)[h0 / 4] = make_float4(b[0], b[1], b[2], b[3]);
}

struct FwdParams {
  const float* s_a;
  const float* s_w;
  const int32_t* rp;
  const int32_t* ci;
  const float* cv;
  const uint16_t* W;
  int64_t ldw;
  void* Y;
  int64_t ldy;
  int y_type;
  int M, N, K;
  const HotInfo* hot;   // null: no tensor-core compensation
  uint32_t* status;
  uint64_t wait_ns;
  int fallback_only;    // run only when dA has more distinct columns than the tensor-core path takes
};

template <int BN, int NACC, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmPh,
                   const __grid_constant__ CUtensorMap tmPl, const __grid_constant__ CUtensorMap tmQh,
                   const __grid_constant__ CUtensorMap tmQl, const FwdParams p) {
  using C = FwdCfg<BN, NACC, PAIR>;
  // as the fallback of the wide kernel: nothing to do unless dA has too many
  // distinct columns for the tensor-core compensation (uniform over the grid)
  if (p.fallback_only && !(p.hot->hc > kHotMax)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::kStages * C::kAStage;
  uint8_t* sOut = smem + C::kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + kEpiWarps * C::kOutBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 2 * NACC + 1);
  float* inv_sw_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + C::kBarBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::kStages;
  const uint32_t accf0 = empty0 + 8 * C::kStages;
  const uint32_t acce0 = accf0 + 8 * NACC;
  const uint32_t done_bar = acce0 + 8 * NACC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // 0: the CTA that issues the MMAs

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmY);
    if (p.hot) {
      prefetch_tmap(&tmPh);
      prefetch_tmap(&tmPl);
      prefetch_tmap(&tmQh);
      prefetch_tmap(&tmQl);
    }
    // full: the leader's counts both CTAs' bytes; empty / acc-full: one multicast
    // commit each; acc-empty (the leader's): the epilogue warps of both CTAs
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < NACC; ++b) {
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

  if (warp >= 2 && warp < 6) {  // unit block scales: every scale byte = 0x7F (2^0)
    const uint32_t lb = uint32_t((warp & 3) * 32) << 16;
    tmem_st8_fill(tmem + lb + C::kSfaCol, 0x7F7F7F7Fu);
    tmem_st8_fill(tmem + lb + C::kSfaCol + 8, 0x7F7F7F7Fu);
    tmem_st8_fill(tmem + lb + C::kSfbCol, 0x7F7F7F7Fu);
    tmem_st8_fill(tmem + lb + C::kSfbCol + 8, 0x7F7F7F7Fu);
    tmem_wait_st();
  }
  tc_fence_before();
  cta_sync<PAIR>();   // (pair) the leader's first MMA reads both CTAs' scale-factor columns
  tc_fence_after();

  constexpr int kTileM = kBM * C::kCtas;   // rows of A per tile (per pair)
  const int num_m = (p.M + kTileM - 1) / kTileM;
  const int num_n = (p.N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int pair_id = int(blockIdx.x) / C::kCtas, npairs = int(gridDim.x) / C::kCtas;
  const int kblocks = (p.K / 2 + kBKBytes - 1) / kBKBytes;
  // tensor-core compensation: 3 stages (hi*hi, hi*lo, lo*hi) per 32 columns of
  // H, or one stage holding all three products when they fit side by side
  // (packed mode: the first stage's loads, chunk 0 of P_hi and Q_hi, are those)
  const bool hot = p.hot != nullptr && p.hot->mode != 0;
  const int hot_stages = hot ? (p.hot->mode == 2 ? 1 : 3 * (p.hot->hp / kHotChunk)) : 0;
  const int nstages = kblocks + hot_stages;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    for (int tile = pair_id; tile < tiles && ok; tile += npairs) {
      const int mb = tile % num_m, nb = tile / num_m;
      const int arow = mb * kTileM + int(rank) * kBM;           // this CTA's 128 rows of A
      const int brow = nb * BN + int(rank) * C::kBRows;         // this CTA's part of the tile's B rows
      for (int kb = 0; kb < nstages; ++kb) {
        if (!mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          // completion is counted on the MMA-issuing CTA's full barrier
          const uint32_t fb = full0 + 8 * stage;
          if (rank == 0) mbar_arrive_expect_tx(fb, C::kCtas * C::kStageBytes);
          const uint32_t da = smem_u32(sA + stage * C::kAStage), db = smem_u32(sB + stage * C::kBStage);
          if (kb < kblocks) {
            tma_load_2d_to<PAIR>(da, &tmA, fb, kb * kBKBytes, arow);
            tma_load_2d_to<PAIR>(db, &tmB, fb, kb * kBKBytes, brow);
          } else {
            // 32 columns of H: P part x Q part, pairs (hi, hi), (hi, lo), (lo, hi);
            // every load names its tensor map directly
            const int hs = kb - kblocks, chunk = hs / 3, pair = hs - 3 * chunk;
            const int x = chunk * kHotChunk;
            if (pair == 2) tma_load_2d_to<PAIR>(da, &tmPl, fb, x, arow);
            else tma_load_2d_to<PAIR>(da, &tmPh, fb, x, arow);
            if (pair == 1) tma_load_2d_to<PAIR>(db, &tmQl, fb, x, brow);
            else tma_load_2d_to<PAIR>(db, &tmQh, fb, x, brow);
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    // every stage this CTA filled has been released by the pair's MMAs (so its
    // loads have landed and no commit is still on its way) before the CTA may exit
    for (int s = 0; s < C::kStages; ++s) {
      const uint32_t n_s = issued / C::kStages + (uint32_t(s) < issued % C::kStages ? 1u : 0u);
      if (n_s > 0 && !mbar_wait_warp(empty0 + 8 * s, (n_s - 1) & 1u, p.wait_ns) && lane == 0)
        atomicOr(p.status, FP4_FLAG_TIMEOUT);
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------ MMA issuer (leader CTA)
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    constexpr uint32_t idesc = idesc_mxf4<BN, PAIR>();
    const uint32_t sfa = tmem + C::kSfaCol, sfb = tmem + C::kSfbCol;
    const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
    for (int tile = pair_id; tile < tiles && ok; tile += npairs) {
      if (!mbar_wait_warp(acce0 + 8 * acc, acc_phase ^ 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + uint32_t(acc * BN);
      for (int kb = 0; kb < nstages; ++kb) {
        if (!mbar_wait_warp(full0 + 8 * stage, phase, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = a_base + stage * C::kAStage, b0 = b_base + stage * C::kBStage;
          // 32 bytes of K per MMA in both kinds: 64 E2M1 values or 8 TF32 values
          if (kb < kblocks) {
#pragma unroll
            for (int k = 0; k < kBKBytes / kMmaKBytes; ++k) {
              const uint64_t ad = smem_desc_sw128(a0 + k * kMmaKBytes, 16, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + k * kMmaKBytes, 16, 1024);
              if constexpr (PAIR) mma_mxf4_pair(d_tmem, ad, bd, idesc, sfa, sfb, (kb | k) != 0 ? 1u : 0u);
              else mma_mxf4(d_tmem, ad, bd, idesc, sfa, sfb, (kb | k) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kBKBytes / kMmaKBytes; ++k) {
              const uint64_t ad = smem_desc_sw128(a0 + k * kMmaKBytes, 16, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + k * kMmaKBytes, 16, 1024);
              if constexpr (PAIR) mma_tf32_pair(d_tmem, ad, bd, idesc_tf32<BN, PAIR>(), 1u);
              else mma_tf32(d_tmem, ad, bd, idesc_tf32<BN, PAIR>(), 1u);
            }
          }
          commit_to<PAIR>(empty0 + 8 * stage, 0x3);   // the stage is free (in both CTAs of a pair)
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) commit_to<PAIR>(accf0 + 8 * acc, 0x3);   // the accumulator(s) are ready
      __syncwarp();
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    // every MMA issued by this thread must finish before TMEM is released
    if (lane == 0) commit_to<PAIR>(done_bar, 0x1);
    __syncwarp();
    if (!mbar_wait_warp(done_bar, 0, p.wait_ns) && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue (both CTAs, own 128 rows)
    constexpr int EC = C::kEpiCols;
    const int q = warp & 3;
    const int c_base = ((warp - 2) / 4) * EC;
    float* inv_sw_w = inv_sw_s + (warp - 2) * EC;
    uint8_t* out_s = sOut + (warp - 2) * C::kOutBytes;
    const int r_local = q * 32 + lane;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const bool raw = (p.y_type == FP4_OUT_RAW_ACC_FP32);
    for (int tile = pair_id; tile < tiles; tile += npairs) {
      const int mb = tile % num_m, nb = tile / num_m;
      const int mrow0 = mb * kTileM + int(rank) * kBM;   // first row of this CTA's rows of the tile
      // this warp's column scales 1/s_W in its own shared-memory slice (no
      // cross-warp barrier, so a warp that gives up on a wait cannot strand others)
      __syncwarp();
      {
        // all of the lane's loads in flight at once, then the reciprocals
        constexpr int kPer = (EC + 31) / 32;
        float sw[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int c = lane + 32 * j, col = nb * BN + c_base + c;
          sw[j] = (c < EC && !raw && col < p.N) ? __ldg(p.s_w + col) : 1.0f;
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j)
          if (lane + 32 * j < EC) inv_sw_w[lane + 32 * j] = 1.0f / sw[j];
      }
      __syncwarp();
      const int row = mrow0 + r_local;
      const bool row_ok = row < p.M;
      float inv_sa = 1.0f;
      int e0 = 0, e1 = 0;
      if (row_ok && !raw) {
        inv_sa = 1.0f / __ldg(p.s_a + row);
        if (p.rp && !hot) {
          e0 = __ldg(p.rp + row);
          e1 = __ldg(p.rp + row + 1);
        }
      }
      const int col_base = nb * BN + c_base;
      int nvalid = p.N - col_base;  // columns of this slice inside the matrix (multiple of 8)
      nvalid = nvalid < 0 ? 0 : (nvalid > EC ? EC : nvalid);
      // compensation sum_e dA[row,k_e] W[k_e, cols] for this row, formed while the
      // tile's main loop still runs (one W row segment per entry, all loads in flight)
      float comp[EC];
#pragma unroll
      for (int c = 0; c < EC; ++c) comp[c] = 0.0f;
      // the (column, value) pairs of the row's first kRegEnt entries are fetched
      // together; W is read in groups of 5 pieces (40 columns) per entry
      constexpr int kRegEnt = 4;
      int kk[kRegEnt];
      float vv[kRegEnt];
#pragma unroll
      for (int j = 0; j < kRegEnt; ++j) {
        kk[j] = 0;
        vv[j] = 0.0f;
        if (e0 + j < e1) {
          kk[j] = __ldg(p.ci + e0 + j);
          vv[j] = __ldg(p.cv + e0 + j);
        }
      }
      for (int e = e0; e < e1; ++e) {
        const int j = e - e0;
        int k;
        float v;
        if (j < kRegEnt) {
          k = kk[0];
          v = vv[0];
#pragma unroll
          for (int i = 1; i < kRegEnt; ++i)
            if (j == i) {
              k = kk[i];
              v = vv[i];
            }
        } else {
          k = __ldg(p.ci + e);
          v = __ldg(p.cv + e);
        }
        if (uint32_t(k) >= uint32_t(p.K)) {   // a column outside W: skipped and reported
          atomicOr(p.status, FP4_FLAG_INTERNAL);
          continue;
        }
        const uint4* wr = reinterpret_cast<const uint4*>(p.W + int64_t(k) * p.ldw + col_base);
#pragma unroll
        for (int g0 = 0; g0 < EC / 8; g0 += 5) {
          uint4 w[5];
#pragma unroll
          for (int g = 0; g < 5; ++g)
            w[g] = (8 * (g0 + g) < nvalid) ? __ldg(wr + g0 + g) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int g = 0; g < 5; ++g) {
            const uint32_t wv[4] = {w[g].x, w[g].y, w[g].z, w[g].w};
#pragma unroll
            for (int t = 0; t < 8; ++t)
              comp[8 * (g0 + g) + t] =
                  fmaf(v, bf16_bits_to_float((wv[t >> 1] >> (16 * (t & 1))) & 0xFFFFu), comp[8 * (g0 + g) + t]);
          }
        }
      }
      // the warp leaves the wait converged and with one verdict (tcgen05.ld is warp-wide)
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(accf0 + 8 * acc, acc_phase, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Y leaves through a per-warp staging buffer (32 rows x 80 bytes) and a TMA
      // store, which writes whole rows and drops what falls outside M x N:
      // 40 columns per pass, as one BF16 store or two fp32 stores of 20 columns.
      const bool bf16_out = (p.y_type == FP4_OUT_BF16);
      const int row0 = mrow0 + q * 32;
      uint8_t* orow = out_s + lane * C::kOutRowBytes;
#pragma unroll
      for (int pc = 0; pc < EC; pc += 40) {
        if (col_base + pc < p.N) {   // warp-uniform
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            if (bf16_out && part == 1) break;
            if (lane == 0) bulk_wait_read_all();   // the previous store has read the buffer
            __syncwarp();
            // 8 columns at a time: read, scale, add, convert and stage
#pragma unroll
            for (int gg = 0; gg < 5; ++gg) {
              // fp32: only the groups that overlap columns 20*part .. +19 of the pass
              if (!bf16_out && !(8 * gg < 20 * part + 20 && 8 * gg + 8 > 20 * part)) continue;
              uint32_t r[8];
              tmem_ld8(tmem + lane_base + uint32_t(acc * BN + c_base + pc + 8 * gg), r);
              tmem_wait_ld();
              float y[8];
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const int c = pc + 8 * gg + t;
                y[t] = raw ? __uint_as_float(r[t]) : __uint_as_float(r[t]) * inv_sa * inv_sw_w[c] + comp[c];
              }
              if (bf16_out) {
                uint32_t pk[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  const __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * t], y[2 * t + 1]);
                  pk[t] = *reinterpret_cast<const uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(orow + 16 * gg) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              } else {
                // fp32: columns 20*part .. +19 of this pass go to the staging row
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                  const int cc = 8 * gg + t - 20 * part;
                  if (cc >= 0 && cc < 20) reinterpret_cast<float*>(orow)[cc] = y[t];
                }
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            const int xcol = col_base + pc + 20 * part;
            if (lane == 0 && row0 < p.M && xcol < p.N) {
              tma_store_2d(&tmY, smem_u32(out_s), xcol, row0);
              bulk_commit_group();
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_on_issuer<PAIR>(acce0 + 8 * acc);   // TMEM buffer free for the next tile
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();
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


// ---------------------------------------------------------------------------
// Wide tiles: 256 x 480 per CTA pair.
//
// The tile's two column halves of 240 share every A stage: per K stage each CTA
// loads its 128 rows of A (16 KB) and 120 rows of W^T for each half (2 x 15 KB),
// and the leader issues one M = 256, N = 240 MMA per half.  Per SM that is
// 46 KB per 960 clk of MMA work (48 B/clk), against 66 B/clk for 256 x 240
// tiles, whose rate the L2 -> shared memory path could barely sustain.  The
// accumulator takes all 480 TMEM columns (plus the 32 scale-factor columns),
// so the next tile cannot start in a second buffer; instead each half has its
// own full / empty barriers and, at a tile's ends, half 0 runs kWLag stages
// ahead of half 1: the epilogue drains half 0 while the tensor core finishes
// half 1, and drains half 1 while the tensor core starts the next tile's half 0.
//
// Work items (host-balanced, see wide_schedule): double tiles (two halves,
// row blocks fastest), then single halves -- the last half of each row block
// when the halves are odd in number, and the doubles of a partial last round
// split in two, so that every pair ends within one half-tile of the others.
// A half narrower than 240 columns (the right edge of W) runs an MMA of that
// width, rounded up to 16; CTA r then loads its W^T rows from r x width / 2.
constexpr int kWHalf = 240;          // columns per half (one MMA)
constexpr int kWBRows = kWHalf / 2;  // W^T rows per CTA per half
constexpr int kWStages = 4;
constexpr int kWLag = 2;             // stages half 0 runs ahead of half 1 at a tile's ends
constexpr int kWEpiWarps = 16;       // 4 per TMEM lane quadrant, each with a column group of each half
constexpr int kWThreads = 64 + 32 * kWEpiWarps;

struct WideCfg {
  static constexpr int kAStage = kBM * kBKBytes;        // 16 KB
  static constexpr int kBPart = kWBRows * kBKBytes;     // 15 KB
  static constexpr int kBStage = 2 * kBPart;
  static constexpr int kStageBytes = kAStage + kBStage;
  static constexpr uint32_t kSfaCol = 2 * kWHalf;       // 480
  static constexpr uint32_t kSfbCol = kSfaCol + 16;
  static constexpr int kNumBars = 2 * kWStages + 4 + 1;
  static constexpr int kBarBytes = 8 * kNumBars + 16;
  static constexpr int kGroupCols = 64;                 // a warp's columns of a half: 64, 64, 64 and 48
  static constexpr int kOutRowBytes = 32;               // staging: 16 BF16 or 8 fp32 columns a row
  static constexpr int kOutBytes = 32 * kOutRowBytes;   // per warp
  static constexpr int kInvSwBytes = kWEpiWarps * 2 * kGroupCols * 4;
  static constexpr int kSmemBytes =
      1024 + kWStages * kStageBytes + kWEpiWarps * kOutBytes + kBarBytes + kInvSwBytes;
  static_assert(kSfbCol + 16 <= kTmemCols, "accumulator and scale factors exceed TMEM");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget exceeded");
  static_assert(3 * kGroupCols < kWHalf && kWHalf - 3 * kGroupCols <= kGroupCols, "column groups");
};

struct WideSched {
  int num_m;     // row blocks of 256
  int num_nh;    // column halves of 240 (the last may be narrower)
  int doubles;   // items [0, doubles): double tiles, row block fastest
  int items;     // all items
};

// MMA width of a half whose first column is `rem` columns before the right edge.
__host__ __device__ __forceinline__ int wide_half_width(int rem) {
  return rem <= 0 ? 0 : (rem >= kWHalf ? kWHalf : (rem + 15) / 16 * 16);
}

__device__ __forceinline__ void wide_item(int i, const WideSched& s, int N, int& mb, int& n0, int& nh0, int& nh1) {
  bool two = false;
  if (i < s.doubles) {
    mb = i % s.num_m;
    n0 = (i / s.num_m) * (2 * kWHalf);
    two = true;
  } else {
    int j = i - s.doubles;
    const int odd = (s.num_nh & 1) ? s.num_m : 0;
    if (j < odd) {                       // the last half of row block j
      mb = j;
      n0 = (s.num_nh - 1) * kWHalf;
    } else {                             // one half of a split double
      j -= odd;
      const int d = s.doubles + (j >> 1);
      mb = d % s.num_m;
      n0 = (d / s.num_m) * (2 * kWHalf) + (j & 1) * kWHalf;
    }
  }
  nh0 = wide_half_width(N - n0);
  nh1 = two ? wide_half_width(N - n0 - kWHalf) : 0;
}

// Instruction descriptors with a run-time N (multiple of 16; M = 256).
__device__ __forceinline__ uint32_t idesc_mxf4_pair_n(int n) {
  return (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (1u << 23) | (uint32_t(256 >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_tf32_pair_n(int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(256 >> 4) << 24);
}

// The 4 MMAs of one half of one stage (K = 256 E2M1 values, or 32 TF32 values),
// into accumulator columns 240 H .. : straight-line code, so that the single
// issuing thread keeps the tensor pipe fed (a version with a per-MMA branch
// between the kinds and a per-MMA accumulate flag ran at about 60 % of the
// instruction rate).
template <int H>
__device__ __forceinline__ void wide_issue(uint32_t tmem, uint32_t a0, uint32_t b0, uint32_t idesc, uint32_t sfa,
                                           uint32_t sfb, bool fp4, bool first) {
  const uint32_t d = tmem + uint32_t(H * kWHalf);
  const uint32_t bb = b0 + uint32_t(H * WideCfg::kBPart);
  if (fp4) {
    mma_mxf4_pair(d, smem_desc_sw128(a0, 16, 1024), smem_desc_sw128(bb, 16, 1024), idesc, sfa, sfb, first ? 0u : 1u);
#pragma unroll
    for (int k = 1; k < kBKBytes / kMmaKBytes; ++k)
      mma_mxf4_pair(d, smem_desc_sw128(a0 + k * kMmaKBytes, 16, 1024), smem_desc_sw128(bb + k * kMmaKBytes, 16, 1024),
                    idesc, sfa, sfb, 1u);
  } else {
#pragma unroll
    for (int k = 0; k < kBKBytes / kMmaKBytes; ++k)
      mma_tf32_pair(d, smem_desc_sw128(a0 + k * kMmaKBytes, 16, 1024), smem_desc_sw128(bb + k * kMmaKBytes, 16, 1024),
                    idesc, 1u);
  }
}

__global__ void __launch_bounds__(kWThreads, 1)
    fp4_fwd_wide_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmPh,
                        const __grid_constant__ CUtensorMap tmPl, const __grid_constant__ CUtensorMap tmQh,
                        const __grid_constant__ CUtensorMap tmQl, const FwdParams p, const WideSched sc) {
  using C = WideCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kWStages * C::kAStage;
  uint8_t* sOut = smem + kWStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + kWEpiWarps * C::kOutBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  float* inv_sw_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + C::kBarBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kWStages;
  const uint32_t accf0 = empty0 + 8 * kWStages;   // per half: accumulator half ready
  const uint32_t acce0 = accf0 + 16;              // per half: accumulator half drained
  const uint32_t done_bar = acce0 + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (p.hot) {
      prefetch_tmap(&tmPh);
      prefetch_tmap(&tmPl);
      prefetch_tmap(&tmQh);
      prefetch_tmap(&tmQl);
    }
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(accf0 + 8 * h, 1);
      mbar_init(acce0 + 8 * h, 2 * kWEpiWarps);   // every epilogue warp of both CTAs
    }
    mbar_init(done_bar, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 1) tmem_alloc_for<true>(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  cta_sync<true>();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 2 && warp < 6) {  // unit block scales: every scale byte = 0x7F (2^0)
    const uint32_t lb = uint32_t((warp & 3) * 32) << 16;
    tmem_st8_fill(tmem + lb + C::kSfaCol, 0x7F7F7F7Fu);
    tmem_st8_fill(tmem + lb + C::kSfaCol + 8, 0x7F7F7F7Fu);
    tmem_st8_fill(tmem + lb + C::kSfbCol, 0x7F7F7F7Fu);
    tmem_st8_fill(tmem + lb + C::kSfbCol + 8, 0x7F7F7F7Fu);
    tmem_wait_st();
  }
  tc_fence_before();
  cta_sync<true>();
  tc_fence_after();

  // with more distinct dA columns than the tensor-core path takes, the
  // fallback kernel (launched after this one) does the whole product
  const bool skip = p.rp != nullptr && p.hot != nullptr && p.hot->hc > kHotMax;
  const bool hot = !skip && p.hot != nullptr && p.hot->mode != 0;
  const int hot_stages = hot ? (p.hot->mode == 2 ? 1 : 3 * (p.hot->hp / kHotChunk)) : 0;
  const int kblocks = (p.K / 2 + kBKBytes - 1) / kBKBytes;
  const int nstages = kblocks + hot_stages;
  const int items = skip ? 0 : sc.items;
  const int pair_id = int(blockIdx.x) >> 1, npairs = int(gridDim.x) >> 1;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int it = pair_id; it < items && ok; it += npairs) {
      int mb, n0, nh0, nh1;
      wide_item(it, sc, p.N, mb, n0, nh0, nh1);
      const int arow = mb * (2 * kBM) + int(rank) * kBM;
      const int b0row = n0 + int(rank) * (nh0 >> 1);
      const int b1row = n0 + kWHalf + int(rank) * (nh1 >> 1);
      const uint32_t bytes = 2u * uint32_t(C::kAStage + (nh0 ? C::kBPart : 0) + (nh1 ? C::kBPart : 0));
      for (int kb = 0; kb < nstages; ++kb) {
        if (!mbar_wait_warp(empty0 + 8 * stage, phase ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = full0 + 8 * stage;
          if (rank == 0) mbar_arrive_expect_tx(fb, bytes);
          const uint32_t da = smem_u32(sA + stage * C::kAStage), db = smem_u32(sB + stage * C::kBStage);
          if (kb < kblocks) {
            tma_load_2d_to<true>(da, &tmA, fb, kb * kBKBytes, arow);
            if (nh0) tma_load_2d_to<true>(db, &tmB, fb, kb * kBKBytes, b0row);
            if (nh1) tma_load_2d_to<true>(db + C::kBPart, &tmB, fb, kb * kBKBytes, b1row);
          } else {
            // 32 columns of H: P part x Q part, pairs (hi, hi), (hi, lo), (lo, hi)
            const int hs = kb - kblocks, chunk = hs / 3, pr = hs - 3 * chunk;
            const int x = chunk * kHotChunk;
            tma_load_2d_to<true>(da, pr == 2 ? &tmPl : &tmPh, fb, x, arow);
            const CUtensorMap* q = pr == 1 ? &tmQl : &tmQh;
            if (nh0) tma_load_2d_to<true>(db, q, fb, x, b0row);
            if (nh1) tma_load_2d_to<true>(db + C::kBPart, q, fb, x, b1row);
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == kWStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    for (int s = 0; s < kWStages; ++s) {
      const uint32_t n_s = issued / kWStages + (uint32_t(s) < issued % kWStages ? 1u : 0u);
      if (n_s > 0 && !mbar_wait_warp(empty0 + 8 * s, (n_s - 1) & 1u, p.wait_ns) && lane == 0)
        atomicOr(p.status, FP4_FLAG_TIMEOUT);
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------ MMA issuer (leader CTA)
    int s0 = 0, s1 = 0;          // ring slot of the next half-0 and half-1 stage
    uint32_t ph0 = 0;            // phase of the next half-0 stage's full barrier
    uint32_t accph = 0;
    bool ok = true;
    const uint32_t sfa = tmem + C::kSfaCol, sfb = tmem + C::kSfbCol;
    const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
    for (int it = pair_id; it < items && ok; it += npairs) {
      int mb, n0, nh0, nh1;
      wide_item(it, sc, p.N, mb, n0, nh0, nh1);
      const uint32_t f0 = idesc_mxf4_pair_n(nh0), f1 = idesc_mxf4_pair_n(nh1);
      const uint32_t t0 = idesc_tf32_pair_n(nh0), t1 = idesc_tf32_pair_n(nh1);
      const int L = nstages < kWLag ? nstages : kWLag;
      const int s_end = nstages - L > L ? nstages - L : L;
      // stage kb of this tile: its full barrier (half 0 only), then lane 0 issues
#define FP4_WIDE_FULL()                                   \
  if (!mbar_wait_warp(full0 + 8 * s0, ph0, p.wait_ns)) {  \
    ok = false;                                           \
    break;                                                \
  }                                                       \
  tc_fence_after();
#define FP4_WIDE_ADV0()   \
  if (++s0 == kWStages) { \
    s0 = 0;               \
    ph0 ^= 1u;            \
  }
#define FP4_WIDE_ADV1() \
  if (++s1 == kWStages) s1 = 0;
      if (!mbar_wait_warp(acce0, accph ^ 1u, p.wait_ns)) {   // half 0 drained
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < L; ++kb) {
        FP4_WIDE_FULL()
        if (lane == 0 && nh0)
          wide_issue<0>(tmem, a_base + s0 * C::kAStage, b_base + s0 * C::kBStage, kb < kblocks ? f0 : t0, sfa, sfb,
                        kb < kblocks, kb == 0);
        __syncwarp();
        FP4_WIDE_ADV0()
      }
      if (!ok) break;
      if (!mbar_wait_warp(acce0 + 8, accph ^ 1u, p.wait_ns)) {   // half 1 drained
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < L; ++kb) {
        if (lane == 0) {
          if (nh1)
            wide_issue<1>(tmem, a_base + s1 * C::kAStage, b_base + s1 * C::kBStage, kb < kblocks ? f1 : t1, sfa, sfb,
                          kb < kblocks, kb == 0);
          commit_to<true>(empty0 + 8 * s1, 0x3);   // the stage is free in both CTAs
        }
        __syncwarp();
        FP4_WIDE_ADV1()
      }
      for (int kb = L; kb < s_end; ++kb) {   // both halves of a stage back to back
        FP4_WIDE_FULL()
        if (lane == 0) {
          const uint32_t a0 = a_base + s0 * C::kAStage, b0 = b_base + s0 * C::kBStage;
          const bool fp4s = kb < kblocks;
          if (nh0) wide_issue<0>(tmem, a0, b0, fp4s ? f0 : t0, sfa, sfb, fp4s, false);
          if (nh1) wide_issue<1>(tmem, a0, b0, fp4s ? f1 : t1, sfa, sfb, fp4s, false);
          commit_to<true>(empty0 + 8 * s0, 0x3);
        }
        __syncwarp();
        FP4_WIDE_ADV0()
        FP4_WIDE_ADV1()
      }
      if (!ok) break;
      for (int kb = s_end; kb < nstages; ++kb) {   // half 0 finishes first
        FP4_WIDE_FULL()
        if (lane == 0 && nh0)
          wide_issue<0>(tmem, a_base + s0 * C::kAStage, b_base + s0 * C::kBStage, kb < kblocks ? f0 : t0, sfa, sfb,
                        kb < kblocks, kb == 0);
        __syncwarp();
        FP4_WIDE_ADV0()
      }
      if (!ok) break;
      if (lane == 0) commit_to<true>(accf0, 0x3);        // half 0 of the accumulator is ready
      __syncwarp();
      for (int kb = s_end; kb < nstages; ++kb) {
        if (lane == 0) {
          if (nh1)
            wide_issue<1>(tmem, a_base + s1 * C::kAStage, b_base + s1 * C::kBStage, kb < kblocks ? f1 : t1, sfa, sfb,
                          kb < kblocks, kb == 0);
          commit_to<true>(empty0 + 8 * s1, 0x3);
        }
        __syncwarp();
        FP4_WIDE_ADV1()
      }
      if (lane == 0) commit_to<true>(accf0 + 8, 0x3);    // half 1 is ready
      __syncwarp();
      accph ^= 1u;
#undef FP4_WIDE_FULL
#undef FP4_WIDE_ADV0
#undef FP4_WIDE_ADV1
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    if (lane == 0) commit_to<true>(done_bar, 0x1);
    __syncwarp();
    if (!mbar_wait_warp(done_bar, 0, p.wait_ns) && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue (both CTAs, own 128 rows)
    // 16 warps; warp w owns TMEM lanes 32 (w % 4) .. +31 (one output row per
    // thread) and column group (w - 2) / 4 of each half: columns 64 g .. of the
    // half, 64 wide (48 for the last).  Per half, for BF16 output: read the
    // group's columns, scale and round them into at most 32 packed registers,
    // release the half, then store.  TMEM is held for the arithmetic alone, about
    // 16 x 64 values a thread-warp, which the tensor core's other half covers.
    constexpr int GC = C::kGroupCols;
    const int e = warp - 2;
    const int g = e >> 2, q = warp & 3;
    const int gw = g < 3 ? GC : kWHalf - 3 * GC;   // this warp's columns of a half
    float* inv_sw_w = inv_sw_s + e * 2 * GC;
    uint8_t* out_s = sOut + e * C::kOutBytes;
    uint8_t* orow = out_s + lane * C::kOutRowBytes;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    const bool raw = (p.y_type == FP4_OUT_RAW_ACC_FP32);
    const bool bf16_out = (p.y_type == FP4_OUT_BF16);
    uint32_t accph = 0;
    bool ok = true;
    for (int it = pair_id; it < items && ok; it += npairs) {
      int mb, n0, nh0, nh1;
      wide_item(it, sc, p.N, mb, n0, nh0, nh1);
      const int row0 = mb * (2 * kBM) + int(rank) * kBM + q * 32;
      const int row = row0 + lane;
      // the row's scale and this warp's column scales of both halves, all loads
      // in flight at once, before the first wait
      float sw[4];
      const float sa = (row < p.M && !raw) ? __ldg(p.s_a + row) : 1.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {   // column c = lane + 32 j of [half 0 group | half 1 group]
        const int c = lane + 32 * j, h = c >= GC, cc = c - h * GC;
        const int col = n0 + h * kWHalf + g * GC + cc;
        sw[j] = (cc < gw && !raw && col < p.N) ? __ldg(p.s_w + col) : 1.0f;
      }
      const float inv_sa = 1.0f / sa;
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) inv_sw_w[lane + 32 * j] = 1.0f / sw[j];
      __syncwarp();
      int ncols[2], col_base[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int nhh = h ? nh1 : nh0;
        ncols[h] = nhh - g * GC < 0 ? 0 : (nhh - g * GC > gw ? gw : nhh - g * GC);   // multiple of 16
        col_base[h] = n0 + h * kWHalf + g * GC;
      }
      if (bf16_out) {
        // both halves into registers, each released as soon as it is read; the
        // stores follow (a store burst between the halves would delay half 1,
        // while after both they overlap the next tile's main loop)
        uint32_t pk[2][GC / 2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(accf0 + 8 * h, accph, p.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tcol = uint32_t(h * kWHalf + g * GC);
#pragma unroll
          for (int c0 = 0; c0 < GC; c0 += 16) {
            if (c0 < ncols[h]) {   // warp-uniform
              uint32_t r[16];
              tmem_ld8(tmem + lane_base + tcol + c0, *reinterpret_cast<uint32_t(*)[8]>(r));
              tmem_ld8(tmem + lane_base + tcol + c0 + 8, *reinterpret_cast<uint32_t(*)[8]>(r + 8));
              tmem_wait_ld();
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                float y0 = __uint_as_float(r[2 * t]), y1 = __uint_as_float(r[2 * t + 1]);
                mul2_rn(y0, y1, inv_sa, inv_sa);
                const float2 w = *reinterpret_cast<const float2*>(inv_sw_w + h * GC + c0 + 2 * t);
                mul2_rn(y0, y1, w.x, w.y);
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(y0, y1);
                pk[h][c0 / 2 + t] = *reinterpret_cast<const uint32_t*>(&b2);
              }
            }
          }
          // the half may be overwritten: its TMEM reads completed at tcgen05.wait::ld
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(acce0 + 8 * h, 0));
        }
        if (!ok) break;
        // stores, 16 columns at a time through the warp's staging rows: each lane
        // writes its row (32 bytes), then the warp stores the block row-major in
        // 16-byte pieces, two lanes to a row
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c0 = 0; c0 < GC; c0 += 16) {
            if (c0 < ncols[h]) {
              __syncwarp();
              *reinterpret_cast<uint4*>(orow) =
                  make_uint4(pk[h][c0 / 2], pk[h][c0 / 2 + 1], pk[h][c0 / 2 + 2], pk[h][c0 / 2 + 3]);
              *reinterpret_cast<uint4*>(orow + 16) =
                  make_uint4(pk[h][c0 / 2 + 4], pk[h][c0 / 2 + 5], pk[h][c0 / 2 + 6], pk[h][c0 / 2 + 7]);
              __syncwarp();
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {   // 64 pieces: piece i is row i / 2, bytes 16 (i % 2) ..
                const int i = lane + 32 * rr;
                const int grow = row0 + (i >> 1), gcol = col_base[h] + c0 + 8 * (i & 1);
                const uint4 v = *reinterpret_cast<const uint4*>(out_s + 16 * i);
                if (grow < p.M && gcol < p.N)
                  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.Y) + int64_t(grow) * p.ldy + gcol) = v;
              }
            }
          }
        }
      } else {
        // fp32 or the raw accumulator: 8 columns (32 bytes a row) at a time,
        // stored while the half is held
        for (int h = 0; h < 2; ++h) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(accf0 + 8 * h, accph, p.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tcol = uint32_t(h * kWHalf + g * GC);
          for (int c0 = 0; c0 < ncols[h]; c0 += 8) {   // warp-uniform
            uint32_t r[8];
            tmem_ld8(tmem + lane_base + tcol + c0, r);
            tmem_wait_ld();
            float y[8];
#pragma unroll
            for (int t = 0; t < 8; t += 2) {
              y[t] = __uint_as_float(r[t]);
              y[t + 1] = __uint_as_float(r[t + 1]);
              if (!raw) {
                mul2_rn(y[t], y[t + 1], inv_sa, inv_sa);
                const float2 w = *reinterpret_cast<const float2*>(inv_sw_w + h * GC + c0 + t);
                mul2_rn(y[t], y[t + 1], w.x, w.y);
              }
            }
            __syncwarp();
            *reinterpret_cast<float4*>(orow) = make_float4(y[0], y[1], y[2], y[3]);
            *reinterpret_cast<float4*>(orow + 16) = make_float4(y[4], y[5], y[6], y[7]);
            __syncwarp();
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int i = lane + 32 * rr;
              const int grow = row0 + (i >> 1), gcol = col_base[h] + c0 + 4 * (i & 1);
              const uint4 v = *reinterpret_cast<const uint4*>(out_s + 16 * i);
              if (grow < p.M && gcol < p.N)
                *reinterpret_cast<uint4*>(static_cast<float*>(p.Y) + int64_t(grow) * p.ldy + gcol) = v;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(acce0 + 8 * h, 0));
        }
        if (!ok) break;
      }
      accph ^= 1u;
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  }

  // neither CTA leaves or frees TMEM while its partner may still signal it
  __syncwarp();
  tc_fence_before();
  cta_sync<true>();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_for<true>(tmem, kTmemCols);
  }
}

constexpr int kFwdBN = 240;
constexpr int kFwdAcc = 2;

}  // namespace
}  // namespace fp4

namespace fp4 {
namespace {
// Workspace of the tensor-core compensation (offsets in bytes).
struct HotLayout {
  size_t info, bitmap, prefix, hlist, p_hi, p_lo, q_hi, q_lo, total;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

HotLayout hot_layout(int64_t M, int64_t N, int64_t K) {
  HotLayout L;
  size_t off = 0;
  L.info = off;
  off += 256;
  L.bitmap = off;   // K/32 bitmap words, then the CTA-done counter (one memset clears both)
  off = align_up(off + size_t(K / 32) * 4 + 4, 256);
  L.prefix = off;
  off = align_up(off + size_t(K / 32) * 4, 256);
  L.hlist = off;
  off = align_up(off + size_t(kHotMax) * 4, 1024);
  L.p_hi = off;
  off = align_up(off + size_t(M) * kHotMax * 4, 1024);
  L.p_lo = off;
  off = align_up(off + size_t(M) * kHotMax * 4, 1024);
  L.q_hi = off;
  off = align_up(off + size_t(N) * kHotMax * 4, 1024);
  L.q_lo = off;
  off = align_up(off + size_t(N) * kHotMax * 4, 1024);
  L.total = off;
  return L;
}
}  // namespace
}  // namespace fp4

FP4_API size_t fp4_linear_fwd_workspace(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || K > 16384 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31))
    return 0;
  return fp4::hot_layout(M, N, K).total;
}

namespace fp4 {
namespace {
// Encodes the B-side tensor maps for the tile shape of PAIR and launches the GEMM
// (as clusters of two CTAs for PAIR), persistent over the tiles.
template <bool PAIR>
fp4_status launch_fwd(const CUtensorMap& tmA, const CUtensorMap& tmY, const uint8_t* w_codes_t, int64_t ldw_codes_bytes,
                      const float* q_hi, const float* q_lo, const float* p_hi, const float* p_lo, FwdParams p, int sms,
                      cudaStream_t cs) {
  using C = FwdCfg<kFwdBN, kFwdAcc, PAIR>;
  fp4_status st;
  CUtensorMap tmB, tmPh = tmA, tmPl = tmA, tmQh = tmA, tmQl = tmA;   // compensation maps unused without p.hot
  if ((st = encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_codes_t, uint64_t(p.K / 2), uint64_t(p.N),
                           uint64_t(ldw_codes_bytes), kBKBytes, C::kBRows, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK)
    return st;
  if (p.hot) {
    const uint32_t row_bytes = kHotMax * 4;
    if ((st = encode_tmap_2d(&tmPh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p_hi, kHotMax, uint64_t(p.M), row_bytes,
                             kHotChunk, kBM, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK ||
        (st = encode_tmap_2d(&tmPl, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p_lo, kHotMax, uint64_t(p.M), row_bytes,
                             kHotChunk, kBM, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK ||
        (st = encode_tmap_2d(&tmQh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, q_hi, kHotMax, uint64_t(p.N), row_bytes,
                             kHotChunk, C::kBRows, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK ||
        (st = encode_tmap_2d(&tmQl, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, q_lo, kHotMax, uint64_t(p.N), row_bytes,
                             kHotChunk, C::kBRows, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK)
      return st;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = fp4_fwd_kernel<kFwdBN, kFwdAcc, PAIR>;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t tiles = ((p.M + kBM * C::kCtas - 1) / (kBM * C::kCtas)) * ((p.N + kFwdBN - 1) / kFwdBN);
  const int64_t units = sms / C::kCtas;
  const int grid = int(C::kCtas * (tiles < units ? tiles : units));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = cs;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(C::kCtas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmY, tmPh, tmPl, tmQh, tmQl, p) != cudaSuccess) return launch_status();
  return launch_status();
}
}  // namespace
}  // namespace fp4


namespace fp4 {
namespace {
// Half-tiles of the busiest pair when items [0, doubles) are double tiles and
// [doubles, doubles + singles) single halves, dealt round robin to `pairs`.
int64_t wide_makespan(int64_t doubles, int64_t singles, int64_t pairs) {
  int64_t worst = 0;
  for (int64_t p = 0; p < pairs && p < doubles + singles; ++p) {
    const int64_t nd = p < doubles ? (doubles - 1 - p) / pairs + 1 : 0;
    // items i in [doubles, doubles + singles) with i = p (mod pairs)
    const int64_t first = doubles + ((p - doubles) % pairs + pairs) % pairs;
    const int64_t ns = first < doubles + singles ? (doubles + singles - 1 - first) / pairs + 1 : 0;
    worst = std::max(worst, 2 * nd + ns);
  }
  return worst;
}

// Work list of the wide kernel: all double tiles, or the last partial round of
// them split into single halves when that shortens the busiest pair's list.
WideSched wide_schedule(int64_t M, int64_t N, int64_t pairs) {
  WideSched s;
  s.num_m = int((M + 2 * kBM - 1) / (2 * kBM));
  s.num_nh = int((N + kWHalf - 1) / kWHalf);
  const int64_t d0 = int64_t(s.num_m) * (s.num_nh / 2);
  const int64_t s0 = (s.num_nh & 1) ? s.num_m : 0;
  const int64_t r = d0 % pairs;
  int64_t split = 0;
  if (r && wide_makespan(d0 - r, s0 + 2 * r, pairs) < wide_makespan(d0, s0, pairs)) split = r;
  s.doubles = int(d0 - split);
  s.items = int(d0 - split + s0 + 2 * split);
  return s;
}

fp4_status launch_fwd_wide(const CUtensorMap& tmA, const uint8_t* w_codes_t,
                           int64_t ldw_codes_bytes, const float* q_hi, const float* q_lo, const float* p_hi,
                           const float* p_lo, FwdParams p, int sms, cudaStream_t cs) {
  using C = WideCfg;
  fp4_status st;
  CUtensorMap tmB, tmPh = tmA, tmPl = tmA, tmQh = tmA, tmQl = tmA;   // compensation maps unused without p.hot
  if ((st = encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_codes_t, uint64_t(p.K / 2), uint64_t(p.N),
                           uint64_t(ldw_codes_bytes), kBKBytes, kWBRows, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK)
    return st;
  if (p.hot) {
    const uint32_t row_bytes = kHotMax * 4;
    if ((st = encode_tmap_2d(&tmPh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p_hi, kHotMax, uint64_t(p.M), row_bytes,
                             kHotChunk, kBM, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK ||
        (st = encode_tmap_2d(&tmPl, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p_lo, kHotMax, uint64_t(p.M), row_bytes,
                             kHotChunk, kBM, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK ||
        (st = encode_tmap_2d(&tmQh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, q_hi, kHotMax, uint64_t(p.N), row_bytes,
                             kHotChunk, kWBRows, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK ||
        (st = encode_tmap_2d(&tmQl, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, q_lo, kHotMax, uint64_t(p.N), row_bytes,
                             kHotChunk, kWBRows, CU_TENSOR_MAP_SWIZZLE_128B)) != FP4_OK)
      return st;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(fp4_fwd_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t pairs = sms / 2;
  const WideSched sc = wide_schedule(p.M, p.N, pairs);
  const int grid = int(2 * (sc.items < pairs ? sc.items : pairs));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = cs;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fp4_fwd_wide_kernel, tmA, tmB, tmPh, tmPl, tmQh, tmQl, p, sc) != cudaSuccess)
    return launch_status();
  return launch_status();
}
}  // namespace
}  // namespace fp4

FP4_API fp4_status fp4_linear_fwd(const uint8_t* a_codes, int64_t lda_codes_bytes, const float* s_a,
                                  const uint8_t* w_codes_t, int64_t ldw_codes_bytes, const float* s_w, int64_t M,
                                  int64_t N, int64_t K, const int32_t* dA_row_ptr, const int32_t* dA_col,
                                  const float* dA_val, const void* W, int64_t ldw, void* Y, int y_type, int64_t ldy,
                                  void* workspace, size_t ws_bytes, fp4_stream_t stream) {
  using namespace fp4;
  if (!a_codes || !w_codes_t || !Y) return FP4_ERR_INVALID_ARG;
  if (y_type != FP4_OUT_BF16 && y_type != FP4_OUT_FP32 && y_type != FP4_OUT_RAW_ACC_FP32) return FP4_ERR_INVALID_ARG;
  const bool raw = (y_type == FP4_OUT_RAW_ACC_FP32);
  if (!raw && (!s_a || !s_w)) return FP4_ERR_INVALID_ARG;
  const int ncsr = (dA_row_ptr != nullptr) + (dA_col != nullptr) + (dA_val != nullptr);
  if (ncsr != 0 && ncsr != 3) return FP4_ERR_INVALID_ARG;
  const bool comp = (ncsr == 3) && !raw;
  if (comp && !W) return FP4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || N % 8 != 0 || M >= (int64_t(1) << 31) ||
      N >= (int64_t(1) << 31) || K > 16384)
    return FP4_ERR_SHAPE;
  if (lda_codes_bytes < K / 2 || ldw_codes_bytes < K / 2 || ldy < N || (comp && ldw < N)) return FP4_ERR_SHAPE;
  if (lda_codes_bytes % 16 || ldw_codes_bytes % 16 || !aligned16(a_codes) || !aligned16(w_codes_t) || !aligned16(Y) ||
      ldy % 8 || (comp && (!aligned16(W) || ldw % 8)))
    return FP4_ERR_ALIGNMENT;
  const HotLayout L = hot_layout(M, N, K);
  const bool use_hot = comp && workspace != nullptr;
  if (use_hot && ws_bytes < L.total) return FP4_ERR_WORKSPACE;
  if (use_hot && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  CUtensorMap tmA;
  st = encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, uint64_t(K / 2), uint64_t(M),
                      uint64_t(lda_codes_bytes), kBKBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;

  CUtensorMap tmY;
  const bool bf16_out = (y_type == FP4_OUT_BF16);
  st = encode_tmap_2d(&tmY, bf16_out ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, Y,
                      uint64_t(N), uint64_t(M), uint64_t(ldy) * (bf16_out ? 2 : 4), bf16_out ? 40 : 20, 32,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != FP4_OK) return st;

  // tensor-core compensation: prep kernels fill the workspace; the GEMM reads
  // HotInfo to learn whether (and over how many columns) to run the TF32 stages
  const HotInfo* hot_info = nullptr;
  float *p_hi = nullptr, *p_lo = nullptr, *q_hi = nullptr, *q_lo = nullptr;
  if (use_hot) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    HotInfo* info = reinterpret_cast<HotInfo*>(ws + L.info);
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(ws + L.bitmap);
    uint32_t* prefix = reinterpret_cast<uint32_t*>(ws + L.prefix);
    int32_t* hlist = reinterpret_cast<int32_t*>(ws + L.hlist);
    p_hi = reinterpret_cast<float*>(ws + L.p_hi);
    p_lo = reinterpret_cast<float*>(ws + L.p_lo);
    q_hi = reinterpret_cast<float*>(ws + L.q_hi);
    q_lo = reinterpret_cast<float*>(ws + L.q_lo);
    const int nwords = int(K / 32);
    uint32_t* done = bitmap + nwords;
    if (cudaMemsetAsync(bitmap, 0, size_t(nwords) * 4 + 4, cs) != cudaSuccess) return launch_status();
    hot_mark_kernel<<<sms / 2, 512, 0, cs>>>(dA_row_ptr, dA_col, int(M), int(K), bitmap, done, prefix, hlist, info,
                                             status_word());
    const int p_ctas = int((M + 7) / 8);
    const int q_ctas = int((N + 255) / 256) * (kHotMax / 4);
    hot_build_kernel<<<p_ctas + q_ctas, 256, 0, cs>>>(dA_row_ptr, dA_col, dA_val, s_a, static_cast<const uint16_t*>(W),
                                                     ldw, s_w, bitmap, prefix, hlist, info, p_hi, p_lo, q_hi, q_lo,
                                                     int(M), int(N), int(K), p_ctas);
    st = launch_status();
    if (st != FP4_OK) return st;
    hot_info = info;
  }

  FwdParams p;
  p.s_a = s_a;
  p.s_w = s_w;
  p.rp = comp ? dA_row_ptr : nullptr;
  p.ci = comp ? dA_col : nullptr;
  p.cv = comp ? dA_val : nullptr;
  p.W = static_cast<const uint16_t*>(W);
  p.ldw = ldw;
  p.Y = Y;
  p.ldy = ldy;
  p.y_type = y_type;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.hot = hot_info;
  p.status = status_word();
  p.wait_ns = kWaitLimitNs;
  p.fallback_only = 0;
  // K >= 4096, without compensation or with it on the tensor cores: the wide
  // kernel (256 x 480 pair tiles; below 16 K stages a tile is too short to
  // hide the drain of its single accumulator, and the double-buffered 240-wide
  // kernel is faster).  The tensor-core path is decided on the device (the
  // distinct dA columns are counted there), so with a workspace the 240-wide
  // kernel follows as a fallback that does the product only when dA has more
  // than kHotMax distinct columns (the wide kernel then does nothing), forming
  // the compensation on its CUDA cores; otherwise that kernel does it all.
  if (K >= 4096 && (!comp || use_hot)) {
    st = launch_fwd_wide(tmA, w_codes_t, ldw_codes_bytes, q_hi, q_lo, p_hi, p_lo, p, sms, cs);
    if (st != FP4_OK || !comp) return st;
    p.fallback_only = 1;
  }
  // CTA pairs once the K loop is long enough (16 FP4 stages, K >= 4096) for the
  // pair's lighter stages to outweigh its shared accumulator hand-off
  if (K >= 4096) return launch_fwd<true>(tmA, tmY, w_codes_t, ldw_codes_bytes, q_hi, q_lo, p_hi, p_lo, p, sms, cs);
  return launch_fwd<false>(tmA, tmY, w_codes_t, ldw_codes_bytes, q_hi, q_lo, p_hi, p_lo, p, sms, cs);
}
