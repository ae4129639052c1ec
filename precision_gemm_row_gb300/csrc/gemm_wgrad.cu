// Weight gradient of the quantized linear layer with the differentiable
// gradient estimator (DGE), on sm_103a tensor cores.
//
// The page "首个 FP4 精度的大模型训练框架来了" (czzqal.com), DGE passage: the
// derivative of the hard quantizer is almost everywhere 0, so the forward pass
// keeps hard quantization while the backward pass refits the quantizer with a
// continuous differentiable function and uses its derivative as a correction
// of the weight gradient (also the abstract of "Optimizing Large Language Model
// Training Using FP4 Quantization").  The function is not printed on the pages;
// the one used is a per-interval power function:
//   x = |fl32(W s_W)|, [lo, lo + delta] the E2M1 interval holding x,
//   u = 2 (x - lo) / delta - 1,  f'(x) = min(clip, (1/k) |u|^(1/k - 1)),  f' = 1/k for x >= 6.
//
// G = A^T dY is a BF16 GEMM with both operands stored with the reduction
// (token) dimension strided, i.e. MN-major: TMA loads [64 tokens x 64
// features] boxes with 128-byte swizzle and tcgen05.mma kind::f16 reads them
// through MN-major descriptors, so no transpose copy is ever made.
//
// Accumulation precision: the tensor core's fp32 accumulation drifts by about
// 1e-9 x (number of accumulated tokens) relative (a biased, truncation-like
// error), which would exceed 1e-5 at 16k tokens.  The token range of every
// tile is therefore split into chunks of kChunkStages x 64 tokens; each chunk
// is accumulated in one of two TMEM buffers and the epilogue warps add it into
// fp32 registers (round to nearest), so the error stays at the chunk level.
// While the epilogue drains one buffer the MMA warp fills the other.
//
// Roles (10 warps): warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer,
// warps 2-9 epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (one dW row per
// thread) and columns (w-2)/4 * 128 .. +127 of the 256-wide tile, adding each
// chunk into fp32 registers.  After the last chunk of a tile the warp computes
// the DGE factors from W and s_W and writes dW = G * f' once, through a swizzled
// staging tile as coalesced row chunks, while the tensor core already fills
// both TMEM buffers with the next tile.  Every mbarrier wait is bounded; on
// expiry the CTA records FP4_FLAG_TIMEOUT, drains its TMA loads and MMAs, frees
// TMEM and exits.
#include "common.cuh"

namespace fp4 {
namespace {

constexpr int kBM = 128;      // rows of dW (input features) per tile
constexpr int kBN = 256;      // columns of dW (output features) per tile
constexpr int kBT = 64;       // tokens per stage
constexpr int kMmaT = 16;     // tokens per MMA (BF16 K = 16)
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kNAcc = 2;
constexpr int kChunkStages = 16;                 // 1024 tokens per TMEM accumulation chunk
constexpr int kEpiCols = kBN / 2;                // columns per epilogue warp
constexpr int kBlk = 32;                         // epilogue block: 32 rows x 32 columns per warp
constexpr uint32_t kTmemCols = 512;
constexpr int kBox = 64;                          // features per TMA box (128 bytes of BF16)
constexpr int kBoxBytes = kBox * kBT * 2;         // 8 KB
// epilogue staging per warp: one dW block of 32 x 32 fp32 (128-byte swizzle),
// written out with coalesced stores (TMA stays free for the main loop's stages)
constexpr int kOutBytes = kBlk * kBlk * 4;        // 4 KB
constexpr int kEpiWarpBytes = kOutBytes;

// PAIR: tiles of 256 x 256 per CTA pair (a cluster of two CTAs on two SMs): each
// CTA loads its 128 dW rows of A and 128 of the tile's 256 dY columns per stage
// (32 KB instead of 48 KB for the same MMA work), the leader issues M = 256
// tcgen05 MMAs (cta_group::2), and each CTA's TMEM holds its 128 rows x 256
// columns.  Short token loops run single-CTA 128 x 256 tiles.
template <bool PAIR>
struct WgCfg {
  static constexpr int kCtas = PAIR ? 2 : 1;
  static constexpr int kBCols = kBN / kCtas;                  // dY columns per CTA
  static constexpr int kAStage = (kBM / kBox) * kBoxBytes;    // 16 KB
  static constexpr int kBStage = (kBCols / kBox) * kBoxBytes; // 16 or 32 KB
  static constexpr int kStageBytes = kAStage + kBStage;
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kDataBytes = kStages * kStageBytes + kEpiWarps * kEpiWarpBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kNAcc + 1;
  static constexpr int kSmemBytes = 1024 + kDataBytes + 8 * kNumBars + 16;
  // Instruction descriptor, kind::f16: fp32 accumulator, A and B BF16, both
  // MN-major, N = 256, M = 128 per CTA.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                                     (uint32_t(kBN >> 3) << 17) | (uint32_t((kBM * kCtas) >> 4) << 24);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget exceeded");
};

struct WgradParams {
  const uint16_t* W;
  int64_t ldw;
  const float* s_w;
  float* dW;
  int64_t lddw;
  int M, N, K;
  float inv_k, expo, clip, pw0;
  uint32_t* status;
  uint64_t wait_ns;
};

// DGE factor f'(x) for the scaled weight magnitude x.  |u|^e uses the fast
// power intrinsic (relative error a few fp32 ulps); u = 0 takes pw0, the limit
// of |u|^e there: +inf for e < 0 (then clipped), 1 for e = 0, 0 for e > 0.
// Written without branches: the interval is found by scaling x with 2/delta
// (a power of two, so s and its fractional part are exact), and every case is
// a select, so a warp never diverges over mixed magnitudes.
__device__ __forceinline__ float dge_factor(float x, float inv_k, float expo, float clip, float pw0) {
  const float two_over_delta = x < 2.0f ? 2.0f : (x < 4.0f ? 1.0f : 0.5f);
  const float s = x * two_over_delta;                        // interval [floor(s), floor(s) + 1)
  const float u = fabsf(fmaf(s - floorf(s), 2.0f, -1.0f));   // |2 (x - lo) / delta - 1|
  const float pw = u > 0.0f ? __powf(u, expo) : pw0;
  const float f = fminf(clip, inv_k * pw);
  return x < 6.0f ? f : inv_k;
}

template <bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_dge_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                     const WgradParams p) {
  using C = WgCfg<PAIR>;
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
    prefetch_tmap(&tmG);
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

  constexpr int kTileR = kBM * C::kCtas;   // dW rows per tile (per pair)
  const int num_r = (p.K + kTileR - 1) / kTileR;
  const int num_n = (p.N + kBN - 1) / kBN;
  const int tiles = num_r * num_n;
  const int tblocks = (p.M + kBT - 1) / kBT;
  const int pair_id = int(blockIdx.x) / C::kCtas, npairs = int(gridDim.x) / C::kCtas;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    for (int tile = pair_id; tile < tiles && ok; tile += npairs) {
      const int rb = tile % num_r, nb = tile / num_r;
      const int arow = rb * kTileR + int(rank) * kBM;          // this CTA's 128 dW rows (A features)
      const int bcol = nb * kBN + int(rank) * C::kBCols;       // this CTA's dY columns of the tile
      for (int tb = 0; tb < tblocks; ++tb) {
        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          // completion is counted on the MMA-issuing CTA's full barrier
          const uint32_t fb = full0 + 8 * stage;
          if (rank == 0) mbar_arrive_expect_tx(fb, C::kCtas * C::kStageBytes);
          const uint32_t a_dst = smem_u32(sA + stage * C::kAStage);
          const uint32_t b_dst = smem_u32(sB + stage * C::kBStage);
#pragma unroll
          for (int h = 0; h < kBM / kBox; ++h) tma_load_2d_to<PAIR>(a_dst + h * kBoxBytes, &tmA, fb, arow + h * kBox, tb * kBT);
#pragma unroll
          for (int h = 0; h < C::kBCols / kBox; ++h) tma_load_2d_to<PAIR>(b_dst + h * kBoxBytes, &tmG, fb, bcol + h * kBox, tb * kBT);
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
      if (n_s > 0 && !mbar_wait(empty0 + 8 * s, (n_s - 1) & 1u, p.wait_ns) && lane == 0)
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
    for (int tile = pair_id; tile < tiles && ok; tile += npairs) {
      for (int tb0 = 0; tb0 < tblocks && ok; tb0 += kChunkStages) {
        const int tb1 = tb0 + kChunkStages < tblocks ? tb0 + kChunkStages : tblocks;
        if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + uint32_t(acc * kBN);
        for (int tb = tb0; tb < tb1; ++tb) {
          if (!mbar_wait(full0 + 8 * stage, phase, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = a_base + stage * C::kAStage, b0 = b_base + stage * C::kBStage;
#pragma unroll
            for (int k = 0; k < kBT / kMmaT; ++k) {
              // MN-major, 128-byte swizzle: 64-feature atoms kBoxBytes apart (LBO),
              // 8-token groups 1024 bytes apart (SBO); 16 tokens = 2048 bytes per MMA.
              const uint64_t ad = smem_desc_sw128(a0 + k * (kMmaT * 128), kBoxBytes, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + k * (kMmaT * 128), kBoxBytes, 1024);
              if constexpr (PAIR) mma_f16_pair(d_tmem, ad, bd, C::kIdesc, (tb != tb0 || k != 0) ? 1u : 0u);
              else mma_f16(d_tmem, ad, bd, C::kIdesc, (tb != tb0 || k != 0) ? 1u : 0u);
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
    if (!mbar_wait(done_bar, 0, p.wait_ns) && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  } else if (warp >= 2) {
    // ------------------------------------------------ chunk promotion + DGE epilogue (own 128 rows)
    const int ew = warp - 2;
    const int q = warp & 3;
    const int c_base = (ew / 4) * kEpiCols;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    uint8_t* out_s = sEpi + ew * kEpiWarpBytes;          // 32 x 32 fp32, 128-byte swizzle
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    constexpr int kNBlk = kEpiCols / kBlk;
    for (int tile = pair_id; tile < tiles && ok; tile += npairs) {
      const int rb = tile % num_r, nb = tile / num_r;
      const int row0 = rb * kTileR + int(rank) * kBM + q * 32;  // first dW row of this warp's 32-row slab
      float sum[kEpiCols];
#pragma unroll
      for (int c = 0; c < kEpiCols; ++c) sum[c] = 0.0f;
      for (int tb0 = 0; tb0 < tblocks; tb0 += kChunkStages) {
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
      // (2) dW = G * f'(|W s_W|): this lane's sums go through the staging tile so
      // that the read of W, the factor, the multiply and the store of dW run on
      // coalesced row chunks: lane l takes 4 columns (chunk l % 8) of rows l / 8 + 4 i.
      // This runs while the tensor core starts the next tile in both TMEM buffers.
      if (row0 >= p.K) continue;
#pragma unroll
      for (int j = 0; j < kNBlk; ++j) {
        const int col0 = nb * kBN + c_base + j * kBlk;
        if (col0 >= p.N) break;  // same for the whole warp
        const int c = lane & 7, gcol = col0 + 4 * c;
        const bool col_ok = gcol < p.N;   // N % 8 == 0: the 4 columns are all in or all out
        // every load of the block first (one memory latency), then the math
        float4 sw = make_float4(1.f, 1.f, 1.f, 1.f);
        if (col_ok) sw = make_float4(__ldg(p.s_w + gcol), __ldg(p.s_w + gcol + 1), __ldg(p.s_w + gcol + 2), __ldg(p.s_w + gcol + 3));
        uint2 w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int grow = row0 + (lane >> 3) + 4 * i;
          w[i] = (col_ok && grow < p.K) ? __ldg(reinterpret_cast<const uint2*>(p.W + int64_t(grow) * p.ldw + gcol))
                                        : make_uint2(0u, 0u);
        }
        __syncwarp();  // the staging tile is free
        uint8_t* orow = out_s + lane * 128;   // this lane's row: chunk k at k ^ (lane & 7)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<float4*>(orow + ((k ^ (lane & 7)) << 4)) =
              make_float4(sum[j * kBlk + 4 * k], sum[j * kBlk + 4 * k + 1], sum[j * kBlk + 4 * k + 2],
                          sum[j * kBlk + 4 * k + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = (lane >> 3) + 4 * i;
          const int grow = row0 + r;
          if (grow < p.K && col_ok) {
            const float4 g = *reinterpret_cast<const float4*>(out_s + r * 128 + ((c ^ (r & 7)) << 4));
            const float f0 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(w[i].x & 0xFFFFu), sw.x)), p.inv_k, p.expo, p.clip, p.pw0);
            const float f1 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(w[i].x >> 16), sw.y)), p.inv_k, p.expo, p.clip, p.pw0);
            const float f2 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(w[i].y & 0xFFFFu), sw.z)), p.inv_k, p.expo, p.clip, p.pw0);
            const float f3 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(w[i].y >> 16), sw.w)), p.inv_k, p.expo, p.clip, p.pw0);
            *reinterpret_cast<float4*>(p.dW + int64_t(grow) * p.lddw + gcol) =
                make_float4(g.x * f0, g.y * f1, g.z * f2, g.w * f3);
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

}  // namespace
}  // namespace fp4

namespace fp4 {
namespace {
template <bool PAIR>
fp4_status launch_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmG, const WgradParams& p, int sms,
                        cudaStream_t cs) {
  using C = WgCfg<PAIR>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = wgrad_dge_kernel<PAIR>;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t tiles = ((int64_t(p.K) + kBM * C::kCtas - 1) / (kBM * C::kCtas)) * ((int64_t(p.N) + kBN - 1) / kBN);
  const int64_t units = sms / C::kCtas;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(unsigned(C::kCtas * (tiles < units ? tiles : units)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = cs;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(C::kCtas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmG, p) != cudaSuccess) return launch_status();
  return launch_status();
}
}  // namespace
}  // namespace fp4

FP4_API fp4_status fp4_linear_wgrad_dge(const void* A, int64_t lda, const void* dY, int64_t lddy, const void* W,
                                        int64_t ldw, const float* s_w, int64_t M, int64_t N, int64_t K, float dge_k,
                                        float dge_clip, float* dW, int64_t lddw, fp4_stream_t stream) {
  using namespace fp4;
  if (!A || !dY || !W || !s_w || !dW) return FP4_ERR_INVALID_ARG;
  if (!(dge_k > 0.0f) || !(dge_clip > 0.0f) || !isfinite(dge_k)) return FP4_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || K < 8 || N % 8 || K % 8 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31))
    return FP4_ERR_SHAPE;
  if (lda < K || lddy < N || ldw < N || lddw < N) return FP4_ERR_SHAPE;
  if (lda % 8 || lddy % 8 || ldw % 8 || lddw % 4 || !aligned16(A) || !aligned16(dY) || !aligned16(W) ||
      !aligned16(dW) || (reinterpret_cast<uintptr_t>(s_w) & 3u))
    return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  CUtensorMap tmA, tmG;
  st = encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, uint64_t(K), uint64_t(M), uint64_t(lda) * 2, kBox,
                      kBT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  st = encode_tmap_2d(&tmG, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, uint64_t(N), uint64_t(M), uint64_t(lddy) * 2, kBox,
                      kBT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  WgradParams p;
  p.W = static_cast<const uint16_t*>(W);
  p.ldw = ldw;
  p.s_w = s_w;
  p.dW = dW;
  p.lddw = lddw;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.inv_k = 1.0f / dge_k;
  p.expo = 1.0f / dge_k - 1.0f;
  p.clip = dge_clip;
  p.pw0 = p.expo < 0.0f ? INFINITY : (p.expo == 0.0f ? 1.0f : 0.0f);
  p.status = status_word();
  p.wait_ns = kWaitLimitNs;
  // CTA pairs once the token loop is long (32 or more stages of 64 tokens); short
  // loops keep single-CTA tiles
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (M >= 2048) return launch_wgrad<true>(tmA, tmG, p, sms, cs);
  return launch_wgrad<false>(tmA, tmG, p, sms, cs);
}
