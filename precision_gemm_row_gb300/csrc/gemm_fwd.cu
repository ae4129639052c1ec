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
#include "common.cuh"

namespace fp4 {
namespace {

constexpr int kBM = 128;          // rows of A per tile (TMEM lanes)
constexpr int kBKBytes = 128;     // bytes of K per stage = 256 E2M1 values (one swizzle row)
constexpr int kMmaKBytes = 32;    // 64 E2M1 values per MMA
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;

template <int BN, int NACC>
struct FwdCfg {
  static constexpr int kAStage = kBM * kBKBytes;
  static constexpr int kBStage = BN * kBKBytes;
  static constexpr int kStageBytes = kAStage + kBStage;
  static constexpr int kStages = (196 * 1024) / kStageBytes;
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
};

// Instruction descriptor, kind::mxf4: A and B E2M1 (format 1), both K-major,
// UE8M0 scale type, M = 128, N = BN, dense K = 64, scale-factor ids 0.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_mxf4() {
  return (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (1u << 23) | (uint32_t(kBM >> 4) << 24);
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
  uint32_t* status;
  uint64_t wait_ns;
};

template <int BN, int NACC>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmY, const FwdParams p) {
  using C = FwdCfg<BN, NACC>;
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

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmY);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
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
  __syncthreads();
  tc_fence_after();

  const int num_m = (p.M + kBM - 1) / kBM;
  const int num_n = (p.N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int kblocks = (p.K / 2 + kBKBytes - 1) / kBKBytes;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      const int mb = tile % num_m, nb = tile / num_m;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = full0 + 8 * stage;
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          tma_load_2d(smem_u32(sA + stage * C::kAStage), &tmA, fb, kb * kBKBytes, mb * kBM);
          tma_load_2d(smem_u32(sB + stage * C::kBStage), &tmB, fb, kb * kBKBytes, nb * BN);
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
    // wait for the last load armed on every stage before the CTA may exit
    for (int s = 0; s < C::kStages; ++s) {
      const uint32_t n_s = issued / C::kStages + (uint32_t(s) < issued % C::kStages ? 1u : 0u);
      if (n_s > 0 && !mbar_wait(full0 + 8 * s, (n_s - 1) & 1u, p.wait_ns) && lane == 0)
        atomicOr(p.status, FP4_FLAG_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    constexpr uint32_t idesc = idesc_mxf4<BN>();
    const uint32_t sfa = tmem + C::kSfaCol, sfb = tmem + C::kSfbCol;
    const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + uint32_t(acc * BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait(full0 + 8 * stage, phase, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = a_base + stage * C::kAStage, b0 = b_base + stage * C::kBStage;
#pragma unroll
          for (int k = 0; k < kBKBytes / kMmaKBytes; ++k) {
            const uint64_t ad = smem_desc_sw128(a0 + k * kMmaKBytes, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b0 + k * kMmaKBytes, 16, 1024);
            mma_mxf4(d_tmem, ad, bd, idesc, sfa, sfb, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(empty0 + 8 * stage);
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(accf0 + 8 * acc);
      __syncwarp();
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    // every MMA issued by this thread must finish before TMEM is released
    if (lane == 0) tc_commit(done_bar);
    __syncwarp();
    if (!mbar_wait(done_bar, 0, p.wait_ns) && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  } else {
    // ------------------------------------------------ epilogue
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
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      const int mb = tile % num_m, nb = tile / num_m;
      // this warp's column scales 1/s_W in its own shared-memory slice (no
      // cross-warp barrier, so a warp that gives up on a wait cannot strand others)
      __syncwarp();
      for (int c = lane; c < EC; c += 32) {
        const int col = nb * BN + c_base + c;
        inv_sw_w[c] = (!raw && col < p.N) ? 1.0f / __ldg(p.s_w + col) : 1.0f;
      }
      __syncwarp();
      const int row = mb * kBM + r_local;
      const bool row_ok = row < p.M;
      float inv_sa = 1.0f;
      int e0 = 0, e1 = 0;
      if (row_ok && !raw) {
        inv_sa = 1.0f / __ldg(p.s_a + row);
        if (p.rp) {
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
      const int row0 = mb * kBM + q * 32;
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
      if (lane == 0) mbar_arrive(acce0 + 8 * acc);   // TMEM buffer free for the next tile
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();
    if (!ok && lane == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

constexpr int kFwdBN = 240;
constexpr int kFwdAcc = 2;

}  // namespace
}  // namespace fp4

FP4_API fp4_status fp4_linear_fwd(const uint8_t* a_codes, int64_t lda_codes_bytes, const float* s_a,
                                  const uint8_t* w_codes_t, int64_t ldw_codes_bytes, const float* s_w, int64_t M,
                                  int64_t N, int64_t K, const int32_t* dA_row_ptr, const int32_t* dA_col,
                                  const float* dA_val, const void* W, int64_t ldw, void* Y, int y_type, int64_t ldy,
                                  fp4_stream_t stream) {
  using namespace fp4;
  using C = FwdCfg<kFwdBN, kFwdAcc>;
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
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;

  CUtensorMap tmA, tmB;
  st = encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, uint64_t(K / 2), uint64_t(M),
                      uint64_t(lda_codes_bytes), kBKBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  st = encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_codes_t, uint64_t(K / 2), uint64_t(N),
                      uint64_t(ldw_codes_bytes), kBKBytes, kFwdBN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;

  CUtensorMap tmY;
  const bool bf16_out = (y_type == FP4_OUT_BF16);
  st = encode_tmap_2d(&tmY, bf16_out ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, Y,
                      uint64_t(N), uint64_t(M), uint64_t(ldy) * (bf16_out ? 2 : 4), bf16_out ? 40 : 20, 32,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != FP4_OK) return st;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = fp4_fwd_kernel<kFwdBN, kFwdAcc>;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set[dev] = true;
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
  p.status = status_word();
  p.wait_ns = kWaitLimitNs;
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kFwdBN - 1) / kFwdBN);
  const int grid = int(tiles < sms ? tiles : sms);
  kern<<<grid, kThreads, C::kSmemBytes, reinterpret_cast<cudaStream_t>(stream)>>>(tmA, tmB, tmY, p);
  return launch_status();
}
