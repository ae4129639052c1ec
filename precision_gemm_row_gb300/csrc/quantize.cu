// Row (token-wise) and column (channel-wise) absmax quantization of BF16 to
// packed E2M1, per the granularity and quantization passages of the page
// "首个 FP4 精度的大模型训练框架来了" (czzqal.com): A per row, W per column,
// scale into the FP4 range, round to the nearest FP4 value.
//
// Both are HBM-bound streaming kernels: 16-byte loads, one row or column strip
// per warp / CTA, absmax by warp shuffles, two codes per byte.
#include <mutex>

#include "common.cuh"

namespace fp4 {
namespace {

constexpr int kRowThreads = 256;  // 8 warps

// Each row is handled by `wpr` warps; each lane keeps up to CH 16-byte chunks
// of the row in registers, so A is read from HBM exactly once.
template <int CH, bool CLAMP>
__global__ void __launch_bounds__(kRowThreads, 2) quantize_rows_kernel(const uint16_t* __restrict__ A, int64_t M,
                                                                       int K, int64_t lda,
                                                                       const float* __restrict__ clamp_t,
                                                                       uint8_t* __restrict__ codes, int64_t ldc,
                                                                       float* __restrict__ scales, int wpr) {
  __shared__ uint32_t red[kRowThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_cta = (kRowThreads / 32) / wpr;
  const int r_in_cta = warp / wpr, w_in_row = warp % wpr;
  const int nchunk = K >> 3;
  // A BF16 threshold (the usual case: the quantile threshold is one) is applied
  // exactly on the bit patterns; any other fp32 threshold in fp32.
  const float tf = CLAMP ? __ldg(clamp_t) : INFINITY;
  const bool t_bits_exact = (__float_as_uint(tf) & 0xFFFFu) == 0u;
  const uint32_t tb = CLAMP ? (__float_as_uint(tf) >> 16) & 0x7FFFu : 0x7FFFu;
  const uint32_t tb2 = tb | (tb << 16);

  for (int64_t row0 = int64_t(blockIdx.x) * rows_per_cta; row0 < M; row0 += int64_t(gridDim.x) * rows_per_cta) {
    const int64_t row = row0 + r_in_cta;
    const bool active = row < M;
    const uint4* src = reinterpret_cast<const uint4*>(A + (active ? row : 0) * lda);
    uint4 v[CH];
    uint32_t mx = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int ci = lane + 32 * (w_in_row + wpr * c);
      v[c] = (active && ci < nchunk) ? __ldcs(src + ci) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) mx = maxmag8(v[c], mx);
    uint32_t amax_bits = warp_max_bits(mx);
    if (wpr > 1) {
      if (lane == 0) red[warp] = amax_bits;
      __syncthreads();
      for (int i = 0; i < wpr; ++i) amax_bits = max(amax_bits, red[r_in_cta * wpr + i]);
      __syncthreads();
    }
    // max over min(|x|, t) = min(max |x|, t)
    const float s = scale_from_absmax(CLAMP ? fminf(bf16_bits_to_float(amax_bits), tf) : bf16_bits_to_float(amax_bits));
    if (active) {
      if (w_in_row == 0 && lane == 0) scales[row] = s;
      uint32_t* dst = reinterpret_cast<uint32_t*>(codes + row * ldc);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int ci = lane + 32 * (w_in_row + wpr * c);
        if (ci < nchunk)
          dst[ci] = (!CLAMP || t_bits_exact) ? quantize8<CLAMP>(v[c], s, tb2) : quantize8_clamp_f32(v[c], s, tf);
      }
    }
  }
}

// Column maxima of |W|: each CTA covers 256 columns (8 per lane) and a slice
// of rows; partial maxima are merged with an atomic max on the fp32 bit
// pattern (valid for non-negative floats).
__global__ void __launch_bounds__(256) col_absmax_kernel(const uint16_t* __restrict__ W, int K, int N, int64_t ldw,
                                                        int rows_per_split, uint32_t* __restrict__ colmax) {
  __shared__ float part[8][256 + 8];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int cchunk = blockIdx.x * 32 + lane;  // 8-column chunk index
  const bool col_ok = cchunk * 8 < N;
  const int k0 = blockIdx.y * rows_per_split;
  const int k1 = min(K, k0 + rows_per_split);
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = 0.0f;
  if (col_ok) {
    constexpr int kU = 4;  // rows in flight per thread
    for (int kb = k0 + grp; kb < k1; kb += 8 * kU) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int k = kb + 8 * u;
        v[u] = k < k1 ? __ldg(reinterpret_cast<const uint4*>(W + int64_t(k) * ldw) + cchunk)
                      : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          m[2 * i] = fmaxf(m[2 * i], fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)));
          m[2 * i + 1] = fmaxf(m[2 * i + 1], fabsf(bf16_bits_to_float(w[i] >> 16)));
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[grp][lane * 8 + i] = m[i];
  __syncthreads();
  const int c = threadIdx.x;  // one column of the 256 per thread
  float r = part[0][c];
#pragma unroll
  for (int g = 1; g < 8; ++g) r = fmaxf(r, part[g][c]);
  const int col = blockIdx.x * 256 + c;
  if (col < N) atomicMax(colmax + col, __float_as_uint(r));
}

// Quantizes a 256 (K) x 32 (N) tile of W with the column scales and writes it
// transposed (codes_t[j][k/2], 128 bytes per column per tile).  The tile comes
// in by one TMA load (row pitch 64 bytes: a warp reading one k for 32 columns
// touches 64 contiguous bytes) and leaves by one TMA store from a 128-byte
// swizzled staging tile (one 128-byte row per column).
constexpr int kColTileK = 256, kColTileN = 32;

__global__ void __launch_bounds__(256) quantize_cols_tma_kernel(const __grid_constant__ CUtensorMap tmW,
                                                               const __grid_constant__ CUtensorMap tmC, int K, int N,
                                                               const uint32_t* __restrict__ colmax,
                                                               float* __restrict__ scales,
                                                               uint32_t* __restrict__ status) {
  __shared__ __align__(1024) uint8_t w_s[kColTileK * kColTileN * 2];
  __shared__ __align__(1024) uint8_t c_s[kColTileN * 128];
  __shared__ float s_col[kColTileN];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  // K tiles in reverse: the rows col_absmax_kernel read last are the likeliest to be in L2
  const int j0 = blockIdx.x * kColTileN, k0 = (int(gridDim.y) - 1 - int(blockIdx.y)) * kColTileK;
  const uint32_t b = smem_u32(&bar);
  if (tid == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(b, kColTileK * kColTileN * 2);
    tma_load_2d(smem_u32(w_s), &tmW, b, j0, k0);
  }
  if (tid < kColTileN) {
    const int j = j0 + tid;
    float sc = 1.0f;
    if (j < N) {
      sc = scale_from_absmax(__uint_as_float(colmax[j]));
      if (k0 == 0) scales[j] = sc;
    }
    s_col[tid] = sc;
  }
  __syncthreads();
  const bool ok = mbar_wait(b, 0, kWaitLimitNs);
  if (!ok && tid == 0) atomicOr(status, FP4_FLAG_TIMEOUT);
  const int j = tid & 31, kq = tid >> 5;  // column, group of 32 rows (one warp per group)
  const float sc = s_col[j];
  const uint16_t* col = reinterpret_cast<const uint16_t*>(w_s) + j;
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t word = 0;
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
      const int k = 32 * kq + 8 * q + 2 * bb;
      const float x0 = bf16_bits_to_float(col[k * kColTileN]);
      const float x1 = bf16_bits_to_float(col[(k + 1) * kColTileN]);
      word |= e2m1x2_encode(__fmul_rn(x0, sc), __fmul_rn(x1, sc)) << (8 * bb);
    }
    out[q] = word;
  }
  *reinterpret_cast<uint4*>(c_s + j * 128 + ((kq ^ (j & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0 && ok) {
    tma_store_2d(&tmC, smem_u32(c_s), k0 / 2, j0);
    bulk_commit_group();
    bulk_wait_all();
  }
}

// Column maxima (atomic max into colmax) then the TMA tile quantizer.
fp4_status launch_cols(const uint16_t* w, int64_t K, int64_t N, int64_t ldw, uint8_t* codes_t, int64_t ldc,
                       float* scales, uint32_t* colmax, int sms, cudaStream_t s) {
  CUtensorMap tmW, tmC;
  fp4_status st = encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, uint64_t(N), uint64_t(K),
                                 uint64_t(ldw) * 2, kColTileN, kColTileK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != FP4_OK) return st;
  st = encode_tmap_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes_t, uint64_t(K / 2), uint64_t(N), uint64_t(ldc), 128,
                      kColTileN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  if (cudaMemsetAsync(colmax, 0, size_t(N) * 4, s) != cudaSuccess) return FP4_ERR_CUDA;
  const int col_blocks = int((N + 255) / 256);
  int splits = (4 * sms + col_blocks - 1) / col_blocks;
  const int max_splits = int((K + 63) / 64);
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  const int rows_per_split = int((K + splits - 1) / splits);
  splits = int((K + rows_per_split - 1) / rows_per_split);
  col_absmax_kernel<<<dim3(col_blocks, splits), 256, 0, s>>>(w, int(K), int(N), ldw, rows_per_split, colmax);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  quantize_cols_tma_kernel<<<dim3(unsigned((N + kColTileN - 1) / kColTileN), unsigned((K + kColTileK - 1) / kColTileK)),
                             256, 0, s>>>(tmW, tmC, int(K), int(N), colmax, scales, status_word());
  return launch_status();
}

template <int CH>
void launch_rows(const uint16_t* A, int64_t M, int K, int64_t lda, const float* clamp_t, uint8_t* codes,
                 int64_t ldc, float* scales, int wpr, int sms, cudaStream_t stream) {
  const int rows_per_cta = 8 / wpr;
  int64_t blocks = (M + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = int64_t(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (clamp_t)
    quantize_rows_kernel<CH, true><<<unsigned(blocks), kRowThreads, 0, stream>>>(A, M, K, lda, clamp_t, codes, ldc,
                                                                               scales, wpr);
  else
    quantize_rows_kernel<CH, false><<<unsigned(blocks), kRowThreads, 0, stream>>>(A, M, K, lda, clamp_t, codes, ldc,
                                                                                scales, wpr);
}

}  // namespace
}  // namespace fp4

FP4_API fp4_status fp4_quantize_rows(const void* A, int64_t M, int64_t K, int64_t lda, const float* clamp_t,
                                     uint8_t* codes, int64_t ldc_bytes, float* scales, fp4_stream_t stream) {
  using namespace fp4;
  if (M < 0 || K <= 0) return FP4_ERR_SHAPE;
  if (M > 0 && (!A || !codes || !scales)) return FP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || K > 16384 || lda < K || ldc_bytes < K / 2) return FP4_ERR_SHAPE;
  if (lda % 8 != 0 || ldc_bytes % 16 != 0 || !aligned16(A) || !aligned16(codes) || !aligned16(scales) ||
      (clamp_t && (reinterpret_cast<uintptr_t>(clamp_t) & 3u)))
    return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  if (M == 0) return FP4_OK;
  const int nchunk = int(K / 8);
  // warps per row and chunks per lane: keep <= 8 chunks (32 registers) per lane
  int wpr = 1;
  while (wpr < 8 && nchunk > 32 * 8 * wpr) wpr *= 2;
  const int per_lane = (nchunk + 32 * wpr - 1) / (32 * wpr);
  auto s = reinterpret_cast<cudaStream_t>(stream);
  const auto* a = static_cast<const uint16_t*>(A);
  if (per_lane <= 1) launch_rows<1>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 2) launch_rows<2>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 4) launch_rows<4>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 8) launch_rows<8>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else return FP4_ERR_SHAPE;
  return launch_status();
}

FP4_API size_t fp4_quantize_cols_workspace(int64_t N) {
  return N > 0 ? size_t((N * 4 + 255) / 256 * 256) : 0;
}

FP4_API fp4_status fp4_quantize_cols(const void* W, int64_t K, int64_t N, int64_t ldw, uint8_t* codes_t,
                                     int64_t ldc_bytes, float* scales, void* workspace, size_t ws_bytes,
                                     fp4_stream_t stream) {
  using namespace fp4;
  if (K <= 0 || N <= 0) return FP4_ERR_SHAPE;
  if (!W || !codes_t || !scales) return FP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || N % 8 != 0 || K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || ldw < N ||
      ldc_bytes < K / 2)
    return FP4_ERR_SHAPE;
  if (ldw % 8 != 0 || ldc_bytes % 16 != 0 || !aligned16(W) || !aligned16(codes_t) || !aligned16(scales))
    return FP4_ERR_ALIGNMENT;
  if (!workspace || ws_bytes < fp4_quantize_cols_workspace(N)) return FP4_ERR_WORKSPACE;
  if (!aligned16(workspace)) return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  return launch_cols(static_cast<const uint16_t*>(W), K, N, ldw, codes_t, ldc_bytes, scales,
                     static_cast<uint32_t*>(workspace), sms, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Column quantization without caller-provided scratch.
//
// Some callers cannot hand the library any scratch memory: code that runs
// inside a framework which owns every device allocation (so it has no handle
// to allocate a workspace), real-time paths that must not call cudaMalloc
// because it can synchronize the device, and embedded users with a fixed
// memory budget.  For them the column maxima live in a fixed device array
// that is part of the library image: every GPU that loads the library holds
// it (256 KiB) until the process exits, and it bounds N.
namespace fp4 {
namespace {
constexpr int64_t kNoAllocMaxN = 65536;
static __device__ __align__(256) uint32_t g_colmax_scratch[kNoAllocMaxN];

std::mutex g_scratch_mu;
uint32_t* g_scratch_ptr[64];

// Device address of g_colmax_scratch for the current device, looked up once
// per device (host code cannot use the symbol itself as a device pointer).
fp4_status scratch_address(uint32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_colmax_scratch) != cudaSuccess || !ptr) return FP4_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint32_t*>(ptr);
  }
  *out = g_scratch_ptr[dev];
  return FP4_OK;
}
}  // namespace
}  // namespace fp4

FP4_API fp4_status fp4_quantize_cols_noalloc(const void* W, int64_t K, int64_t N, int64_t ldw, uint8_t* codes_t,
                                             int64_t ldc_bytes, float* scales, fp4_stream_t stream) {
  using namespace fp4;
  if (K <= 0 || N <= 0) return FP4_ERR_SHAPE;
  if (!W || !codes_t || !scales) return FP4_ERR_INVALID_ARG;
  if (N > kNoAllocMaxN) return FP4_ERR_SHAPE;  // the built-in scratch holds at most 65536 column maxima
  if (K % 32 != 0 || N % 8 != 0 || K >= (int64_t(1) << 31) || ldw < N || ldc_bytes < K / 2) return FP4_ERR_SHAPE;
  if (ldw % 8 != 0 || ldc_bytes % 16 != 0 || !aligned16(W) || !aligned16(codes_t) || !aligned16(scales))
    return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  uint32_t* colmax = nullptr;
  st = scratch_address(&colmax);
  if (st != FP4_OK) return st;
  // the maxima are merged with atomic max, so launch_cols clears the shared array on every call
  return launch_cols(static_cast<const uint16_t*>(W), K, N, ldw, codes_t, ldc_bytes, scales, colmax, sms,
                     reinterpret_cast<cudaStream_t>(stream));
}
