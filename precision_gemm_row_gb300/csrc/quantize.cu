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

// Scales 8 BF16 values by s after clamping |x| to t, and packs their 8 E2M1
// codes into one 32-bit word (element 0 in the lowest nibble).
template <bool CLAMP>
__device__ __forceinline__ uint32_t quantize8(const uint4 v, float s, float t) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo = bf16_bits_to_float(w[i] & 0xFFFFu);
    float hi = bf16_bits_to_float(w[i] >> 16);
    if (CLAMP) {
      if (fabsf(lo) > t) lo = copysignf(t, lo);
      if (fabsf(hi) > t) hi = copysignf(t, hi);
    }
    out |= e2m1x2_encode(__fmul_rn(lo, s), __fmul_rn(hi, s)) << (8 * i);
  }
  return out;
}

__device__ __forceinline__ float absmax8(const uint4 v, float t) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fminf(fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)), t));
    m = fmaxf(m, fminf(fabsf(bf16_bits_to_float(w[i] >> 16)), t));
  }
  return m;
}

// Each row is handled by `wpr` warps; each lane keeps up to CH 16-byte chunks
// of the row in registers, so A is read from HBM exactly once.
template <int CH, bool CLAMP>
__global__ void __launch_bounds__(kRowThreads) quantize_rows_kernel(const uint16_t* __restrict__ A, int64_t M,
                                                                    int K, int64_t lda,
                                                                    const float* __restrict__ clamp_t,
                                                                    uint8_t* __restrict__ codes, int64_t ldc,
                                                                    float* __restrict__ scales, int wpr) {
  __shared__ float red[kRowThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_cta = (kRowThreads / 32) / wpr;
  const int r_in_cta = warp / wpr, w_in_row = warp % wpr;
  const int nchunk = K >> 3;
  const float t = CLAMP ? __ldg(clamp_t) : INFINITY;

  for (int64_t row0 = int64_t(blockIdx.x) * rows_per_cta; row0 < M; row0 += int64_t(gridDim.x) * rows_per_cta) {
    const int64_t row = row0 + r_in_cta;
    const bool active = row < M;
    const uint4* src = reinterpret_cast<const uint4*>(A + (active ? row : 0) * lda);
    uint4 v[CH];
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int ci = lane + 32 * (w_in_row + wpr * c);
      v[c] = (active && ci < nchunk) ? __ldcs(src + ci) : make_uint4(0u, 0u, 0u, 0u);
      amax = fmaxf(amax, absmax8(v[c], t));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (wpr > 1) {
      if (lane == 0) red[warp] = amax;
      __syncthreads();
      for (int i = 0; i < wpr; ++i) amax = fmaxf(amax, red[r_in_cta * wpr + i]);
      __syncthreads();
    }
    const float s = scale_from_absmax(amax);
    if (active) {
      if (w_in_row == 0 && lane == 0) scales[row] = s;
      uint32_t* dst = reinterpret_cast<uint32_t*>(codes + row * ldc);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int ci = lane + 32 * (w_in_row + wpr * c);
        if (ci < nchunk) dst[ci] = quantize8<CLAMP>(v[c], s, t);
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
    for (int k = k0 + grp; k < k1; k += 8) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(W + int64_t(k) * ldw) + cchunk);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m[2 * i] = fmaxf(m[2 * i], fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)));
        m[2 * i + 1] = fmaxf(m[2 * i + 1], fabsf(bf16_bits_to_float(w[i] >> 16)));
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

// Quantizes a 64 (K) x 64 (N) tile of W with the column scales and writes it
// transposed: codes_t[j][k/2], 32 bytes per column per tile.
__global__ void __launch_bounds__(256) quantize_cols_kernel(const uint16_t* __restrict__ W, int K, int N,
                                                           int64_t ldw, const uint32_t* __restrict__ colmax,
                                                           uint8_t* __restrict__ codes_t, int64_t ldc,
                                                           float* __restrict__ scales) {
  __shared__ float s_col[64];
  __shared__ uint8_t tile[64][64 + 16];  // [column][k] one code per byte
  const int tid = threadIdx.x;
  const int j0 = blockIdx.x * 64, k0 = blockIdx.y * 64;
  if (tid < 64) {
    const int j = j0 + tid;
    float s = 1.0f;
    if (j < N) {
      s = scale_from_absmax(__uint_as_float(colmax[j]));
      if (blockIdx.y == 0) scales[j] = s;
    }
    s_col[tid] = s;
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int r = (tid >> 3) + 32 * it;  // k within tile
    const int cc = tid & 7;              // 8-column chunk within tile
    const int k = k0 + r, j = j0 + cc * 8;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (k < K && j < N) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(W + int64_t(k) * ldw + j));
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float x0 = bf16_bits_to_float(w[i >> 1] & 0xFFFFu);
      const float x1 = bf16_bits_to_float(w[i >> 1] >> 16);
      const uint32_t c2 = e2m1x2_encode(__fmul_rn(x0, s_col[cc * 8 + i]), __fmul_rn(x1, s_col[cc * 8 + i + 1]));
      tile[cc * 8 + i][r] = static_cast<uint8_t>(c2 & 0xFu);
      tile[cc * 8 + i + 1][r] = static_cast<uint8_t>(c2 >> 4);
    }
  }
  __syncthreads();
  if (tid < 128) {
    const int c = tid >> 1, h = tid & 1;  // column, which 32-k half
    const int j = j0 + c, k = k0 + 32 * h;
    if (j < N && k < K) {
      uint32_t out[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t wv = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) wv |= uint32_t(tile[c][32 * h + 8 * q + b]) << (4 * b);
        out[q] = wv;
      }
      *reinterpret_cast<uint4*>(codes_t + int64_t(j) * ldc + (k >> 1)) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
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
  if (K % 32 != 0 || K > (1 << 30) || lda < K || ldc_bytes < K / 2) return FP4_ERR_SHAPE;
  if (lda % 8 != 0 || ldc_bytes % 16 != 0 || !aligned16(A) || !aligned16(codes) || !aligned16(scales) ||
      (clamp_t && (reinterpret_cast<uintptr_t>(clamp_t) & 3u)))
    return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  if (M == 0) return FP4_OK;
  const int nchunk = int(K / 8);
  // warps per row and chunks per lane: keep <= 16 chunks (64 registers) per lane
  int wpr = 1;
  while (wpr < 8 && nchunk > 32 * 16 * wpr) wpr *= 2;
  const int per_lane = (nchunk + 32 * wpr - 1) / (32 * wpr);
  auto s = reinterpret_cast<cudaStream_t>(stream);
  const auto* a = static_cast<const uint16_t*>(A);
  if (per_lane <= 1) launch_rows<1>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 2) launch_rows<2>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 4) launch_rows<4>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 8) launch_rows<8>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 12) launch_rows<12>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
  else if (per_lane <= 16) launch_rows<16>(a, M, int(K), lda, clamp_t, codes, ldc_bytes, scales, wpr, sms, s);
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
  auto s = reinterpret_cast<cudaStream_t>(stream);
  auto* colmax = static_cast<uint32_t*>(workspace);
  if (cudaMemsetAsync(colmax, 0, size_t(N) * 4, s) != cudaSuccess) return FP4_ERR_CUDA;
  const int col_blocks = int((N + 255) / 256);
  int splits = (4 * sms + col_blocks - 1) / col_blocks;
  const int max_splits = int((K + 63) / 64);
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  const int rows_per_split = int((K + splits - 1) / splits);
  splits = int((K + rows_per_split - 1) / rows_per_split);
  const auto* w = static_cast<const uint16_t*>(W);
  col_absmax_kernel<<<dim3(col_blocks, splits), 256, 0, s>>>(w, int(K), int(N), ldw, rows_per_split, colmax);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  quantize_cols_kernel<<<dim3(unsigned((N + 63) / 64), unsigned((K + 63) / 64)), 256, 0, s>>>(
      w, int(K), int(N), ldw, colmax, codes_t, ldc_bytes, scales);
  return launch_status();
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
  auto s = reinterpret_cast<cudaStream_t>(stream);
  // the maxima are merged with atomic max, so the shared array must start at zero on every call
  if (cudaMemsetAsync(colmax, 0, size_t(N) * 4, s) != cudaSuccess) return FP4_ERR_CUDA;
  const int col_blocks = int((N + 255) / 256);
  int splits = (4 * sms + col_blocks - 1) / col_blocks;
  const int max_splits = int((K + 63) / 64);
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  const int rows_per_split = int((K + splits - 1) / splits);
  splits = int((K + rows_per_split - 1) / rows_per_split);
  const auto* w = static_cast<const uint16_t*>(W);
  col_absmax_kernel<<<dim3(col_blocks, splits), 256, 0, s>>>(w, int(K), int(N), ldw, rows_per_split, colmax);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  quantize_cols_kernel<<<dim3(unsigned((N + 63) / 64), unsigned((K + 63) / 64)), 256, 0, s>>>(
      w, int(K), int(N), ldw, colmax, codes_t, ldc_bytes, scales);
  return launch_status();
}
