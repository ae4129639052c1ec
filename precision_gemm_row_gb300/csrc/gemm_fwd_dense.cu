// Forward of the quantized linear layer for a dense compensation matrix, on
// sm_103a tensor cores.
//
// Page "Microsoft Research bringt den ersten FP4-Genauigkeitsrahmen ..."
// (topaibox.com), "Peak-Dämpfung und -Kompensation von Ausreißern", and the
// outlier passage of page "首个 FP4 精度的大模型训练框架来了" (czzqal.com): the
// clamped activation goes through the FP4 GEMM and the sparse matrix
// dA = A - A_clamped is multiplied in higher precision and added:
//   Y = (qA qW^T) / (s_A s_W^T) + dA W.
// When the clamp quantile is low (a few percent of A clamped), dA has entries
// in every column of every 128 x 64 tile, and its product is a dense GEMM.
// Here it runs on the BF16 tensor cores, exactly:
//   1. every fp32 entry of dA is split into BF16 parts whose sum is the entry,
//      written densely as D = [part 1 | part 2 | ...] (M x parts K): with the
//      clamp threshold t given, two parts, A and -sign(A) t (each entry is
//      A - sign(A) t with A and t BF16); without it, three (round to nearest
//      at each step: 3 x 8 significant bits cover the 24 of an fp32 value);
//   2. W^T (N x K, BF16) is written once, since the engine reads its operands
//      with the reduction dimension contiguous;
//   3. the FP4 product without compensation is written in fp32 to the
//      workspace (the forward kernel, unchanged);
//   4. the backward BF16 engine forms D (W^T)^T over the parts x K reduction, reading
//      W^T again for each part (reduction index modulo K), with its chunked
//      fp32 accumulation, and its epilogue adds the fp32 FP4 product and
//      rounds once to the caller's output type.
#include "bwd_gemm.cuh"

namespace fp4 {
namespace {

constexpr int kDensifyWarps = 8;

// BF16 of an fp32 value, round to nearest even (finite inputs).
__device__ __forceinline__ uint32_t bf16_rn_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// One warp per row of dA: the row of D is zeroed (PARTS K-wide parts), then
// the row's entries are split and written at columns k, K + k (, 2K + k).
// __syncwarp orders the zeros before the entries (same warp, same addresses).
//  PARTS = 3: hi + mid + lo = the fp32 entry (each part rounded to nearest from
//             what is left; the remainders are exact);
//  PARTS = 2: the entry is A - sign(A) t with A and t BF16 values (a clamp at
//             t), so A = entry + sign t (exact in fp32) and -sign t are its two
//             exact BF16 parts; an entry for which A is not a BF16 value breaks
//             that premise: it is written as hi + lo rounded and reported.
template <int PARTS>
__global__ void __launch_bounds__(32 * kDensifyWarps)
    densify_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
                   const float* __restrict__ val, const float* __restrict__ t_ptr, int M, int K,
                   uint16_t* __restrict__ D, uint32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * kDensifyWarps + warp;
  if (m >= M) return;   // whole warps only
  uint16_t* row = D + int64_t(m) * PARTS * K;
  uint4* row4 = reinterpret_cast<uint4*>(row);
  const int n4 = PARTS * K / 8;
  for (int i = lane; i < n4; i += 32) row4[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  const float t = PARTS == 2 ? __ldg(t_ptr) : 0.0f;
  const int e0 = __ldg(row_ptr + m), e1 = __ldg(row_ptr + m + 1);
  bool bad = false;
  for (int e = e0 + lane; e < e1; e += 32) {
    const int k = __ldg(col + e);
    if (k < 0 || k >= K) {
      bad = true;   // the forward skips a column outside [0, K) and reports it
      continue;
    }
    const float v = __ldg(val + e);
    if constexpr (PARTS == 2) {
      const float st = copysignf(t, v);
      const float a = v + st;                          // A itself when the premise holds
      uint32_t hi = __float_as_uint(a) >> 16, lo = bf16_rn_bits(-st);
      if ((__float_as_uint(a) & 0xFFFFu) != 0u || bf16_bits_to_float(lo) != -st) {
        bad = true;
        hi = bf16_rn_bits(v);
        lo = bf16_rn_bits(v - bf16_bits_to_float(hi));
      }
      row[k] = uint16_t(hi);
      row[K + k] = uint16_t(lo);
    } else {
      const uint32_t hi = bf16_rn_bits(v);
      const float r1 = v - bf16_bits_to_float(hi);    // exact: v minus its own rounding
      const uint32_t mid = bf16_rn_bits(r1);
      const float r2 = r1 - bf16_bits_to_float(mid);  // exact again
      const uint32_t lo = bf16_rn_bits(r2);
      row[k] = uint16_t(hi);
      row[K + k] = uint16_t(mid);
      row[2 * K + k] = uint16_t(lo);
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(status, FP4_FLAG_INTERNAL);
}

// W (K x N, ldw) -> WT (N x K), 64 x 64 tiles through shared memory.
__global__ void __launch_bounds__(256)
    transpose_bf16_kernel(const uint16_t* __restrict__ W, int64_t ldw, int K, int N, uint16_t* __restrict__ WT) {
  __shared__ uint16_t t[64][66];
  const int k0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int k = k0 + ty + 8 * i;
    const int n = n0 + 2 * tx;
    uint32_t v = 0u;
    if (k < K && n < N) v = *reinterpret_cast<const uint32_t*>(W + int64_t(k) * ldw + n);   // N % 8 == 0
    t[ty + 8 * i][2 * tx] = uint16_t(v & 0xFFFFu);
    t[ty + 8 * i][2 * tx + 1] = uint16_t(v >> 16);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = n0 + ty + 8 * i;
    const int k = k0 + 2 * tx;
    if (n < N && k < K) {
      const uint32_t v = uint32_t(t[2 * tx][ty + 8 * i]) | (uint32_t(t[2 * tx + 1][ty + 8 * i]) << 16);
      *reinterpret_cast<uint32_t*>(WT + int64_t(n) * K + k) = v;                           // K % 64 == 0
    }
  }
}

// Y = round(C + Y0): C the engine's fp32 sum (dA W), Y0 the fp32 FP4 product.
struct AddEpilogue {
  const float* y0;
  int64_t ld0;
  void* out;
  int64_t ld;
  int rows, cols;
  bool bf16;

  __device__ __forceinline__ void prefetch(int row0, int col0, int lane) const {
    const int grow = row0 + lane;
    if (grow < rows && col0 < cols) prefetch_l2(y0 + int64_t(grow) * ld0 + col0);
  }
  struct Pre {
    float4 y[4];
  };
  __device__ __forceinline__ Pre load(int row0, int gcol, bool col_ok, int lane) const {
    Pre pr;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int grow = row0 + (lane >> 3) + 4 * i;
      pr.y[i] = (col_ok && grow < rows) ? __ldg(reinterpret_cast<const float4*>(y0 + int64_t(grow) * ld0 + gcol))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return pr;
  }
  __device__ __forceinline__ void store(const Pre& pr, int i, int grow, int gcol, float4 g) const {
    const float4 y = make_float4(pr.y[i].x + g.x, pr.y[i].y + g.y, pr.y[i].z + g.z, pr.y[i].w + g.w);
    const int64_t off = int64_t(grow) * ld + gcol;
    if (bf16) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(y.x, y.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(y.z, y.w);
      uint2 v;
      v.x = *reinterpret_cast<const uint32_t*>(&lo);
      v.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + off) = v;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = y;
    }
  }
};

template <bool PAIR>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    dense_comp_kernel(const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmWT,
                      const bwd::Shape s, const AddEpilogue e) {
  bwd::run<true, PAIR>(tmD, tmWT, s, e);
}

// Workspace: [Y0 fp32 M x N][D bf16 M x 3K (or 2K)][WT bf16 N x K][engine split tail], 256-byte aligned parts.
struct DenseLayout {
  size_t y0, d, wt, tail, total;
};

size_t round256d(size_t x) { return (x + 255) / 256 * 256; }

DenseLayout dense_layout(int64_t M, int64_t N, int64_t K, int sms) {
  DenseLayout L;
  size_t off = 0;
  L.y0 = off; off += round256d(size_t(M) * size_t(N) * 4);
  L.d = off; off += round256d(size_t(M) * size_t(3 * K) * 2);
  L.wt = off; off += round256d(size_t(N) * size_t(K) * 2);
  const size_t t2 = bwd::plan_split(M, N, 2 * K, sms).total, t3 = bwd::plan_split(M, N, 3 * K, sms).total;
  L.tail = off; off += round256d(t2 > t3 ? t2 : t3);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace fp4

FP4_API size_t fp4_linear_fwd_dense_workspace(int64_t M, int64_t N, int64_t K) {
  using namespace fp4;
  int sms = 0;
  if (M < 1 || N < 1 || K < 64 || K % 64 || check_device(&sms) != FP4_OK) return 0;
  return dense_layout(M, N, K, sms).total;
}

FP4_API fp4_status fp4_linear_fwd_dense(const uint8_t* a_codes, int64_t lda_codes_bytes, const float* s_a,
                                        const uint8_t* w_codes_t, int64_t ldw_codes_bytes, const float* s_w,
                                        int64_t M, int64_t N, int64_t K, const int32_t* dA_row_ptr,
                                        const int32_t* dA_col, const float* dA_val, const float* dA_t,
                                        const void* W, int64_t ldw, void* Y, int y_type, int64_t ldy,
                                        void* workspace, size_t ws_bytes, fp4_stream_t stream) {
  using namespace fp4;
  if (!a_codes || !s_a || !w_codes_t || !s_w || !dA_row_ptr || !dA_col || !dA_val || !W || !Y || !workspace)
    return FP4_ERR_INVALID_ARG;
  if (y_type != FP4_OUT_BF16 && y_type != FP4_OUT_FP32) return FP4_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || N % 8 || K < 64 || K % 64 || K > 16384 || M >= (int64_t(1) << 31) ||
      N >= (int64_t(1) << 31))
    return FP4_ERR_SHAPE;
  if (ldw < N || ldy < N) return FP4_ERR_SHAPE;
  if (ldw % 8 || ldy % 8 || !aligned16(W) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      (reinterpret_cast<uintptr_t>(dA_t) & 3u))
    return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  const DenseLayout L = dense_layout(M, N, K, sms);
  if (ws_bytes < L.total) return FP4_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* y0 = reinterpret_cast<float*>(ws + L.y0);
  uint16_t* D = reinterpret_cast<uint16_t*>(ws + L.d);
  uint16_t* WT = reinterpret_cast<uint16_t*>(ws + L.wt);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  // the FP4 product alone, fp32 (checks the code and scale arguments itself)
  st = fp4_linear_fwd(a_codes, lda_codes_bytes, s_a, w_codes_t, ldw_codes_bytes, s_w, M, N, K, nullptr, nullptr,
                      nullptr, nullptr, 0, y0, FP4_OUT_FP32, N, nullptr, 0, stream);
  if (st != FP4_OK) return st;
  const int parts = dA_t ? 2 : 3;
  const unsigned dgrid = unsigned((M + kDensifyWarps - 1) / kDensifyWarps);
  if (parts == 2)
    densify_kernel<2><<<dgrid, 32 * kDensifyWarps, 0, cs>>>(dA_row_ptr, dA_col, dA_val, dA_t, int(M), int(K), D,
                                                            status_word());
  else
    densify_kernel<3><<<dgrid, 32 * kDensifyWarps, 0, cs>>>(dA_row_ptr, dA_col, dA_val, nullptr, int(M), int(K), D,
                                                            status_word());
  transpose_bf16_kernel<<<dim3(unsigned((N + 63) / 64), unsigned(K / 64)), 256, 0, cs>>>(
      static_cast<const uint16_t*>(W), ldw, int(K), int(N), WT);
  st = launch_status();
  if (st != FP4_OK) return st;

  CUtensorMap tmD, tmWT;
  st = encode_tmap_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, uint64_t(parts * K), uint64_t(M),
                      uint64_t(parts * K) * 2,
                      bwd::kBT, bwd::kBox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  st = encode_tmap_2d(&tmWT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, WT, uint64_t(K), uint64_t(N), uint64_t(K) * 2,
                      bwd::kBT, bwd::kBox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  AddEpilogue e;
  e.y0 = y0;
  e.ld0 = N;
  e.out = Y;
  e.ld = ldy;
  e.rows = int(M);
  e.cols = int(N);
  e.bf16 = (y_type == FP4_OUT_BF16);
  bwd::Shape s;
  s.R = int(M);
  s.C = int(N);
  s.L = int(parts * K);
  s.q_wrap = int(K);
  s.status = status_word();
  s.wait_ns = kWaitLimitNs;
  st = bwd::schedule(s, bwd::plan_split(M, N, parts * K, sms), ws + L.tail, ws_bytes - L.tail, cs);
  if (st != FP4_OK) return st;
  if (bwd::use_pairs(parts * K)) return bwd::launch<true, true>(dense_comp_kernel<true>, s, sms, cs, tmD, tmWT, s, e);
  return bwd::launch<true, false>(dense_comp_kernel<false>, s, sms, cs, tmD, tmWT, s, e);
}
