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
// G = A^T dY runs on the backward BF16 engine (bwd_gemm.cuh) with both
// operands MN-major (the token dimension strided); its epilogue loads W and
// s_W for each 32 x 32 block of dW, computes the factors and writes dW = G f'
// once.
#include <cmath>

#include "bwd_gemm.cuh"

namespace fp4 {
namespace {

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Constants of the DGE factor for one call.
struct DgeConst {
  float inv_k;        // 1/k
  float expo;         // 1/k - 1
  float log2_inv_k;   // log2(1/k)
  float clip;
  float f_mid;        // the factor at u = 0: min(clip, (1/k) lim |u|^expo), +inf, 1 or 0 before clipping
};

// DGE factor f'(x) for the scaled weight magnitude x.  (1/k)|u|^expo is taken
// as 2^(expo log2 u + log2(1/k)) on the special-function unit (relative error
// about 1e-6 at the largest exponents, far inside the 1e-5 bound of dW); u is
// 0 or at least 2^-23 here, so flushing subnormals changes nothing, and u = 0
// (an interval midpoint) takes the precomputed limit.  The interval is found
// by scaling x with 2/delta (a power of two, so s and its fractional part are
// exact), and every case is a select, so a warp never diverges over mixed
// magnitudes.
__device__ __forceinline__ float dge_factor(float x, const DgeConst& c) {
  const float two_over_delta = x < 2.0f ? 2.0f : (x < 4.0f ? 1.0f : 0.5f);
  const float s = x * two_over_delta;                        // interval [floor(s), floor(s) + 1)
  const float u = fabsf(fmaf(s - floorf(s), 2.0f, -1.0f));   // |2 (x - lo) / delta - 1|
  const float f = fminf(c.clip, ex2_approx(fmaf(c.expo, lg2_approx(u), c.log2_inv_k)));
  const float fu = u > 0.0f ? f : c.f_mid;
  return x < 6.0f ? fu : c.inv_k;
}

// Two E4M3 bytes of fl32 values (lo at the lower address), round to nearest
// even, magnitudes past 448 saturated to 448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// dW[k, n] = G[k, n] * f'(|fl32(W[k, n] s_W[n])|): fp32, or (FP8) the E4M3
// codes of fl32(dW * scale) with max |dW| kept per thread (amax) and folded
// into *amax_out at the end of the kernel (finish).
template <bool FP8>
struct DgeEpilogue {
  const uint16_t* W;
  int64_t ldw;
  const float* s_w;
  void* dW;
  int64_t lddw;
  int rows, cols;   // K, N
  DgeConst dge;
  const float* scale;   // FP8: device, per-tensor
  float* amax_out;      // FP8: device, zeroed before the launch
  mutable float amax;   // FP8: this thread's max |dW| so far

  // W rows row0..row0+31 (columns col0..col0+63: one 128-byte line per row)
  // and s_w[col0..col0+63] (two lines) into L2
  __device__ __forceinline__ void prefetch(int row0, int col0, int lane) const {
    const int grow = row0 + lane;
    if (grow < rows && col0 < cols) prefetch_l2(W + int64_t(grow) * ldw + col0);
    if (lane < 2 && col0 + 32 * lane < cols) prefetch_l2(s_w + col0 + 32 * lane);
  }

  struct Pre {
    float4 sw;
    uint2 w[4];
  };
  __device__ __forceinline__ Pre load(int row0, int gcol, bool col_ok, int lane) const {
    Pre pr;
    pr.sw = make_float4(1.f, 1.f, 1.f, 1.f);
    if (col_ok) pr.sw = make_float4(__ldg(s_w + gcol), __ldg(s_w + gcol + 1), __ldg(s_w + gcol + 2), __ldg(s_w + gcol + 3));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int grow = row0 + (lane >> 3) + 4 * i;
      pr.w[i] = (col_ok && grow < rows) ? __ldg(reinterpret_cast<const uint2*>(W + int64_t(grow) * ldw + gcol))
                                        : make_uint2(0u, 0u);
    }
    return pr;
  }
  __device__ __forceinline__ void store(const Pre& pr, int i, int grow, int gcol, float4 g) const {
    const float f0 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(pr.w[i].x & 0xFFFFu), pr.sw.x)), dge);
    const float f1 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(pr.w[i].x >> 16), pr.sw.y)), dge);
    const float f2 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(pr.w[i].y & 0xFFFFu), pr.sw.z)), dge);
    const float f3 = dge_factor(fabsf(__fmul_rn(bf16_bits_to_float(pr.w[i].y >> 16), pr.sw.w)), dge);
    const float4 d = make_float4(g.x * f0, g.y * f1, g.z * f2, g.w * f3);
    if constexpr (FP8) {
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(d.x), fabsf(d.y)), fmaxf(fabsf(d.z), fabsf(d.w))));
      const float sc = __ldg(scale);
      const uint32_t q = e4m3x2(__fmul_rn(d.x, sc), __fmul_rn(d.y, sc)) |
                         (e4m3x2(__fmul_rn(d.z, sc), __fmul_rn(d.w, sc)) << 16);
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(dW) + int64_t(grow) * lddw + gcol) = q;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(dW) + int64_t(grow) * lddw + gcol) = d;
    }
  }

  // every thread of the block, after the engine: one atomic per warp
  __device__ __forceinline__ void finish() const {
    if constexpr (FP8) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax));   // amax >= 0: order of bits
      if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(reinterpret_cast<unsigned int*>(amax_out), m);
    }
  }
};

template <bool PAIR, bool FP8>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    wgrad_dge_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                     const bwd::Shape s, const DgeEpilogue<FP8> e) {
  if constexpr (FP8) {
    DgeEpilogue<FP8> el = e;   // a per-thread copy carries the running max
    el.amax = 0.0f;
    bwd::run<false, PAIR>(tmA, tmG, s, el);
    el.finish();
  } else {
    bwd::run<false, PAIR>(tmA, tmG, s, e);
  }
}

}  // namespace
}  // namespace fp4

FP4_API fp4_status fp4_linear_wgrad_dge(const void* A, int64_t lda, const void* dY, int64_t lddy, const void* W,
                                        int64_t ldw, const float* s_w, int64_t M, int64_t N, int64_t K, float dge_k,
                                        float dge_clip, void* dW, int dw_type, int64_t lddw, const float* dw_scale,
                                        float* dw_amax, void* workspace, size_t ws_bytes, fp4_stream_t stream) {
  using namespace fp4;
  if (!A || !dY || !W || !s_w || !dW) return FP4_ERR_INVALID_ARG;
  if (!(dge_k > 0.0f) || !(dge_clip > 0.0f) || !isfinite(dge_k)) return FP4_ERR_INVALID_ARG;
  if (dw_type != FP4_DW_FP32 && dw_type != FP4_DW_E4M3) return FP4_ERR_INVALID_ARG;
  const bool fp8 = dw_type == FP4_DW_E4M3;
  if (fp8 && (!dw_scale || !dw_amax)) return FP4_ERR_INVALID_ARG;
  if (fp8 && ((reinterpret_cast<uintptr_t>(dw_scale) & 3u) || (reinterpret_cast<uintptr_t>(dw_amax) & 3u)))
    return FP4_ERR_ALIGNMENT;
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
  st = encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, uint64_t(K), uint64_t(M), uint64_t(lda) * 2,
                      bwd::kBox, bwd::kBT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  st = encode_tmap_2d(&tmG, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, uint64_t(N), uint64_t(M), uint64_t(lddy) * 2,
                      bwd::kBox, bwd::kBT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  if (fp8) {
    // the running maximum must not land in dW (it is zeroed before the launch)
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dW), d1 = d0 + uintptr_t((K - 1) * lddw + N);
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(dw_amax);
    if (a0 + sizeof(float) > d0 && a0 < d1) return FP4_ERR_INVALID_ARG;
  }
  DgeEpilogue<false> e;
  e.W = static_cast<const uint16_t*>(W);
  e.ldw = ldw;
  e.s_w = s_w;
  e.dW = dW;
  e.lddw = lddw;
  e.rows = int(K);
  e.cols = int(N);
  e.dge.inv_k = 1.0f / dge_k;
  e.dge.expo = 1.0f / dge_k - 1.0f;
  e.dge.log2_inv_k = std::log2(1.0f / dge_k);
  e.dge.clip = dge_clip;
  // lim_{u -> 0} |u|^expo: +inf for expo < 0 (clipped), 1 for expo = 0, 0 for expo > 0
  const float lim = e.dge.expo < 0.0f ? INFINITY : (e.dge.expo == 0.0f ? 1.0f : 0.0f);
  e.dge.f_mid = std::fmin(dge_clip, e.dge.inv_k * lim);
  bwd::Shape s;
  s.R = int(K);
  s.C = int(N);
  s.L = int(M);
  s.q_wrap = 0;
  s.status = status_word();
  s.wait_ns = kWaitLimitNs;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  st = bwd::schedule(s, bwd::plan_split(K, N, M, sms), workspace, ws_bytes, cs);
  if (st != FP4_OK) return st;
  const bool pairs = bwd::use_pairs(M);
  if (!fp8) {
    e.scale = nullptr;
    e.amax_out = nullptr;
    e.amax = 0.0f;
    if (pairs) return bwd::launch<false, true>(wgrad_dge_kernel<true, false>, s, sms, cs, tmA, tmG, s, e);
    return bwd::launch<false, false>(wgrad_dge_kernel<false, false>, s, sms, cs, tmA, tmG, s, e);
  }
  DgeEpilogue<true> e8;
  e8.W = e.W;
  e8.ldw = e.ldw;
  e8.s_w = e.s_w;
  e8.dW = e.dW;
  e8.lddw = e.lddw;
  e8.rows = e.rows;
  e8.cols = e.cols;
  e8.dge = e.dge;
  e8.scale = dw_scale;
  e8.amax_out = dw_amax;
  e8.amax = 0.0f;
  if (cudaMemsetAsync(dw_amax, 0, sizeof(float), cs) != cudaSuccess) return launch_status();
  if (pairs) return bwd::launch<false, true>(wgrad_dge_kernel<true, true>, s, sms, cs, tmA, tmG, s, e8);
  return bwd::launch<false, false>(wgrad_dge_kernel<false, true>, s, sms, cs, tmA, tmG, s, e8);
}

FP4_API size_t fp4_linear_wgrad_dge_workspace(int64_t M, int64_t N, int64_t K) {
  using namespace fp4;
  int sms = 0;
  if (M < 1 || N < 1 || K < 1 || check_device(&sms) != FP4_OK) return 0;
  return bwd::plan_split(K, N, M, sms).total;
}
