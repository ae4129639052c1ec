// Input gradient of the linear layer, dX = dY W^T, on sm_103a tensor cores.
//
// The pages give the forward pass and the DGE-corrected weight gradient but not
// the input gradient.  The plainest reading that closes the linear's backward
// is the chain rule of Y = A W through the same BF16 tensor-core engine as the
// weight gradient: dX[m, k] = sum_n dY[m, n] W[k, n], with the BF16 W the
// caller passes (the unquantized weight, as the compensation term uses), fp32
// accumulation, and dX in BF16 (round to nearest even) or fp32.
//
// Both operands keep the reduction dimension (the N outputs) contiguous, so
// the engine (bwd_gemm.cuh) reads them K-major: dY rows are the tile's 128
// (or 256 per CTA pair) output rows, W rows its 256 output columns.  The
// epilogue only converts and stores.
#include "bwd_gemm.cuh"

namespace fp4 {
namespace {

struct StoreEpilogue {
  void* out;
  int64_t ld;   // elements
  bool bf16;

  __device__ __forceinline__ void prefetch(int, int, int) const {}
  struct Pre {};
  __device__ __forceinline__ Pre load(int, int, bool, int) const { return Pre{}; }
  __device__ __forceinline__ void store(const Pre&, int, int grow, int gcol, float4 g) const {
    const int64_t off = int64_t(grow) * ld + gcol;
    if (bf16) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(g.x, g.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(g.z, g.w);
      uint2 v;
      v.x = *reinterpret_cast<const uint32_t*>(&lo);
      v.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + off) = v;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = g;
    }
  }
};

template <bool PAIR>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    dgrad_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmW,
                 const bwd::Shape s, const StoreEpilogue e) {
  bwd::run<true, PAIR>(tmG, tmW, s, e);
}

}  // namespace
}  // namespace fp4

FP4_API fp4_status fp4_linear_dgrad(const void* dY, int64_t lddy, const void* W, int64_t ldw, int64_t M, int64_t N,
                                    int64_t K, void* dX, int dx_type, int64_t lddx, void* workspace, size_t ws_bytes,
                                    fp4_stream_t stream) {
  using namespace fp4;
  if (!dY || !W || !dX) return FP4_ERR_INVALID_ARG;
  if (dx_type != FP4_OUT_BF16 && dx_type != FP4_OUT_FP32) return FP4_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || K < 8 || N % 8 || K % 8 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31))
    return FP4_ERR_SHAPE;
  if (lddy < N || ldw < N || lddx < K) return FP4_ERR_SHAPE;
  if (lddy % 8 || ldw % 8 || lddx % 8 || !aligned16(dY) || !aligned16(W) || !aligned16(dX)) return FP4_ERR_ALIGNMENT;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  CUtensorMap tmG, tmW;
  st = encode_tmap_2d(&tmG, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, uint64_t(N), uint64_t(M), uint64_t(lddy) * 2,
                      bwd::kBT, bwd::kBox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  st = encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, uint64_t(N), uint64_t(K), uint64_t(ldw) * 2,
                      bwd::kBT, bwd::kBox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FP4_OK) return st;
  StoreEpilogue e;
  e.out = dX;
  e.ld = lddx;
  e.bf16 = (dx_type == FP4_OUT_BF16);
  bwd::Shape s;
  s.R = int(M);
  s.C = int(K);
  s.L = int(N);
  s.q_wrap = 0;
  s.status = status_word();
  s.wait_ns = kWaitLimitNs;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  st = bwd::schedule(s, bwd::plan_split(M, K, N, sms), workspace, ws_bytes, cs);
  if (st != FP4_OK) return st;
  if (bwd::use_pairs(N)) return bwd::launch<true, true>(dgrad_kernel<true>, s, sms, cs, tmG, tmW, s, e);
  return bwd::launch<true, false>(dgrad_kernel<false>, s, sms, cs, tmG, tmW, s, e);
}

FP4_API size_t fp4_linear_dgrad_workspace(int64_t M, int64_t N, int64_t K) {
  using namespace fp4;
  int sms = 0;
  if (M < 1 || N < 1 || K < 1 || check_device(&sms) != FP4_OK) return 0;
  return bwd::plan_split(M, K, N, sms).total;
}
