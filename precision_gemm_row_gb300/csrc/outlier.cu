// Quantile outlier clamp and sparse compensation matrix, per the outlier
// passage of the page "首个 FP4 精度的大模型训练框架来了" (czzqal.com): a quantile
// search finds the largest-magnitude outliers of A, they are clamped to the
// threshold (A_clamped), and dA = A - A_clamped is kept as a sparse matrix that
// is nonzero only where clamping happened.
//
// Kernels (all HBM-bound, no spin-waits):
//  1. histogram_select: one 32768-bin histogram of the 15-bit BF16 magnitude
//     pattern per CTA in shared memory, merged into a global histogram; the
//     last CTA to finish (atomic ticket) scans it for the exact k-th order
//     statistic t.
//  2. stage: one warp per row counts |A| > t, reserves space in a staging area
//     with one atomic per row and writes (column, A - sign(A) t) in column
//     order; optionally writes A_clamped.
//  3. row_scan: exclusive scan of the per-row counts -> row_ptr (one CTA).
//  4. gather: copies every row's staged entries to its CSR position.
#include <cmath>

#include "common.cuh"

namespace fp4 {
namespace {

constexpr int kBins = 32768;
constexpr int kHistThreads = 1024;

struct Ctrl {
  uint32_t done;          // CTAs finished with the histogram
  uint32_t t_bits;        // 15-bit magnitude pattern of t
  unsigned long long cursor;     // next free staging slot
  unsigned long long nnz_expect; // number of |A| > t from the histogram
};

struct WsLayout {
  size_t hist, ctrl, cnt, start, scol, sval, total;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

WsLayout ws_layout(int64_t M, int64_t cap) {
  WsLayout L;
  size_t off = 0;
  L.hist = off; off += round256(size_t(kBins) * 4);
  L.ctrl = off; off += round256(sizeof(Ctrl));
  L.cnt = off; off += round256(size_t(M) * 4);
  L.start = off; off += round256(size_t(M) * 8);
  L.scol = off; off += round256(size_t(cap) * 4);
  L.sval = off; off += round256(size_t(cap) * 4);
  L.total = off;
  return L;
}

__global__ void __launch_bounds__(kHistThreads, 1)
    histogram_select_kernel(const uint16_t* __restrict__ A, int64_t M, int K, int64_t lda, int64_t k_rank,
                            uint32_t* __restrict__ ghist, Ctrl* __restrict__ ctrl, float* __restrict__ t_out) {
  extern __shared__ uint32_t hist[];  // kBins counters
  __shared__ uint32_t part[kHistThreads];
  __shared__ int is_last;
  for (int b = threadIdx.x; b < kBins; b += kHistThreads) hist[b] = 0;
  __syncthreads();

  const int cpr = K >> 3;  // 16-byte chunks per row
  const int64_t total = M * cpr;
  const bool dense = (lda == K);
  for (int64_t g = int64_t(blockIdx.x) * kHistThreads + threadIdx.x; g < total;
       g += int64_t(gridDim.x) * kHistThreads) {
    const uint4* p;
    if (dense) {
      p = reinterpret_cast<const uint4*>(A) + g;
    } else {
      const int64_t r = g / cpr;
      p = reinterpret_cast<const uint4*>(A + r * lda) + (g - r * cpr);
    }
    const uint4 v = __ldcs(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      atomicAdd(&hist[w[i] & 0x7FFFu], 1u);
      atomicAdd(&hist[(w[i] >> 16) & 0x7FFFu], 1u);
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kBins; b += kHistThreads) {
    const uint32_t c = hist[b];
    if (c) atomicAdd(ghist + b, c);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(&ctrl->done, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Exact order statistic: the smallest bin b with cumulative count >= k_rank.
  constexpr int kPer = kBins / kHistThreads;  // 32 bins per thread
  const int b0 = threadIdx.x * kPer;
  uint32_t local[kPer];
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    local[i] = __ldcg(ghist + b0 + i);
    sum += local[i];
  }
  part[threadIdx.x] = sum;
  __syncthreads();
  // inclusive scan over the 1024 partial sums (Hillis-Steele in shared memory, 64-bit safe via two halves)
  for (int off = 1; off < kHistThreads; off <<= 1) {
    const uint32_t add = threadIdx.x >= off ? part[threadIdx.x - off] : 0u;
    __syncthreads();
    part[threadIdx.x] += add;
    __syncthreads();
  }
  const uint64_t incl = part[threadIdx.x];
  const uint64_t excl = incl - sum;
  if (excl < uint64_t(k_rank) && uint64_t(k_rank) <= incl) {
    uint64_t run = excl;
    int sel = b0 + kPer - 1;
    for (int i = 0; i < kPer; ++i) {
      run += local[i];
      if (run >= uint64_t(k_rank)) {
        sel = b0 + i;
        break;
      }
    }
    const uint64_t n = uint64_t(M) * uint64_t(K);
    ctrl->t_bits = uint32_t(sel);
    ctrl->nnz_expect = n - run;
    *t_out = bf16_bits_to_float(uint32_t(sel));
  }
}

// One warp per row: count entries with magnitude pattern > t_bits, reserve a
// contiguous run in the staging area, then write them in column order.
__global__ void __launch_bounds__(256) stage_kernel(const uint16_t* __restrict__ A, int64_t M, int K, int64_t lda,
                                                   Ctrl* ctrl,
                                                   const float* __restrict__ t_ptr, int64_t cap,
                                                   int32_t* __restrict__ row_cnt, int64_t* __restrict__ row_start,
                                                   int32_t* __restrict__ scol, float* __restrict__ sval,
                                                   uint16_t* __restrict__ A_c, int64_t ldac,
                                                   uint32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const uint32_t tb = ctrl->t_bits;
  const float t = *t_ptr;
  const int cpr = K >> 3;
  for (int64_t row = warp_global; row < M; row += nwarps) {
    const uint4* src = reinterpret_cast<const uint4*>(A + row * lda);
    uint32_t cnt = 0;
    for (int c = lane; c < cpr; c += 32) {
      const uint4 v = __ldg(src + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t cw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
        const bool olo = (lo & 0x7FFFu) > tb, ohi = (hi & 0x7FFFu) > tb;
        cnt += uint32_t(olo) + uint32_t(ohi);
        cw[i] = (olo ? ((lo & 0x8000u) | tb) : lo) | ((ohi ? ((hi & 0x8000u) | tb) : hi) << 16);
      }
      if (A_c) reinterpret_cast<uint4*>(A_c + row * ldac)[c] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    unsigned long long base = 0;
    if (cnt && lane == 0) base = atomicAdd(&ctrl->cursor, (unsigned long long)cnt);
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (lane == 0) {
      row_cnt[row] = int32_t(cnt);
      row_start[row] = int64_t(base);
    }
    if (cnt == 0) continue;
    if (int64_t(base + cnt) > cap) {
      if (lane == 0) atomicOr(status, FP4_FLAG_CAPACITY);
      continue;
    }
    // second pass (row is L1/L2 resident): write entries in column order
    unsigned long long run = base;
    for (int c0 = 0; c0 < cpr; c0 += 32) {
      const int c = c0 + lane;
      uint32_t mask = 0;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (c < cpr) {
        v = __ldg(src + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mask |= uint32_t((w[i] & 0x7FFFu) > tb) << (2 * i);
          mask |= uint32_t(((w[i] >> 16) & 0x7FFFu) > tb) << (2 * i + 1);
        }
      }
      const uint32_t n = __popc(mask);
      uint32_t incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
      if (n) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        unsigned long long pos = run + (incl - n);
        for (int e = 0; e < 8; ++e) {
          if (mask & (1u << e)) {
            const float x = bf16_bits_to_float((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
            scol[pos] = c * 8 + e;
            sval[pos] = __fsub_rn(x, copysignf(t, x));
            ++pos;
          }
        }
      }
      run += total;
    }
  }
}

// row_ptr[0] = 0, row_ptr[i+1] = sum of counts of rows <= i; checks the total
// against the histogram's count.
__global__ void __launch_bounds__(1024) row_scan_kernel(const int32_t* __restrict__ row_cnt, int64_t M,
                                                       int32_t* __restrict__ row_ptr, int64_t* __restrict__ nnz_out,
                                                       const Ctrl* __restrict__ ctrl, int64_t cap,
                                                       uint32_t* __restrict__ status) {
  __shared__ long long part[1024];
  const int64_t per = (M + 1023) / 1024;
  const int64_t r0 = int64_t(threadIdx.x) * per;
  const int64_t r1 = r0 + per < M ? r0 + per : M;
  long long s = 0;
  for (int64_t r = r0; r < r1; ++r) s += row_cnt[r];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const long long add = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += add;
    __syncthreads();
  }
  long long run = part[threadIdx.x] - s;
  if (threadIdx.x == 0) row_ptr[0] = 0;
  for (int64_t r = r0; r < r1; ++r) {
    run += row_cnt[r];
    row_ptr[r + 1] = int32_t(run);
  }
  if (threadIdx.x == 1023) {
    const long long total = part[1023];
    if (nnz_out) *nnz_out = total;
    if (uint64_t(total) != ctrl->nnz_expect && total <= cap) atomicOr(status, FP4_FLAG_INTERNAL);
  }
}

__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ row_cnt,
                                                    const int64_t* __restrict__ row_start,
                                                    const int32_t* __restrict__ row_ptr, int64_t M,
                                                    const int32_t* __restrict__ scol, const float* __restrict__ sval,
                                                    int32_t* __restrict__ col_idx, float* __restrict__ vals,
                                                    int64_t cap) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = warp_global; row < M; row += nwarps) {
    const int32_t n = row_cnt[row];
    const int64_t src = row_start[row];
    const int64_t dst = row_ptr[row];
    if (src + n > cap || dst + n > cap) continue;
    for (int e = lane; e < n; e += 32) {
      col_idx[dst + e] = scol[src + e];
      vals[dst + e] = sval[src + e];
    }
  }
}

}  // namespace
}  // namespace fp4

FP4_API int64_t outlier_max_nnz(int64_t M, int64_t K, double q) {
  if (M <= 0 || K <= 0 || !(q > 0.0) || !(q <= 1.0)) return 0;
  const int64_t n = M * K;
  double kd = std::ceil(q * double(n));
  int64_t k = kd < 1.0 ? 1 : (kd > double(n) ? n : int64_t(kd));
  return n - k;
}

FP4_API size_t outlier_clamp_quantile_workspace(int64_t M, int64_t K, int64_t nnz_capacity) {
  if (M <= 0 || K <= 0 || nnz_capacity < 0) return 0;
  return fp4::ws_layout(M, nnz_capacity).total;
}

FP4_API fp4_status outlier_clamp_quantile(const void* A, int64_t M, int64_t K, int64_t lda, double q, float* t_out,
                                          int32_t* row_ptr, int32_t* col_idx, float* vals, int64_t nnz_capacity,
                                          int64_t* nnz_out, void* A_clamped, int64_t ldac, void* workspace,
                                          size_t ws_bytes, fp4_stream_t stream) {
  using namespace fp4;
  if (!A || !t_out || !row_ptr || !workspace) return FP4_ERR_INVALID_ARG;
  if (!(q > 0.0) || !(q <= 1.0)) return FP4_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0 || K % 8 != 0 || lda < K || K > (1 << 30) || M >= (int64_t(1) << 31) ||
      M * K >= (int64_t(1) << 32))
    return FP4_ERR_SHAPE;
  if (A_clamped && ldac < K) return FP4_ERR_SHAPE;
  if (lda % 8 != 0 || !aligned16(A) || !aligned16(workspace) || (A_clamped && (!aligned16(A_clamped) || ldac % 8)))
    return FP4_ERR_ALIGNMENT;
  const int64_t need = outlier_max_nnz(M, K, q);
  if (nnz_capacity < need || nnz_capacity >= (int64_t(1) << 31)) return FP4_ERR_CAPACITY;
  if (nnz_capacity > 0 && (!col_idx || !vals)) return FP4_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(M, nnz_capacity);
  if (ws_bytes < L.total) return FP4_ERR_WORKSPACE;
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  auto* ws = static_cast<uint8_t*>(workspace);
  auto* ghist = reinterpret_cast<uint32_t*>(ws + L.hist);
  auto* ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  auto* row_cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  auto* row_start = reinterpret_cast<int64_t*>(ws + L.start);
  auto* scol = reinterpret_cast<int32_t*>(ws + L.scol);
  auto* sval = reinterpret_cast<float*>(ws + L.sval);
  uint32_t* status = status_word();

  const int64_t n = M * K;
  const int64_t k_rank = n - need;
  if (cudaMemsetAsync(ws, 0, L.cnt, s) != cudaSuccess) return FP4_ERR_CUDA;  // histogram + control block

  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t hist_smem = size_t(kBins) * 4;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(histogram_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(hist_smem)) !=
        cudaSuccess)
      return FP4_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t chunks = n / 8;
  int64_t hblocks = (chunks + kHistThreads * 4 - 1) / (kHistThreads * 4);
  if (hblocks > sms) hblocks = sms;
  if (hblocks < 1) hblocks = 1;
  histogram_select_kernel<<<unsigned(hblocks), kHistThreads, hist_smem, s>>>(
      static_cast<const uint16_t*>(A), M, int(K), lda, k_rank, ghist, ctrl, t_out);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;

  int64_t sblocks = (M + 7) / 8;
  if (sblocks > int64_t(sms) * 8) sblocks = int64_t(sms) * 8;
  stage_kernel<<<unsigned(sblocks), 256, 0, s>>>(static_cast<const uint16_t*>(A), M, int(K), lda, ctrl, t_out,
                                                  nnz_capacity, row_cnt, row_start, scol, sval,
                                                  static_cast<uint16_t*>(A_clamped), ldac, status);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  row_scan_kernel<<<1, 1024, 0, s>>>(row_cnt, M, row_ptr, nnz_out, ctrl, nnz_capacity, status);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  if (nnz_capacity > 0) {
    gather_kernel<<<unsigned(sblocks), 256, 0, s>>>(row_cnt, row_start, row_ptr, M, scol, sval, col_idx, vals,
                                                    nnz_capacity);
    if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  }
  return FP4_OK;
}
