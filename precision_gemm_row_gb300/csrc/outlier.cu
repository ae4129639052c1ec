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
//  2. rows_outlier: one row per warp (or several warps for long rows), held in
//     registers: counts |A| > t per 16-byte chunk and writes the row's count
//     and its first kRowSlots entries (column, A - sign(A) t), in column order,
//     into fixed per-row slots (no atomics); optionally writes A_clamped, and
//     in the fused variant also the row's E2M1 codes and scale (the clamp
//     applied), so A is read once here.
//  3. row_scan: scan of the per-row counts -> row_ptr (one CTA, coalesced tiles).
//  4. gather: copies every row's slots to its CSR position; a row with more
//     than kRowSlots entries is read again from A and emitted in full.
#include <cmath>

#include "common.cuh"

namespace fp4 {
namespace {

constexpr int kBins = 32768;
constexpr int kHistThreads = 1024;

constexpr int kRowSlots = 16;  // entries per row kept by the row pass (more are re-read from A)

struct Ctrl {
  uint32_t done;          // CTAs finished with the histogram
  uint32_t t_bits;        // 15-bit magnitude pattern of t
  unsigned long long nnz_expect; // number of |A| > t from the histogram
};

struct WsLayout {
  size_t hist, ctrl, cnt, scol, sval, total;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

WsLayout ws_layout(int64_t M) {
  WsLayout L;
  size_t off = 0;
  L.hist = off; off += round256(size_t(kBins) * 4);
  L.ctrl = off; off += round256(sizeof(Ctrl));
  L.cnt = off; off += round256(size_t(M) * 4);
  L.scol = off; off += round256(size_t(M) * kRowSlots * 4);
  L.sval = off; off += round256(size_t(M) * kRowSlots * 4);
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
  const int64_t stride = int64_t(gridDim.x) * kHistThreads;
  constexpr int kU = 8;  // loads in flight per thread
  for (int64_t g0 = int64_t(blockIdx.x) * kHistThreads + threadIdx.x; g0 < total; g0 += stride * kU) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t g = g0 + u * stride;
      if (g < total) {
        const uint4* p;
        if (dense) {
          p = reinterpret_cast<const uint4*>(A) + g;
        } else {
          const int64_t r = g / cpr;
          p = reinterpret_cast<const uint4*>(A + r * lda) + (g - r * cpr);
        }
        v[u] = __ldcs(p);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (g0 + u * stride < total) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          atomicAdd(&hist[w[i] & 0x7FFFu], 1u);
          atomicAdd(&hist[(w[i] >> 16) & 0x7FFFu], 1u);
        }
      }
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
  // The merged histogram comes into this CTA's shared memory with coalesced
  // 16-byte loads; thread t then owns bins 32 t .. 32 t + 31 (summed in a
  // lane-skewed order, so a warp's 32 reads fall in 32 different banks).
  constexpr int kPer = kBins / kHistThreads;  // 32 bins per thread
#pragma unroll
  for (int j = 0; j < kBins / 4 / kHistThreads; ++j) {
    const int i4 = threadIdx.x + j * kHistThreads;
    reinterpret_cast<uint4*>(hist)[i4] = __ldcg(reinterpret_cast<const uint4*>(ghist) + i4);
  }
  __syncthreads();
  const int b0 = threadIdx.x * kPer;
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) sum += hist[b0 + ((i + threadIdx.x) & (kPer - 1))];
  // inclusive scan of the 1024 partial sums: within each warp by shuffles, then
  // over the 32 warp totals (counts fit 32 bits: n < 2^32)
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) part[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t wv = part[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, wv, o);
      if (lane >= o) wv += y;
    }
    part[lane] = wv;
  }
  __syncthreads();
  const uint64_t incl = uint64_t(x) + (wid ? part[wid - 1] : 0u);
  const uint64_t excl = incl - sum;
  if (excl < uint64_t(k_rank) && uint64_t(k_rank) <= incl) {
    uint64_t run = excl;
    int sel = b0 + kPer - 1;
    for (int i = 0; i < kPer; ++i) {
      run += hist[b0 + i];
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

constexpr int kMaxRowWarps = 16;   // warps per CTA of the row pass

// 8-bit mask of the elements of a 16-byte BF16 chunk whose magnitude pattern exceeds tb.
__device__ __forceinline__ uint32_t outlier_mask8(const uint4 v, uint32_t tb) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m |= uint32_t((w[i] & 0x7FFFu) > tb) << (2 * i);
    m |= uint32_t(((w[i] >> 16) & 0x7FFFu) > tb) << (2 * i + 1);
  }
  return m;
}

// Each row is handled by `wpr` warps; lane l of warp w holds the row's 16-byte
// chunks ci = l + 32 (w + wpr c), c < CH, in registers.  Column order of the
// entries is chunk-slot c first, then warp, then lane, which is what the
// offsets below follow.  A CTA holds blockDim.x / 32 / wpr rows.
template <int CH, bool CODES>
__global__ void __launch_bounds__(512, 1) rows_outlier_kernel(
    const uint16_t* __restrict__ A, int64_t M, int K, int64_t lda, Ctrl* ctrl, const float* __restrict__ t_ptr,
    int32_t* __restrict__ row_cnt, int32_t* __restrict__ scol, float* __restrict__ sval, uint16_t* __restrict__ A_c,
    int64_t ldac, uint8_t* __restrict__ codes, int64_t ldc, float* __restrict__ scales, int wpr) {
  __shared__ uint32_t red[kMaxRowWarps];
  __shared__ uint32_t tcnt[kMaxRowWarps][CH];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_cta = int(blockDim.x >> 5) / wpr;
  const int r_in_cta = warp / wpr, w_in_row = warp % wpr;
  const int wrow0 = r_in_cta * wpr;  // first warp of this row
  const int nchunk = K >> 3;
  const uint32_t tb = ctrl->t_bits;
  const uint32_t tb2 = tb | (tb << 16);
  const float t = *t_ptr;
  // persistent over row groups; the next group's chunks are loaded before the
  // current group is processed, so every warp keeps one row's loads in flight
  const int64_t gstride = int64_t(gridDim.x) * rows_per_cta;
  uint4 v[CH];
  {
    const int64_t row = int64_t(blockIdx.x) * rows_per_cta + r_in_cta;
    const uint4* src = reinterpret_cast<const uint4*>(A + (row < M ? row : 0) * lda);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int ci = lane + 32 * (w_in_row + wpr * c);
      v[c] = (row < M && ci < nchunk) ? __ldcs(src + ci) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  for (int64_t row0 = int64_t(blockIdx.x) * rows_per_cta; row0 < M; row0 += gstride) {
    const int64_t row = row0 + r_in_cta;
    const bool active = row < M;
    uint4 vn[CH];
    {
      const int64_t nrow = row + gstride;
      const uint4* nsrc = reinterpret_cast<const uint4*>(A + (nrow < M ? nrow : 0) * lda);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int ci = lane + 32 * (w_in_row + wpr * c);
        vn[c] = (nrow < M && ci < nchunk) ? __ldcs(nsrc + ci) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    uint32_t msk[CH], excl[CH];
    uint32_t mx = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      // one packed maximum per chunk serves the row's absmax and the outlier test
      const uint32_t m2 = chunk_maxmag(v[c]);
      if (CODES) mx = bf2_max(mx, m2);
      const uint32_t g = bf2_gt_mask(m2, tb2);
      msk[c] = 0;
      excl[c] = 0;
      uint32_t tot = 0;
      if (__any_sync(0xFFFFFFFFu, g != 0)) {  // rare: some lane has an outlier in this slot
        msk[c] = g ? outlier_mask8(v[c], tb) : 0u;
        const uint32_t n = __popc(msk[c]);
        uint32_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        excl[c] = incl - n;
      }
      if (lane == 0) tcnt[warp][c] = tot;
    }
    if (CODES) {
      const uint32_t mb = warp_max_bits(mx);
      if (lane == 0) red[warp] = mb;
    }
    __syncthreads();
    if (active && w_in_row == 0 && lane == 0) {
      uint32_t total = 0;
      for (int c = 0; c < CH; ++c)
        for (int w = 0; w < wpr; ++w) total += tcnt[wrow0 + w][c];
      row_cnt[row] = int32_t(total);
    }
    if (active) {
      // the row's first kRowSlots entries go to its slots; a longer row is
      // emitted again from A by the gather pass
      uint32_t off = 0;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        uint32_t pos = off + excl[c];
        for (int w = 0; w < w_in_row; ++w) pos += tcnt[wrow0 + w][c];
        uint32_t m = msk[c];
        if (m && pos < uint32_t(kRowSlots)) {
          const int ci = lane + 32 * (w_in_row + wpr * c);
          const uint4 vc = v[c];
          while (m && pos < uint32_t(kRowSlots)) {  // set bits in ascending column order
            const int e = __ffs(m) - 1;
            m &= m - 1;
            const uint32_t word = e < 4 ? (e < 2 ? vc.x : vc.y) : (e < 6 ? vc.z : vc.w);
            const float x = bf16_bits_to_float((word >> (16 * (e & 1))) & 0xFFFFu);
            scol[row * kRowSlots + pos] = ci * 8 + e;
            sval[row * kRowSlots + pos] = __fsub_rn(x, copysignf(t, x));
            ++pos;
          }
        }
        for (int w = 0; w < wpr; ++w) off += tcnt[wrow0 + w][c];
      }
    }
    if (active && A_c) {
      uint4* dst = reinterpret_cast<uint4*>(A_c + row * ldac);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int ci = lane + 32 * (w_in_row + wpr * c);
        if (ci < nchunk) {
          const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
          uint32_t cw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
            cw[i] = (((lo & 0x7FFFu) > tb) ? ((lo & 0x8000u) | tb) : lo) |
                    ((((hi & 0x7FFFu) > tb) ? ((hi & 0x8000u) | tb) : hi) << 16);
          }
          dst[ci] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        }
      }
    }
    if (CODES) {
      uint32_t amax_bits = 0;
      for (int i = 0; i < wpr; ++i) amax_bits = max(amax_bits, red[wrow0 + i]);
      // max over min(|x|, t) = min(max |x|, t)
      const float sc = scale_from_absmax(bf16_bits_to_float(min(amax_bits, tb)));
      if (active) {
        if (w_in_row == 0 && lane == 0) scales[row] = sc;
        uint32_t* dst = reinterpret_cast<uint32_t*>(codes + row * ldc);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int ci = lane + 32 * (w_in_row + wpr * c);
          if (ci < nchunk) dst[ci] = quantize8<true>(v[c], sc, tb2);   // the clamp is a no-op without outliers
        }
      }
    }
    __syncthreads();  // tcnt / red are reused by the next row group
#pragma unroll
    for (int c = 0; c < CH; ++c) v[c] = vn[c];
  }
}

// row_ptr[0] = 0, row_ptr[i+1] = sum of counts of rows <= i, in tiles of 4096
// rows (coalesced loads); checks the total against the histogram's count.
__global__ void __launch_bounds__(1024) row_scan_kernel(const int32_t* __restrict__ row_cnt, int64_t M,
                                                       int32_t* __restrict__ row_ptr, int64_t* __restrict__ nnz_out,
                                                       const Ctrl* __restrict__ ctrl, int64_t cap,
                                                       uint32_t* __restrict__ status) {
  __shared__ long long wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long carry = 0;
  if (tid == 0) row_ptr[0] = 0;
  for (int64_t base = 0; base < M; base += 4096) {
    const int64_t idx = base + 4 * tid;
    int c[4];
    if (idx + 3 < M) {
      const int4 q = *reinterpret_cast<const int4*>(row_cnt + idx);
      c[0] = q.x; c[1] = q.y; c[2] = q.z; c[3] = q.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = (idx + i < M) ? row_cnt[idx + i] : 0;
    }
    const long long s0 = c[0], s1 = s0 + c[1], s2 = s1 + c[2], s3 = s2 + c[3];
    long long x = s3;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      long long w = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      wsum[lane] = w;
    }
    __syncthreads();
    const long long excl = carry + (warp ? wsum[warp - 1] : 0) + x - s3;
    const long long incl4[4] = {s0, s1, s2, s3};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (idx + i < M) row_ptr[idx + i + 1] = int32_t(excl + incl4[i]);
    carry += wsum[31];
    __syncthreads();
  }
  if (tid == 0) {
    if (nnz_out) *nnz_out = carry;
    if (carry > cap) atomicOr(status, FP4_FLAG_CAPACITY);
    else if (uint64_t(carry) != ctrl->nnz_expect) atomicOr(status, FP4_FLAG_INTERNAL);
  }
}

// One warp per row: the row's slots to its CSR position, or, for a row with
// more than kRowSlots entries, the row read again from A and emitted in column
// order (a warp prefix over the lanes' 16-byte chunks).
__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ row_cnt,
                                                    const int32_t* __restrict__ row_ptr, int64_t M,
                                                    const int32_t* __restrict__ scol, const float* __restrict__ sval,
                                                    const uint16_t* __restrict__ A, int K, int64_t lda,
                                                    const Ctrl* __restrict__ ctrl, const float* __restrict__ t_ptr,
                                                    int32_t* __restrict__ col_idx, float* __restrict__ vals,
                                                    int64_t cap) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const uint32_t tb = ctrl->t_bits;
  const float t = *t_ptr;
  const int nchunk = K >> 3;
  for (int64_t row = warp_global; row < M; row += nwarps) {
    const int32_t n = row_cnt[row];
    const int64_t dst = row_ptr[row];
    if (dst + n > cap) continue;   // flagged by the scan
    if (n <= kRowSlots) {
      if (lane < n) {
        col_idx[dst + lane] = scol[row * kRowSlots + lane];
        vals[dst + lane] = sval[row * kRowSlots + lane];
      }
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(A + row * lda);
    int64_t base = dst;
    constexpr int kDepth = 4;   // 32-chunk groups loaded before any is scanned
    for (int c00 = 0; c00 < nchunk; c00 += 32 * kDepth) {
      uint4 vv[kDepth];
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int ci = c00 + 32 * u + lane;
        vv[u] = ci < nchunk ? __ldg(src + ci) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int ci = c00 + 32 * u + lane;
        const uint4 v = vv[u];
        uint32_t m = ci < nchunk ? outlier_mask8(v, tb) : 0u;
        const uint32_t cnt = __popc(m);
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        int64_t pos = base + (incl - cnt);
        while (m) {
          const int e = __ffs(m) - 1;
          m &= m - 1;
          const uint32_t word = e < 4 ? (e < 2 ? v.x : v.y) : (e < 6 ? v.z : v.w);
          const float x = bf16_bits_to_float((word >> (16 * (e & 1))) & 0xFFFFu);
          col_idx[pos] = ci * 8 + e;
          vals[pos] = __fsub_rn(x, copysignf(t, x));
          ++pos;
        }
        base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
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
  return fp4::ws_layout(M).total;
}

namespace fp4 {
namespace {

template <bool CODES>
void launch_rows_outlier(int ch, int wpr, unsigned blocks, unsigned threads, cudaStream_t s, const uint16_t* A,
                         int64_t M, int K, int64_t lda, Ctrl* ctrl, const float* t, int32_t* row_cnt,
                         int32_t* scol, float* sval, uint16_t* A_c, int64_t ldac, uint8_t* codes, int64_t ldc,
                         float* scales) {
#define FP4_ROWS_OUTLIER(CHV)                                                                                     \
  rows_outlier_kernel<CHV, CODES><<<blocks, threads, 0, s>>>(A, M, K, lda, ctrl, t, row_cnt, scol, sval, A_c, ldac, \
                                                             codes, ldc, scales, wpr)
  switch (ch) {
    case 1: FP4_ROWS_OUTLIER(1); break;
    case 2: FP4_ROWS_OUTLIER(2); break;
    case 4: FP4_ROWS_OUTLIER(4); break;
    default: FP4_ROWS_OUTLIER(8); break;
  }
#undef FP4_ROWS_OUTLIER
}

// Histogram + threshold, fused row pass (CSR staging, optional A_clamped, optional
// codes / scales), row scan and gather.  Arguments are validated by the callers.
fp4_status run_outlier_pipeline(const void* A, int64_t M, int64_t K, int64_t lda, double q, float* t_out,
                                int32_t* row_ptr, int32_t* col_idx, float* vals, int64_t nnz_capacity,
                                int64_t* nnz_out, void* A_clamped, int64_t ldac, uint8_t* codes, int64_t ldc,
                                float* scales, void* workspace, cudaStream_t s) {
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  const WsLayout L = ws_layout(M);
  auto* ws = static_cast<uint8_t*>(workspace);
  auto* ghist = reinterpret_cast<uint32_t*>(ws + L.hist);
  auto* ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  auto* row_cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  auto* scol = reinterpret_cast<int32_t*>(ws + L.scol);
  auto* sval = reinterpret_cast<float*>(ws + L.sval);
  uint32_t* status = status_word();
  const auto* a = static_cast<const uint16_t*>(A);

  const int64_t n = M * K;
  const int64_t k_rank = n - outlier_max_nnz(M, K, q);
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
  int64_t hblocks = (chunks + kHistThreads * 8 - 1) / (kHistThreads * 8);
  if (hblocks > sms) hblocks = sms;
  if (hblocks < 1) hblocks = 1;
  histogram_select_kernel<<<unsigned(hblocks), kHistThreads, hist_smem, s>>>(a, M, int(K), lda, k_rank, ghist, ctrl,
                                                                             t_out);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;

  // fused row pass: ch chunks per lane and wpr warps per row, chosen to cover the
  // row's 16-byte chunks with the least padding (ties: 4 chunks per lane;
  // K <= 16384 fits 16 warps x 4 chunks); CTAs of about 8 warps, as many per
  // SM as fit in 16 warps; persistent over row groups
  const int nchunk = int(K / 8);
  int ch = 1, wpr = (nchunk + 31) / 32, waste = wpr * 32 - nchunk;
  for (int c : {2, 8, 4}) {
    const int w = (nchunk + 32 * c - 1) / (32 * c);
    const int x = w * 32 * c - nchunk;
    if (w <= kMaxRowWarps && (wpr > kMaxRowWarps || x < waste || (x == waste && c == 4))) {
      ch = c;
      wpr = w;
      waste = x;
    }
  }
  const int rows_per_cta = wpr >= 8 ? 1 : 8 / wpr;
  const int ctas_per_sm = kMaxRowWarps / (wpr * rows_per_cta) > 0 ? kMaxRowWarps / (wpr * rows_per_cta) : 1;
  const unsigned threads = unsigned(32 * wpr * rows_per_cta);
  int64_t rblocks = (M + rows_per_cta - 1) / rows_per_cta;
  if (rblocks > int64_t(sms) * ctas_per_sm) rblocks = int64_t(sms) * ctas_per_sm;
  if (codes)
    launch_rows_outlier<true>(ch, wpr, unsigned(rblocks), threads, s, a, M, int(K), lda, ctrl, t_out, row_cnt, scol,
                              sval, static_cast<uint16_t*>(A_clamped), ldac, codes, ldc, scales);
  else
    launch_rows_outlier<false>(ch, wpr, unsigned(rblocks), threads, s, a, M, int(K), lda, ctrl, t_out, row_cnt, scol,
                               sval, static_cast<uint16_t*>(A_clamped), ldac, nullptr, 0, nullptr);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  row_scan_kernel<<<1, 1024, 0, s>>>(row_cnt, M, row_ptr, nnz_out, ctrl, nnz_capacity, status);
  if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  if (nnz_capacity > 0) {
    int64_t gblocks = (M + 7) / 8;
    if (gblocks > int64_t(sms) * 8) gblocks = int64_t(sms) * 8;
    gather_kernel<<<unsigned(gblocks), 256, 0, s>>>(row_cnt, row_ptr, M, scol, sval, a, int(K), lda, ctrl, t_out,
                                                    col_idx, vals, nnz_capacity);
    if (launch_status() != FP4_OK) return FP4_ERR_CUDA;
  }
  return FP4_OK;
}

fp4_status validate_outlier_args(const void* A, int64_t M, int64_t K, int64_t lda, double q, const float* t_out,
                                 const int32_t* row_ptr, const int32_t* col_idx, const float* vals,
                                 int64_t nnz_capacity, const void* workspace, size_t ws_bytes) {
  if (!A || !t_out || !row_ptr || !workspace) return FP4_ERR_INVALID_ARG;
  if (!(q > 0.0) || !(q <= 1.0)) return FP4_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0 || K % 8 != 0 || lda < K || K > 16384 || M >= (int64_t(1) << 31) ||
      M * K >= (int64_t(1) << 32))
    return FP4_ERR_SHAPE;
  if (lda % 8 != 0 || !aligned16(A) || !aligned16(workspace)) return FP4_ERR_ALIGNMENT;
  const int64_t need = outlier_max_nnz(M, K, q);
  if (nnz_capacity < need || nnz_capacity >= (int64_t(1) << 31)) return FP4_ERR_CAPACITY;
  if (nnz_capacity > 0 && (!col_idx || !vals)) return FP4_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(M).total) return FP4_ERR_WORKSPACE;
  return FP4_OK;
}

}  // namespace
}  // namespace fp4

FP4_API fp4_status outlier_clamp_quantile(const void* A, int64_t M, int64_t K, int64_t lda, double q, float* t_out,
                                          int32_t* row_ptr, int32_t* col_idx, float* vals, int64_t nnz_capacity,
                                          int64_t* nnz_out, void* A_clamped, int64_t ldac, void* workspace,
                                          size_t ws_bytes, fp4_stream_t stream) {
  using namespace fp4;
  fp4_status st = validate_outlier_args(A, M, K, lda, q, t_out, row_ptr, col_idx, vals, nnz_capacity, workspace,
                                        ws_bytes);
  if (st != FP4_OK) return st;
  if (A_clamped && ldac < K) return FP4_ERR_SHAPE;
  if (A_clamped && (!aligned16(A_clamped) || ldac % 8)) return FP4_ERR_ALIGNMENT;
  return run_outlier_pipeline(A, M, K, lda, q, t_out, row_ptr, col_idx, vals, nnz_capacity, nnz_out, A_clamped, ldac,
                              nullptr, 0, nullptr, workspace, reinterpret_cast<cudaStream_t>(stream));
}

FP4_API fp4_status fp4_quantize_rows_outliers(const void* A, int64_t M, int64_t K, int64_t lda, double q,
                                              uint8_t* codes, int64_t ldc_bytes, float* scales, float* t_out,
                                              int32_t* row_ptr, int32_t* col_idx, float* vals, int64_t nnz_capacity,
                                              int64_t* nnz_out, void* workspace, size_t ws_bytes,
                                              fp4_stream_t stream) {
  using namespace fp4;
  fp4_status st = validate_outlier_args(A, M, K, lda, q, t_out, row_ptr, col_idx, vals, nnz_capacity, workspace,
                                        ws_bytes);
  if (st != FP4_OK) return st;
  if (!codes || !scales) return FP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || ldc_bytes < K / 2) return FP4_ERR_SHAPE;
  if (ldc_bytes % 16 != 0 || !aligned16(codes) || !aligned16(scales)) return FP4_ERR_ALIGNMENT;
  return run_outlier_pipeline(A, M, K, lda, q, t_out, row_ptr, col_idx, vals, nnz_capacity, nnz_out, nullptr, 0, codes,
                              ldc_bytes, scales, workspace, reinterpret_cast<cudaStream_t>(stream));
}
