// Quantile outlier clamp and sparse compensation matrix, per the outlier
// passage of the page "首个 FP4 精度的大模型训练框架来了" (czzqal.com): a quantile
// search finds the largest-magnitude outliers of A, they are clamped to the
// threshold (A_clamped), and dA = A - A_clamped is kept as a sparse matrix that
// is nonzero only where clamping happened.
//
// One cooperative kernel does it all (rowcall_kernel, below; HBM-bound): a
// coarse pilot histogram of every 64th row gives a floor under the threshold,
// a full pass histograms only the magnitudes above the floor and records each
// row's largest magnitude (a second pass fills in the rest when the pilot
// misleads), every CTA selects the exact k-th order statistic t, a streaming
// row pass writes the row codes / scales, A_clamped on request and each row's
// first kRowSlots entries (column, A - sign(A) t) into per-row slots, and
// row_ptr and the CSR follow from per-CTA totals.  Its three or four grid
// barriers are bounded waits.
#include <cmath>

#include "common.cuh"

namespace fp4 {
namespace {

constexpr int kBins = 32768;

constexpr int kRowSlots = 32;  // entries per row kept by the row pass (more are re-read from A)

struct Ctrl {
  uint32_t unused;
  uint32_t t_bits;        // 15-bit magnitude pattern of t
  unsigned long long nnz_expect; // number of |A| > t from the histogram
};

struct WsLayout {
  size_t hist, hist2, ctrl, fctrl, cta_total, cnt, rmax, scol, sval, total;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

constexpr int kMaxCtas = 1024;   // CTA totals of the fused row call (one CTA per SM)

// The histograms and both control blocks come first: one memset clears them.
WsLayout ws_layout(int64_t M) {
  WsLayout L;
  size_t off = 0;
  L.hist = off; off += round256(size_t(kBins) * 4);
  L.hist2 = off; off += round256(size_t(kBins) * 4);
  L.ctrl = off; off += round256(sizeof(Ctrl));
  L.fctrl = off; off += 256;
  L.cta_total = off; off += round256(size_t(kMaxCtas) * 8);
  L.cnt = off; off += round256(size_t(M) * 4);
  L.rmax = off; off += round256(size_t(M) * 4);
  L.scol = off; off += round256(size_t(M) * kRowSlots * 4);
  L.sval = off; off += round256(size_t(M) * kRowSlots * 4);
  L.total = off;
  return L;
}


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

// ---------------------------------------------------------------------------
// The fused row call: threshold, clamp, CSR of dA and (optionally) the row
// codes / scales and A_clamped in ONE cooperative kernel (one CTA of 512
// threads per SM, all resident; grid barriers are bounded waits).
//
//  1. pilot: every 64th row of each CTA's row block in a coarse 512-bin
//     histogram (exponent and the first mantissa bit), merged into g_pilot;
//                                                               -- barrier
//  2. every CTA derives the same floor F from the pilot: the lower edge of the
//     coarse bin holding the sample's magnitude with 4x the requested
//     exceedance (plus 16) above it, so t >= F unless the sample misleads
//     (then step 4 fills the rest in);
//  3. main pass over the CTA's rows: a histogram of the magnitudes >= F only
//     (a chunk whose 8 magnitudes are all below F costs three packed maxima,
//     no atomics), merged into g_main, and each row's largest magnitude;
//                                                               -- barrier
//  4. every CTA selects t = the largest bin b with #{|A| >= b} >= n - k + 1
//     (the k-th smallest); if the bins >= F hold fewer than n - k + 1 values,
//     a second pass counts the magnitudes < F, and t is selected over all bins;
//  5. row pass over the CTA's rows in reverse order (the rows read last in
//     step 3 are still in L2): one warp per row in one streaming sweep -- the
//     row's largest magnitude was recorded in step 3, so the scale of the
//     clamped row, min(max |A|, t), comes first -- codes, A_clamped, the
//     outlier count and the row's first kRowSlots entries (column order) into
//     its slots;                                                -- barrier
//  6. row_ptr from the per-CTA totals and a block scan; the slots (or, for a
//     longer row, A read again) go to their CSR positions.
constexpr int kRThreads = 512;
constexpr int kRWarps = kRThreads / 32;
constexpr int kPilotStride = 64;
constexpr int kCoarseShift = 6;                      // pilot bins: magnitude pattern >> 6 (exponent + 1 mantissa bit)
constexpr int kCoarseBins = kBins >> kCoarseShift;  // 512
constexpr int kRU = 8;   // 16-byte chunks a lane per step of the row pass (two steps in flight)
constexpr int kHU = 16;  // 16-byte loads in flight per lane (histogram passes)

struct FCtrl {
  uint32_t bar_count;   // CTAs arrived at the current grid barrier
  uint32_t bar_gen;     // barrier generation
};

struct RowCallParams {
  const uint16_t* A;
  int64_t M;
  int K;
  int64_t lda;
  int64_t k_rank;          // 1-based rank of t among |A| ascending
  int64_t n_pilot;         // values in the pilot sample (every kPilotStride-th row of each CTA's block)
  uint32_t* g_pilot;       // 32768 bins, zeroed
  uint32_t* g_main;        // 32768 bins, zeroed
  FCtrl* fctrl;            // zeroed
  Ctrl* ctrl;              // t_bits and nnz_expect for the caller-visible checks
  int64_t* cta_total;      // one per CTA
  int32_t* row_cnt;
  uint32_t* rmax;          // per row: the largest magnitude pattern (main histogram pass)
  int32_t* scol;
  float* sval;
  float* t_out;
  int32_t* row_ptr;
  int32_t* col_idx;
  float* vals;
  int64_t cap;
  int64_t* nnz_out;
  uint16_t* A_c;
  int64_t ldac;
  uint8_t* codes;
  int64_t ldc;
  float* scales;
  uint32_t* status;
  uint64_t wait_ns;
};

// Grid barrier over co-resident CTAs (sense by generation), bounded: false when
// the limit ran out (the caller records FP4_FLAG_TIMEOUT and stops).
__device__ bool grid_sync(FCtrl* c, uint64_t limit_ns) {
  __syncthreads();
  int ok = 1;
  if (threadIdx.x == 0) {
    volatile uint32_t* gen = &c->bar_gen;
    const uint32_t g = *gen;
    __threadfence();
    if (atomicAdd(&c->bar_count, 1u) == gridDim.x - 1) {
      c->bar_count = 0u;
      __threadfence();
      atomicAdd(&c->bar_gen, 1u);
    } else {
      const uint64_t t0 = global_timer_ns();
      while (*gen == g) {
        if (global_timer_ns() - t0 > limit_ns) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  return __syncthreads_and(ok) != 0;
}

// Counts the magnitude patterns in [lo, hi) of rows r (r_begin <= r < r_end,
// r - r_begin a multiple of `stride`, one warp per row) into hist (shared).
__device__ void rows_histogram(const RowCallParams& p, int64_t r_begin, int64_t r_end, int stride, uint32_t lo,
                               uint32_t hi, uint32_t* hist, uint32_t* rmax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = p.K >> 3;
  for (int64_t row = r_begin + int64_t(warp) * stride; row < r_end; row += int64_t(kRWarps) * stride) {
    const uint4* src = reinterpret_cast<const uint4*>(p.A + row * p.lda);
    uint32_t mx = 0;   // the row's largest magnitude pattern (rmax given)
    for (int c00 = 0; c00 < nchunk; c00 += 32 * kHU) {   // every lane takes every step
      uint4 v[kHU];
#pragma unroll
      for (int u = 0; u < kHU; ++u) {
        const int c = c00 + 32 * u + lane;
        v[u] = c < nchunk ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kHU; ++u) {
        if (c00 + 32 * u + lane >= nchunk) continue;
        const uint32_t m2 = chunk_maxmag(v[u]);
        const uint32_t m1 = max(m2 & 0xFFFFu, m2 >> 16);
        mx = max(mx, m1);
        if (m1 < lo) continue;   // all 8 below the range: no atomics
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t k0 = w[i] & 0x7FFFu, k1 = (w[i] >> 16) & 0x7FFFu;
          if (k0 >= lo && k0 < hi) atomicAdd(hist + k0, 1u);
          if (k1 >= lo && k1 < hi) atomicAdd(hist + k1, 1u);
        }
      }
    }
    if (rmax) {
      mx = __reduce_max_sync(0xFFFFFFFFu, mx);
      if (lane == 0) rmax[row] = mx;
    }
  }
}

// Pilot: coarse histogram (kCoarseBins bins of the magnitude pattern >>
// kCoarseShift) of every kPilotStride-th row of [r0, r1), one warp per row,
// each warp counting into its own kCoarseBins words of `hist` (shared), then
// merged into g (global).
__device__ void pilot_phase(const RowCallParams& p, int64_t r0, int64_t r1, uint32_t* hist, uint32_t* g) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = threadIdx.x; b < kRWarps * kCoarseBins; b += kRThreads) hist[b] = 0u;
  __syncthreads();
  uint32_t* mine = hist + warp * kCoarseBins;
  const int nchunk = p.K >> 3;
  for (int64_t row = r0 + int64_t(warp) * kPilotStride; row < r1; row += int64_t(kRWarps) * kPilotStride) {
    const uint4* src = reinterpret_cast<const uint4*>(p.A + row * p.lda);
    for (int c00 = 0; c00 < nchunk; c00 += 32 * kRU) {   // every lane takes every step
      uint4 v[kRU];
#pragma unroll
      for (int u = 0; u < kRU; ++u) {
        const int c = c00 + 32 * u + lane;
        v[u] = c < nchunk ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kRU; ++u) {
        if (c00 + 32 * u + lane >= nchunk) continue;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          atomicAdd(mine + ((w[i] & 0x7FFFu) >> kCoarseShift), 1u);
          atomicAdd(mine + (((w[i] >> 16) & 0x7FFFu) >> kCoarseShift), 1u);
        }
      }
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kCoarseBins; b += kRThreads) {
    uint32_t c = 0;
    for (int w = 0; w < kRWarps; ++w) c += hist[w * kCoarseBins + b];
    if (c) atomicAdd(g + b, c);
  }
}

// Over the kCoarseBins bins of g (global, complete): the lower edge (a
// magnitude pattern) of the largest coarse bin B with #{coarse bins >= B} >=
// target, or 0 when there is none.  Computed by warp 0, returned to all
// threads of the CTA.
__device__ uint32_t coarse_floor(const uint32_t* g, uint64_t target) {
  __shared__ uint32_t s_floor;
  constexpr int kPer = kCoarseBins / 32;   // 16 bins a lane
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t c[kPer];
    unsigned long long sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      c[i] = __ldcg(g + lane * kPer + i);
      sum += c[i];
    }
    // suffix over the lanes above: the bins of lanes lane+1 .. 31
    unsigned long long incl = sum;   // sum of lanes lane .. 31
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
      if (lane + o < 32) incl += y;
    }
    const unsigned long long above = incl - sum;
    uint32_t f = 0u;
    bool found = false;
    if (above < target && incl >= target) {   // the crossing is in this lane's bins
      unsigned long long run = above;
      for (int i = kPer - 1; i >= 0; --i) {
        run += c[i];
        if (run >= target) {
          f = uint32_t(lane * kPer + i) << kCoarseShift;
          found = true;
          break;
        }
      }
    }
    const uint32_t who = __ballot_sync(0xFFFFFFFFu, found);
    f = who ? __shfl_sync(0xFFFFFFFFu, f, __ffs(who) - 1) : 0u;
    if (lane == 0) s_floor = f;
  }
  __syncthreads();
  const uint32_t r = s_floor;
  __syncthreads();
  return r;
}

// Zeroes hist[lo, hi) (shared), histograms the CTA's rows into it and adds the
// nonzero bins to g (global).
__device__ void histogram_phase(const RowCallParams& p, int64_t r0, int64_t r1, int stride, uint32_t lo,
                                uint32_t hi, uint32_t* hist, uint32_t* g, uint32_t* rmax = nullptr) {
  for (uint32_t b = lo + threadIdx.x; b < hi; b += kRThreads) hist[b] = 0u;
  __syncthreads();
  rows_histogram(p, r0, r1, stride, lo, hi, hist, rmax);
  __syncthreads();
  for (uint32_t b = lo + threadIdx.x; b < hi; b += kRThreads) {
    const uint32_t c = hist[b];
    if (c) atomicAdd(g + b, c);
  }
}

// Over bins [lo, 32768) of g (global, complete there): finds the largest bin b
// with suffix(b) = sum of bins >= b at least `target`.  Returns b, or -1 when
// suffix(lo) < target; *total = suffix(lo), *above = suffix(b + 1).  Uniform
// over the CTA (uses `scratch`: kBins words of shared memory).
__device__ int suffix_select(const uint32_t* g, uint32_t lo, uint64_t target, uint32_t* scratch, uint64_t* total,
                             uint64_t* above) {
  __shared__ int sel;
  __shared__ unsigned long long sel_above;
  constexpr int kPer = kBins / kRThreads;   // 64 bins a thread
  {
    // all of a thread's loads in flight at once, then the stores (a load-then-store
    // loop would wait out one L2 round trip per 16 bytes)
    constexpr int kLd = kBins / 4 / kRThreads;   // 16
    uint4 v[kLd];
#pragma unroll
    for (int j = 0; j < kLd; ++j) {
      const int i = threadIdx.x + j * kRThreads;
      v[j] = (4u * uint32_t(i) + 3u < lo) ? make_uint4(0u, 0u, 0u, 0u) : __ldcg(reinterpret_cast<const uint4*>(g) + i);
    }
#pragma unroll
    for (int j = 0; j < kLd; ++j) reinterpret_cast<uint4*>(scratch)[threadIdx.x + j * kRThreads] = v[j];
  }
  if (threadIdx.x == 0) sel = -1;
  __syncthreads();
  // bins below lo are not counted (a partially covered word had them zeroed above only if fully below)
  const int b0 = threadIdx.x * kPer;
  unsigned long long sum = 0;
  for (int i = 0; i < kPer; ++i) {
    const int b = b0 + ((i + threadIdx.x) & (kPer - 1));
    if (uint32_t(b) >= lo) sum += scratch[b];
  }
  // suffix sums over the 512 partial sums (from the top), one thread per partial
  unsigned long long suf = 0;   // sum of partials of threads > this one
  {
    // a simple two-level scan: each warp sums its 32 partials, then warps from the top
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_down_sync(0xFFFFFFFFu, x, o);
      if (lane + o < 32) x += y;
    }
    // x = sum of partials lane..31 of this warp
    __shared__ unsigned long long wsum[kRWarps];
    if (lane == 0) wsum[wid] = x;
    __syncthreads();
    unsigned long long higher = 0;
    for (int w = wid + 1; w < kRWarps; ++w) higher += wsum[w];
    suf = higher + x - sum;   // partials strictly above this thread
    if (threadIdx.x == 0) *total = higher + x;
  }
  // the crossing: suffix at the top of this thread's range is suf, at its bottom suf + sum
  if (suf < target && suf + sum >= target) {
    unsigned long long run = suf;
    for (int i = kPer - 1; i >= 0; --i) {
      const int b = b0 + i;
      const unsigned long long c = uint32_t(b) >= lo ? scratch[b] : 0u;
      if (run + c >= target) {
        sel = b;
        sel_above = run;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
  *above = sel_above;
  const int r = sel;
  __syncthreads();
  return r;
}

// The row's entries in chunk j (lane's 16-byte chunk c = column chunk): the warp
// numbers them in column order (chunk index c ascending across the lanes) and
// writes those with position < kRowSlots into the row's slots.  `pos` (warp-
// uniform) is the number of entries in earlier chunks; every lane must call.
__device__ __noinline__ void emit_slots(const RowCallParams& p, int64_t row, int c, bool valid, const uint4 v,
                                        uint32_t tbits, float t, uint32_t& pos) {
  const int lane = threadIdx.x & 31;
  uint32_t m = valid ? outlier_mask8(v, tbits) : 0u;
  const uint32_t nm = __popc(m);
  if (!__any_sync(0xFFFFFFFFu, nm != 0)) return;
  uint32_t incl = nm;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t ps = pos + incl - nm;
  while (m && ps < uint32_t(kRowSlots)) {   // set bits in ascending column order
    const int e = __ffs(m) - 1;
    m &= m - 1;
    const uint32_t word = e < 4 ? (e < 2 ? v.x : v.y) : (e < 6 ? v.z : v.w);
    const float x = bf16_bits_to_float((word >> (16 * (e & 1))) & 0xFFFFu);
    p.scol[row * kRowSlots + ps] = c * 8 + e;
    p.sval[row * kRowSlots + ps] = __fsub_rn(x, copysignf(t, x));
    ++ps;
  }
  pos += __shfl_sync(0xFFFFFFFFu, incl, 31);
}

// Codes and A_clamped of one 16-byte chunk; `has` says whether some value of the
// chunk exceeds t (without one the clamp changes nothing and is skipped).
__device__ __noinline__ void chunk_outputs_clamped(uint32_t* cdst, uint4* adst, int c, const uint4 v, float sc,
                                                 uint32_t tb2) {
  if (cdst) cdst[c] = quantize8<true>(v, sc, tb2);
  if (adst) adst[c] = make_uint4(clamp_pair(v.x, tb2), clamp_pair(v.y, tb2), clamp_pair(v.z, tb2), clamp_pair(v.w, tb2));
}
// (the rare paths are out of line: a fully unrolled row pass with them inlined
// outgrew the instruction cache)
__device__ __forceinline__ void chunk_outputs(uint32_t* cdst, uint4* adst, int c, const uint4 v, float sc, uint32_t tb2,
                                              bool has) {
  if (has) {
    chunk_outputs_clamped(cdst, adst, c, v, sc, tb2);
    return;
  }
  if (cdst) cdst[c] = quantize8_packed(v, sc);
  if (adst) adst[c] = v;
}

__device__ __noinline__ uint32_t count_outliers(const uint4 v, uint32_t tbits) { return __popc(outlier_mask8(v, tbits)); }

// Loads step s of a row: chunks c = 32 (kRU s + u) + lane (zero past the row).
__device__ __forceinline__ void load_step(const uint4* src, int s, int nchunk, uint4 (&v)[kRU]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < kRU; ++u) {
    const int c = 32 * (kRU * s + u) + lane;
    v[u] = c < nchunk ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Codes, A_clamped, outlier count and slots of step s's chunks (the scale is
// known).  Every lane calls.
__device__ __forceinline__ void row_step(const RowCallParams& p, int64_t row, int s, int nchunk, const uint4 (&v)[kRU],
                                         uint32_t* cdst, uint4* adst, float sc, uint32_t tbits, uint32_t tb2, float t,
                                         uint32_t& cnt, uint32_t& pos) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < kRU; ++u) {
    const int c = 32 * (kRU * s + u) + lane;
    const bool has = bf2_gt_mask(chunk_maxmag(v[u]), tb2);   // zero chunks past the row: never
    if (c < nchunk) chunk_outputs(cdst, adst, c, v[u], sc, tb2, has);
    if (has) cnt += count_outliers(v[u], tbits);
    if (pos < uint32_t(kRowSlots) && __any_sync(0xFFFFFFFFu, has)) emit_slots(p, row, c, has, v[u], tbits, t, pos);
  }
}

// One row in a single streaming sweep: its largest magnitude is known from the
// main histogram pass, so the scale comes first, and every chunk is quantized,
// clamped and searched for outliers as it arrives (two steps of kRU chunks a
// lane in flight).  Every lane of the warp calls; returns the outlier count.
__device__ uint32_t row_pass(const RowCallParams& p, int64_t row, int nchunk, uint32_t tbits, float t) {
  const uint32_t tb2 = tbits | (tbits << 16);
  const uint4* src = reinterpret_cast<const uint4*>(p.A + row * p.lda);
  const int nsteps = (nchunk + 32 * kRU - 1) / (32 * kRU);
  uint4 a[kRU], b[kRU];
  load_step(src, 0, nchunk, a);
  // max over min(|x|, t) = min(max |x|, t)
  const float sc = scale_from_absmax(bf16_bits_to_float(min(__ldcg(p.rmax + row), tbits)));
  if ((threadIdx.x & 31) == 0 && p.scales) p.scales[row] = sc;
  uint32_t* cdst = p.codes ? reinterpret_cast<uint32_t*>(p.codes + row * p.ldc) : nullptr;
  uint4* adst = p.A_c ? reinterpret_cast<uint4*>(p.A_c + row * p.ldac) : nullptr;
  uint32_t cnt = 0, pos = 0;
  for (int s = 0; s < nsteps; s += 2) {   // warp-uniform
    if (s + 1 < nsteps) load_step(src, s + 1, nchunk, b);
    row_step(p, row, s, nchunk, a, cdst, adst, sc, tbits, tb2, t, cnt, pos);
    if (s + 1 < nsteps) {
      if (s + 2 < nsteps) load_step(src, s + 2, nchunk, a);
      row_step(p, row, s + 1, nchunk, b, cdst, adst, sc, tbits, tb2, t, cnt, pos);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
  if ((threadIdx.x & 31) == 0) p.row_cnt[row] = int32_t(cnt);
  return cnt;
}

__global__ void __launch_bounds__(kRThreads, 1) rowcall_kernel(const RowCallParams p) {
  extern __shared__ uint32_t hist[];   // kBins words
  __shared__ uint64_t s_above;
  __shared__ unsigned long long red64[kRWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n = p.M * int64_t(p.K);
  const int64_t r0 = p.M * blockIdx.x / gridDim.x, r1 = p.M * (blockIdx.x + 1) / gridDim.x;
  const uint64_t e_rank = uint64_t(n - p.k_rank + 1);   // t is the e_rank-th largest magnitude
  bool ok = true;

  // ---- 1-2: pilot histogram and the floor F
  uint32_t F = 0;
  const bool use_pilot = e_rank * 4 <= uint64_t(n);   // q > 0.75: the threshold sits in the tail
  if (use_pilot) {
    pilot_phase(p, r0, r1, hist, p.g_pilot);
    ok = grid_sync(p.fctrl, p.wait_ns);
    if (ok) {
      const uint64_t n_pilot = uint64_t(p.n_pilot);
      const double want = 4.0 * double(e_rank) * double(n_pilot) / double(n) + 16.0;
      if (n_pilot >= 4096 && want < double(n_pilot)) F = coarse_floor(p.g_pilot, uint64_t(want));
    }
  }
  // ---- 3-4: histogram of the magnitudes >= F, then t
  int tb = -1;
  uint64_t nnz_expect = 0;
  if (ok) {
    histogram_phase(p, r0, r1, 1, F, uint32_t(kBins), hist, p.g_main, p.rmax);   // every row: its max too
    ok = grid_sync(p.fctrl, p.wait_ns);
  }
  if (ok) {
    uint64_t tot = 0, above = 0;
    tb = suffix_select(p.g_main, F, e_rank, hist, &tot, &above);
    if (threadIdx.x == 0) s_above = above;
    __syncthreads();
    if (tb < 0 && F > 0) {   // the pilot misled: count the magnitudes below F as well
      histogram_phase(p, r0, r1, 1, 0u, F, hist, p.g_main);
      ok = grid_sync(p.fctrl, p.wait_ns);
      if (ok) {
        tb = suffix_select(p.g_main, 0u, e_rank, hist, &tot, &above);
        if (threadIdx.x == 0) s_above = above;
        __syncthreads();
      }
    }
    nnz_expect = s_above;
  }
  if (!ok) {   // a grid barrier ran out: report, produce nothing
    if (threadIdx.x == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    return;
  }
  if (tb < 0) {   // cannot happen with a complete histogram: report, produce nothing
    if (threadIdx.x == 0) atomicOr(p.status, FP4_FLAG_INTERNAL);
    return;
  }
  const uint32_t tbits = uint32_t(tb);
  const float t = bf16_bits_to_float(tbits);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *p.t_out = t;
    p.ctrl->t_bits = tbits;
    p.ctrl->nnz_expect = nnz_expect;
  }

  // ---- 5: row pass, one warp per row, the CTA's rows in reverse order
  const int nchunk = p.K >> 3;
  long long cta_cnt = 0;
  for (int64_t i = warp; r1 - 1 - i >= r0; i += kRWarps) {
    const uint32_t cnt = row_pass(p, r1 - 1 - i, nchunk, tbits, t);
    cta_cnt += cnt;
  }
  // the CTA's total
  if (lane == 0) red64[warp] = (unsigned long long)cta_cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long s = 0;
    for (int w = 0; w < kRWarps; ++w) s += red64[w];
    p.cta_total[blockIdx.x] = int64_t(s);
  }
  if (!grid_sync(p.fctrl, p.wait_ns)) {
    if (threadIdx.x == 0) atomicOr(p.status, FP4_FLAG_TIMEOUT);
    return;
  }

  // ---- 6: row_ptr and the gather
  __shared__ long long s_base;
  {
    long long b = 0;
    for (int c = threadIdx.x; c < int(blockIdx.x); c += kRThreads) b += __ldcg(p.cta_total + c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
    if (lane == 0) red64[warp] = (unsigned long long)b;
    __syncthreads();
    if (threadIdx.x == 0) {
      long long s = 0;
      for (int w = 0; w < kRWarps; ++w) s += (long long)red64[w];
      s_base = s;
    }
    __syncthreads();
  }
  const long long base = s_base;
  // row_ptr[r0] is also the previous CTA's last value; writing it here (the same
  // number) lets the gather below read only this CTA's own entries
  if (threadIdx.x == 0 && (r0 < r1 || blockIdx.x == 0)) p.row_ptr[r0] = int32_t(base);
  // block scan of the counts of rows r0 .. r1 - 1, kRThreads at a time
  long long carry = 0;
  for (int64_t tile = r0; tile < r1; tile += kRThreads) {
    const int64_t row = tile + threadIdx.x;
    const long long c = row < r1 ? __ldcg(p.row_cnt + row) : 0;
    long long x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) red64[warp] = (unsigned long long)x;
    __syncthreads();
    long long before = 0, tile_total = 0;
    for (int w = 0; w < kRWarps; ++w) {
      if (w < warp) before += (long long)red64[w];
      tile_total += (long long)red64[w];
    }
    if (row < r1) {
      const long long end = base + carry + before + x;
      p.row_ptr[row + 1] = int32_t(end);
      // a row whose entries all fit in its slots is copied to its CSR position
      // here, by its own thread (longer rows are read again from A below)
      if (p.cap > 0 && c > 0 && c <= kRowSlots && end <= p.cap) {
        const long long dst = end - c;
        for (int e0 = 0; e0 < int(c); e0 += 8) {
          int32_t ci[8];
          float cv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (e0 + u < int(c)) {
              ci[u] = __ldcg(p.scol + row * kRowSlots + e0 + u);
              cv[u] = __ldcg(p.sval + row * kRowSlots + e0 + u);
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (e0 + u < int(c)) {
              p.col_idx[dst + e0 + u] = ci[u];
              p.vals[dst + e0 + u] = cv[u];
            }
          }
        }
      }
    }
    carry += tile_total;
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    const long long total = base + carry;
    if (p.nnz_out) *p.nnz_out = total;
    if (total > p.cap) atomicOr(p.status, FP4_FLAG_CAPACITY);
    else if (uint64_t(total) != p.ctrl->nnz_expect) atomicOr(p.status, FP4_FLAG_INTERNAL);
  }
  __syncthreads();   // this CTA's row_ptr entries are visible to all its threads
  if (p.cap == 0) return;
  // rows with more entries than slots: read again from A, one warp per row;
  // warp w takes rows r0 + w + kRWarps t, finding the long ones among 32
  // values of t at a time (so all warps share the work when every row is long)
  for (int64_t first = r0 + warp; first < r1; first += 32 * int64_t(kRWarps)) {
    const int64_t myrow = first + int64_t(kRWarps) * lane;
    const int32_t myc = myrow < r1 ? __ldcg(p.row_cnt + myrow) : 0;
    uint32_t longrows = __ballot_sync(0xFFFFFFFFu, myc > kRowSlots);
    while (longrows) {   // warp-uniform
      const int l = __ffs(longrows) - 1;
      longrows &= longrows - 1;
      const int64_t row = first + int64_t(kRWarps) * l;
      const int32_t nr = __shfl_sync(0xFFFFFFFFu, myc, l);
      const int64_t dst = p.row_ptr[row];
      if (dst + nr > p.cap) continue;   // beyond the capacity: flagged above
      const uint4* src = reinterpret_cast<const uint4*>(p.A + row * p.lda);
      int64_t b = dst;
      constexpr int kDepth = 4;   // 32-chunk groups loaded before any is scanned
      for (int c00 = 0; c00 < nchunk; c00 += 32 * kDepth) {   // every lane takes every step
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
          uint32_t m = ci < nchunk ? outlier_mask8(v, tbits) : 0u;
          const uint32_t nm = __popc(m);
          uint32_t incl = nm;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
          }
          int64_t ps = b + (incl - nm);
          while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1;
            const uint32_t word = e < 4 ? (e < 2 ? v.x : v.y) : (e < 6 ? v.z : v.w);
            const float x = bf16_bits_to_float((word >> (16 * (e & 1))) & 0xFFFFu);
            p.col_idx[ps] = ci * 8 + e;
            p.vals[ps] = __fsub_rn(x, copysignf(t, x));
            ++ps;
          }
          b += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
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

// The fused row call (rowcall_kernel): threshold, clamp, CSR staging, optional
// A_clamped and codes / scales, row_ptr and gather in one cooperative launch of
// one CTA per SM, after one memset of the histograms and control blocks.
// Arguments are validated by the callers.
fp4_status run_outlier_pipeline(const void* A, int64_t M, int64_t K, int64_t lda, double q, float* t_out,
                                int32_t* row_ptr, int32_t* col_idx, float* vals, int64_t nnz_capacity,
                                int64_t* nnz_out, void* A_clamped, int64_t ldac, uint8_t* codes, int64_t ldc,
                                float* scales, void* workspace, cudaStream_t s) {
  int sms = 0;
  fp4_status st = check_device(&sms);
  if (st != FP4_OK) return st;
  const WsLayout L = ws_layout(M);
  auto* ws = static_cast<uint8_t*>(workspace);
  const int64_t n = M * K;
  if (cudaMemsetAsync(ws, 0, L.cta_total, s) != cudaSuccess) return FP4_ERR_CUDA;

  static int ctas_per_sm[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = size_t(kBins) * 4;
  if (dev < 0 || dev >= 64) return FP4_ERR_CUDA;
  if (!ctas_per_sm[dev]) {
    if (cudaFuncSetAttribute(rowcall_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return FP4_ERR_CUDA;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, rowcall_kernel, kRThreads, smem) != cudaSuccess || nb < 1)
      return FP4_ERR_CUDA;
    ctas_per_sm[dev] = nb;
  }
  RowCallParams prm;
  prm.A = static_cast<const uint16_t*>(A);
  prm.M = M;
  prm.K = int(K);
  prm.lda = lda;
  prm.k_rank = n - outlier_max_nnz(M, K, q);
  prm.g_pilot = reinterpret_cast<uint32_t*>(ws + L.hist);
  prm.g_main = reinterpret_cast<uint32_t*>(ws + L.hist2);
  prm.fctrl = reinterpret_cast<FCtrl*>(ws + L.fctrl);
  prm.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  prm.cta_total = reinterpret_cast<int64_t*>(ws + L.cta_total);
  prm.row_cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  prm.rmax = reinterpret_cast<uint32_t*>(ws + L.rmax);
  prm.scol = reinterpret_cast<int32_t*>(ws + L.scol);
  prm.sval = reinterpret_cast<float*>(ws + L.sval);
  prm.t_out = t_out;
  prm.row_ptr = row_ptr;
  prm.col_idx = col_idx;
  prm.vals = vals;
  prm.cap = nnz_capacity;
  prm.nnz_out = nnz_out;
  prm.A_c = static_cast<uint16_t*>(A_clamped);
  prm.ldac = ldac;
  prm.codes = codes;
  prm.ldc = ldc;
  prm.scales = scales;
  prm.status = status_word();
  prm.wait_ns = kWaitLimitNs;
  // one CTA per SM (every CTA resident: the grid barriers need it)
  int grid = sms < kMaxCtas ? sms : kMaxCtas;
  prm.n_pilot = 0;
  for (int c = 0; c < grid; ++c) {
    const int64_t a = M * c / grid, b = M * (c + 1) / grid;
    prm.n_pilot += (b - a + kPilotStride - 1) / kPilotStride * K;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, rowcall_kernel, prm) != cudaSuccess) return launch_status();
  return launch_status();
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
