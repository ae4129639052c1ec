// Internal helpers of the sm_103a FP4 linear-layer library: host-side device
// checks and tensor-map encoding, device-side wrappers for mbarrier, TMA and
// tcgen05 (inline PTX), and the E2M1 encoder shared by the quantize kernels.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; the driver entry point is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp4lin.h"

#define FP4_API extern "C" __attribute__((visibility("default")))

namespace fp4 {

// ------------------------------------------------------------------ host side

// Checks that the current device is compute capability 10.3 and returns its SM count.
fp4_status check_device(int* num_sms);
// Device address of the sticky status word of the current device.
uint32_t* status_word();
// Encodes a 2-D tiled tensor map (row-major, dim0 contiguous) with the given swizzle.
fp4_status encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                          uint64_t dim1, uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                          CUtensorMapSwizzle swizzle);
// Maps the last launch error to FP4_ERR_CUDA (and remembers its text for this thread).
fp4_status launch_status();
const char* last_cuda_error();
// Default limit for bounded mbarrier waits, in nanoseconds.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ device side

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with the given parity has completed, for at most
// limit_ns of wall time.  Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// mbar_wait by every lane of a warp, with one verdict for the whole warp (a lane
// that gave up at the limit while another saw the phase complete would otherwise
// leave the warp divergent before its next warp-wide operation).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, limit_ns));
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// 2-D tiled TMA store shared -> global (bulk-group completion).  Elements of the
// box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until every committed bulk store of this thread but the most recent one
// has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Hint: bring the global-memory line holding `ptr` into L1 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr));
}
// 32-byte read-only global load (sm_100 and later); the address must be 32-byte aligned.
__device__ __forceinline__ void ld_nc_v8(const void* ptr, uint4& lo, uint4& hi) {
  asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
               : "l"(ptr));
}
// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Makes this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 (5th-generation tensor core, tensor memory)

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// D(tmem) (+)= A(smem desc) x B(smem desc), BF16/FP16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D(tmem) (+)= A x B with TF32 operands (fp32 values whose low 13 mantissa bits are zero).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D(tmem) (+)= A x B with E2M1 operands and per-32-element UE8M0 block scales read from tmem.
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// ---------------------------------------------------------------- CTA pairs (cluster of 2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the object at shared::cta address `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Barrier over every thread of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Relaxed arrive on an mbarrier of a CTA of the cluster: no release of this
// thread's prior memory operations (for signals that order only tensor-memory
// reads already completed by tcgen05.wait::ld, so outstanding global stores
// are not waited for).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMEM allocation for a CTA pair: one warp of each CTA executes it; both get the same columns.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
// 2-D tiled TMA load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
// Pair MMAs (issued by one thread of the leader CTA): M = 256, A rows split by CTA,
// B's N split by CTA; each CTA's TMEM holds its 128 rows of D.
__device__ __forceinline__ void mma_mxf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on the mbarrier at offset `bar` in every CTA of `cta_mask` when the pair's
// previously issued tcgen05 operations complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Single-CTA (PAIR = false) and CTA-pair forms of the pipeline operations.
// TMA load whose completion is counted on `bar` of the MMA-issuing CTA (rank 0).
template <bool PAIR>
__device__ __forceinline__ void tma_load_2d_to(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                               int32_t y) {
  if constexpr (PAIR) tma_load_2d_pair(dst, map, mapa_shared(bar, 0), x, y);
  else tma_load_2d(dst, map, bar, x, y);
}
// Commit of the issued MMAs to `bar` (in the CTAs of `mask`, for a pair).
template <bool PAIR>
__device__ __forceinline__ void commit_to(uint32_t bar, uint16_t mask) {
  if constexpr (PAIR) tc_commit_pair(bar, mask);
  else tc_commit(bar);
}
// Arrive on `bar` of the MMA-issuing CTA (rank 0).
template <bool PAIR>
__device__ __forceinline__ void arrive_on_issuer(uint32_t bar) {
  if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(bar, 0));
  else mbar_arrive(bar);
}
// Block barrier, or cluster barrier for a pair.
template <bool PAIR>
__device__ __forceinline__ void cta_sync() {
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
}
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc_for(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (PAIR) {
    tmem_alloc_pair(dst_smem, ncols);
    tmem_relinquish_pair();
  } else {
    tmem_alloc(dst_smem, ncols);
    tmem_relinquish();
  }
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc_for(uint32_t taddr, uint32_t ncols) {
  if constexpr (PAIR) tmem_dealloc_pair(taddr, ncols);
  else tmem_dealloc(taddr, ncols);
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// Each thread of the warp reads 8 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// (a, b) *= (x, y) as one packed fp32 multiply (each half rounded to nearest, as two fmul.rn).
__device__ __forceinline__ void mul2_rn(float& a, float& b, float x, float y) {
  uint64_t r;
  const uint64_t ab = (uint64_t(__float_as_uint(b)) << 32) | __float_as_uint(a);
  const uint64_t xy = (uint64_t(__float_as_uint(y)) << 32) | __float_as_uint(x);
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ab), "l"(xy));
  a = __uint_as_float(uint32_t(r));
  b = __uint_as_float(uint32_t(r >> 32));
}

// Named barrier over `nthreads` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  // the warp reconverges first; the non-aligned form also tolerates callers
  // that reach the barrier from divergent code
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Each thread of the warp writes 8 consecutive 32-bit columns of its own TMEM lane with `v`.
__device__ __forceinline__ void tmem_st8_fill(uint32_t taddr, uint32_t v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(taddr), "r"(v)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for tcgen05.mma: 128-byte swizzle, the
// given leading / stride byte offsets, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // version
  d |= 2ull << 61;  // SWIZZLE_128B
  return d;
}

// ---- quantizer arithmetic

// s = 6 / absmax as one IEEE fp32 division; 1 when absmax is 0 or the quotient is not finite.
__device__ __forceinline__ float scale_from_absmax(float absmax) {
  const float s = __fdiv_rn(6.0f, absmax);
  return (absmax == 0.0f || !isfinite(s)) ? 1.0f : s;
}

// Two E2M1 codes in one byte (lo in bits 3..0, hi in bits 7..4) by the hardware
// conversion (round to nearest even, saturating to +-6).  On sm_103a it keeps
// the sign of -0 and of negative values that round to zero (code 0x8), as the
// quantizer's definition requires; the exhaustive BF16-pattern tests check it.
__device__ __forceinline__ uint32_t e2m1x2_encode(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return uint32_t(r);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Scales 8 BF16 values by s after clamping |x| to t, and packs their 8 E2M1
// codes into one 32-bit word (element 0 in the lowest nibble).
// Packed BF16 helpers: a 32-bit word holds two BF16 values, element 2i in the
// low half.  Magnitudes compare as unsigned 15-bit integers (sign cleared).

// Packed BF16 pair operations on the hardware's bf16x2 units.  The operands are
// magnitude patterns (sign cleared, finite), for which the BF16 order is the
// unsigned integer order of the 15-bit patterns.
__device__ __forceinline__ uint32_t bf2_gt_mask(uint32_t a, uint32_t b) {   // 0xFFFF per half where a > b
  return __hgt2_mask(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
}
__device__ __forceinline__ uint32_t bf2_min(uint32_t a, uint32_t b) {
  const __nv_bfloat162 m = __hmin2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&m);
}
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  const __nv_bfloat162 m = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&m);
}

// sign(x) min(|x|, t) for both halves, with tb2 = t's 15-bit pattern in both
// halves: exact, since t is itself a BF16 value.
__device__ __forceinline__ uint32_t clamp_pair(uint32_t w, uint32_t tb2) {
  return (w & 0x80008000u) | bf2_min(w & 0x7FFF7FFFu, tb2);
}

// Two E2M1 codes (one byte) of the fp32 products x * s of a BF16 pair.
__device__ __forceinline__ uint32_t quantize_pair(uint32_t w, float s) {
  return e2m1x2_encode(__fmul_rn(__uint_as_float(w << 16), s), __fmul_rn(__uint_as_float(w & 0xFFFF0000u), s));
}

// Eight codes of a 16-byte chunk of BF16 values (no clamp), the products x * s
// formed two at a time by the packed fp32 multiply (each rounded as fmul.rn).
__device__ __forceinline__ uint32_t quantize8_packed(const uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
    mul2_rn(lo, hi, s, s);
    out |= e2m1x2_encode(lo, hi) << (8 * i);
  }
  return out;
}

// Eight codes of a 16-byte chunk of BF16 values, element 0 in the lowest nibble;
// with CLAMP the values are first clamped to t (tb2 as for clamp_pair).
template <bool CLAMP>
__device__ __forceinline__ uint32_t quantize8(const uint4 v, float s, uint32_t tb2) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) out |= quantize_pair(CLAMP ? clamp_pair(w[i], tb2) : w[i], s) << (8 * i);
  return out;
}

// As quantize8<true> for a clamp threshold t that need not be a BF16 value:
// the clamp sign(x) min(|x|, t) is taken in fp32.
__device__ __forceinline__ uint32_t quantize8_clamp_f32(const uint4 v, float s, float t) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
    if (fabsf(lo) > t) lo = copysignf(t, lo);
    if (fabsf(hi) > t) hi = copysignf(t, hi);
    out |= e2m1x2_encode(__fmul_rn(lo, s), __fmul_rn(hi, s)) << (8 * i);
  }
  return out;
}

// Largest 15-bit magnitude pattern of a chunk, per 16-bit half.
__device__ __forceinline__ uint32_t chunk_maxmag(const uint4 v) {
  return bf2_max(bf2_max(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu), bf2_max(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
}

// Running maximum of the magnitude patterns of a chunk, per 16-bit half.
__device__ __forceinline__ uint32_t maxmag8(const uint4 v, uint32_t acc) { return bf2_max(acc, chunk_maxmag(v)); }

// Largest magnitude pattern of a warp's packed maxima, as an fp32 value.
__device__ __forceinline__ uint32_t warp_max_bits(uint32_t acc2) {
  uint32_t m = max(acc2 & 0xFFFFu, acc2 >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  return m;
}

}  // namespace fp4
