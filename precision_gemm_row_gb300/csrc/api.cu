// Host-side plumbing of the C ABI: status strings, device checks, the sticky
// device status word, tensor-map encoding, and the bounded-wait self-test.
#include <mutex>

#include "common.cuh"

namespace fp4 {

namespace {
// Sticky error flags (FP4_FLAG_*), one word per device that loads the library.
__device__ uint32_t g_status_flags;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_checked[kMaxDevices];          // 0 unknown, 1 ok, -1 unsupported
int g_sms[kMaxDevices];
uint32_t* g_status_ptr[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;
}  // namespace

fp4_status check_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_checked[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FP4_ERR_CUDA;
    if (major != 10 || minor != 3) {
      g_checked[dev] = -1;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_flags) != cudaSuccess) return FP4_ERR_CUDA;
      g_status_ptr[dev] = static_cast<uint32_t*>(p);
      g_sms[dev] = sms;
      g_checked[dev] = 1;
    }
  }
  if (g_checked[dev] < 0) return FP4_ERR_DEVICE_UNSUPPORTED;
  if (num_sms) *num_sms = g_sms[dev];
  return FP4_OK;
}

uint32_t* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_status_ptr[dev];
}

fp4_status encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                          uint64_t dim1, uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                          CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode_tried) {
      g_encode_tried = true;
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
              cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  if (!g_encode) return FP4_ERR_CUDA;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP4_OK : FP4_ERR_CUDA;
}

namespace {
thread_local const char* t_last_cuda_error = "no CUDA error";
}  // namespace

fp4_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return FP4_OK;
  t_last_cuda_error = cudaGetErrorString(e);
  return FP4_ERR_CUDA;
}

const char* last_cuda_error() { return t_last_cuda_error; }

namespace {
// One CTA waits on an mbarrier that is never arrived on; the bounded wait
// gives up after limit_ns and records FP4_FLAG_TIMEOUT.
__global__ void bounded_wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(b, 0, limit_ns)) atomicOr(status, FP4_FLAG_TIMEOUT);
  }
  __syncthreads();
}
}  // namespace

}  // namespace fp4

FP4_API const char* fp4_status_string(fp4_status s) {
  switch (s) {
    case FP4_OK: return "FP4_OK";
    case FP4_ERR_INVALID_ARG: return "FP4_ERR_INVALID_ARG";
    case FP4_ERR_SHAPE: return "FP4_ERR_SHAPE";
    case FP4_ERR_ALIGNMENT: return "FP4_ERR_ALIGNMENT";
    case FP4_ERR_WORKSPACE: return "FP4_ERR_WORKSPACE";
    case FP4_ERR_CAPACITY: return "FP4_ERR_CAPACITY";
    case FP4_ERR_TIMEOUT: return "FP4_ERR_TIMEOUT";
    case FP4_ERR_DEVICE_UNSUPPORTED: return "FP4_ERR_DEVICE_UNSUPPORTED";
    case FP4_ERR_CUDA: return "FP4_ERR_CUDA";
    case FP4_ERR_INTERNAL: return "FP4_ERR_INTERNAL";
  }
  return "FP4_ERR_UNKNOWN";
}

FP4_API int fp4_abi_version(void) { return 2; }   // 2: fp4_linear_wgrad_dge takes dw_type, dw_scale, dw_amax

FP4_API const char* fp4_last_cuda_error(void) { return fp4::last_cuda_error(); }

FP4_API fp4_status fp4_device_status(fp4_stream_t stream, uint32_t* flags_out) {
  fp4_status st = fp4::check_device(nullptr);
  if (st != FP4_OK) return st;
  uint32_t* word = fp4::status_word();
  uint32_t flags = 0;
  const uint32_t zero = 0;
  if (cudaMemcpyAsync(&flags, word, sizeof(flags), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemcpyAsync(word, &zero, sizeof(zero), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FP4_ERR_CUDA;
  if (flags_out) *flags_out = flags;
  if (flags & FP4_FLAG_TIMEOUT) return FP4_ERR_TIMEOUT;
  if (flags & FP4_FLAG_CAPACITY) return FP4_ERR_CAPACITY;
  if (flags & FP4_FLAG_INTERNAL) return FP4_ERR_INTERNAL;
  return FP4_OK;
}

FP4_API fp4_status fp4_selftest_bounded_wait(uint32_t timeout_us, fp4_stream_t stream) {
  if (timeout_us == 0 || timeout_us > 1000000u) return FP4_ERR_INVALID_ARG;
  fp4_status st = fp4::check_device(nullptr);
  if (st != FP4_OK) return st;
  fp4::bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(fp4::status_word(), uint64_t(timeout_us) * 1000ull);
  return fp4::launch_status();
}
