// Library runtime: the device error word, status strings, SM count, tensor-map encoding.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"

// One error word per device. A __device__ symbol: every GPU that loads the library holds it; no allocation.
static __device__ unsigned int g_mv_error_word[2];

unsigned int* mv_error_word() {
  static std::mutex mu;
  static unsigned int* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mv_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

int mv_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

bool mv_pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("MV_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

int mv_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

bool mv_set_smem_once(const void* func, int bytes, int* flags) {
  const int dev = mv_device();
  if (dev < 0 || dev >= 64) return false;
  if (flags[dev] >= bytes) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  flags[dev] = bytes;
  return true;
}

mv_status mv_last_launch(const char* what) {
  (void)what;
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MV_OK : MV_ERR_CUDA;
}

extern "C" mv_status mv_get_error(uint32_t* code) {
  unsigned int* w = mv_error_word();
  if (!w) return MV_ERR_CUDA;
  unsigned int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return MV_ERR_CUDA;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MV_ERR_CUDA;
  if (code) *code = v;
  if (v != 0) {
    unsigned int z[2] = {0, 0};
    if (cudaMemcpy(w, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return MV_ERR_CUDA;
    return MV_ERR_DEVICE;
  }
  return MV_OK;
}

namespace {

// The two bounded waits every kernel of the path relies on, run with a short limit on a counter and an mbarrier
// that nothing completes: the counter wait of the projection chain's phase boundaries and the mbarrier wait of
// the TMA / bulk-copy rings. Each must give up, report MV_DEVERR_TIMEOUT and let the kernel return.
__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t* out, unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  unsigned int* counter = reinterpret_cast<unsigned int*>(out + 2);  // nothing bumps it
  if (threadIdx.x == 0) {
    *counter = 0u;
    __threadfence();
    mbar_init(&bar, 1);  // count 1, and nothing arrives
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = mv_globaltimer();
    const bool c = wait_count(counter, 1u, limit_ns);
    const bool m = mbar_wait(&bar, 0u, limit_ns);
    const uint64_t t1 = mv_globaltimer();
    out[0] = c ? 1 : 0;
    out[1] = m ? 1 : 0;
    out[3] = (int32_t)min((uint64_t)0x7fffffff, (t1 - t0) / 1000u);  // microseconds both waits took
    if (!c || !m) mv_set_error_detail(err, 20, MV_DEVERR_TIMEOUT, (c ? 0u : 1u) | (m ? 0u : 2u));
  }
}

}  // namespace

extern "C" mv_status mv_selftest_wait_timeout(uint32_t limit_ns, int32_t* d_out, mv_stream stream) {
  if (!d_out || limit_ns < 1000u || limit_ns > 10000000u) return MV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_out) & 3) return MV_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, d_out, mv_error_word());
  return mv_last_launch("selftest_wait");
}

extern "C" mv_status mv_get_error_detail(uint32_t* detail) {
  unsigned int* w = mv_error_word();
  if (!w || !detail) return MV_ERR_INVALID_ARG;
  if (cudaMemcpy(detail, w + 1, sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess) return MV_ERR_CUDA;
  return MV_OK;
}

extern "C" const char* mv_status_string(mv_status s) {
  switch (s) {
    case MV_OK: return "ok";
    case MV_ERR_INVALID_ARG: return "invalid argument";
    case MV_ERR_SHAPE: return "unsupported or inconsistent shape";
    case MV_ERR_TREE: return "malformed tree";
    case MV_ERR_CAPACITY: return "capacity exceeded";
    case MV_ERR_CUDA: return "CUDA error";
    case MV_ERR_DEVICE: return "device error word set";
    case MV_ERR_UNSUPPORTED: return "unsupported";
  }
  return "unknown status";
}

bool mv_encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                    const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                    CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!encode) return false;
  cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  CUresult r = encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), (const cuuint64_t*)dims,
                      (const cuuint64_t*)strides_bytes, (const cuuint32_t*)box, elem_strides,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
