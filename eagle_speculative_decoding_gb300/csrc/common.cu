// Host-side helpers and the status/launch-count entry points.
#include <atomic>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"

namespace eagle {

namespace {
std::atomic<uint64_t> g_launches{0};
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// cuTensorMapEncodeTiled through the runtime's entry-point query (no -lcuda)
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}
}  // namespace

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int v = g_sm_count[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  g_sm_count[dev].store(v, std::memory_order_relaxed);
  return v;
}

eagle_status last_launch_status() {
  return cudaGetLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void* ws_carve(char*& cursor, size_t bytes) {
  uintptr_t p = reinterpret_cast<uintptr_t>(cursor);
  p = (p + 255u) & ~uintptr_t(255u);
  cursor = reinterpret_cast<char*>(p + bytes);
  return reinterpret_cast<void*>(p);
}

bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t rows,
                  uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  if (!encoder()) return false;
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  if (!encoder()) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
// Self-test of the bounded wait every kernel uses: thread 0 waits on an
// mbarrier that nothing ever arrives on, with a limit of limit_ns, and must
// give up with EAGLE_ERR_TIMEOUT; thread 32 waits on a second such barrier
// with the ordinary 2 s limit and must end early, through the abort flag the
// first waiter raises (status[1] = 1).
__global__ void __launch_bounds__(64) wait_selftest_kernel(unsigned long long limit_ns,
                                                           int32_t* status) {
  __shared__ uint64_t never_a, never_b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&never_a), 1);
    mbar_init(smem_u32(&never_b), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(smem_u32(&never_a), 0, &abort_flag, limit_ns)) set_status(status, EAGLE_ERR_TIMEOUT);
  } else if (threadIdx.x == 32) {
    const unsigned long long t0 = globaltimer_ns();
    const bool done = mbar_wait(smem_u32(&never_b), 0, &abort_flag);
    if (!done && abort_flag && globaltimer_ns() - t0 < kWaitLimitNs / 2) status[1] = 1;
  }
  __syncthreads();
}
}  // namespace

}  // namespace eagle

extern "C" {

int eagle_selftest_wait_timeout(unsigned int limit_us, int32_t* dev_status, void* stream) {
  if (!dev_status || limit_us == 0 || limit_us > 1000000u) return EAGLE_ERR_INVALID_ARG;
  eagle::launch(eagle::wait_selftest_kernel, 1, 64, 0, static_cast<cudaStream_t>(stream),
                (unsigned long long)limit_us * 1000ull, dev_status);
  eagle::note_launch();
  return eagle::last_launch_status();
}


const char* eagle_status_string(int status) {
  switch (status) {
    case EAGLE_OK: return "EAGLE_OK";
    case EAGLE_ERR_INVALID_ARG: return "EAGLE_ERR_INVALID_ARG";
    case EAGLE_ERR_UNSUPPORTED: return "EAGLE_ERR_UNSUPPORTED";
    case EAGLE_ERR_WORKSPACE: return "EAGLE_ERR_WORKSPACE";
    case EAGLE_ERR_CUDA: return "EAGLE_ERR_CUDA";
    case EAGLE_ERR_BAD_TREE: return "EAGLE_ERR_BAD_TREE";
    case EAGLE_ERR_BAD_KV: return "EAGLE_ERR_BAD_KV";
    case EAGLE_ERR_NONFINITE: return "EAGLE_ERR_NONFINITE";
    case EAGLE_ERR_TIMEOUT: return "EAGLE_ERR_TIMEOUT";
    default: return "EAGLE_ERR_UNKNOWN";
  }
}

int eagle_read_status(const int32_t* dev_status, void* stream, int32_t* host_status) {
  if (!dev_status || !host_status) return EAGLE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_status, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return EAGLE_ERR_CUDA;
  return *host_status;
}

uint64_t eagle_launch_count(void) { return eagle::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
