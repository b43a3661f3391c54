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
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
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
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
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

}  // namespace eagle

extern "C" {

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
