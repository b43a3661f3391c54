// Lossless tree verification (greedy longest accepted path; multi-round
// speculative sampling with deterministic top-k proposals).
//
// Source: "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty"
// (paper summary), section "Verification Phase: Multi-Round Speculative Sampling
// on Trees" (the paper's Algorithm 1); "EAGLE-3: Scaling up Inference
// Acceleration of Large Language Models via Training-Time Test", "Stage 2:
// Verification".
//
// Two kernels:
//   rowstats : one CTA per (row, request): max and sum-exp of z/T (stochastic)
//              or the argmax (greedy without a caller-provided argmax).
//   walk     : one CTA per request: thread 0 walks the tree from the seed
//              using the row statistics and the target logit of each child's
//              token; then the whole CTA runs the exponential race over the
//              stop row for the bonus token.
#include <math.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int kStatThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kMaxVerifyRows = 1024;
constexpr float kLog2e = 1.4426950408889634f;

struct RowStat {
  float m;  // max_v z/T
  float s;  // sum_v exp(z/T - m)
};

__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (better(v2, i2, v, i)) {
    v = v2;
    i = i2;
  }
}

__global__ void __launch_bounds__(kStatThreads) verify_rowstats_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ n_rows, int R, int V,
    float inv_t, int want_argmax, RowStat* __restrict__ stats, int32_t* __restrict__ amax,
    int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x % R, b = blockIdx.x / R;
  const int n = n_rows ? n_rows[b] : R;
  if (r >= n || r >= R) return;
  const float* z = logits + ((size_t)b * R + r) * V;
  __shared__ float sh_v[kStatThreads / 32];
  __shared__ float sh_s[kStatThreads / 32];
  __shared__ int sh_i[kStatThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  bool nan_seen = false;
  if (want_argmax) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int v = threadIdx.x; v < V; v += kStatThreads) {
      const float x = z[v];
      nan_seen |= isnan(x);
      argmax_merge(bv, bi, x, v);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(bv, bi, ov, oi);
    }
    if (lane == 0) {
      sh_v[warp] = bv;
      sh_i[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kStatThreads / 32; ++w) argmax_merge(bv, bi, sh_v[w], sh_i[w]);
      amax[(size_t)b * R + r] = bi;
    }
  } else {
    // online max / sum-exp of y = z / T
    float m = -INFINITY, s = 0.f;
    for (int v = threadIdx.x; v < V; v += kStatThreads) {
      const float y = z[v] * inv_t;
      nan_seen |= isnan(y);
      if (y > m) {
        s = s * exp2f((m - y) * kLog2e) + 1.f;
        m = y;
      } else {
        s += exp2f((y - m) * kLog2e);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, o);
      const float os = __shfl_xor_sync(0xffffffffu, s, o);
      const float nm = fmaxf(m, om);
      s = (m == -INFINITY ? 0.f : s * exp2f((m - nm) * kLog2e)) +
          (om == -INFINITY ? 0.f : os * exp2f((om - nm) * kLog2e));
      m = nm;
    }
    if (lane == 0) {
      sh_v[warp] = m;
      sh_s[warp] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float M = sh_v[0];
      for (int w = 1; w < kStatThreads / 32; ++w) M = fmaxf(M, sh_v[w]);
      float S = 0.f;
      for (int w = 0; w < kStatThreads / 32; ++w)
        if (sh_v[w] != -INFINITY) S += sh_s[w] * exp2f((sh_v[w] - M) * kLog2e);
      stats[(size_t)b * R + r] = RowStat{M, S};
    }
  }
  if (nan_seen) set_status(dev_status, EAGLE_ERR_NONFINITE);
}

__global__ void __launch_bounds__(kWalkThreads) verify_walk_kernel(
    int R, int V, const int32_t* __restrict__ parent_row, const int32_t* __restrict__ token,
    const int32_t* __restrict__ n_rows, const float* __restrict__ logits,
    const int32_t* __restrict__ target_argmax, const RowStat* __restrict__ stats,
    const int32_t* __restrict__ ws_argmax, int greedy, float inv_t, uint32_t key0, uint32_t key1,
    uint32_t ctr2_accept, uint32_t ctr3, const float* __restrict__ uniforms_override,
    int max_depth, int32_t* __restrict__ accept_len, int32_t* __restrict__ path_rows,
    int32_t* __restrict__ out_tokens, int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  __shared__ int s_parent[kMaxVerifyRows];
  __shared__ int s_token[kMaxVerifyRows];
  __shared__ int s_path[65];
  __shared__ int s_excl[kMaxVerifyRows];
  __shared__ int s_nexcl, s_stop, s_plen, s_bad, s_bonus;
  __shared__ float s_rv[kWalkThreads / 32];
  __shared__ int s_ri[kWalkThreads / 32];

  const int n = n_rows ? n_rows[b] : R;
  if (threadIdx.x == 0) {
    s_bad = (n < 1 || n > R) ? 1 : 0;
    s_nexcl = 0;
  }
  __syncthreads();
  const int nn = s_bad ? 1 : n;
  for (int i = threadIdx.x; i < nn; i += kWalkThreads) {
    const int p = parent_row[(size_t)b * R + i];
    const int t = token[(size_t)b * R + i];
    s_parent[i] = p;
    s_token[i] = t;
    const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i && t >= 0 && t < V);
    if (!ok) atomicExch(&s_bad, 1);
  }
  __syncthreads();

  if (threadIdx.x == 0) {
    int plen = 1, cur = 0, bad = s_bad;
    s_path[0] = 0;
    while (!bad) {
      int accepted = -1;
      if (greedy) {
        const int a = target_argmax ? target_argmax[(size_t)b * R + cur]
                                    : ws_argmax[(size_t)b * R + cur];
        for (int c = cur + 1; c < nn; ++c)
          if (s_parent[c] == cur && s_token[c] == a) {
            accepted = c;
            break;
          }
      } else {
        const RowStat st = stats[(size_t)b * R + cur];
        const float* z = logits + ((size_t)b * R + cur) * V;
        float rem = 1.f;  // probability mass not yet rejected
        s_nexcl = 0;
        for (int c = cur + 1; c < nn; ++c) {
          if (s_parent[c] != cur) continue;
          const int t = s_token[c];
          bool dup = false;
          for (int e = 0; e < s_nexcl; ++e) dup |= (s_excl[e] == t);
          const float pt = dup ? 0.f : exp2f((z[t] * inv_t - st.m) * kLog2e) / st.s;
          const float ratio = pt / rem;
          float u;
          if (uniforms_override) {
            u = uniforms_override[(size_t)b * R + c];
          } else {
            const uint4 w = philox4x32_10(make_uint4((uint32_t)c, (uint32_t)b, ctr2_accept, ctr3),
                                          key0, key1);
            u = bits_to_uniform(w.x);
          }
          if (u < ratio) {
            accepted = c;
            break;
          }
          if (!dup && rem - pt > 0.f) {
            rem -= pt;
            s_excl[s_nexcl++] = t;
          }
        }
      }
      if (accepted < 0) break;
      if (plen > max_depth) {
        bad = 2;
        break;
      }
      s_path[plen++] = accepted;
      cur = accepted;
    }
    s_stop = cur;
    s_plen = plen;
    if (bad) s_bad = bad;
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      set_status(dev_status, EAGLE_ERR_BAD_TREE);
      accept_len[b] = 0;
    }
    for (int i = threadIdx.x; i <= max_depth; i += kWalkThreads) {
      path_rows[(size_t)b * (max_depth + 1) + i] = (i == 0) ? 0 : -1;
      out_tokens[(size_t)b * (max_depth + 1) + i] = -1;
    }
    return;
  }

  const int stop = s_stop;
  if (greedy) {
    if (threadIdx.x == 0)
      s_bonus = target_argmax ? target_argmax[(size_t)b * R + stop] : ws_argmax[(size_t)b * R + stop];
  } else {
    // exponential race over the ids not rejected at the stop row:
    // bonus = argmax_y z_y/T - log(-log u_y)  (ties to the lower id)
    const float* z = logits + ((size_t)b * R + stop) * V;
    const int nex = s_nexcl;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    bool nan_seen = false;
    const uint32_t ctr2_race = ctr2_accept + 1u;
    for (int g = threadIdx.x; g * 4 < V; g += kWalkThreads) {
      const uint4 w = philox4x32_10(make_uint4((uint32_t)g, (uint32_t)b, ctr2_race, ctr3), key0, key1);
      const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int y = g * 4 + j;
        if (y >= V) break;
        bool ex = false;
        for (int e = 0; e < nex; ++e) ex |= (s_excl[e] == y);
        if (ex) continue;
        const float zy = z[y];
        nan_seen |= isnan(zy);
        const float u = bits_to_uniform(words[j]);
        const float key = zy * inv_t - logf(-logf(u));
        argmax_merge(bv, bi, key, y);
      }
    }
    if (nan_seen) set_status(dev_status, EAGLE_ERR_NONFINITE);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(bv, bi, ov, oi);
    }
    if ((threadIdx.x & 31) == 0) {
      s_rv[threadIdx.x >> 5] = bv;
      s_ri[threadIdx.x >> 5] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kWalkThreads / 32; ++w) argmax_merge(bv, bi, s_rv[w], s_ri[w]);
      s_bonus = bi;
    }
  }
  __syncthreads();
  const int plen = s_plen;
  for (int i = threadIdx.x; i <= max_depth; i += kWalkThreads) {
    const size_t o = (size_t)b * (max_depth + 1) + i;
    path_rows[o] = i < plen ? s_path[i] : -1;
    out_tokens[o] = i + 1 < plen ? s_token[s_path[i + 1]] : (i + 1 == plen ? s_bonus : -1);
  }
  if (threadIdx.x == 0) accept_len[b] = plen - 1;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_verify_workspace_size(int B, int R, int V) {
  (void)V;
  if (B <= 0 || R <= 0) return 0;
  return round_up((size_t)B * R * sizeof(RowStat), 256) + round_up((size_t)B * R * 4, 256) + 512;
}

extern "C" int eagle_tree_verify(int B, int R, int V, const int32_t* parent_row,
                                 const int32_t* token, const int32_t* n_rows,
                                 const float* target_logits, const int32_t* target_argmax,
                                 const float* draft_logits, float temperature, int proposal_mode,
                                 uint64_t seed, uint64_t offset, const float* uniforms_override,
                                 int max_depth, int32_t* accept_len, int32_t* path_rows,
                                 int32_t* out_tokens, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, void* stream) {
  (void)draft_logits;
  if (B <= 0 || R <= 0 || V < 2 || max_depth < 0) return EAGLE_ERR_INVALID_ARG;
  if (!parent_row || !token || !accept_len || !path_rows || !out_tokens) return EAGLE_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || isinf(temperature)) return EAGLE_ERR_INVALID_ARG;
  if (proposal_mode != EAGLE_PROPOSAL_DETERMINISTIC && proposal_mode != EAGLE_PROPOSAL_SAMPLED)
    return EAGLE_ERR_INVALID_ARG;
  const bool greedy = temperature == 0.f;
  if (proposal_mode == EAGLE_PROPOSAL_SAMPLED) return greedy ? EAGLE_ERR_INVALID_ARG : EAGLE_ERR_UNSUPPORTED;
  if (greedy && !target_logits && !target_argmax) return EAGLE_ERR_INVALID_ARG;
  if (!greedy && !target_logits) return EAGLE_ERR_INVALID_ARG;
  if (R > kMaxVerifyRows || max_depth > 64) return EAGLE_ERR_UNSUPPORTED;
  if ((offset >> 63) != 0) return EAGLE_ERR_INVALID_ARG;
  const bool need_stats = !greedy || !target_argmax;
  if (need_stats && (!ws || ws_bytes < eagle_tree_verify_workspace_size(B, R, V)))
    return EAGLE_ERR_WORKSPACE;
  if ((long long)B * R > 2147483647LL) return EAGLE_ERR_UNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* cur = static_cast<char*>(ws);
  RowStat* stats = nullptr;
  int32_t* amax = nullptr;
  if (need_stats) {
    stats = static_cast<RowStat*>(ws_carve(cur, (size_t)B * R * sizeof(RowStat)));
    amax = static_cast<int32_t*>(ws_carve(cur, (size_t)B * R * 4));
  }
  const float inv_t = greedy ? 0.f : 1.f / temperature;
  if (need_stats) {
    launch(verify_rowstats_kernel, (unsigned)(B * R), kStatThreads, 0, s,
        target_logits, n_rows, R, V, inv_t, greedy ? 1 : 0, stats, amax, dev_status);
    note_launch();
  }
  const uint32_t off_hi = (uint32_t)(offset >> 32), off_lo = (uint32_t)offset;
  launch(verify_walk_kernel, B, kWalkThreads, 0, s,
      R, V, parent_row, token, n_rows, target_logits, target_argmax, stats, amax, greedy ? 1 : 0,
      inv_t, (uint32_t)seed, (uint32_t)(seed >> 32), 2u * off_hi, off_lo, uniforms_override,
      max_depth, accept_len, path_rows, out_tokens, dev_status);
  note_launch();
  return last_launch_status();
}

// ---------------------------------------------------------------------------
// eagle_tree_verify_noalloc: the same verification for callers that cannot
// allocate device memory (for instance a plugin whose host framework owns
// every device allocation and hands it only the input and output tensors, or
// a latency-critical loop that may not call cudaMalloc because of its implicit
// device-wide synchronisation).  The row statistics that eagle_tree_verify
// keeps in the caller's workspace live here in one library-owned buffer of
// fixed capacity, allocated statically when the library is loaded.
namespace eagle {
namespace {

constexpr int kNoAllocMaxRows = 65536;  // B * R rows of statistics
constexpr size_t kNoAllocScratchBytes =
    ((size_t)kNoAllocMaxRows * sizeof(RowStat) + 255) / 256 * 256 + (size_t)kNoAllocMaxRows * 4;

// One copy per GPU that loads the library, kept until the process exits.
// Every call on a device shares it: two calls whose kernels overlap on that
// device (for example on two streams) race on it.  Nothing in it needs to
// start at zero: every statistic is written before it is read.
static __device__ __align__(256) unsigned char g_verify_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kNoAllocMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_verify_scratch on the current device.  In host code the
// symbol's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress once per device, with that device current.
void* noalloc_scratch(eagle_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    *st = EAGLE_ERR_CUDA;
    return nullptr;
  }
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) {
      *st = EAGLE_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace
}  // namespace eagle

extern "C" int eagle_tree_verify_noalloc(int B, int R, int V, const int32_t* parent_row,
                                         const int32_t* token, const int32_t* n_rows,
                                         const float* target_logits, const int32_t* target_argmax,
                                         const float* draft_logits, float temperature,
                                         int proposal_mode, uint64_t seed, uint64_t offset,
                                         const float* uniforms_override, int max_depth,
                                         int32_t* accept_len, int32_t* path_rows,
                                         int32_t* out_tokens, int32_t* dev_status, void* stream) {
  (void)draft_logits;
  if (B <= 0 || R <= 0 || V < 2 || max_depth < 0) return EAGLE_ERR_INVALID_ARG;
  if (!parent_row || !token || !accept_len || !path_rows || !out_tokens) return EAGLE_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || isinf(temperature)) return EAGLE_ERR_INVALID_ARG;
  if (proposal_mode != EAGLE_PROPOSAL_DETERMINISTIC && proposal_mode != EAGLE_PROPOSAL_SAMPLED)
    return EAGLE_ERR_INVALID_ARG;
  const bool greedy = temperature == 0.f;
  if (proposal_mode == EAGLE_PROPOSAL_SAMPLED) return greedy ? EAGLE_ERR_INVALID_ARG : EAGLE_ERR_UNSUPPORTED;
  if (greedy && !target_logits && !target_argmax) return EAGLE_ERR_INVALID_ARG;
  if (!greedy && !target_logits) return EAGLE_ERR_INVALID_ARG;
  if (R > kMaxVerifyRows || max_depth > 64) return EAGLE_ERR_UNSUPPORTED;
  if ((offset >> 63) != 0) return EAGLE_ERR_INVALID_ARG;
  // the built-in scratch holds statistics for at most kNoAllocMaxRows rows
  if ((long long)B * R > kNoAllocMaxRows) return EAGLE_ERR_WORKSPACE;
  const bool need_stats = !greedy || !target_argmax;
  RowStat* stats = nullptr;
  int32_t* amax = nullptr;
  if (need_stats) {
    eagle_status st = EAGLE_OK;
    char* base = static_cast<char*>(noalloc_scratch(&st));
    if (!base) return st;
    stats = reinterpret_cast<RowStat*>(base);
    amax = reinterpret_cast<int32_t*>(base + ((size_t)kNoAllocMaxRows * sizeof(RowStat) + 255) / 256 * 256);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float inv_t = greedy ? 0.f : 1.f / temperature;
  if (need_stats) {
    launch(verify_rowstats_kernel, (unsigned)(B * R), kStatThreads, 0, s,
        target_logits, n_rows, R, V, inv_t, greedy ? 1 : 0, stats, amax, dev_status);
    note_launch();
  }
  const uint32_t off_hi = (uint32_t)(offset >> 32), off_lo = (uint32_t)offset;
  launch(verify_walk_kernel, B, kWalkThreads, 0, s,
      R, V, parent_row, token, n_rows, target_logits, target_argmax, stats, amax, greedy ? 1 : 0,
      inv_t, (uint32_t)seed, (uint32_t)(seed >> 32), 2u * off_hi, off_lo, uniforms_override,
      max_depth, accept_len, path_rows, out_tokens, dev_status);
  note_launch();
  return last_launch_status();
}
