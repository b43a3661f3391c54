// EAGLE-2 dynamic draft-tree expansion, global rerank and flatten.
//
// Source: "M7.5 - EAGLE Feature Drafting: Uncertainty, Dynamic Trees, HASS, and
// EAGLE-3", sections 0x06A "Path Value Derivation" (log V(u) = sum over the
// path of log max(c_j, eps), eps = 1e-12; a child never outranks its parent),
// 0x06B "Expansion And Reranking" (expand the top-width nodes of the latest
// layer by (-log V, depth, node_id); rerank all non-seed nodes by the same key
// and keep the verification budget) and 0x05C "Target Verification" (flatten
// with ancestry-aware positions and a tree mask).
//
// One CTA per request (the step body is expand_step_block, expand_step.cuh).
// A step ranks its (at most width*k) new nodes by counting smaller 64-bit
// order-preserving keys (unique: node ids differ); the final rerank ranks or
// bitonic-sorts the keys of all stored nodes.  log V is accumulated in fp32
// with one correctly rounded addition per level.
#include <math.h>

#include "common.cuh"
#include "expand_step.cuh"
#include "lm_merge.cuh"

namespace eagle {
namespace {

constexpr int kExpandThreads = 512;
constexpr int kMaxCand = 1024;  // width * k
constexpr int kMaxNodes = kExpandMaxNodes;

// One expansion step per CTA (request blockIdx.x); see expand_step_block.
// The next kernel (an LM head that prefetches its weights) is let in only at
// the end: its prefetch would otherwise queue ahead of this kernel's few
// latency-bound loads.
template <bool MERGE>
__global__ void __launch_bounds__(kExpandThreads) expand_step_kernel(const ExpandArgs a, const LmPartials lp,
                                                                     int stage_rows) {
  __shared__ ExpandSmem<kMaxCand> sm;
  extern __shared__ __align__(16) unsigned char stage[];
  pdl_wait();
  expand_step_block<kExpandThreads, kMaxCand, MERGE>(a, blockIdx.x, sm, lp, stage, stage_rows);
  pdl_trigger();
}

__global__ void __launch_bounds__(kExpandThreads) expand_finalize_kernel(
    int max_nodes, int budget, int R, const int32_t* __restrict__ node_parent,
    const int32_t* __restrict__ node_token, const float* __restrict__ node_logv,
    const int32_t* __restrict__ node_depth, const int32_t* __restrict__ node_count,
    const int32_t* __restrict__ ctx_lens, int32_t* __restrict__ token,
    int32_t* __restrict__ parent_row, int32_t* __restrict__ depth, uint64_t* __restrict__ mask,
    int32_t* __restrict__ node_id, int32_t* __restrict__ position, int32_t* __restrict__ n_rows,
    int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int32_t* np_ = node_parent + (size_t)b * max_nodes;
  const int32_t* nt_ = node_token + (size_t)b * max_nodes;
  const float* nv_ = node_logv + (size_t)b * max_nodes;
  const int32_t* nd_ = node_depth + (size_t)b * max_nodes;
  __shared__ unsigned long long s_key[kMaxNodes];
  __shared__ unsigned long long s_sel[64];  // the selected nodes' keys, rank order
  __shared__ int s_row_of[kMaxNodes];
  __shared__ int s_prow[64];
  __shared__ int s_bad;
  // the stored nodes' log V and depth are read beside the node count instead
  // of after it (every slot of the store; those past the count go unused)
  constexpr int kPer = kMaxNodes / kExpandThreads;
  float lv[kPer];
  int dp[kPer];
#pragma unroll
  for (int h = 0; h < kPer; ++h) {
    const int i = h * kExpandThreads + threadIdx.x;
    if (i + 1 < max_nodes) {
      lv[h] = nv_[i + 1];
      dp[h] = nd_[i + 1];
    }
  }
  int count = node_count[b];
  count = count < 1 ? 1 : (count > max_nodes ? max_nodes : count);
  const int n = count - 1;  // candidates (the seed excluded)
  const int nsel = min(budget, n);
  const int ctx = ctx_lens ? ctx_lens[b] : 0;
  int P = 1;
  while (P < n) P <<= 1;
#pragma unroll
  for (int h = 0; h < kPer; ++h) {
    const int i = h * kExpandThreads + threadIdx.x;
    if (i < P) s_key[i] = i < n ? node_key(lv[h], dp[h], i + 1) : ~0ull;
  }
  for (int i = threadIdx.x; i < count; i += kExpandThreads) s_row_of[i] = -1;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if (n > 64 && P <= kExpandThreads) {
    // one key per thread: each warp sorts its 32 keys (shuffle bitonic),
    // and a key's rank is its place in its warp plus, for every other warp,
    // how many of that warp's sorted keys are smaller (binary search); keys
    // of nodes are unique, and the padding (~0) sorts after all of them.
    // (Measured: 8.65 -> 7.73 µs per call with 510 candidates; with a few
    // dozen, counting is cheaper than the sort's barriers.)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool mine = (int)threadIdx.x < P;
    unsigned long long key = mine ? s_key[threadIdx.x] : ~0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, stride);
        const bool keep_min = ((lane & stride) == 0) == ((lane & size) == 0 || size == 32);
        key = keep_min ? (other < key ? other : key) : (other > key ? other : key);
      }
    }
    __syncthreads();  // every key is in registers before the sorted runs overwrite them
    if (mine) s_key[threadIdx.x] = key;
    __syncthreads();
    if (mine && key != ~0ull) {
      int rank = lane;
      for (int w = 0; w * 32 < P; ++w) {
        if (w == warp) continue;
        const unsigned long long* run = s_key + w * 32;
        int lo = 0, hi = 32;  // keys of run w below `key`: the first index whose key is >= it
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (run[mid] < key)
            lo = mid + 1;
          else
            hi = mid;
        }
        rank += lo;
      }
      if (rank < nsel) s_sel[rank] = key;
    }
  } else if (n <= 1024) {
    // the rank of each candidate = how many keys are smaller (keys are
    // unique); branch-free, every thread reads the same key at a time
    for (int i = threadIdx.x; i < n; i += kExpandThreads) {
      const unsigned long long mk = s_key[i];
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < n; ++j) rank += s_key[j] < mk ? 1 : 0;
      if (rank < nsel) s_sel[rank] = mk;
    }
  } else {
    // bitonic sort of the keys (ascending)
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < P / 2; i += kExpandThreads) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const unsigned long long a = s_key[lo], c = s_key[hi];
          if ((a > c) == up) {
            s_key[lo] = c;
            s_key[hi] = a;
          }
        }
        __syncthreads();
      }
    }
    for (int r = threadIdx.x; r < nsel; r += kExpandThreads) s_sel[r] = s_key[r];
  }
  __syncthreads();
  for (int r = 1 + threadIdx.x; r <= nsel; r += kExpandThreads)
    s_row_of[(int)(s_sel[r - 1] & 0xFFFFu)] = r;
  if (threadIdx.x == 0) s_row_of[0] = 0;
  __syncthreads();
  // parent rows (a parent always precedes its child in key order)
  for (int r = threadIdx.x; r < 64 && r <= nsel; r += kExpandThreads) {
    if (r == 0) {
      s_prow[0] = -1;
      continue;
    }
    const int nd = (int)(s_sel[r - 1] & 0xFFFFu);
    const int p = np_[nd];
    int pr = (p >= 0 && p < count) ? s_row_of[p] : -1;
    if (pr < 0 || pr >= r) {
      atomicExch(&s_bad, 1);
      pr = 0;
    }
    s_prow[r] = pr;
  }
  __syncthreads();
  const size_t o = (size_t)b * R;
  for (int r = threadIdx.x; r < R; r += kExpandThreads) {
    if (r <= nsel) {
      const int nd = r == 0 ? 0 : (int)(s_sel[r - 1] & 0xFFFFu);
      uint64_t m = 1ull << r;
      int j = r, guard = 0;
      while (j != 0 && guard++ < 64) {  // ancestry bits by walking the parent rows
        j = s_prow[j];
        m |= 1ull << j;
      }
      const int dd = r == 0 ? 0 : nd_[nd];
      token[o + r] = nt_[nd];
      parent_row[o + r] = s_prow[r];
      depth[o + r] = dd;
      mask[o + r] = m;
      node_id[o + r] = nd;
      position[o + r] = ctx + dd;
    } else {
      token[o + r] = -1;
      parent_row[o + r] = -1;
      depth[o + r] = 0;
      mask[o + r] = 1ull << r;
      node_id[o + r] = -1;
      position[o + r] = ctx;
    }
  }
  if (threadIdx.x == 0) {
    n_rows[b] = nsel + 1;
    if (s_bad) set_status(dev_status, EAGLE_ERR_BAD_TREE);
  }
}

}  // namespace
}  // namespace eagle

using namespace eagle;

namespace {
// Dynamic shared memory the merging expansion stages partial lists in.
constexpr size_t kStageBytes = 192 * 1024;

int expand_launch(int B, int step, int width, int k, int max_nodes, const int32_t* fanout,
                  const int32_t* cand_ids, const float* cand_logprobs, const LmPartials* lp,
                  const int32_t* root_token, int32_t* node_parent, int32_t* node_token, float* node_logv,
                  int32_t* node_depth, int32_t* node_count, int32_t* frontier, int32_t* n_frontier,
                  int32_t* dev_status, void* stream) {
  if (B <= 0 || step < 0 || width < 1 || k < 1 || max_nodes < 1) return EAGLE_ERR_INVALID_ARG;
  if ((!lp && (!cand_ids || !cand_logprobs)) || !node_parent || !node_token || !node_logv || !node_depth ||
      !node_count || !frontier || !n_frontier)
    return EAGLE_ERR_INVALID_ARG;
  if (step == 0 && !root_token) return EAGLE_ERR_INVALID_ARG;
  const int chk = expand_check(B, step, width, k, max_nodes, kMaxCand);
  if (chk != EAGLE_OK) return chk;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ExpandArgs a{step,      width,       k,          max_nodes,  cand_ids,   cand_logprobs, root_token,
                     node_parent, node_token, node_logv, node_depth, node_count, frontier,      n_frontier,
                     fanout,    dev_status};
  if (lp) {
    const size_t row_bytes = ((size_t)lp->cpg * k * 8 + (size_t)lp->cpg * 4 + 15) / 16 * 16;
    const int P = step == 0 ? 1 : width;
    int rows = (int)(kStageBytes / row_bytes);
    rows = rows < kExpandThreads / 32 ? rows : kExpandThreads / 32;
    rows = rows < P ? rows : P;
    if (rows < 1) return EAGLE_ERR_UNSUPPORTED;
    const size_t smem = (size_t)rows * row_bytes;
    cudaFuncSetAttribute(expand_step_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch(expand_step_kernel<true>, B, kExpandThreads, smem, s, a, *lp, rows);
  } else {
    launch(expand_step_kernel<false>, B, kExpandThreads, 0, s, a, LmPartials{}, 0);
  }
  note_launch();
  return last_launch_status();
}
}  // namespace

extern "C" int eagle_tree_expand(int B, int step, int width, int k, int max_nodes,
                                 const int32_t* cand_ids, const float* cand_logprobs,
                                 const int32_t* root_token, int32_t* node_parent,
                                 int32_t* node_token, float* node_logv, int32_t* node_depth,
                                 int32_t* node_count, int32_t* frontier, int32_t* n_frontier,
                                 int32_t* dev_status, void* stream) {
  return expand_launch(B, step, width, k, max_nodes, nullptr, cand_ids, cand_logprobs, nullptr, root_token,
                       node_parent, node_token, node_logv, node_depth, node_count, frontier, n_frontier,
                       dev_status, stream);
}

extern "C" int eagle_tree_expand_lmhead(int B, int step, int width, int k, int max_nodes,
                                        const void* lm_ws, size_t lm_ws_bytes, int d, int V,
                                        float temperature, int dtype, const int32_t* root_token,
                                        int32_t* node_parent, int32_t* node_token, float* node_logv,
                                        int32_t* node_depth, int32_t* node_count, int32_t* frontier,
                                        int32_t* n_frontier, int32_t* dev_status, void* stream) {
  if (B <= 0 || width < 1 || step < 0) return EAGLE_ERR_INVALID_ARG;
  const long long M = (long long)B * (step == 0 ? 1 : width);
  if (M > 2048) return EAGLE_ERR_UNSUPPORTED;
  LmPartials lp;
  if (!lm_partials_view(const_cast<void*>(lm_ws), lm_ws_bytes, (int)M, d, V, k, dtype, temperature, &lp))
    return lm_ws ? EAGLE_ERR_WORKSPACE : EAGLE_ERR_INVALID_ARG;
  return expand_launch(B, step, width, k, max_nodes, nullptr, nullptr, nullptr, &lp, root_token, node_parent,
                       node_token, node_logv, node_depth, node_count, frontier, n_frontier, dev_status,
                       stream);
}

extern "C" int eagle_tree_expand_static(int B, int step, int width, int k, int max_nodes,
                                        const int32_t* fanout, const int32_t* cand_ids,
                                        const float* cand_logprobs, const int32_t* root_token,
                                        int32_t* node_parent, int32_t* node_token, float* node_logv,
                                        int32_t* node_depth, int32_t* node_count, int32_t* frontier,
                                        int32_t* n_frontier, int32_t* dev_status, void* stream) {
  if (!fanout) return EAGLE_ERR_INVALID_ARG;
  return expand_launch(B, step, width, k, max_nodes, fanout, cand_ids, cand_logprobs, nullptr, root_token,
                       node_parent, node_token, node_logv, node_depth, node_count, frontier, n_frontier,
                       dev_status, stream);
}

extern "C" int eagle_tree_expand_finalize(int B, int max_nodes, int budget, int R,
                                          const int32_t* node_parent, const int32_t* node_token,
                                          const float* node_logv, const int32_t* node_depth,
                                          const int32_t* node_count, const int32_t* ctx_lens,
                                          int32_t* token, int32_t* parent_row, int32_t* depth,
                                          uint64_t* mask, int32_t* node_id, int32_t* position,
                                          int32_t* n_rows, int32_t* dev_status, void* stream) {
  if (B <= 0 || max_nodes < 1 || budget < 0 || R < 1) return EAGLE_ERR_INVALID_ARG;
  if (!node_parent || !node_token || !node_logv || !node_depth || !node_count || !token ||
      !parent_row || !depth || !mask || !node_id || !position || !n_rows)
    return EAGLE_ERR_INVALID_ARG;
  if (R > 64 || max_nodes > kMaxNodes || B > 65535) return EAGLE_ERR_UNSUPPORTED;
  if (R < 1 + budget) return EAGLE_ERR_INVALID_ARG;
  launch(expand_finalize_kernel, B, kExpandThreads, 0, static_cast<cudaStream_t>(stream),
      max_nodes, budget, R, node_parent, node_token, node_logv, node_depth, node_count, ctx_lens,
      token, parent_row, depth, mask, node_id, position, n_rows, dev_status);
  note_launch();
  return last_launch_status();
}
