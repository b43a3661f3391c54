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
// One CTA per request.  A step ranks its (at most width*k) new nodes by
// counting smaller keys (keys are unique: node ids differ); the final rerank
// bitonic-sorts 64-bit order-preserving keys of all stored nodes.  log V is
// accumulated in fp32 with one correctly rounded addition per level.
#include <math.h>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int kExpandThreads = 512;
constexpr int kMaxCand = 1024;      // width * k
constexpr int kMaxNodes = 2048;
// log(1e-12) rounded to fp32: the ranking floor of a zero confidence.
constexpr float kLogEps = -27.631021115928547f;
constexpr float kMassTol = 1e-4f;

// key(a) < key(b): larger log V first, then shallower, then smaller node id.
__device__ __forceinline__ bool key_less(float va, int da, int ia, float vb, int db, int ib) {
  if (va != vb) return va > vb;
  if (da != db) return da < db;
  return ia < ib;
}

// Order-preserving 64-bit sort key of a node: ascending key = descending
// log V, then ascending depth, then ascending node id.
__device__ __forceinline__ unsigned long long node_key(float v, int d, int id) {
  uint32_t f = __float_as_uint(v);
  f = (f & 0x80000000u) ? ~f : (f | 0x80000000u);  // ascending as unsigned
  return ((unsigned long long)(~f) << 32) | ((unsigned long long)(uint32_t)d << 16) |
         (unsigned long long)(uint32_t)id;
}

// Exclusive prefix sum of 0/1 flags over n <= kMaxCand entries (block-wide).
__device__ __forceinline__ int block_exclusive_scan(const int* flags, int* out, int n) {
  __shared__ int s_warp[kExpandThreads / 32 * 2];
  __shared__ int s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kW = kExpandThreads / 32;
  int pref[2], v[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = h * kExpandThreads + threadIdx.x;
    v[h] = t < n ? flags[t] : 0;
    const unsigned bal = __ballot_sync(0xffffffffu, v[h]);
    pref[h] = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) s_warp[h * kW + warp] = __popc(bal);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int w = 0; w < 2 * kW; ++w) {
      const int c = s_warp[w];
      s_warp[w] = acc;
      acc += c;
    }
    s_total = acc;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = h * kExpandThreads + threadIdx.x;
    if (t < n) out[t] = s_warp[h * kW + warp] + pref[h];
  }
  __syncthreads();
  return s_total;
}

__global__ void __launch_bounds__(kExpandThreads) expand_step_kernel(
    int step, int width, int k, int max_nodes, const int32_t* __restrict__ cand_ids,
    const float* __restrict__ cand_lp, const int32_t* __restrict__ root_token,
    int32_t* __restrict__ node_parent, int32_t* __restrict__ node_token,
    float* __restrict__ node_logv, int32_t* __restrict__ node_depth,
    int32_t* __restrict__ node_count, int32_t* __restrict__ frontier,
    int32_t* __restrict__ n_frontier, const int32_t* __restrict__ fanout, int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int P = step == 0 ? 1 : width;
  int32_t* np_ = node_parent + (size_t)b * max_nodes;
  int32_t* nt_ = node_token + (size_t)b * max_nodes;
  float* nv_ = node_logv + (size_t)b * max_nodes;
  int32_t* nd_ = node_depth + (size_t)b * max_nodes;

  __shared__ int s_par[64];  // expanded parent node ids (slot j)
  __shared__ float s_parv[64];
  __shared__ int s_pard[64];
  __shared__ float s_mass[64];
  __shared__ int s_valid[kMaxCand];
  __shared__ int s_scan[kMaxCand];
  __shared__ float s_v[kMaxCand];
  __shared__ int s_id[kMaxCand];
  __shared__ float s_lp[kMaxCand];
  __shared__ int s_bad;
  __shared__ int s_fan[64];  // static tree: children kept per parent slot

  const int npar = step == 0 ? 1 : max(0, min(width, n_frontier[b]));
  const int count0 = step == 0 ? 1 : node_count[b];
  const int ncand = npar * k;
  if (threadIdx.x == 0) s_bad = 0;
  if (threadIdx.x < 64) s_mass[threadIdx.x] = 0.f;
  __syncthreads();  // the error word is reset before any thread can raise it
  if (threadIdx.x < npar) {
    int f = k;
    if (fanout) {
      f = fanout[threadIdx.x];
      if (f < 0 || f > k) {
        atomicCAS(&s_bad, 0, EAGLE_ERR_BAD_TREE);
        f = 0;
      }
    }
    s_fan[threadIdx.x] = f;
  }
  // the expanded parents, loaded in parallel
  if (threadIdx.x < npar) {
    const int j = threadIdx.x;
    if (step == 0) {
      s_par[0] = 0;
      s_parv[0] = 0.f;
      s_pard[0] = 0;
      np_[0] = -1;
      nt_[0] = root_token ? root_token[b] : -1;
      nv_[0] = 0.f;
      nd_[0] = 0;
    } else {
      int p = frontier[(size_t)b * width + j];
      if (p < 0 || p >= count0) {
        atomicCAS(&s_bad, 0, EAGLE_ERR_BAD_TREE);
        p = 0;
      }
      s_par[j] = p;
      s_parv[j] = nv_[p];
      s_pard[j] = nd_[p];
    }
  }
  for (int t = threadIdx.x; t < ncand; t += kExpandThreads) {
    const int j = t / k, i = t % k;
    const size_t src = ((size_t)b * P + j) * k + i;
    s_id[t] = cand_ids[src];
    s_lp[t] = cand_lp[src];
  }
  __syncthreads();
  // validation (duplicates, non-finite values, sibling mass) and values
  for (int t = threadIdx.x; t < ncand; t += kExpandThreads) {
    const int j = t / k, i = t % k;
    const int id = s_id[t];
    float lp = s_lp[t];
    int valid = id >= 0 && i < s_fan[j];
    if (valid) {
      if (isnan(lp) || lp == INFINITY) {
        atomicCAS(&s_bad, 0, EAGLE_ERR_NONFINITE);
        valid = 0;
      }
      for (int i2 = 0; i2 < i; ++i2)
        if (s_id[j * k + i2] == id) atomicCAS(&s_bad, 0, EAGLE_ERR_BAD_TREE);
      lp = fminf(lp, 0.f);
      atomicAdd(&s_mass[j], expf(lp));
      // log V(child) = log V(parent) + log max(c, eps): one fp32 addition
      s_v[t] = __fadd_rn(s_parv[j], fmaxf(lp, kLogEps));
    }
    s_valid[t] = valid;
  }
  __syncthreads();
  if (threadIdx.x < npar && s_mass[threadIdx.x] > 1.f + kMassTol) atomicCAS(&s_bad, 0, EAGLE_ERR_BAD_TREE);
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      set_status(dev_status, s_bad);
      n_frontier[b] = 0;
      if (step == 0) node_count[b] = 1;
    }
    return;
  }
  // creation-ordered node ids (slot, then rank) via a block prefix sum
  const int nnew = block_exclusive_scan(s_valid, s_scan, ncand);
  if (count0 + nnew > max_nodes) {
    if (threadIdx.x == 0) {
      set_status(dev_status, EAGLE_ERR_INVALID_ARG);
      n_frontier[b] = 0;
    }
    return;
  }
  for (int t = threadIdx.x; t < ncand; t += kExpandThreads) {
    if (!s_valid[t]) continue;
    const int j = t / k;
    const int node = count0 + s_scan[t];
    np_[node] = s_par[j];
    nt_[node] = s_id[t];
    nv_[node] = s_v[t];
    nd_[node] = s_pard[j] + 1;
    // next frontier: rank of this node among the new nodes (same depth) by
    // key; a static tree keeps creation order
    int rank = s_scan[t];
    if (!fanout) {
      const float v = s_v[t];
      rank = 0;
      for (int u = 0; u < ncand; ++u) {
        if (!s_valid[u] || u == t) continue;
        rank += key_less(s_v[u], 0, count0 + s_scan[u], v, 0, node) ? 1 : 0;
      }
    }
    if (rank < width) frontier[(size_t)b * width + rank] = node;
  }
  if (threadIdx.x == 0) {
    if (fanout && nnew > width) set_status(dev_status, EAGLE_ERR_BAD_TREE);  // a depth wider than the frontier
    n_frontier[b] = nnew < width ? nnew : width;
    node_count[b] = count0 + nnew;
  }
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
  __shared__ int s_row_of[kMaxNodes];
  __shared__ int s_prow[64];
  __shared__ int s_bad;
  int count = node_count[b];
  count = count < 1 ? 1 : (count > max_nodes ? max_nodes : count);
  const int n = count - 1;  // candidates (the seed excluded)
  const int nsel = min(budget, n);
  const int ctx = ctx_lens ? ctx_lens[b] : 0;
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = threadIdx.x; i < P; i += kExpandThreads)
    s_key[i] = i < n ? node_key(nv_[i + 1], nd_[i + 1], i + 1) : ~0ull;
  for (int i = threadIdx.x; i < count; i += kExpandThreads) s_row_of[i] = -1;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
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
  for (int r = 1 + threadIdx.x; r <= nsel; r += kExpandThreads)
    s_row_of[(int)(s_key[r - 1] & 0xFFFFu)] = r;
  if (threadIdx.x == 0) s_row_of[0] = 0;
  __syncthreads();
  // parent rows (a parent always precedes its child in key order)
  for (int r = threadIdx.x; r < 64 && r <= nsel; r += kExpandThreads) {
    if (r == 0) {
      s_prow[0] = -1;
      continue;
    }
    const int nd = (int)(s_key[r - 1] & 0xFFFFu);
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
      const int nd = r == 0 ? 0 : (int)(s_key[r - 1] & 0xFFFFu);
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
int expand_launch(int B, int step, int width, int k, int max_nodes, const int32_t* fanout,
                  const int32_t* cand_ids, const float* cand_logprobs, const int32_t* root_token,
                  int32_t* node_parent, int32_t* node_token, float* node_logv, int32_t* node_depth,
                  int32_t* node_count, int32_t* frontier, int32_t* n_frontier, int32_t* dev_status,
                  void* stream) {
  if (B <= 0 || step < 0 || width < 1 || k < 1 || max_nodes < 1) return EAGLE_ERR_INVALID_ARG;
  if (!cand_ids || !cand_logprobs || !node_parent || !node_token || !node_logv || !node_depth ||
      !node_count || !frontier || !n_frontier)
    return EAGLE_ERR_INVALID_ARG;
  if (step == 0 && !root_token) return EAGLE_ERR_INVALID_ARG;
  if (width > 64 || k > 32 || width * k > kMaxCand || max_nodes > kMaxNodes || B > 65535)
    return EAGLE_ERR_UNSUPPORTED;
  if ((long long)max_nodes < 1LL + k + (long long)step * width * k) return EAGLE_ERR_INVALID_ARG;
  launch(expand_step_kernel, B, kExpandThreads, 0, static_cast<cudaStream_t>(stream),
      step, width, k, max_nodes, cand_ids, cand_logprobs, root_token, node_parent, node_token,
      node_logv, node_depth, node_count, frontier, n_frontier, fanout, dev_status);
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
  return expand_launch(B, step, width, k, max_nodes, nullptr, cand_ids, cand_logprobs, root_token,
                       node_parent, node_token, node_logv, node_depth, node_count, frontier, n_frontier,
                       dev_status, stream);
}

extern "C" int eagle_tree_expand_static(int B, int step, int width, int k, int max_nodes,
                                        const int32_t* fanout, const int32_t* cand_ids,
                                        const float* cand_logprobs, const int32_t* root_token,
                                        int32_t* node_parent, int32_t* node_token, float* node_logv,
                                        int32_t* node_depth, int32_t* node_count, int32_t* frontier,
                                        int32_t* n_frontier, int32_t* dev_status, void* stream) {
  if (!fanout) return EAGLE_ERR_INVALID_ARG;
  return expand_launch(B, step, width, k, max_nodes, fanout, cand_ids, cand_logprobs, root_token,
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
