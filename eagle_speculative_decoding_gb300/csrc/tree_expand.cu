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
// One CTA per request.  Ranks are computed by counting, for each node, the
// nodes with a smaller key: keys are unique (node ids differ), so the ranks
// are a permutation and need no sort network.  log V is accumulated in fp32
// with one correctly rounded addition per level.
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

__global__ void __launch_bounds__(kExpandThreads) expand_step_kernel(
    int step, int width, int k, int max_nodes, const int32_t* __restrict__ cand_ids,
    const float* __restrict__ cand_lp, const int32_t* __restrict__ root_token,
    int32_t* __restrict__ node_parent, int32_t* __restrict__ node_token,
    float* __restrict__ node_logv, int32_t* __restrict__ node_depth,
    int32_t* __restrict__ node_count, int32_t* __restrict__ frontier,
    int32_t* __restrict__ n_frontier, int32_t* dev_status) {
  const int b = blockIdx.x;
  const int P = step == 0 ? 1 : width;
  int32_t* np_ = node_parent + (size_t)b * max_nodes;
  int32_t* nt_ = node_token + (size_t)b * max_nodes;
  float* nv_ = node_logv + (size_t)b * max_nodes;
  int32_t* nd_ = node_depth + (size_t)b * max_nodes;

  __shared__ int s_par[64];       // expanded parent node ids (slot j)
  __shared__ float s_parv[64];
  __shared__ int s_pard[64];
  __shared__ int s_npar, s_count0, s_bad;
  __shared__ int s_valid[kMaxCand];
  __shared__ int s_scan[kMaxCand];
  __shared__ float s_v[kMaxCand];
  __shared__ int s_id[kMaxCand];
  __shared__ float s_mass[64];

  if (threadIdx.x == 0) {
    s_bad = 0;
    if (step == 0) {
      np_[0] = -1;
      nt_[0] = root_token ? root_token[b] : -1;
      nv_[0] = 0.f;
      nd_[0] = 0;
      s_npar = 1;
      s_count0 = 1;
      s_par[0] = 0;
      s_parv[0] = 0.f;
      s_pard[0] = 0;
    } else {
      int np = n_frontier[b];
      np = np < 0 ? 0 : (np > width ? width : np);
      s_npar = np;
      s_count0 = node_count[b];
      for (int j = 0; j < np; ++j) {
        int p = frontier[(size_t)b * width + j];
        if (p < 0 || p >= s_count0) {
          s_bad = EAGLE_ERR_BAD_TREE;
          p = 0;
        }
        s_par[j] = p;
        s_parv[j] = nv_[p];
        s_pard[j] = nd_[p];
      }
    }
  }
  if (threadIdx.x < 64) s_mass[threadIdx.x] = 0.f;
  __syncthreads();
  const int npar = s_npar, ncand = npar * k, count0 = s_count0;

  // candidates: validity, duplicates, non-finite values, sibling mass
  for (int t = threadIdx.x; t < ncand; t += kExpandThreads) {
    const int j = t / k, i = t % k;
    const size_t src = ((size_t)b * P + j) * k + i;
    const int id = cand_ids[src];
    float lp = cand_lp[src];
    int valid = id >= 0;
    if (valid) {
      if (isnan(lp) || lp == INFINITY) {
        atomicCAS(&s_bad, 0, EAGLE_ERR_NONFINITE);
        valid = 0;
      }
      for (int i2 = 0; i2 < i; ++i2)
        if (cand_ids[((size_t)b * P + j) * k + i2] == id) atomicCAS(&s_bad, 0, EAGLE_ERR_BAD_TREE);
      lp = fminf(lp, 0.f);
      atomicAdd(&s_mass[j], expf(lp));
      // log V(child) = log V(parent) + log max(c, eps): one fp32 addition
      s_v[t] = __fadd_rn(s_parv[j], fmaxf(lp, kLogEps));
    }
    s_valid[t] = valid;
    s_id[t] = id;
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
  // exclusive scan of validity -> creation-ordered node ids (slot, then rank)
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int t = 0; t < ncand; ++t) {
      s_scan[t] = acc;
      acc += s_valid[t];
    }
    if (count0 + acc > max_nodes) s_bad = EAGLE_ERR_INVALID_ARG;
    s_count0 = acc;  // reuse: number of new nodes
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      set_status(dev_status, s_bad);
      n_frontier[b] = 0;
    }
    return;
  }
  const int nnew = s_count0;
  for (int t = threadIdx.x; t < ncand; t += kExpandThreads) {
    if (!s_valid[t]) continue;
    const int j = t / k;
    const int node = count0 + s_scan[t];
    np_[node] = s_par[j];
    nt_[node] = s_id[t];
    nv_[node] = s_v[t];
    nd_[node] = s_pard[j] + 1;
  }
  // next frontier: the top-`width` new nodes by key (all at the same depth)
  for (int t = threadIdx.x; t < ncand; t += kExpandThreads) {
    if (!s_valid[t]) continue;
    const int node = count0 + s_scan[t];
    const float v = s_v[t];
    int rank = 0;
    for (int u = 0; u < ncand; ++u) {
      if (!s_valid[u] || u == t) continue;
      const int nu = count0 + s_scan[u];
      rank += key_less(s_v[u], 0, nu, v, 0, node) ? 1 : 0;
    }
    if (rank < width) frontier[(size_t)b * width + rank] = node;
  }
  if (threadIdx.x == 0) {
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
  const int b = blockIdx.x;
  const int32_t* np_ = node_parent + (size_t)b * max_nodes;
  const int32_t* nt_ = node_token + (size_t)b * max_nodes;
  const float* nv_ = node_logv + (size_t)b * max_nodes;
  const int32_t* nd_ = node_depth + (size_t)b * max_nodes;
  __shared__ float s_v[kMaxNodes];
  __shared__ int s_d[kMaxNodes];
  __shared__ int s_row_of[kMaxNodes];
  __shared__ int s_sel[64];
  __shared__ int s_bad;
  int count = node_count[b];
  count = count < 1 ? 1 : (count > max_nodes ? max_nodes : count);
  const int nsel = min(budget, count - 1);
  const int ctx = ctx_lens ? ctx_lens[b] : 0;
  for (int n = threadIdx.x; n < count; n += kExpandThreads) {
    s_v[n] = nv_[n];
    s_d[n] = nd_[n];
    s_row_of[n] = -1;
  }
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int n = 1 + threadIdx.x; n < count; n += kExpandThreads) {
    const float v = s_v[n];
    const int d = s_d[n];
    int rank = 0;
    for (int u = 1; u < count; ++u) rank += key_less(s_v[u], s_d[u], u, v, d, n) ? 1 : 0;
    if (rank < nsel) {
      s_sel[rank] = n;
      s_row_of[n] = rank + 1;
    }
  }
  if (threadIdx.x == 0) s_row_of[0] = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    // rows in key order; a parent always precedes its child
    uint64_t m[64];
    m[0] = 1ull;
    const size_t o = (size_t)b * R;
    token[o] = nt_[0];
    parent_row[o] = -1;
    depth[o] = 0;
    mask[o] = 1ull;
    node_id[o] = 0;
    position[o] = ctx;
    for (int r = 1; r <= nsel; ++r) {
      const int n = s_sel[r - 1];
      const int p = np_[n];
      int pr = (p >= 0 && p < count) ? s_row_of[p] : -1;
      if (pr < 0 || pr >= r) {
        s_bad = 1;
        pr = 0;
      }
      m[r] = m[pr] | (1ull << r);
      token[o + r] = nt_[n];
      parent_row[o + r] = pr;
      depth[o + r] = s_d[n];
      mask[o + r] = m[r];
      node_id[o + r] = n;
      position[o + r] = ctx + s_d[n];
    }
    for (int r = nsel + 1; r < R; ++r) {
      token[o + r] = -1;
      parent_row[o + r] = -1;
      depth[o + r] = 0;
      mask[o + r] = 1ull << r;
      node_id[o + r] = -1;
      position[o + r] = ctx;
    }
    n_rows[b] = nsel + 1;
    if (s_bad) set_status(dev_status, EAGLE_ERR_BAD_TREE);
  }
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" int eagle_tree_expand(int B, int step, int width, int k, int max_nodes,
                                 const int32_t* cand_ids, const float* cand_logprobs,
                                 const int32_t* root_token, int32_t* node_parent,
                                 int32_t* node_token, float* node_logv, int32_t* node_depth,
                                 int32_t* node_count, int32_t* frontier, int32_t* n_frontier,
                                 int32_t* dev_status, void* stream) {
  if (B <= 0 || step < 0 || width < 1 || k < 1 || max_nodes < 1) return EAGLE_ERR_INVALID_ARG;
  if (!cand_ids || !cand_logprobs || !node_parent || !node_token || !node_logv || !node_depth ||
      !node_count || !frontier || !n_frontier)
    return EAGLE_ERR_INVALID_ARG;
  if (step == 0 && !root_token) return EAGLE_ERR_INVALID_ARG;
  if (width > 64 || k > 32 || width * k > kMaxCand || max_nodes > kMaxNodes || B > 65535)
    return EAGLE_ERR_UNSUPPORTED;
  if ((long long)max_nodes < 1LL + k + (long long)step * width * k) return EAGLE_ERR_INVALID_ARG;
  expand_step_kernel<<<B, kExpandThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      step, width, k, max_nodes, cand_ids, cand_logprobs, root_token, node_parent, node_token,
      node_logv, node_depth, node_count, frontier, n_frontier, dev_status);
  note_launch();
  return last_launch_status();
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
  expand_finalize_kernel<<<B, kExpandThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      max_nodes, budget, R, node_parent, node_token, node_logv, node_depth, node_count, ctx_lens,
      token, parent_row, depth, mask, node_id, position, n_rows, dev_status);
  note_launch();
  return last_launch_status();
}
