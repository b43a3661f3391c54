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
// counting smaller 64-bit order-preserving keys (unique: node ids differ);
// the final rerank bitonic-sorts the keys of all stored nodes.  log V is
// accumulated in fp32 with one correctly rounded addition per level.
#include <math.h>

#include "common.cuh"
#include "lm_merge.cuh"

namespace eagle {
namespace {

constexpr int kExpandThreads = 512;
constexpr int kMaxCand = 1024;      // width * k
constexpr int kMaxNodes = 2048;
// log(1e-12) rounded to fp32: the ranking floor of a zero confidence.
constexpr float kLogEps = -27.631021115928547f;
constexpr float kMassTol = 1e-4f;

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
  static_assert(2 * kW == 32, "one warp scans the warp totals");
  if (warp == 0) {  // exclusive scan of the 32 warp totals by shuffles
    const int c = s_warp[lane];
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    s_warp[lane] = inc - c;
    if (lane == 31) s_total = inc;
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

// One expansion step.  MERGE: the candidate lists are not read from
// cand_ids / cand_lp but merged here from the per-CTA partials an LM-head call
// left (lp; row b * P + j holds parent slot j of request b): stage_rows rows
// at a time are staged in dynamic shared memory by all threads, then one warp
// per row merges them straight into the candidate arrays.
template <bool MERGE>
__global__ void __launch_bounds__(kExpandThreads) expand_step_kernel(
    int step, int width, int k, int max_nodes, const int32_t* __restrict__ cand_ids,
    const float* __restrict__ cand_lp, const LmPartials lp, int stage_rows,
    const int32_t* __restrict__ root_token,
    int32_t* __restrict__ node_parent, int32_t* __restrict__ node_token,
    float* __restrict__ node_logv, int32_t* __restrict__ node_depth,
    int32_t* __restrict__ node_count, int32_t* __restrict__ frontier,
    int32_t* __restrict__ n_frontier, const int32_t* __restrict__ fanout, int32_t* dev_status) {
  // the next kernel (an LM head that prefetches its weights) is let in only
  // at the end: its prefetch would otherwise queue ahead of this kernel's
  // few latency-bound loads
  pdl_wait();
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
  // s_lp and s_valid share their bytes with the 64-bit ranking keys, which
  // are written only after both are consumed
  __shared__ __align__(16) unsigned char s_kbuf[kMaxCand * 8];
  float* s_lp = reinterpret_cast<float*>(s_kbuf);
  int* s_valid = reinterpret_cast<int*>(s_kbuf) + kMaxCand;
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(s_kbuf);
  __shared__ int s_scan[kMaxCand];
  __shared__ float s_v[kMaxCand];
  __shared__ int s_id[kMaxCand];
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
  if (MERGE) {
    extern __shared__ __align__(16) unsigned char stage[];
    const int nc = lp.cpg, n = nc * k, warp = threadIdx.x >> 5;
    const size_t row_bytes = ((size_t)n * 8 + (size_t)nc * 4 + 15) / 16 * 16;
    for (int j0 = 0; j0 < npar; j0 += stage_rows) {
      const int nb = min(stage_rows, npar - j0);
      // the batch's lists are contiguous ([row][cta][K] from row b * P + j0):
      // 16-byte loads when the rows keep 16-byte alignment, four in flight
      // per thread before any store
      const size_t m0 = (size_t)b * P + j0;
      if ((n & 3) == 0) {
        const int n4 = n / 4, tot = nb * n4;
        const float4* gv = reinterpret_cast<const float4*>(lp.v + m0 * n);
        const int4* gi = reinterpret_cast<const int4*>(lp.id + m0 * n);
        for (int f0 = threadIdx.x; f0 < tot; f0 += 4 * kExpandThreads) {
          float4 v[4];
          int4 id[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int f = f0 + u * kExpandThreads;
            if (f < tot) {
              v[u] = __ldcg(gv + f);
              id[u] = __ldcg(gi + f);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int f = f0 + u * kExpandThreads;
            if (f < tot) {
              const int r = f / n4, e = f % n4;
              float4* sv = reinterpret_cast<float4*>(stage + r * row_bytes);
              sv[e] = v[u];
              reinterpret_cast<int4*>(sv + n4)[e] = id[u];
            }
          }
        }
      } else {
        const int tot = nb * n;
        for (int f0 = threadIdx.x; f0 < tot; f0 += 4 * kExpandThreads) {
          float v[4];
          int id[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int f = f0 + u * kExpandThreads;
            if (f < tot) {
              v[u] = __ldcg(lp.v + m0 * n + f);
              id[u] = __ldcg(lp.id + m0 * n + f);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int f = f0 + u * kExpandThreads;
            if (f < tot) {
              const int r = f / n, e = f % n;
              float* sv = reinterpret_cast<float*>(stage + r * row_bytes);
              sv[e] = v[u];
              reinterpret_cast<int*>(sv + n)[e] = id[u];
            }
          }
        }
      }
      for (int f = threadIdx.x; f < nb * nc; f += kExpandThreads) {
        const int r = f / nc, c = f % nc;
        const size_t m = (size_t)b * P + j0 + r;
        int* sc = reinterpret_cast<int*>(stage + r * row_bytes) + 2 * n;
        sc[c] = __ldcg(lp.cnt + m * nc + c);
      }
      __syncthreads();
      if (warp < nb) {
        const float* sv = reinterpret_cast<const float*>(stage + warp * row_bytes);
        const int* si = reinterpret_cast<const int*>(sv + n);
        lm_merge_row(lp, b * P + j0 + warp, sv, si, si + n, s_id + (j0 + warp) * k, s_lp + (j0 + warp) * k,
                     nullptr, nullptr);
      }
      __syncthreads();
    }
  } else {
    for (int t = threadIdx.x; t < ncand; t += kExpandThreads) {
      const int j = t / k, i = t % k;
      const size_t src = ((size_t)b * P + j) * k + i;
      s_id[t] = cand_ids[src];
      s_lp[t] = cand_lp[src];
    }
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
    pdl_trigger();
    return;
  }
  // creation-ordered node ids (slot, then rank) via a block prefix sum
  const int nnew = block_exclusive_scan(s_valid, s_scan, ncand);
  if (count0 + nnew > max_nodes) {
    if (threadIdx.x == 0) {
      set_status(dev_status, EAGLE_ERR_INVALID_ARG);
      n_frontier[b] = 0;
    }
    pdl_trigger();
    return;
  }
  // the ranking key of each new node (all of the same depth): larger log V
  // first, then smaller node id; a discarded candidate sorts last
  constexpr int kPerT = kMaxCand / kExpandThreads;
  unsigned long long key[kPerT];
#pragma unroll
  for (int h = 0; h < kPerT; ++h) {
    const int t = h * kExpandThreads + threadIdx.x;
    key[h] = ~0ull;
    if (t < ncand && s_valid[t]) key[h] = node_key(s_v[t] + 0.f, 0, count0 + s_scan[t]);
  }
  __syncthreads();  // s_valid and s_lp are read: their bytes become the keys
#pragma unroll
  for (int h = 0; h < kPerT; ++h) {
    const int t = h * kExpandThreads + threadIdx.x;
    if (t < ncand) s_key[t] = key[h];
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kPerT; ++h) {
    const int t = h * kExpandThreads + threadIdx.x;
    const unsigned long long mk = key[h];
    if (t >= ncand || mk == ~0ull) continue;
    const int j = t / k;
    const int node = count0 + s_scan[t];
    np_[node] = s_par[j];
    nt_[node] = s_id[t];
    nv_[node] = s_v[t];
    nd_[node] = s_pard[j] + 1;
    // next frontier: rank of this node among the new nodes by key (keys are
    // unique: node ids differ); a static tree keeps creation order
    int rank = s_scan[t];
    if (!fanout) {
      rank = 0;
#pragma unroll 8
      for (int u = 0; u < ncand; ++u) rank += s_key[u] < mk ? 1 : 0;
    }
    if (rank < width) frontier[(size_t)b * width + rank] = node;
  }
  if (threadIdx.x == 0) {
    if (fanout && nnew > width) set_status(dev_status, EAGLE_ERR_BAD_TREE);  // a depth wider than the frontier
    n_frontier[b] = nnew < width ? nnew : width;
    node_count[b] = count0 + nnew;
  }
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
  if (n <= 1024) {
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
  if (width > 64 || k > 32 || width * k > kMaxCand || max_nodes > kMaxNodes || B > 65535)
    return EAGLE_ERR_UNSUPPORTED;
  if ((long long)max_nodes < 1LL + k + (long long)step * width * k) return EAGLE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (lp) {
    const size_t row_bytes = ((size_t)lp->cpg * k * 8 + (size_t)lp->cpg * 4 + 15) / 16 * 16;
    const int P = step == 0 ? 1 : width;
    int rows = (int)(kStageBytes / row_bytes);
    rows = rows < kExpandThreads / 32 ? rows : kExpandThreads / 32;
    rows = rows < P ? rows : P;
    if (rows < 1) return EAGLE_ERR_UNSUPPORTED;
    const size_t smem = (size_t)rows * row_bytes;
    cudaFuncSetAttribute(expand_step_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch(expand_step_kernel<true>, B, kExpandThreads, smem, s, step, width, k, max_nodes, cand_ids,
           cand_logprobs, *lp, rows, root_token, node_parent, node_token, node_logv, node_depth, node_count,
           frontier, n_frontier, fanout, dev_status);
  } else {
    launch(expand_step_kernel<false>, B, kExpandThreads, 0, s, step, width, k, max_nodes, cand_ids,
           cand_logprobs, LmPartials{}, 0, root_token, node_parent, node_token, node_logv, node_depth,
           node_count, frontier, n_frontier, fanout, dev_status);
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
