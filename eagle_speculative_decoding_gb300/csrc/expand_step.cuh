// One EAGLE-2 expansion step of one request, as a block-wide device function
// (the body of the expansion kernel, for a block of NT threads and up to MAXC
// candidates).
//
// Source: "M7.5 - EAGLE Feature Drafting: Uncertainty, Dynamic Trees, HASS, and
// EAGLE-3", sections 0x06A "Path Value Derivation" (log V(u) = sum over the
// path of log max(c_j, eps), eps = 1e-12; a child never outranks its parent)
// and 0x06B "Expansion And Reranking" (the top-width nodes of the latest
// layer by (-log V, depth, node_id) are the next frontier); "EAGLE:
// Speculative Sampling Requires Rethinking Feature Uncertainty",
// "Tree-Structured Draft Generation" (top-k tokens become the children).
//
// The new nodes (at most width * k) get creation-ordered ids by a block prefix
// sum over the kept candidates and are ranked by counting smaller 64-bit
// order-preserving keys (unique: node ids differ).  log V is accumulated in
// fp32 with one correctly rounded addition per level.
#pragma once

#include "common.cuh"
#include "lm_merge.cuh"

namespace eagle {

constexpr int kExpandMaxNodes = 2048;
constexpr int kExpandMaxWidth = 64;
// log(1e-12) rounded to fp32: the ranking floor of a zero confidence.
constexpr float kExpandLogEps = -27.631021115928547f;
constexpr float kExpandMassTol = 1e-4f;

// Order-preserving 64-bit sort key of a node: ascending key = descending
// log V, then ascending depth, then ascending node id.
__device__ __forceinline__ unsigned long long node_key(float v, int d, int id) {
  uint32_t f = __float_as_uint(v);
  f = (f & 0x80000000u) ? ~f : (f | 0x80000000u);  // ascending as unsigned
  return ((unsigned long long)(~f) << 32) | ((unsigned long long)(uint32_t)d << 16) |
         (unsigned long long)(uint32_t)id;
}

// The tree state of a batch and the inputs of one step (node arrays are
// [B, max_nodes], frontier [B, width]).
struct ExpandArgs {
  int step, width, k, max_nodes;
  const int32_t* cand_ids;  // [B, P, k] merged candidate lists (unless merged in the step)
  const float* cand_lp;
  const int32_t* root_token;
  int32_t* node_parent;
  int32_t* node_token;
  float* node_logv;
  int32_t* node_depth;
  int32_t* node_count;
  int32_t* frontier;
  int32_t* n_frontier;
  const int32_t* fanout;  // static tree: children kept per parent slot, or null
  int32_t* status;
};

// Shared memory of one step with up to MAXC candidates.
template <int MAXC>
struct ExpandSmem {
  int par[kExpandMaxWidth];  // expanded parent node ids (slot j)
  float parv[kExpandMaxWidth];
  int pard[kExpandMaxWidth];
  float mass[kExpandMaxWidth];
  int fan[kExpandMaxWidth];
  // the candidates' log-probs ([0, MAXC) as floats) and kept flags
  // ([MAXC, 2 MAXC) as ints) share their bytes with the 64-bit ranking keys,
  // which are written only after both are consumed
  unsigned long long kbuf[MAXC];
  int scan[MAXC];
  float v[MAXC];
  int id[MAXC];
  int warp_tot[32];
  int total;
  int bad;
};

// Host-side argument checks of a step (0 = OK, else an eagle_status).
inline int expand_check(int B, int step, int width, int k, int max_nodes, int max_cand) {
  if (B <= 0 || step < 0 || width < 1 || k < 1 || max_nodes < 1) return EAGLE_ERR_INVALID_ARG;
  if (width > kExpandMaxWidth || k > 32 || width * k > max_cand || max_nodes > kExpandMaxNodes || B > 65535)
    return EAGLE_ERR_UNSUPPORTED;
  if ((long long)max_nodes < 1LL + k + (long long)step * width * k) return EAGLE_ERR_INVALID_ARG;
  return EAGLE_OK;
}

// Exclusive prefix sum of 0/1 flags over n <= MAXC entries (block of NT
// threads); returns the total.
template <int NT, int MAXC>
__device__ __forceinline__ int expand_scan(ExpandSmem<MAXC>& s, const int* flags, int* out, int n) {
  constexpr int kW = NT / 32, kH = (MAXC + NT - 1) / NT;
  static_assert(kW * kH <= 32, "one warp scans the warp totals");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int pref[kH], v[kH];
#pragma unroll
  for (int h = 0; h < kH; ++h) {
    const int t = h * NT + threadIdx.x;
    v[h] = t < n ? flags[t] : 0;
    const unsigned bal = __ballot_sync(0xffffffffu, v[h]);
    pref[h] = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) s.warp_tot[h * kW + warp] = __popc(bal);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the warp totals by shuffles
    const int c = lane < kW * kH ? s.warp_tot[lane] : 0;
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane < kW * kH) s.warp_tot[lane] = inc - c;
    if (lane == 31) s.total = inc;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kH; ++h) {
    const int t = h * NT + threadIdx.x;
    if (t < n) out[t] = s.warp_tot[h * kW + warp] + pref[h];
  }
  __syncthreads();
  return s.total;
}

// One expansion step of request b by a block of NT threads.  MERGE: the
// candidate lists are merged here from the per-CTA partials an LM-head call
// left (lp; row b * P + j holds parent slot j of request b): stage_rows rows
// at a time (at most NT / 32) are staged in `stage` by all threads, then one
// warp per row merges them.  Errors go to a.status; the request is then left
// with an empty frontier.
template <int NT, int MAXC, bool MERGE>
__device__ void expand_step_block(const ExpandArgs& a, int b, ExpandSmem<MAXC>& s, const LmPartials& lp,
                                  unsigned char* stage, int stage_rows) {
  constexpr int kU = 4;  // 16-byte loads of each kind in flight per thread
  const int step = a.step, width = a.width, k = a.k;
  const int P = step == 0 ? 1 : width;
  int32_t* np_ = a.node_parent + (size_t)b * a.max_nodes;
  int32_t* nt_ = a.node_token + (size_t)b * a.max_nodes;
  float* nv_ = a.node_logv + (size_t)b * a.max_nodes;
  int32_t* nd_ = a.node_depth + (size_t)b * a.max_nodes;
  float* s_lp = reinterpret_cast<float*>(s.kbuf);
  int* s_valid = reinterpret_cast<int*>(s.kbuf) + MAXC;

  // Loads whose addresses need only the arguments go out first, beside the
  // frontier count they would otherwise wait for: the frontier's node ids
  // ([B, width]) and the candidate lists ([B, P, k]); entries past the count
  // are read but not used.
  constexpr int kCandPerThread = (MAXC + NT - 1) / NT;
  int fr = 0;
  if (step > 0 && threadIdx.x < width) fr = a.frontier[(size_t)b * width + threadIdx.x];
  int cid[kCandPerThread];
  float clp[kCandPerThread];
  if (!MERGE) {
#pragma unroll
    for (int h = 0; h < kCandPerThread; ++h) {
      const int t = h * NT + threadIdx.x;
      if (t < P * k) {
        cid[h] = a.cand_ids[(size_t)b * P * k + t];
        clp[h] = a.cand_lp[(size_t)b * P * k + t];
      }
    }
  }

  const int npar = step == 0 ? 1 : max(0, min(width, a.n_frontier[b]));
  const int count0 = step == 0 ? 1 : a.node_count[b];
  const int ncand = npar * k;
  if (threadIdx.x == 0) s.bad = 0;
  if (threadIdx.x < kExpandMaxWidth) s.mass[threadIdx.x] = 0.f;
  __syncthreads();  // the error word is reset before any thread can raise it
  if (threadIdx.x < npar) {
    int f = k;
    if (a.fanout) {
      f = a.fanout[threadIdx.x];
      if (f < 0 || f > k) {
        atomicCAS(&s.bad, 0, EAGLE_ERR_BAD_TREE);
        f = 0;
      }
    }
    s.fan[threadIdx.x] = f;
  }
  // the expanded parents, loaded in parallel
  if (threadIdx.x < npar) {
    const int j = threadIdx.x;
    if (step == 0) {
      s.par[0] = 0;
      s.parv[0] = 0.f;
      s.pard[0] = 0;
      np_[0] = -1;
      nt_[0] = a.root_token ? a.root_token[b] : -1;
      nv_[0] = 0.f;
      nd_[0] = 0;
    } else {
      int p = fr;
      if (p < 0 || p >= count0) {
        atomicCAS(&s.bad, 0, EAGLE_ERR_BAD_TREE);
        p = 0;
      }
      s.par[j] = p;
      s.parv[j] = nv_[p];
      s.pard[j] = nd_[p];
    }
  }
  if (MERGE) {
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
        for (int f0 = threadIdx.x; f0 < tot; f0 += kU * NT) {
          float4 v[kU];
          int4 id[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int f = f0 + u * NT;
            if (f < tot) {
              v[u] = __ldcg(gv + f);
              id[u] = __ldcg(gi + f);
            }
          }
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int f = f0 + u * NT;
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
        for (int f0 = threadIdx.x; f0 < tot; f0 += kU * NT) {
          float v[kU];
          int id[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int f = f0 + u * NT;
            if (f < tot) {
              v[u] = __ldcg(lp.v + m0 * n + f);
              id[u] = __ldcg(lp.id + m0 * n + f);
            }
          }
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int f = f0 + u * NT;
            if (f < tot) {
              const int r = f / n, e = f % n;
              float* sv = reinterpret_cast<float*>(stage + r * row_bytes);
              sv[e] = v[u];
              reinterpret_cast<int*>(sv + n)[e] = id[u];
            }
          }
        }
      }
      for (int f = threadIdx.x; f < nb * nc; f += NT) {
        const int r = f / nc, c = f % nc;
        const size_t m = (size_t)b * P + j0 + r;
        int* sc = reinterpret_cast<int*>(stage + r * row_bytes) + 2 * n;
        sc[c] = __ldcg(lp.cnt + m * nc + c);
      }
      __syncthreads();
      if (warp < nb) {
        const float* sv = reinterpret_cast<const float*>(stage + warp * row_bytes);
        const int* si = reinterpret_cast<const int*>(sv + n);
        lm_merge_row(lp, b * P + j0 + warp, sv, si, si + n, s.id + (j0 + warp) * k, s_lp + (j0 + warp) * k,
                     nullptr, nullptr);
      }
      __syncthreads();
    }
  } else {
#pragma unroll
    for (int h = 0; h < kCandPerThread; ++h) {
      const int t = h * NT + threadIdx.x;
      if (t < ncand) {
        s.id[t] = cid[h];
        s_lp[t] = clp[h];
      }
    }
  }
  __syncthreads();
  // validation (duplicates, non-finite values, sibling mass) and values
  for (int t = threadIdx.x; t < ncand; t += NT) {
    const int j = t / k, i = t % k;
    const int id = s.id[t];
    float lpv = s_lp[t];
    int valid = id >= 0 && i < s.fan[j];
    if (valid) {
      if (isnan(lpv) || lpv == INFINITY) {
        atomicCAS(&s.bad, 0, EAGLE_ERR_NONFINITE);
        valid = 0;
      }
      for (int i2 = 0; i2 < i; ++i2)
        if (s.id[j * k + i2] == id) atomicCAS(&s.bad, 0, EAGLE_ERR_BAD_TREE);
      lpv = fminf(lpv, 0.f);
      atomicAdd(&s.mass[j], expf(lpv));
      // log V(child) = log V(parent) + log max(c, eps): one fp32 addition
      s.v[t] = __fadd_rn(s.parv[j], fmaxf(lpv, kExpandLogEps));
    }
    s_valid[t] = valid;
  }
  __syncthreads();
  if (threadIdx.x < npar && s.mass[threadIdx.x] > 1.f + kExpandMassTol) atomicCAS(&s.bad, 0, EAGLE_ERR_BAD_TREE);
  __syncthreads();
  if (s.bad) {
    if (threadIdx.x == 0) {
      set_status(a.status, s.bad);
      a.n_frontier[b] = 0;
      if (step == 0) a.node_count[b] = 1;
    }
    return;
  }
  // creation-ordered node ids (slot, then rank) via a block prefix sum
  const int nnew = expand_scan<NT, MAXC>(s, s_valid, s.scan, ncand);
  if (count0 + nnew > a.max_nodes) {
    if (threadIdx.x == 0) {
      set_status(a.status, EAGLE_ERR_INVALID_ARG);
      a.n_frontier[b] = 0;
    }
    return;
  }
  // the ranking key of each new node (all of the same depth): larger log V
  // first, then smaller node id; a discarded candidate sorts last
  constexpr int kPerT = (MAXC + NT - 1) / NT;
  unsigned long long key[kPerT];
#pragma unroll
  for (int h = 0; h < kPerT; ++h) {
    const int t = h * NT + threadIdx.x;
    key[h] = ~0ull;
    if (t < ncand && s_valid[t]) key[h] = node_key(s.v[t] + 0.f, 0, count0 + s.scan[t]);
  }
  __syncthreads();  // s_valid and s_lp are read: their bytes become the keys
#pragma unroll
  for (int h = 0; h < kPerT; ++h) {
    const int t = h * NT + threadIdx.x;
    if (t < ncand) s.kbuf[t] = key[h];
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kPerT; ++h) {
    const int t = h * NT + threadIdx.x;
    const unsigned long long mk = key[h];
    if (t >= ncand || mk == ~0ull) continue;
    const int j = t / k;
    const int node = count0 + s.scan[t];
    np_[node] = s.par[j];
    nt_[node] = s.id[t];
    nv_[node] = s.v[t];
    nd_[node] = s.pard[j] + 1;
    // next frontier: rank of this node among the new nodes by key (keys are
    // unique: node ids differ); a static tree keeps creation order
    int rank = s.scan[t];
    if (!a.fanout) {
      rank = 0;
#pragma unroll 8
      for (int u = 0; u < ncand; ++u) rank += s.kbuf[u] < mk ? 1 : 0;
    }
    if (rank < width) a.frontier[(size_t)b * width + rank] = node;
  }
  if (threadIdx.x == 0) {
    if (a.fanout && nnew > width) set_status(a.status, EAGLE_ERR_BAD_TREE);  // a depth wider than the frontier
    a.n_frontier[b] = nnew < width ? nnew : width;
    a.node_count[b] = count0 + nnew;
  }
}

}  // namespace eagle
