// Lossless tree verification (greedy longest accepted path; multi-round
// speculative sampling with deterministic top-k proposals).
//
// Source: "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty"
// (paper summary), section "Verification Phase: Multi-Round Speculative Sampling
// on Trees" (the paper's Algorithm 1); "EAGLE-3: Scaling up Inference
// Acceleration of Large Language Models via Training-Time Test", "Stage 2:
// Verification".
//
// Deterministic proposals and greedy verification take up to three kernels:
//   rowstats : one CTA per (row, request): max and sum-exp of z/T (stochastic)
//              or the argmax (greedy without a caller-provided argmax),
//              streamed with 16-byte loads, four in flight per thread.
//   walk     : one CTA per request: every per-row input of the walk (parents,
//              tokens, row statistics or argmax, the target logit of each
//              child's token at its parent row, the accept-test uniform) is
//              gathered into shared memory in parallel, then one warp walks the
//              tree from the seed without touching global memory.
//   race     : (stochastic only) the exponential race for the bonus token at
//              the stop row, split over 4096-id chunks of the vocabulary; each
//              CTA reduces its chunk and the last CTA of a request (atomic
//              ticket, no waiting) merges the chunk winners.
// Sampled proposals take one kernel, a cluster of CTAs per request that reads
// only the target and draft rows its walk visits (verify_walk_sampled_kernel).
#include <math.h>

#include <atomic>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int kStatThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kRaceThreads = 256;
constexpr int kRaceChunk = 4096;  // vocabulary ids per race CTA
constexpr int kMaxVerifyRows = 1024;
constexpr float kLog2e = 1.4426950408889634f;

struct RowStat {
  float m;  // max_v z/T
  float s;  // sum_v exp(z/T - m)
};

// Walk result of one request, read by the race kernel.
struct VerifyReq {
  int stop;    // row where the walk stopped; -1 = no race (bad tree)
  int plen;    // rows on the accepted path (seed included)
  int nexcl;   // tokens rejected at the stop row
  int ticket;  // race CTAs of this request that have finished
};

struct RacePart {
  float key;
  int id;
};

__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (better(v2, i2, v, i)) {
    v = v2;
    i = i2;
  }
}

// Online max / sum-exp of four values of y = z/T.
__device__ __forceinline__ void lse_add4(float& m, float& s, float y0, float y1, float y2, float y3) {
  const float m4 = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
  if (m4 > m) {
    s *= exp2f((m - m4) * kLog2e);
    m = m4;
  }
  if (m != -INFINITY)
    s += exp2f((y0 - m) * kLog2e) + exp2f((y1 - m) * kLog2e) + exp2f((y2 - m) * kLog2e) +
         exp2f((y3 - m) * kLog2e);
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
  float m = -INFINITY, s = 0.f;     // stochastic: online max / sum-exp of z/T
  float bv = -INFINITY;             // greedy: argmax (ties to the lower id)
  int bi = 0x7fffffff;
  auto take4 = [&](float z0, float z1, float z2, float z3, int y) {
    nan_seen |= isnan(z0) | isnan(z1) | isnan(z2) | isnan(z3);
    if (want_argmax) {
      argmax_merge(bv, bi, z0, y);
      argmax_merge(bv, bi, z1, y + 1);
      argmax_merge(bv, bi, z2, y + 2);
      argmax_merge(bv, bi, z3, y + 3);
    } else {
      lse_add4(m, s, z0 * inv_t, z1 * inv_t, z2 * inv_t, z3 * inv_t);
    }
  };
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    const int n4 = V >> 2;
    constexpr int kU = 4;  // 16-byte loads in flight per thread
    for (int i0 = threadIdx.x; i0 < n4; i0 += kStatThreads * kU) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kStatThreads;
        v[u] = i < n4 ? __ldcs(z4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kStatThreads;
        if (i < n4) take4(v[u].x, v[u].y, v[u].z, v[u].w, 4 * i);
      }
    }
  } else {
    for (int y = threadIdx.x; y < V; y += kStatThreads) {
      const float x = z[y];
      nan_seen |= isnan(x);
      if (want_argmax) {
        argmax_merge(bv, bi, x, y);
      } else {
        const float yv = x * inv_t;
        lse_add4(m, s, yv, -INFINITY, -INFINITY, -INFINITY);
      }
    }
  }
  if (want_argmax) {
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
    int32_t* __restrict__ out_tokens, VerifyReq* __restrict__ req, int32_t* __restrict__ excl_out,
    const float* __restrict__ st_max, const float* __restrict__ st_sumexp,
    const float* __restrict__ child_logit, const int32_t* __restrict__ race_ids, int race_k,
    int32_t* dev_status) {
  // statistics mode (race_ids != NULL): row max / sum-exp, the target logit
  // of each child's token and each row's sorted race candidates come from
  // the verification LM head; no logits are read
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  __shared__ int s_parent[kMaxVerifyRows];
  __shared__ int s_token[kMaxVerifyRows];
  __shared__ int s_amax[kMaxVerifyRows];      // greedy: argmax of row i
  __shared__ float s_zt[kMaxVerifyRows];      // z[parent(i), token(i)]
  __shared__ RowStat s_stat[kMaxVerifyRows];  // (max, sum-exp) of row i
  __shared__ float s_u[kMaxVerifyRows];       // accept-test uniform of row i
  __shared__ int s_excl[kMaxVerifyRows];
  __shared__ int s_ch[kMaxVerifyRows];         // children of the current row
  __shared__ int s_path[65];
  __shared__ int s_nexcl, s_stop, s_plen, s_bad;

  // the [B, R] row arrays are read for all R rows beside the row count, not
  // after it (rows past the count go unused)
  constexpr int kRowsPerThread = kMaxVerifyRows / kWalkThreads;
  const int32_t* am_src = target_argmax ? target_argmax : ws_argmax;
  int pre_p[kRowsPerThread], pre_t[kRowsPerThread], pre_a[kRowsPerThread];
  float pre_m[kRowsPerThread], pre_s[kRowsPerThread], pre_z[kRowsPerThread];
#pragma unroll
  for (int h = 0; h < kRowsPerThread; ++h) {
    const int i = h * kWalkThreads + threadIdx.x;
    if (i < R) {
      const size_t gi = (size_t)b * R + i;
      pre_p[h] = parent_row[gi];
      pre_t[h] = token[gi];
      if (greedy) {
        pre_a[h] = am_src[gi];
      } else if (race_ids) {
        pre_m[h] = st_max[gi];
        pre_s[h] = st_sumexp[gi];
        pre_z[h] = child_logit[gi];
      }
    }
  }
  const int n = n_rows ? n_rows[b] : R;
  if (threadIdx.x == 0) s_bad = (n < 1 || n > R) ? 1 : 0;
  __syncthreads();
  const int nn = s_bad ? 1 : n;
#pragma unroll
  for (int h = 0; h < kRowsPerThread; ++h) {
    const int i = h * kWalkThreads + threadIdx.x;
    if (i >= nn) continue;
    const size_t gi = (size_t)b * R + i;
    const int p = pre_p[h];
    const int t = pre_t[h];
    s_parent[i] = p;
    s_token[i] = t;
    const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i && t >= 0 && t < V);
    if (!ok) atomicExch(&s_bad, 1);
    if (greedy) {
      s_amax[i] = pre_a[h];
    } else if (race_ids) {
      s_stat[i] = RowStat{pre_m[h], pre_s[h]};
      s_zt[i] = pre_z[h];
    } else {
      s_stat[i] = stats[gi];
      s_zt[i] = (i > 0 && ok) ? logits[((size_t)b * R + p) * V + t] : 0.f;
    }
    if (!greedy) {
      if (uniforms_override) {
        s_u[i] = uniforms_override[gi];
      } else {
        const uint4 w =
            philox4x32_10(make_uint4((uint32_t)i, (uint32_t)b, ctr2_accept, ctr3), key0, key1);
        s_u[i] = bits_to_uniform(w.x);
      }
    }
  }
  __syncthreads();

  // the walk, by warp 0: the children of the current row are found 32 rows at
  // a time with ballots; the stochastic accept chain over them runs on lane 0
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int plen = 1, cur = 0, bad = s_bad, nex = 0;
    if (lane == 0) s_path[0] = 0;
    while (!bad) {
      int accepted = -1;
      if (greedy) {
        const int a = s_amax[cur];
        for (int c0 = cur + 1; c0 < nn && accepted < 0; c0 += 32) {
          const int c = c0 + lane;
          const unsigned hit =
              __ballot_sync(0xffffffffu, c < nn && s_parent[c] == cur && s_token[c] == a);
          if (hit) accepted = c0 + __ffs(hit) - 1;
        }
      } else {
        int nch = 0;  // children of cur, in row order, into s_ch
        for (int c0 = cur + 1; c0 < nn; c0 += 32) {
          const int c = c0 + lane;
          const bool is_child = c < nn && s_parent[c] == cur;
          const unsigned m = __ballot_sync(0xffffffffu, is_child);
          if (is_child) s_ch[nch + __popc(m & ((1u << lane) - 1u))] = c;
          nch += __popc(m);
        }
        __syncwarp();
        if (lane == 0) {
          const RowStat st = s_stat[cur];
          float rem = 1.f;  // probability mass not yet rejected
          nex = 0;
          for (int j = 0; j < nch; ++j) {
            const int c = s_ch[j];
            const int t = s_token[c];
            bool dup = false;
            for (int e = 0; e < nex; ++e) dup |= (s_excl[e] == t);
            const float pt = dup ? 0.f : exp2f((s_zt[c] * inv_t - st.m) * kLog2e) / st.s;
            const float ratio = pt / rem;
            if (s_u[c] < ratio) {
              accepted = c;
              break;
            }
            if (!dup && rem - pt > 0.f) {
              rem -= pt;
              s_excl[nex++] = t;
            }
          }
        }
        accepted = __shfl_sync(0xffffffffu, accepted, 0);
        nex = __shfl_sync(0xffffffffu, nex, 0);
        __syncwarp();
      }
      if (accepted < 0) break;
      if (plen > max_depth) {
        bad = 2;
        break;
      }
      if (lane == 0) s_path[plen] = accepted;
      ++plen;
      cur = accepted;
    }
    if (lane == 0) {
      s_stop = cur;
      s_plen = plen;
      s_nexcl = greedy ? 0 : nex;
      if (bad) s_bad = bad;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      set_status(dev_status, EAGLE_ERR_BAD_TREE);
      accept_len[b] = 0;
      if (req) req[b] = VerifyReq{-1, 0, 0, 0};
    }
    for (int i = threadIdx.x; i <= max_depth; i += kWalkThreads) {
      path_rows[(size_t)b * (max_depth + 1) + i] = (i == 0) ? 0 : -1;
      out_tokens[(size_t)b * (max_depth + 1) + i] = -1;
    }
    return;
  }
  const int plen = s_plen, stop = s_stop;
  if (!greedy && race_ids && threadIdx.x == 0) {
    // the race winner at the stop row: its first candidate not rejected there
    const int nex = s_nexcl;
    int bonus = -1;
    for (int j = 0; j < race_k && bonus < 0; ++j) {
      const int y = race_ids[((size_t)b * R + stop) * race_k + j];
      bool ex = y < 0;
      for (int e = 0; e < nex; ++e) ex |= (s_excl[e] == y);
      if (!ex) bonus = y;
    }
    if (bonus < 0) set_status(dev_status, EAGLE_ERR_INVALID_ARG);  // race_k too small
    s_amax[stop] = bonus;
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= max_depth; i += kWalkThreads) {
    const size_t o = (size_t)b * (max_depth + 1) + i;
    path_rows[o] = i < plen ? s_path[i] : -1;
    if (i + 1 < plen)
      out_tokens[o] = s_token[s_path[i + 1]];
    else if (i + 1 > plen)
      out_tokens[o] = -1;
    else if (greedy || race_ids)
      out_tokens[o] = s_amax[stop];  // the bonus token; the race kernel writes it otherwise
  }
  if (!greedy && !race_ids) {
    const int nex = s_nexcl;
    for (int e = threadIdx.x; e < nex; e += kWalkThreads) excl_out[(size_t)b * R + e] = s_excl[e];
    if (threadIdx.x == 0) req[b] = VerifyReq{stop, plen, nex, 0};
  }
  if (threadIdx.x == 0) accept_len[b] = plen - 1;
}

// Exponential race over the ids not rejected at the stop row:
// bonus = argmax_y z_y/T - log(-log u_y), ties to the lower id.
__global__ void __launch_bounds__(kRaceThreads) verify_race_kernel(
    int R, int V, const float* __restrict__ logits, VerifyReq* __restrict__ req,
    const int32_t* __restrict__ excl, RacePart* __restrict__ part, float inv_t, uint32_t key0,
    uint32_t key1, uint32_t ctr2_race, uint32_t ctr3, int max_depth,
    int32_t* __restrict__ out_tokens, int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, cx = blockIdx.y, C = gridDim.y;
  const VerifyReq q = req[b];
  if (q.stop < 0) return;
  const int lo = cx * kRaceChunk, hi = min(V, lo + kRaceChunk);
  __shared__ uint32_t s_bits[kRaceChunk / 32];  // excluded ids of this chunk
  __shared__ float s_rv[kRaceThreads / 32];
  __shared__ int s_ri[kRaceThreads / 32];
  __shared__ int s_last;
  for (int i = threadIdx.x; i < kRaceChunk / 32; i += kRaceThreads) s_bits[i] = 0u;
  __syncthreads();
  for (int e = threadIdx.x; e < q.nexcl; e += kRaceThreads) {
    const int y = excl[(size_t)b * R + e];
    if (y >= lo && y < hi) atomicOr(&s_bits[(y - lo) >> 5], 1u << ((y - lo) & 31));
  }
  __syncthreads();
  const float* z = logits + ((size_t)b * R + q.stop) * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool nan_seen = false;
  for (int g = lo / 4 + threadIdx.x; g * 4 < hi; g += kRaceThreads) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)g, (uint32_t)b, ctr2_race, ctr3), key0, key1);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int y = g * 4 + j;
      if (y >= hi) break;
      if ((s_bits[(y - lo) >> 5] >> ((y - lo) & 31)) & 1u) continue;
      const float zy = z[y];
      nan_seen |= isnan(zy);
      const float u = bits_to_uniform(words[j]);
      argmax_merge(bv, bi, zy * inv_t - logf(-logf(u)), y);
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
    for (int w = 1; w < kRaceThreads / 32; ++w) argmax_merge(bv, bi, s_rv[w], s_ri[w]);
    part[(size_t)b * C + cx] = RacePart{bv, bi};
    __threadfence();
    s_last = atomicAdd(&req[b].ticket, 1) == C - 1;
  }
  __syncthreads();
  if (!s_last) return;
  // the last chunk of this request to finish merges the chunk winners
  __threadfence();
  float mv = -INFINITY;
  int mi = 0x7fffffff;
  for (int c = threadIdx.x; c < C; c += kRaceThreads) {
    const float pk = __ldcg(&part[(size_t)b * C + c].key);
    const int pi = __ldcg(&part[(size_t)b * C + c].id);
    argmax_merge(mv, mi, pk, pi);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, mv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
    argmax_merge(mv, mi, ov, oi);
  }
  if ((threadIdx.x & 31) == 0) {
    s_rv[threadIdx.x >> 5] = mv;
    s_ri[threadIdx.x >> 5] = mi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kRaceThreads / 32; ++w) argmax_merge(mv, mi, s_rv[w], s_ri[w]);
    out_tokens[(size_t)b * (max_depth + 1) + q.plen - 1] = mi;
    req[b].ticket = 0;
  }
}

// Sampled proposals ([E1] Algorithm 1 verbatim): the siblings under a row
// were drawn i.i.d. from q = softmax(draft logits / T) of that row.  Child t
// is accepted when u < p(t) / q(t), with p the current target distribution;
// after a rejection p <- norm(max(0, p - q)) (p unchanged when that mass is
// 0); if every child is rejected the bonus token is the exponential race
// argmax_y p(y) / E_y, E_y = -log u_y, over the final p (the race in ratio
// form: the same argmax as log p(y) - log(-log u_y)).
//
// The residual is never stored.  All siblings of a row share q, so after r
// rejections p_r = max(0, p_0 - c_r q) / S_r exactly, with c_0 = 0, S_0 = 1,
// c_{r+1} = c_r + S_r and S_{r+1} = sum_y max(0, p_0(y) - c_{r+1} q(y)) (the
// step is skipped when that sum is 0): by induction, max(0, p_r - q) =
// max(0, p_0 - (c_r + S_r) q) / S_r, since p_0 - c_r q <= 0 implies
// p_0 - (c_r + S_r) q < 0.  The race drops the common 1 / S_r.
//
// One thread-block cluster of `cs` CTAs per request (cs = 1..8, chosen so
// that the clusters fill the SMs); CTA k of the cluster owns the k-th slice
// of the vocabulary (16-byte groups of 4 ids).  Every CTA runs the whole walk
// in step; a vocabulary-wide quantity is reduced per CTA and the cs partials
// are exchanged through distributed shared memory behind one cluster barrier
// (two exchange slots used alternately, so one barrier per exchange
// suffices), each CTA combining them in rank order, so all CTAs take the same
// decisions.  Per visited row: one pass for the row statistics of p_0 and q
// (max and sum of 2^(z T^-1 log2 e - max), both rows), then per rejection one
// pass for S_{r+1}; the last rejection's pass is folded into the race pass,
// which keeps the race winners for both c_r and c_{r+1}.  Rows the walk does
// not visit are never read.
constexpr int kSampThreads = 1024;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kSampMaxCluster = 8;
constexpr int kSampUnroll = 4;         // 16-byte loads per logit row in flight per thread
constexpr int kRaceUnroll = 2;         // the same in the race pass (Philox keeps more registers live)
constexpr int kSampMinGroups = 256;    // vocabulary groups per CTA, at least (host choice of cs)
constexpr int kNoWinner = 0x7fffffff;
static_assert(kSampWarps == 32, "cluster_reduce folds one value per warp in warp 0");

// Online (max, sum 2^(y - max)) of four base-2 values.
__device__ __forceinline__ void lse2_add4(float& m, float& s, float y0, float y1, float y2, float y3) {
  const float m4 = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
  if (m4 > m) {
    s *= exp2f(m - m4);
    m = m4;
  }
  if (m != -INFINITY) s += exp2f(y0 - m) + exp2f(y1 - m) + exp2f(y2 - m) + exp2f(y3 - m);
}
__device__ __forceinline__ void lse2_merge(float& m, float& s, float om, float os) {
  const float nm = fmaxf(m, om);
  s = (m == -INFINITY ? 0.f : s * exp2f(m - nm)) + (om == -INFINITY ? 0.f : os * exp2f(om - nm));
  m = nm;
}

// Combination rules of the exchanged float4s (commutative, so a butterfly
// leaves every lane with the same value).
struct CombLse {  // (max, sum) of the target row in .xy, of the draft row in .zw
  __device__ void operator()(float4& a, const float4& b) const {
    lse2_merge(a.x, a.y, b.x, b.y);
    lse2_merge(a.z, a.w, b.z, b.w);
  }
};
struct CombSum {
  __device__ void operator()(float4& a, const float4& b) const { a.x += b.x; }
};
struct CombRace {  // two (key, id) winners: .xy and .zw, ids as bit patterns
  __device__ void operator()(float4& a, const float4& b) const {
    int i0 = __float_as_int(a.y), i1 = __float_as_int(a.w);
    argmax_merge(a.x, i0, b.x, __float_as_int(b.y));
    argmax_merge(a.z, i1, b.z, __float_as_int(b.w));
    a.y = __int_as_float(i0);
    a.w = __int_as_float(i1);
  }
};

__device__ __forceinline__ float4 shfl_xor4(float4 v, int o) {
  return make_float4(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o),
                     __shfl_xor_sync(0xffffffffu, v.z, o), __shfl_xor_sync(0xffffffffu, v.w, o));
}

// Reduces v over the CTA, exchanges the CTA results through slot `xb` of
// every CTA of the cluster and returns their rank-order combination (the
// same value in every thread of every CTA).  Every thread must call it.
template <class Op>
__device__ __forceinline__ float4 cluster_reduce(float4 v, Op op, float4* s_red, float4* s_x, int& xb,
                                                 int cs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) op(v, shfl_xor4(v, o));
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = s_red[lane];
#pragma unroll
    for (int o = 16; o; o >>= 1) op(v, shfl_xor4(v, o));
    if (lane == 0) s_x[xb] = v;
  }
  cluster_barrier();
  float4 r = ld_cluster_f4(&s_x[xb], 0);
  for (int k = 1; k < cs; ++k) op(r, ld_cluster_f4(&s_x[xb], (uint32_t)k));
  xb ^= 1;
  return r;
}

// Streams groups [g0, g1) of two logit rows, U 16-byte loads per row in
// flight per thread, and calls f(z4, zd4, g) per group; ids >= V read as -inf.
template <int U, class F>
__device__ __forceinline__ void stream_rows(const float* z, const float* zd, int g0, int g1, int V, bool vec,
                                            F&& f) {
  const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  auto ld = [&](const float* row, int g) -> float4 {
    if (vec) return __ldg(reinterpret_cast<const float4*>(row) + g);
    const int y = 4 * g;
    return make_float4(row[y], y + 1 < V ? row[y + 1] : -INFINITY, y + 2 < V ? row[y + 2] : -INFINITY,
                       y + 3 < V ? row[y + 3] : -INFINITY);
  };
  for (int i0 = g0 + (int)threadIdx.x; i0 < g1; i0 += kSampThreads * U) {
    float4 a[U], d[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = i0 + u * kSampThreads;
      a[u] = g < g1 ? ld(z, g) : ninf;
      d[u] = g < g1 ? ld(zd, g) : ninf;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = i0 + u * kSampThreads;
      if (g < g1) f(a[u], d[u], g);
    }
  }
}

__global__ void __launch_bounds__(kSampThreads, 1) verify_walk_sampled_kernel(
    int R, int V, int cs, const int32_t* __restrict__ parent_row, const int32_t* __restrict__ token,
    const int32_t* __restrict__ n_rows, const float* __restrict__ logits,
    const float* __restrict__ draft, float inv_t, uint32_t key0, uint32_t key1, uint32_t ctr2_accept,
    uint32_t ctr3, const float* __restrict__ uniforms_override, int max_depth,
    int32_t* __restrict__ accept_len, int32_t* __restrict__ path_rows, int32_t* __restrict__ out_tokens,
    int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x / cs, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster_ctarank();
  __shared__ int s_parent[kMaxVerifyRows];
  __shared__ int s_token[kMaxVerifyRows];
  __shared__ float s_u[kMaxVerifyRows];
  __shared__ int s_ch[kMaxVerifyRows];
  __shared__ int s_path[65];
  __shared__ float4 s_red[kSampWarps];
  __shared__ float4 s_x[2];
  __shared__ int s_bad, s_nch, s_acc;

  const int n = n_rows ? n_rows[b] : R;
  if (tid == 0) s_bad = (n < 1 || n > R) ? 1 : 0;
  __syncthreads();
  const int nn = s_bad ? 1 : n;
  for (int i = tid; i < nn; i += kSampThreads) {
    const size_t gi = (size_t)b * R + i;
    const int p = parent_row[gi], t = token[gi];
    s_parent[i] = p;
    s_token[i] = t;
    if (!((i == 0) ? (p == -1) : (p >= 0 && p < i && t >= 0 && t < V))) atomicExch(&s_bad, 1);
    if (uniforms_override) {
      s_u[i] = uniforms_override[gi];
    } else {
      const uint4 w = philox4x32_10(make_uint4((uint32_t)i, (uint32_t)b, ctr2_accept, ctr3), key0, key1);
      s_u[i] = bits_to_uniform(w.x);
    }
  }
  __syncthreads();
  // this CTA's vocabulary slice, in groups of 4 ids
  const int G = (V + 3) / 4;
  const int g0 = (int)((long long)G * rank / cs), g1 = (int)((long long)G * (rank + 1) / cs);
  const float at = inv_t * kLog2e;  // z T^-1 in base 2
  const bool vec = (V & 3) == 0;
  int xb = 0;  // exchange slot of the next cluster_reduce
  int bad = s_bad, cur = 0, plen = 1;
  bool nan_seen = false;
  // row cur: p_0(y) = 2^(z at - pm) ips, q(y) = 2^(zd at - qm) iqs; the
  // residual is max(0, p_0 - c q) / S; `pending`: the last child was rejected
  // and S_{r+1} is not formed yet
  float pm = 0.f, ips = 1.f, qm = 0.f, iqs = 1.f, c = 0.f, S = 1.f;
  bool pending = false;
  if (tid == 0) s_path[0] = 0;
  while (!bad) {
    // the children of cur in row order (warp 0, by ballots)
    if (warp == 0) {
      int nch = 0;
      for (int c0 = cur + 1; c0 < nn; c0 += 32) {
        const int ch = c0 + lane;
        const bool is_child = ch < nn && s_parent[ch] == cur;
        const unsigned m = __ballot_sync(0xffffffffu, is_child);
        if (is_child) s_ch[nch + __popc(m & ((1u << lane) - 1u))] = ch;
        nch += __popc(m);
      }
      if (lane == 0) s_nch = nch;
    }
    const float* z = logits + ((size_t)b * R + cur) * V;
    const float* zd = draft + ((size_t)b * R + cur) * V;
    {  // row statistics of p_0 and q
      float4 v = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      stream_rows<kSampUnroll>(z, zd, g0, g1, V, vec, [&](const float4& a, const float4& d, int) {
        nan_seen |= isnan(a.x) | isnan(a.y) | isnan(a.z) | isnan(a.w) | isnan(d.x) | isnan(d.y) |
                    isnan(d.z) | isnan(d.w);
        lse2_add4(v.x, v.y, a.x * at, a.y * at, a.z * at, a.w * at);
        lse2_add4(v.z, v.w, d.x * at, d.y * at, d.z * at, d.w * at);
      });
      v = cluster_reduce(v, CombLse{}, s_red, s_x, xb, cs);  // also publishes s_nch, s_ch
      pm = v.x;
      ips = 1.f / v.y;
      qm = v.z;
      iqs = 1.f / v.w;
    }
    const int nch = s_nch;
    c = 0.f;
    S = 1.f;
    pending = false;
    int accepted = -1;
    for (int j = 0; j < nch; ++j) {
      if (pending) {  // S_{r+1} = sum_y max(0, p_0 - (c + S) q)
        const float c2 = c + S;
        float acc = 0.f;
        stream_rows<kSampUnroll>(z, zd, g0, g1, V, vec, [&](const float4& a, const float4& d, int) {
          acc += fmaxf(0.f, fmaf(-c2, exp2f(fmaf(d.x, at, -qm)) * iqs, exp2f(fmaf(a.x, at, -pm)) * ips));
          acc += fmaxf(0.f, fmaf(-c2, exp2f(fmaf(d.y, at, -qm)) * iqs, exp2f(fmaf(a.y, at, -pm)) * ips));
          acc += fmaxf(0.f, fmaf(-c2, exp2f(fmaf(d.z, at, -qm)) * iqs, exp2f(fmaf(a.z, at, -pm)) * ips));
          acc += fmaxf(0.f, fmaf(-c2, exp2f(fmaf(d.w, at, -qm)) * iqs, exp2f(fmaf(a.w, at, -pm)) * ips));
        });
        const float tot = cluster_reduce(make_float4(acc, 0.f, 0.f, 0.f), CombSum{}, s_red, s_x, xb, cs).x;
        if (tot > 0.f) {  // a zero mass keeps p (a probability-zero event in exact arithmetic)
          c = c2;
          S = tot;
        }
        pending = false;
      }
      if (tid == 0) {
        const int ch = s_ch[j], t = s_token[ch];
        const float p0 = exp2f(fmaf(z[t], at, -pm)) * ips;
        const float q = exp2f(fmaf(zd[t], at, -qm)) * iqs;
        const float pv = fmaxf(0.f, fmaf(-c, q, p0)) / S;
        const float ratio = q > 0.f ? pv / q : (pv > 0.f ? INFINITY : 0.f);
        s_acc = s_u[ch] < ratio ? ch : -1;
      }
      __syncthreads();
      accepted = s_acc;
      __syncthreads();  // s_acc is rewritten by the next test
      if (accepted >= 0) break;
      pending = true;
    }
    if (accepted < 0) break;
    if (plen > max_depth) {
      bad = 2;
      break;
    }
    if (tid == 0) s_path[plen] = accepted;
    ++plen;
    cur = accepted;
  }
  int bonus = -1;
  if (!bad) {
    // bonus: argmax_y max(0, p_0 - c q) / E_y at the stop row, and with
    // c + S when a rejection is pending (used when its mass is positive)
    const float* z = logits + ((size_t)b * R + cur) * V;
    const float* zd = draft + ((size_t)b * R + cur) * V;
    const float c2 = c + S;
    float4 v = make_float4(-INFINITY, __int_as_float(kNoWinner), -INFINITY, __int_as_float(kNoWinner));
    int bi = kNoWinner, bi2 = kNoWinner;
    stream_rows<kRaceUnroll>(z, zd, g0, g1, V, vec, [&](const float4& a, const float4& d, int g) {
      const uint4 w = philox4x32_10(make_uint4((uint32_t)g, (uint32_t)b, ctr2_accept + 1u, ctr3), key0, key1);
      const uint32_t words[4] = {w.x, w.y, w.z, w.w};
      const float za[4] = {a.x, a.y, a.z, a.w}, zq[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int y = 4 * g + k;
        const float p0 = exp2f(fmaf(za[k], at, -pm)) * ips, q = exp2f(fmaf(zq[k], at, -qm)) * iqs;
        const float r = 1.f / -logf(bits_to_uniform(words[k]));
        const float a1 = fmaf(-c, q, p0);
        if (a1 > 0.f && y < V) argmax_merge(v.x, bi, a1 * r, y);
        if (pending) {
          const float a2 = fmaf(-c2, q, p0);
          if (a2 > 0.f && y < V) argmax_merge(v.z, bi2, a2 * r, y);
        }
      }
    });
    v.y = __int_as_float(bi);
    v.w = __int_as_float(bi2);
    v = cluster_reduce(v, CombRace{}, s_red, s_x, xb, cs);
    bi = __float_as_int(v.y);
    bi2 = __float_as_int(v.w);
    const int win = (pending && bi2 != kNoWinner) ? bi2 : bi;
    bonus = win == kNoWinner ? -1 : win;
  }
  if (nan_seen) set_status(dev_status, EAGLE_ERR_NONFINITE);
  if (rank == 0) {
    if (bad) {
      if (tid == 0) {
        set_status(dev_status, EAGLE_ERR_BAD_TREE);
        accept_len[b] = 0;
      }
      for (int i = tid; i <= max_depth; i += kSampThreads) {
        path_rows[(size_t)b * (max_depth + 1) + i] = (i == 0) ? 0 : -1;
        out_tokens[(size_t)b * (max_depth + 1) + i] = -1;
      }
    } else {
      __syncthreads();  // s_path
      for (int i = tid; i <= max_depth; i += kSampThreads) {
        const size_t o = (size_t)b * (max_depth + 1) + i;
        path_rows[o] = i < plen ? s_path[i] : -1;
        out_tokens[o] = i + 1 < plen ? s_token[s_path[i + 1]] : (i + 1 == plen ? bonus : -1);
      }
      if (tid == 0) accept_len[b] = plen - 1;
    }
  }
  cluster_barrier();  // no CTA leaves while a peer may still read its exchange slots
}

int race_chunks(int V) { return (V + kRaceChunk - 1) / kRaceChunk; }

// Workspace layout shared by eagle_tree_verify (caller buffer) and the
// allocation-free variant (library buffer).
struct VerifyScratch {
  RowStat* stats;
  int32_t* amax;
  int32_t* excl;
  VerifyReq* req;
  RacePart* part;
};


size_t scratch_bytes(int B, int R, int V) {
  return round_up((size_t)B * R * sizeof(RowStat), 256) + round_up((size_t)B * R * 4, 256) * 2 +
         round_up((size_t)B * sizeof(VerifyReq), 256) +
         round_up((size_t)B * race_chunks(V) * sizeof(RacePart), 256) + 256;
}

VerifyScratch carve_scratch(void* base, int B, int R, int V, bool race) {
  char* cur = static_cast<char*>(base);
  VerifyScratch w;
  w.stats = static_cast<RowStat*>(ws_carve(cur, (size_t)B * R * sizeof(RowStat)));
  w.amax = static_cast<int32_t*>(ws_carve(cur, (size_t)B * R * 4));
  w.excl = static_cast<int32_t*>(ws_carve(cur, (size_t)B * R * 4));
  w.req = static_cast<VerifyReq*>(ws_carve(cur, (size_t)B * sizeof(VerifyReq)));
  w.part = race ? static_cast<RacePart*>(ws_carve(cur, (size_t)B * race_chunks(V) * sizeof(RacePart)))
               : nullptr;
  return w;
}

// Host-side argument checks common to both entry points.
int verify_check(int B, int R, int V, const int32_t* parent_row, const int32_t* token,
                 const float* target_logits, const int32_t* target_argmax,
                 const float* draft_logits, float temperature,
                 int proposal_mode, uint64_t offset, int max_depth, const int32_t* accept_len,
                 const int32_t* path_rows, const int32_t* out_tokens) {
  if (B <= 0 || R <= 0 || V < 2 || max_depth < 0) return EAGLE_ERR_INVALID_ARG;
  if (!parent_row || !token || !accept_len || !path_rows || !out_tokens) return EAGLE_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || isinf(temperature)) return EAGLE_ERR_INVALID_ARG;
  if (proposal_mode != EAGLE_PROPOSAL_DETERMINISTIC && proposal_mode != EAGLE_PROPOSAL_SAMPLED)
    return EAGLE_ERR_INVALID_ARG;
  const bool greedy = temperature == 0.f;
  if (proposal_mode == EAGLE_PROPOSAL_SAMPLED && (greedy || !draft_logits)) return EAGLE_ERR_INVALID_ARG;
  if (greedy && !target_logits && !target_argmax) return EAGLE_ERR_INVALID_ARG;
  if (!greedy && !target_logits) return EAGLE_ERR_INVALID_ARG;
  if (R > kMaxVerifyRows || max_depth > 64) return EAGLE_ERR_UNSUPPORTED;
  if ((offset >> 63) != 0) return EAGLE_ERR_INVALID_ARG;
  if ((long long)B * R > 2147483647LL) return EAGLE_ERR_UNSUPPORTED;
  if (!greedy && race_chunks(V) > 65535) return EAGLE_ERR_UNSUPPORTED;
  return EAGLE_OK;
}

// Enqueues the kernels of one verification (arguments already checked).
int verify_enqueue(int B, int R, int V, const int32_t* parent_row, const int32_t* token,
                   const int32_t* n_rows, const float* target_logits,
                   const int32_t* target_argmax, const float* draft_logits, int proposal_mode,
                   float temperature, uint64_t seed, uint64_t offset,
                   const float* uniforms_override, int max_depth, int32_t* accept_len,
                   int32_t* path_rows, int32_t* out_tokens, const VerifyScratch& w,
                   int32_t* dev_status, cudaStream_t s) {
  const bool greedy = temperature == 0.f;
  const bool need_stats = !greedy || !target_argmax;
  const float inv_t = greedy ? 0.f : 1.f / temperature;
  const uint32_t off_hi = (uint32_t)(offset >> 32), off_lo = (uint32_t)offset;
  const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
  if (proposal_mode == EAGLE_PROPOSAL_SAMPLED) {
    // a cluster of cs CTAs per request: clusters that fill the SMs, at least
    // kSampMinGroups vocabulary groups per CTA
    const int G = (V + 3) / 4, sms = sm_count();
    int cs = 1;
    while (cs < kSampMaxCluster && 2LL * B * cs <= sms && 2LL * cs * kSampMinGroups <= G) cs *= 2;
    launch_cluster(verify_walk_sampled_kernel, (unsigned)(B * cs), kSampThreads, dim3((unsigned)cs), 0, s, R, V,
                   cs, parent_row, token, n_rows, target_logits, draft_logits, inv_t, key0, key1,
                   2u * off_hi, off_lo, uniforms_override, max_depth, accept_len, path_rows, out_tokens,
                   dev_status);
    note_launch();
    return last_launch_status();
  }
  if (need_stats) {
    launch(verify_rowstats_kernel, (unsigned)(B * R), kStatThreads, 0, s, target_logits, n_rows, R,
           V, inv_t, greedy ? 1 : 0, w.stats, w.amax, dev_status);
    note_launch();
  }
  launch(verify_walk_kernel, B, kWalkThreads, 0, s, R, V, parent_row, token, n_rows, target_logits,
         target_argmax, need_stats ? w.stats : nullptr, need_stats ? w.amax : nullptr,
         greedy ? 1 : 0, inv_t, key0, key1, 2u * off_hi, off_lo, uniforms_override, max_depth,
         accept_len, path_rows, out_tokens, greedy ? nullptr : w.req,
         greedy ? nullptr : w.excl, (const float*)nullptr, (const float*)nullptr,
         (const float*)nullptr, (const int32_t*)nullptr, 0, dev_status);
  note_launch();
  if (!greedy) {
    launch(verify_race_kernel, dim3((unsigned)B, (unsigned)race_chunks(V)), kRaceThreads, 0, s, R,
           V, target_logits, w.req, w.excl, w.part, inv_t, key0, key1, 2u * off_hi + 1u, off_lo,
           max_depth, out_tokens, dev_status);
    note_launch();
  }
  return last_launch_status();
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_verify_workspace_size(int B, int R, int V) {
  if (B <= 0 || R <= 0 || V < 2) return 0;
  return scratch_bytes(B, R, V);
}

extern "C" int eagle_tree_verify(int B, int R, int V, const int32_t* parent_row,
                                 const int32_t* token, const int32_t* n_rows,
                                 const float* target_logits, const int32_t* target_argmax,
                                 const float* draft_logits, float temperature, int proposal_mode,
                                 uint64_t seed, uint64_t offset, const float* uniforms_override,
                                 int max_depth, int32_t* accept_len, int32_t* path_rows,
                                 int32_t* out_tokens, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, void* stream) {
  const int chk = verify_check(B, R, V, parent_row, token, target_logits, target_argmax,
                               draft_logits, temperature, proposal_mode, offset, max_depth,
                               accept_len, path_rows, out_tokens);
  if (chk != EAGLE_OK) return chk;
  const bool need_ws = temperature != 0.f || !target_argmax;
  VerifyScratch w{};
  if (need_ws) {
    if (!ws || ws_bytes < eagle_tree_verify_workspace_size(B, R, V)) return EAGLE_ERR_WORKSPACE;
    w = carve_scratch(ws, B, R, V, temperature != 0.f);
  }
  return verify_enqueue(B, R, V, parent_row, token, n_rows, target_logits, target_argmax,
                        draft_logits, proposal_mode, temperature, seed, offset, uniforms_override,
                        max_depth, accept_len,
                        path_rows, out_tokens, w, dev_status, static_cast<cudaStream_t>(stream));
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

constexpr int kNoAllocMaxRows = 65536;    // B * R rows of statistics
constexpr int kNoAllocMaxChunks = 65536;  // B * ceil(V / 4096) race chunks
constexpr size_t kNoAllocScratchBytes =
    (size_t)kNoAllocMaxRows * sizeof(RowStat) + (size_t)kNoAllocMaxRows * 4 * 2 +
    (size_t)kNoAllocMaxRows * sizeof(VerifyReq) + (size_t)kNoAllocMaxChunks * sizeof(RacePart) +
    5 * 256;

// One copy per GPU that loads the library, kept until the process exits.
// Every call on a device shares it: two calls whose kernels overlap on that
// device (for example on two streams) race on it.  Nothing in it needs to
// start at zero: every statistic is written before it is read.
static __device__ __align__(256) unsigned char g_verify_scratch[kNoAllocScratchBytes];

// The buffer's device address belongs to the module loaded in one CUDA
// context, so it is cached per context, never per device ordinal: a caller
// may make a non-primary context current, and cudaDeviceReset destroys the
// primary context (a new one can even reuse the old handle).  A call made
// outside stream capture therefore looks the address up again and refreshes
// its context's entry; a call made during capture, when no lookup should be
// issued, uses the entry that an earlier call in the same context left, and
// fails cleanly if there is none.
constexpr int kNoAllocMaxContexts = 64;
struct ScratchEntry {
  CUcontext ctx;
  void* ptr;
};
ScratchEntry g_scratch_cache[kNoAllocMaxContexts];
int g_scratch_used = 0;
std::mutex g_scratch_mu;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

bool current_context(CUcontext* ctx) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  *ctx = nullptr;
  return g_ctx_current && g_ctx_current(ctx) == CUDA_SUCCESS && *ctx;
}

// Device address of g_verify_scratch in the current context, or nullptr with
// *st set.  In host code the symbol's name is only a host-side stand-in, so
// the address comes from cudaGetSymbolAddress, issued with the caller's
// device current.  A failed runtime call's error is taken out of the
// runtime's last-error slot, so that a later launch check does not report it.
void* noalloc_scratch(cudaStream_t stream, eagle_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    (void)cudaGetLastError();
    *st = EAGLE_ERR_CUDA;
    return nullptr;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    *st = EAGLE_ERR_CUDA;
    return nullptr;
  }
  CUcontext ctx = nullptr;
  if (!current_context(&ctx)) {
    // the runtime has not made a context current yet: only a lookup (which
    // initialises the primary context) can give the address
    if (cap != cudaStreamCaptureStatusNone) {
      *st = EAGLE_ERR_INVALID_ARG;
      return nullptr;
    }
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap != cudaStreamCaptureStatusNone) {
    for (int i = 0; i < g_scratch_used; ++i)
      if (g_scratch_cache[i].ctx == ctx) return g_scratch_cache[i].ptr;
    *st = EAGLE_ERR_INVALID_ARG;  // no call outside capture has run in this context
    return nullptr;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) {
    (void)cudaGetLastError();
    *st = EAGLE_ERR_CUDA;
    return nullptr;
  }
  if (!ctx && !current_context(&ctx)) return p;  // nothing to key the cache by
  for (int i = 0; i < g_scratch_used; ++i)
    if (g_scratch_cache[i].ctx == ctx) {
      g_scratch_cache[i].ptr = p;
      return p;
    }
  if (g_scratch_used < kNoAllocMaxContexts) {
    g_scratch_cache[g_scratch_used++] = ScratchEntry{ctx, p};
  } else {  // a full table: recycle the oldest slot
    for (int i = 1; i < kNoAllocMaxContexts; ++i) g_scratch_cache[i - 1] = g_scratch_cache[i];
    g_scratch_cache[kNoAllocMaxContexts - 1] = ScratchEntry{ctx, p};
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
  const int chk = verify_check(B, R, V, parent_row, token, target_logits, target_argmax,
                               draft_logits, temperature, proposal_mode, offset, max_depth,
                               accept_len, path_rows, out_tokens);
  if (chk != EAGLE_OK) return chk;
  // the built-in scratch holds kNoAllocMaxRows rows and kNoAllocMaxChunks
  // race chunks
  if ((long long)B * R > kNoAllocMaxRows ||
      (temperature != 0.f && (long long)B * race_chunks(V) > kNoAllocMaxChunks))
    return EAGLE_ERR_WORKSPACE;
  VerifyScratch w{};
  if (temperature != 0.f || !target_argmax) {
    eagle_status st = EAGLE_OK;
    void* base = noalloc_scratch(static_cast<cudaStream_t>(stream), &st);
    if (!base) return st;
    w = carve_scratch(base, B, R, V, temperature != 0.f);
  }
  return verify_enqueue(B, R, V, parent_row, token, n_rows, target_logits, target_argmax,
                        draft_logits, proposal_mode, temperature, seed, offset, uniforms_override,
                        max_depth, accept_len,
                        path_rows, out_tokens, w, dev_status, static_cast<cudaStream_t>(stream));
}

extern "C" int eagle_tree_verify_stats(int B, int R, int V, const int32_t* parent_row,
                                       const int32_t* token, const int32_t* n_rows,
                                       const float* row_max, const float* row_sumexp,
                                       const float* child_logit, const int32_t* race_ids,
                                       int race_k, float temperature, uint64_t seed,
                                       uint64_t offset, const float* uniforms_override,
                                       int max_depth, int32_t* accept_len, int32_t* path_rows,
                                       int32_t* out_tokens, int32_t* dev_status, void* stream) {
  if (B <= 0 || R <= 0 || V < 2 || max_depth < 0 || race_k < 1) return EAGLE_ERR_INVALID_ARG;
  if (!parent_row || !token || !row_max || !row_sumexp || !child_logit || !race_ids ||
      !accept_len || !path_rows || !out_tokens)
    return EAGLE_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || isinf(temperature)) return EAGLE_ERR_INVALID_ARG;
  if (R > kMaxVerifyRows || max_depth > 64) return EAGLE_ERR_UNSUPPORTED;
  if ((offset >> 63) != 0) return EAGLE_ERR_INVALID_ARG;
  if ((long long)B * R > 2147483647LL) return EAGLE_ERR_UNSUPPORTED;
  const uint32_t off_hi = (uint32_t)(offset >> 32), off_lo = (uint32_t)offset;
  launch(verify_walk_kernel, B, kWalkThreads, 0, static_cast<cudaStream_t>(stream), R, V,
         parent_row, token, n_rows, (const float*)nullptr, (const int32_t*)nullptr,
         (const RowStat*)nullptr, (const int32_t*)nullptr, 0, 1.f / temperature, (uint32_t)seed,
         (uint32_t)(seed >> 32), 2u * off_hi, off_lo, uniforms_override, max_depth, accept_len,
         path_rows, out_tokens, (VerifyReq*)nullptr, (int32_t*)nullptr, row_max, row_sumexp,
         child_logit, race_ids, race_k, dev_status);
  note_launch();
  return last_launch_status();
}
