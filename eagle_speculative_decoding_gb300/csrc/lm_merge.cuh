// Merge of the LM head's per-CTA partial results for one activation row,
// shared by the LM head's merge kernel and the EAGLE-2 expansion step that
// consumes the partials directly.
//
// Source: "EAGLE-3: Scaling up Inference Acceleration of Large Language
// Models via Training-Time Test", "Output path to LM head"; "M7.5 - EAGLE
// Feature Drafting ...", section 0x06B (confidence = the conditional token
// probability under the full vocabulary: log-prob = z / T - log sum exp(z / T)).
//
// Every CTA of the row's activation group left, for that row: the running
// (max of z/T, sum of exp(z/T - max)) over its vocabulary slice, its sorted
// top-K list (z descending, id ascending) and the list's length.
#pragma once

#include "common.cuh"

namespace eagle {

constexpr int kLmMaxCtas = 256;  // CTAs per activation group, at most

// Where one LM-head call left its partials ([row][cta] counts and (max, sum)
// pairs, [row][cta][K] values and ids), and how to read them.
struct LmPartials {
  const float2* ms;
  const float* v;
  const int* id;
  const int* cnt;
  int cpg;      // CTAs per activation group (lists per row)
  int K;        // list length
  float inv_t;  // 1 / temperature
  int race;     // race keys instead of logits (log-probs are not formed)
};

// Host side (gemm_tc.cu): the partials an eagle_lmhead_topk_partial call of
// shape (M, d, V, k, dtype, temperature) left in `ws`.  Returns false when the
// shape is outside the LM head's limits or the workspace is too small.
bool lm_partials_view(void* ws, size_t ws_bytes, int M, int d, int V, int k, int dtype,
                      float temperature, LmPartials* out);

// Order-preserving key of a non-NaN float: a larger value gets a larger key;
// -0 and +0 get the same key (they compare equal as floats).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp merges row m, whose lists were staged in shared memory (sv, si:
// [cpg][K]; sc: [cpg]) (lm_merge_row_ms below, with lm_merge_row loading
// the row's (max, sum) pairs first).  Log-sum-exp by max / rescale over the CTAs, then the
// top-K by K rounds of "best head among the CTAs' sorted lists".  Lane 0
// writes ids (-1 past the available candidates) and log-probs (z/T - lse, or
// the race key) to out_ids / out_lp (global or shared), and the row's max and
// sum when the pointers are set.  Every lane of the warp must call it.  The
// lists hold no NaN (the LM head never lists one).
constexpr int kLmMergePer = kLmMaxCtas / 32;  // lists owned per lane of the merging warp

// The (max, sum) pairs of row m's CTAs, lane-strided: lane l holds CTA
// l + 32 i in ms[i].  Issued by the merging warp; the loads may go out before
// the lists are staged.
__device__ __forceinline__ void lm_load_ms(const LmPartials& p, int m, float2 (&ms)[kLmMergePer]) {
  const int lane = threadIdx.x & 31;
  const float2* gms = p.ms + (size_t)m * p.cpg;
#pragma unroll
  for (int i = 0; i < kLmMergePer; ++i) {
    const int c = lane + 32 * i;
    ms[i] = c < p.cpg ? __ldcg(gms + c) : make_float2(-INFINITY, 0.f);
  }
}

// lm_merge_row with the row's (max, sum) pairs already loaded (lm_load_ms).
__device__ __forceinline__ void lm_merge_row_ms(const LmPartials& p, int m, const float2 (&ms)[kLmMergePer],
                                                const float* sv, const int* si, const int* sc, int32_t* out_ids,
                                                float* out_lp, float* row_max, float* row_sumexp) {
  const int lane = threadIdx.x & 31;
  const int K = p.K, nc = p.cpg;
  constexpr int kPer = kLmMergePer;
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) M = fmaxf(M, ms[i].x);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float S = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (ms[i].x != -INFINITY) S += ms[i].y * exp2f((ms[i].x - M) * 1.4426950408889634f);
#pragma unroll
  for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  float hv[kPer];
  int hi[kPer], hp[kPer], hc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int c = lane + 32 * i;
    hp[i] = 0;
    hc[i] = c < nc ? sc[c] : 0;
    hv[i] = hc[i] > 0 ? sv[c * K] : -INFINITY;
    hi[i] = hc[i] > 0 ? si[c * K] : 0x7fffffff;
  }
  const float lse = M + logf(S);
  // each lane keeps its best head (bv, bi) of list bs (-1: none left); only
  // the lane whose head wins a round advances that list and rescans its heads
  float bv;
  int bi, bs;
  auto lane_best = [&]() {
    bv = -INFINITY;
    bi = 0x7fffffff;
    bs = -1;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (hp[i] < hc[i] && better(hv[i], hi[i], bv, bi)) {
        bv = hv[i];
        bi = hi[i];
        bs = i;
      }
  };
  lane_best();
  for (int rnd = 0; rnd < K; ++rnd) {
    // the round's winner: the largest value (order-preserving key, -0 = +0),
    // then the smallest id among equal values
    const uint32_t key = bs >= 0 ? order_key(bv) : 0u;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const unsigned tie = __ballot_sync(0xffffffffu, bs >= 0 && key == kmax);
    if (tie == 0) {  // every list is exhausted
      if (lane == 0) {
        out_ids[rnd] = -1;
        out_lp[rnd] = -INFINITY;
      }
      continue;
    }
    int owner = __ffs(tie) - 1;
    if (tie & (tie - 1)) {
      const bool in = (tie >> lane) & 1u;
      const unsigned mid = __reduce_min_sync(0xffffffffu, in ? (unsigned)bi : 0xffffffffu);
      owner = __ffs(__ballot_sync(0xffffffffu, in && (unsigned)bi == mid)) - 1;
    }
    if (lane == owner) {
      out_ids[rnd] = bi;
      out_lp[rnd] = p.race ? bv : bv * p.inv_t - lse;
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (i == bs) {
          const int c = lane + 32 * i;
          ++hp[i];
          if (hp[i] < hc[i]) {
            hv[i] = sv[c * K + hp[i]];
            hi[i] = si[c * K + hp[i]];
          }
        }
      lane_best();
    }
  }
  if (lane == 0) {
    if (row_max) row_max[m] = M;
    if (row_sumexp) row_sumexp[m] = S;
  }
}

__device__ __forceinline__ void lm_merge_row(const LmPartials& p, int m, const float* sv, const int* si,
                                             const int* sc, int32_t* out_ids, float* out_lp, float* row_max,
                                             float* row_sumexp) {
  float2 ms[kLmMergePer];
  lm_load_ms(p, m, ms);
  lm_merge_row_ms(p, m, ms, sv, si, sc, out_ids, out_lp, row_max, row_sumexp);
}

}  // namespace eagle
