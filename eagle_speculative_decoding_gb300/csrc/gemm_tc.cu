// Tensor-core (tcgen05 + TMEM + TMA) GEMMs of the EAGLE hot path:
//   * eagle_lmhead_topk : z = W_U x with a per-row top-k / log-sum-exp
//     epilogue, so the [M, V] logits never reach HBM.
//   * eagle_fuse_proj   : g = W_proj [h_low; h_mid; h_high], the concatenation
//     walked by the K loop (three tensor maps), stream-K balanced.
//
// Sources: "EAGLE-3: Scaling up Inference Acceleration of Large Language
// Models via Training-Time Test", section 3.4 ("Change 2: The fusion FC
// layer"; "Output path to LM head"); "M7.5 - EAGLE Feature Drafting ...",
// sections 0x08B "Multi-Layer Feature Fusion" and 0x06B (confidence is the
// conditional token probability under the full vocabulary); "EAGLE: Speculative
// Sampling Requires Rethinking Feature Uncertainty", "Tree-Structured Draft
// Generation" (top-k tokens become the children).
//
// Both products are computed "swap-AB": the weight matrix is the MMA's A
// operand (M = 128 weight rows per tile) and the few activation rows are the
// B operand (N = 16..256 rows), so small batches waste no tensor-core rows and
// the kernel is a pure weight stream.  CTA layout (192 threads):
//   warp 0      TMA producer (one elected lane): weight + activation tiles,
//               128-byte swizzled, into an S-stage mbarrier ring
//   warp 1      TMEM allocator + MMA issuer (one lane): 4 MMAs per 128-byte K
//               chunk, accumulators double-buffered in tensor memory
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (lane = weight row)
// Every wait is bounded (2 s); on expiry the CTA records EAGLE_ERR_TIMEOUT,
// drains its copies and MMAs, frees tensor memory and exits.
// fp32 operands run on the CUDA cores in exact fp32 (the tensor cores would
// truncate them to TF32): small SIMT kernels that share the top-k epilogue.
#include <math.h>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kTileA = 128 * 128;  // bytes of one A (weight) stage: 128 rows x 128 B
constexpr int kMaxCtas = 256;      // upper bound used for workspace sizing
constexpr float kLog2e = 1.4426950408889634f;

struct Seg {
  int a_row;  // first weight row of the tile
  int b_row;  // first activation row
  int k0, k1; // K-chunk range [k0, k1)
  int tile;   // tile index (fuse_proj) / vocab tile (lmhead)
};

struct CtaShared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;  // raised by any role whose bounded wait ran out
  int epi_abort;   // epilogue-wide decision, read only after a named barrier
  int flag;
};

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

__host__ __device__ inline uint32_t tmem_cols_for(int bn) {
  uint32_t need = 2u * (uint32_t)bn, c = 32;
  while (c < need) c <<= 1;
  return c;
}

// ------------------------------------------------------------ shared pipeline
template <bool TF32, class Sched>
__device__ __forceinline__ void run_producer(const Sched& sc, CtaShared& sh, uint32_t sA, uint32_t sB,
                                             int stages, int bn) {
  constexpr int kBke = TF32 ? 32 : 64;  // elements per 128-byte chunk
  const uint64_t pol_w = l2_policy_evict_first();
  const uint64_t pol_x = l2_policy_evict_last();
  const uint32_t b_bytes = (uint32_t)bn * 128u;
  int it = 0;
  Seg sg;
  for (int si = 0; sc.seg(si, sg); ++si) {
    for (int kc = sg.k0; kc < sg.k1; ++kc, ++it) {
      const int s = it % stages;
      const uint32_t ph = (uint32_t)(it / stages) & 1u;
      if (!mbar_wait(smem_u32(&sh.empty[s]), ph ^ 1u, &sh.abort_flag)) goto drain;
      const uint32_t fb = smem_u32(&sh.full[s]);
      mbar_arrive_expect_tx(fb, (uint32_t)kTileA + b_bytes);
      tma_load_2d(sA + s * kTileA, sc.map_a(), fb, kc * kBke, sg.a_row, pol_w);
      tma_load_2d(sB + s * b_bytes, sc.map_b(kc), fb, sc.b_x(kc), sg.b_row, pol_x);
    }
  }
  return;
drain:
  // wait (bounded) for the copies this thread issued into each stage
  {
    const int last = it - 1;
    for (int s = 0; s < stages && s <= last; ++s) {
      const int i_s = last - ((last - s) % stages);  // last iteration that used stage s
      const uint32_t ph = (uint32_t)(i_s / stages) & 1u;
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&sh.full[s]), ph) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  }
}

template <bool TF32, class Sched>
__device__ __forceinline__ void run_mma(const Sched& sc, CtaShared& sh, uint32_t sA, uint32_t sB,
                                        int stages, int bn) {
  const uint32_t idesc = mma_idesc(TF32 ? 2 : 1, 128, bn);
  const uint32_t b_bytes = (uint32_t)bn * 128u;
  int it = 0, acc = 0;
  bool ok = true;
  Seg sg;
  for (int si = 0; ok && sc.seg(si, sg); ++si, ++acc) {
    const int buf = acc & 1;
    const uint32_t aph = (uint32_t)(acc >> 1) & 1u;
    if (!mbar_wait(smem_u32(&sh.acc_empty[buf]), aph ^ 1u, &sh.abort_flag)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = sh.tmem_base + (uint32_t)(buf * bn);
    for (int kc = sg.k0; kc < sg.k1; ++kc, ++it) {
      const int s = it % stages;
      const uint32_t ph = (uint32_t)(it / stages) & 1u;
      if (!mbar_wait(smem_u32(&sh.full[s]), ph, &sh.abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t da = smem_desc_sw128(sA + s * kTileA);
      const uint64_t db = smem_desc_sw128(sB + s * b_bytes);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t accum = (kc == sg.k0 && kk == 0) ? 0u : 1u;
        // +32 bytes along K inside the 128-byte swizzle atom = +2 in the
        // descriptor's (address >> 4) field
        if (TF32)
          mma_tf32(d_tmem, da + 2u * kk, db + 2u * kk, idesc, accum);
        else
          mma_bf16(d_tmem, da + 2u * kk, db + 2u * kk, idesc, accum);
      }
      mma_commit(smem_u32(&sh.empty[s]));
    }
    if (ok) mma_commit(smem_u32(&sh.acc_full[buf]));
  }
  if (!ok) {
    // drain: all MMAs issued so far complete before tensor memory is freed
    mma_commit(smem_u32(&sh.drain));
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&sh.drain), 0) && globaltimer_ns() - t0 < 100000000ull) {
    }
  }
}

// Epilogue warps wait for an accumulator buffer together: the four warps take
// one decision (continue / abort) so that none is left alone at a named barrier.
__device__ __forceinline__ bool epi_wait(CtaShared& sh, uint32_t bar, uint32_t parity) {
  bool ok = mbar_wait(bar, parity, &sh.abort_flag);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) atomicExch(&sh.epi_abort, 1);
  named_bar(1, kEpiThreads);
  return !*reinterpret_cast<volatile int*>(&sh.epi_abort);
}

// Kernel prologue/epilogue shared by both GEMMs.
__device__ __forceinline__ void cta_setup(CtaShared& sh, int stages, uint32_t tmem_cols) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh.acc_full[b]), 1);
      mbar_init(smem_u32(&sh.acc_empty[b]), 4);  // one arrive per epilogue warp
    }
    mbar_init(smem_u32(&sh.drain), 1);
    sh.abort_flag = 0;
    sh.epi_abort = 0;
    sh.flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem_base), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ void cta_teardown(CtaShared& sh, uint32_t tmem_cols, int32_t* status) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    tc_fence_after();
    tmem_dealloc(sh.tmem_base, tmem_cols);
  }
  if (threadIdx.x == 0 && sh.abort_flag) set_status(status, EAGLE_ERR_TIMEOUT);
}

// ====================================================================== LM head
struct LmParams {
  int M, V, K, bn, groups, ctas_per_group, n_vtiles, nk, stages;
  float inv_t;
  const float* bias;
  int32_t* topk_ids;
  float* topk_lp;
  float* row_max;
  float* row_sumexp;
  float2* part_ms;   // [cta][bn]       (max of z/T, sum exp)
  float* part_v;     // [cta][bn][K]    top-k logits (z)
  int* part_i;       // [cta][bn][K]
  int* part_cnt;     // [cta][bn]
  int* counters;     // [groups]
  int32_t* status;
};

template <bool TF32>
struct LmSched {
  const CUtensorMap* mw;
  const CUtensorMap* mx;
  int t0, t1, b_row, nk;
  __device__ bool seg(int i, Seg& s) const {
    const int t = t0 + i;
    if (t >= t1) return false;
    s.a_row = t * 128;
    s.b_row = b_row;
    s.k0 = 0;
    s.k1 = nk;
    s.tile = t;
    return true;
  }
  __device__ const CUtensorMap* map_a() const { return mw; }
  __device__ const CUtensorMap* map_b(int) const { return mx; }
  __device__ int b_x(int kc) const { return kc * (TF32 ? 32 : 64); }
};

// Insert-into-list merge of the candidates held by a warp.  Lane j < cnt holds
// entry j of the column's sorted top-K list (lv, li).  Candidate values come
// in per lane (up to 4 per lane, flagged by `cand`); the best remaining
// candidate is inserted until none beats the list's K-th entry.
template <int NPL>
__device__ __forceinline__ void warp_topk_merge(float (&z)[NPL], int (&id)[NPL], bool (&cand)[NPL],
                                                float& lv, int& li, int& cnt, int K) {
  const int lane = threadIdx.x & 31;
  float tv = -INFINITY;
  int ti = 0x7fffffff;
  if (cnt == K) {
    tv = __shfl_sync(0xffffffffu, lv, K - 1);
    ti = __shfl_sync(0xffffffffu, li, K - 1);
#pragma unroll
    for (int i = 0; i < NPL; ++i) cand[i] = cand[i] && better(z[i], id[i], tv, ti);
  }
  for (;;) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (cand[i] && better(z[i], id[i], bv, bi)) {
        bv = z[i];
        bi = id[i];
      }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi == 0x7fffffff) break;
    const unsigned ahead = __ballot_sync(0xffffffffu, lane < cnt && better(lv, li, bv, bi));
    const int pos = __popc(ahead);
    const float nv = __shfl_up_sync(0xffffffffu, lv, 1);
    const int ni = __shfl_up_sync(0xffffffffu, li, 1);
    if (lane > pos) {
      lv = nv;
      li = ni;
    }
    if (lane == pos) {
      lv = bv;
      li = bi;
    }
    cnt = min(cnt + 1, K);
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (cand[i] && id[i] == bi && z[i] == bv) cand[i] = false;
    if (cnt == K) {
      tv = __shfl_sync(0xffffffffu, lv, K - 1);
      ti = __shfl_sync(0xffffffffu, li, K - 1);
#pragma unroll
      for (int i = 0; i < NPL; ++i) cand[i] = cand[i] && better(z[i], id[i], tv, ti);
    }
  }
}

// Per-column running state of the LM-head epilogue (one column = one
// activation row): online max / sum-exp of z/T and a sorted top-K list.
struct LmEpi {
  float* T;      // [16][128] transpose buffer: 16 columns x 128 vocab rows
  float* col_m;  // [bn]
  float* col_s;  // [bn]
  int* col_c;    // [bn] entries in the list
  float* top_v;  // [bn][K]
  int* top_i;    // [bn][K]
  int K;
  float inv_t;
};

__device__ __forceinline__ LmEpi lm_epi_carve(unsigned char* p, int bn, int K, float inv_t) {
  LmEpi E;
  E.T = reinterpret_cast<float*>(p);
  E.col_m = E.T + 16 * 128;
  E.col_s = E.col_m + bn;
  E.col_c = reinterpret_cast<int*>(E.col_s + bn);
  E.top_v = reinterpret_cast<float*>(E.col_c + bn);
  E.top_i = reinterpret_cast<int*>(E.top_v + bn * K);
  E.K = K;
  E.inv_t = inv_t;
  return E;
}

// Fold 16 columns of one 128-row vocabulary tile into the running state.
// Called by the 128 epilogue threads together: thread e holds v[j] = z of
// vocabulary row v0+e for column c16*16+j.  Warp ew then owns columns
// ew*4..ew*4+3 of the chunk.
__device__ __forceinline__ void lm_chunk(const LmEpi& E, const float (&v)[16], int e, int ew,
                                         int lane, int v0, int c16, int ncol) {
  const int K = E.K;
#pragma unroll
  for (int j = 0; j < 16; ++j) E.T[j * 128 + e] = v[j];
  named_bar(1, kEpiThreads);
#pragma unroll 1
  for (int jj = 0; jj < 4; ++jj) {
    const int j = ew * 4 + jj, col = c16 * 16 + j;
    if (col >= ncol) continue;
    float z[4];
    int id[4];
    bool cand[4];
    float tmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      z[i] = E.T[j * 128 + lane + 32 * i];
      id[i] = v0 + lane + 32 * i;
      tmax = fmaxf(tmax, z[i] * E.inv_t);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    float ts = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) ts += exp2f((z[i] * E.inv_t - tmax) * kLog2e);
#pragma unroll
    for (int o = 16; o; o >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, o);
    int cnt = E.col_c[col];
    float lv = lane < cnt ? E.top_v[col * K + lane] : -INFINITY;
    int li = lane < cnt ? E.top_i[col * K + lane] : 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 4; ++i) cand[i] = !isnan(z[i]);
    warp_topk_merge<4>(z, id, cand, lv, li, cnt, K);
    if (lane < cnt) {
      E.top_v[col * K + lane] = lv;
      E.top_i[col * K + lane] = li;
    }
    if (lane == 0) {
      const float om = E.col_m[col];
      const float nm = fmaxf(om, tmax);
      E.col_s[col] = (om == -INFINITY ? 0.f : E.col_s[col] * exp2f((om - nm) * kLog2e)) +
                     ts * exp2f((tmax - nm) * kLog2e);
      E.col_m[col] = nm;
      E.col_c[col] = cnt;
    }
    __syncwarp();
  }
  named_bar(1, kEpiThreads);
}

// Publish this CTA's per-column partial state; the last CTA of the group
// (atomic ticket, no waiting) merges all partials of the group and writes the
// final top-k ids, log-probs and row statistics.
__device__ __forceinline__ void lm_publish_merge(const LmParams& p, const LmEpi& E, int* flag, int g,
                                                 int m0, int ncol, int et, int ew, int lane) {
  const int cta = blockIdx.x, bn = p.bn, K = p.K;
  for (int c = et; c < ncol; c += kEpiThreads) {
    p.part_ms[(size_t)cta * bn + c] = make_float2(E.col_m[c], E.col_s[c]);
    p.part_cnt[(size_t)cta * bn + c] = E.col_c[c];
  }
  for (int x = et; x < ncol * K; x += kEpiThreads) {
    p.part_v[(size_t)cta * bn * K + x] = E.top_v[x];
    p.part_i[(size_t)cta * bn * K + x] = E.top_i[x];
  }
  __threadfence();
  named_bar(1, kEpiThreads);
  if (et == 0) *flag = (atomicAdd(&p.counters[g], 1) == p.ctas_per_group - 1) ? 1 : 0;
  named_bar(1, kEpiThreads);
  if (!*reinterpret_cast<volatile int*>(flag)) return;
  __threadfence();
  const int c0 = g * p.ctas_per_group, nc = p.ctas_per_group;
  for (int col = ew; col < ncol; col += 4) {
    float M = -INFINITY;
    for (int c = lane; c < nc; c += 32) M = fmaxf(M, p.part_ms[(size_t)(c0 + c) * bn + col].x);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float S = 0.f;
    for (int c = lane; c < nc; c += 32) {
      const float2 ms = p.part_ms[(size_t)(c0 + c) * bn + col];
      if (ms.x != -INFINITY) S += ms.y * exp2f((ms.x - M) * kLog2e);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    float lv = -INFINITY;
    int li = 0x7fffffff, cnt = 0;
    for (int f0 = 0; f0 < nc * K; f0 += 32) {
      const int f = f0 + lane;
      float z[1] = {-INFINITY};
      int id[1] = {0x7fffffff};
      bool cand[1] = {false};
      if (f < nc * K) {
        const int c = f / K, j = f % K;
        if (j < p.part_cnt[(size_t)(c0 + c) * bn + col]) {
          z[0] = p.part_v[((size_t)(c0 + c) * bn + col) * K + j];
          id[0] = p.part_i[((size_t)(c0 + c) * bn + col) * K + j];
          cand[0] = true;
        }
      }
      warp_topk_merge<1>(z, id, cand, lv, li, cnt, K);
    }
    const int row = m0 + col;
    const float lse = M + logf(S);
    if (lane < K) {
      p.topk_ids[(size_t)row * K + lane] = lane < cnt ? li : -1;
      p.topk_lp[(size_t)row * K + lane] = lane < cnt ? lv * p.inv_t - lse : -INFINITY;
    }
    if (lane == 0) {
      if (p.row_max) p.row_max[row] = M;
      if (p.row_sumexp) p.row_sumexp[row] = S;
    }
  }
}

template <bool TF32>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_topk_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                       const LmParams p) {
  __shared__ CtaShared sh;
  extern __shared__ unsigned char dsmem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bn = p.bn, stages = p.stages;
  const uint32_t tmem_cols = tmem_cols_for(bn);
  const uint32_t base = align1024(smem_u32(dsmem));
  const uint32_t sA = base, sB = sA + stages * kTileA;
  unsigned char* gbase = dsmem + (base - smem_u32(dsmem));
  const LmEpi E = lm_epi_carve(gbase + stages * (kTileA + bn * 128), bn, p.K, p.inv_t);

  const int g = blockIdx.x / p.ctas_per_group, ci = blockIdx.x % p.ctas_per_group;
  LmSched<TF32> sc;
  sc.mw = &map_w;
  sc.mx = &map_x;
  sc.t0 = (int)((long long)ci * p.n_vtiles / p.ctas_per_group);
  sc.t1 = (int)((long long)(ci + 1) * p.n_vtiles / p.ctas_per_group);
  sc.b_row = g * bn;
  sc.nk = p.nk;
  const int m0 = g * bn;
  const int ncol = min(bn, p.M - m0);

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_x);
  }
  for (int c = threadIdx.x; c < bn; c += kThreads) {
    E.col_m[c] = -INFINITY;
    E.col_s[c] = 0.f;
    E.col_c[c] = 0;
  }
  cta_setup(sh, stages, tmem_cols);

  if (warp == 0) {
    if (lane == 0) run_producer<TF32>(sc, sh, sA, sB, stages, bn);
  } else if (warp == 1) {
    if (lane == 0) run_mma<TF32>(sc, sh, sA, sB, stages, bn);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter of this warp
    const int e = q * 32 + lane;      // weight row inside the tile
    const int ew = warp - 2;          // epilogue warp 0..3
    int acc = 0;
    Seg sg;
    for (int si = 0; sc.seg(si, sg); ++si, ++acc) {
      const int buf = acc & 1;
      const uint32_t aph = (uint32_t)(acc >> 1) & 1u;
      if (!epi_wait(sh, smem_u32(&sh.acc_full[buf]), aph)) break;
      tc_fence_after();
      const int v0 = sg.tile * 128;
      const float bias_e = p.bias ? p.bias[v0 + e] : 0.f;
      const uint32_t taddr = sh.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * bn);
      for (int c16 = 0; c16 * 16 < ncol; ++c16) {
        float v[16];
        tmem_ld16(taddr + c16 * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += bias_e;
        lm_chunk(E, v, e, ew, lane, v0, c16, ncol);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[buf]));
    }
    named_bar(1, kEpiThreads);
    if (!*reinterpret_cast<volatile int*>(&sh.epi_abort))
      lm_publish_merge(p, E, &sh.flag, g, m0, ncol, threadIdx.x - 64, ew, lane);
  }
  cta_teardown(sh, tmem_cols, p.status);
}

// fp32 LM head on the CUDA cores (exact fp32 products and sums).  Same
// schedule and epilogue as the tensor-core kernel; 128 threads, thread e
// computes vocabulary row v0+e against 16 activation rows at a time from
// shared-memory tiles of 32 K-elements.
constexpr int kF32Kc = 32;
__global__ void __launch_bounds__(kEpiThreads)
    lmhead_topk_f32_kernel(const float* __restrict__ x, const float* __restrict__ w, int d,
                           const LmParams p) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ int flag;
  float* Ws = reinterpret_cast<float*>(dsm);         // [128][kF32Kc + 1]
  float* Xs = Ws + 128 * (kF32Kc + 1);                // [16][kF32Kc]
  const LmEpi E = lm_epi_carve(reinterpret_cast<unsigned char*>(Xs + 16 * kF32Kc), p.bn, p.K, p.inv_t);
  const int e = threadIdx.x, lane = e & 31, ew = e >> 5;
  const int g = blockIdx.x / p.ctas_per_group, ci = blockIdx.x % p.ctas_per_group;
  const int t0 = (int)((long long)ci * p.n_vtiles / p.ctas_per_group);
  const int t1 = (int)((long long)(ci + 1) * p.n_vtiles / p.ctas_per_group);
  const int m0 = g * p.bn, ncol = min(p.bn, p.M - m0);
  for (int c = e; c < p.bn; c += kEpiThreads) {
    E.col_m[c] = -INFINITY;
    E.col_s[c] = 0.f;
    E.col_c[c] = 0;
  }
  __syncthreads();
  for (int t = t0; t < t1; ++t) {
    const int v0 = t * 128;
    const float bias_e = p.bias ? p.bias[v0 + e] : 0.f;
    for (int c16 = 0; c16 * 16 < ncol; ++c16) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.f;
      for (int k0 = 0; k0 < d; k0 += kF32Kc) {
        __syncthreads();
        for (int i = e; i < 128 * kF32Kc; i += kEpiThreads) {
          const int r = i / kF32Kc, c = i % kF32Kc;
          Ws[r * (kF32Kc + 1) + c] = w[(size_t)(v0 + r) * d + k0 + c];
        }
        for (int i = e; i < 16 * kF32Kc; i += kEpiThreads) {
          const int r = i / kF32Kc, c = i % kF32Kc, m = m0 + c16 * 16 + r;
          Xs[i] = (c16 * 16 + r < ncol) ? x[(size_t)m * d + k0 + c] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < kF32Kc; ++c) {
          const float wv = Ws[e * (kF32Kc + 1) + c];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = fmaf(wv, Xs[j * kF32Kc + c], v[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] += bias_e;
      lm_chunk(E, v, e, ew, lane, v0, c16, ncol);
    }
  }
  named_bar(1, kEpiThreads);
  lm_publish_merge(p, E, &flag, g, m0, ncol, e, ew, lane);
}

// ==================================================================== fuse_proj
struct FpParams {
  int M, d, bn, groups, n_otiles, nk, nkd, n_tiles, n_ctas, max_contrib, stages;
  long long W;  // total chunks = n_tiles * nk
  const float* bias;
  void* out;
  float* part;    // [n_tiles][max_contrib][bn][128]
  int* counters;  // [n_tiles]
  int32_t* status;
};

__host__ __device__ inline long long sk_lo(long long c, long long W, int n) { return c * W / n; }
// CTA whose stream-K range holds chunk x
__device__ inline int sk_owner(long long x, long long W, int n) {
  int c = (int)((x * n) / W);
  while (c + 1 < n && sk_lo(c + 1, W, n) <= x) ++c;
  while (c > 0 && sk_lo(c, W, n) > x) --c;
  return c;
}

template <bool TF32>
struct FpSched {
  const CUtensorMap* mw;
  const CUtensorMap* mx[3];
  long long lo, hi;
  int nk, nkd, n_otiles, bn;
  __device__ bool seg(int i, Seg& s) const {
    if (lo >= hi) return false;
    const int t = (int)(lo / nk) + i;
    const long long a = (long long)t * nk;
    if (a >= hi) return false;
    s.tile = t;
    s.k0 = (int)(max(lo, a) - a);
    s.k1 = (int)(min(hi, a + nk) - a);
    s.a_row = (t % n_otiles) * 128;
    s.b_row = (t / n_otiles) * bn;
    return true;
  }
  __device__ const CUtensorMap* map_a() const { return mw; }
  __device__ const CUtensorMap* map_b(int kc) const { return mx[kc / nkd]; }
  __device__ int b_x(int kc) const { return (kc % nkd) * (TF32 ? 32 : 64); }
};

template <bool TF32>
__global__ void __launch_bounds__(kThreads, 1)
    fuse_proj_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_l,
                     const __grid_constant__ CUtensorMap map_m, const __grid_constant__ CUtensorMap map_h,
                     const FpParams p) {
  __shared__ CtaShared sh;
  extern __shared__ unsigned char dsmem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bn = p.bn, stages = p.stages;
  const uint32_t tmem_cols = tmem_cols_for(bn);
  const uint32_t base = align1024(smem_u32(dsmem));
  const uint32_t sA = base, sB = sA + stages * kTileA;

  FpSched<TF32> sc;
  sc.mw = &map_w;
  sc.mx[0] = &map_l;
  sc.mx[1] = &map_m;
  sc.mx[2] = &map_h;
  sc.lo = sk_lo(blockIdx.x, p.W, p.n_ctas);
  sc.hi = sk_lo(blockIdx.x + 1, p.W, p.n_ctas);
  sc.nk = p.nk;
  sc.nkd = p.nkd;
  sc.n_otiles = p.n_otiles;
  sc.bn = bn;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_l);
    tma_prefetch_desc(&map_m);
    tma_prefetch_desc(&map_h);
  }
  cta_setup(sh, stages, tmem_cols);

  if (warp == 0) {
    if (lane == 0) run_producer<TF32>(sc, sh, sA, sB, stages, bn);
  } else if (warp == 1) {
    if (lane == 0) run_mma<TF32>(sc, sh, sA, sB, stages, bn);
  } else {
    const int q = warp & 3, e = q * 32 + lane, et = threadIdx.x - 64;
    int acc = 0;
    Seg sg;
    for (int si = 0; sc.seg(si, sg); ++si, ++acc) {
      const int buf = acc & 1;
      const uint32_t aph = (uint32_t)(acc >> 1) & 1u;
      if (!epi_wait(sh, smem_u32(&sh.acc_full[buf]), aph)) break;
      tc_fence_after();
      const int ot = sg.tile % p.n_otiles, gr = sg.tile / p.n_otiles;
      const int o = ot * 128 + e, m0 = gr * bn, ncol = min(bn, p.M - m0);
      const uint32_t taddr = sh.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * bn);
      const bool whole = sg.k0 == 0 && sg.k1 == p.nk;
      const float bias_o = p.bias ? p.bias[o] : 0.f;
      if (whole) {
        for (int c16 = 0; c16 * 16 < ncol; ++c16) {
          float v[16];
          tmem_ld16(taddr + c16 * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c16 * 16 + j;
            if (col < ncol) {
              const size_t idx = (size_t)(m0 + col) * p.d + o;
              if (TF32)
                reinterpret_cast<float*>(p.out)[idx] = v[j] + bias_o;
              else
                reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16(v[j] + bias_o);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[buf]));
      } else {
        // stream-K partial: write, then the last contributor of the tile reduces
        const long long x0 = (long long)sg.tile * p.nk;
        const int c_first = sk_owner(x0, p.W, p.n_ctas);
        const int c_last = sk_owner(x0 + p.nk - 1, p.W, p.n_ctas);
        const int slot = blockIdx.x - c_first;
        float* part = p.part + (((size_t)sg.tile * p.max_contrib + slot) * bn) * 128;
        for (int c16 = 0; c16 * 16 < ncol; ++c16) {
          float v[16];
          tmem_ld16(taddr + c16 * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c16 * 16 + j;
            if (col < ncol) part[(size_t)col * 128 + e] = v[j];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[buf]));
        __threadfence();
        named_bar(1, kEpiThreads);
        if (et == 0)
          sh.flag = (atomicAdd(&p.counters[sg.tile], sg.k1 - sg.k0) + (sg.k1 - sg.k0) == p.nk) ? 1 : 0;
        named_bar(1, kEpiThreads);
        if (sh.flag) {
          __threadfence();
          const int ncontrib = c_last - c_first + 1;
          const float* pbase = p.part + ((size_t)sg.tile * p.max_contrib * bn) * 128;
          for (int col = 0; col < ncol; ++col) {
            float s = 0.f;
            for (int k = 0; k < ncontrib; ++k) s += pbase[((size_t)k * bn + col) * 128 + e];
            const size_t idx = (size_t)(m0 + col) * p.d + o;
            if (TF32)
              reinterpret_cast<float*>(p.out)[idx] = s + bias_o;
            else
              reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16(s + bias_o);
          }
        }
        named_bar(1, kEpiThreads);
      }
    }
  }
  cta_teardown(sh, tmem_cols, p.status);
}

// fp32 fused projection on the CUDA cores (exact fp32): one warp per output
// element g[m, o]; lanes stride the 3d inputs of the concatenation.
__global__ void __launch_bounds__(256)
    fuse_proj_f32_kernel(const float* __restrict__ hl, const float* __restrict__ hm,
                         const float* __restrict__ hh, const float* __restrict__ w,
                         const float* __restrict__ bias, float* __restrict__ g, int M, int d) {
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)M * d) return;
  const int m = (int)(gw / d), o = (int)(gw % d);
  const float* wr = w + (size_t)o * 3 * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) {
    acc = fmaf(wr[c], hl[(size_t)m * d + c], acc);
    acc = fmaf(wr[d + c], hm[(size_t)m * d + c], acc);
    acc = fmaf(wr[2 * d + c], hh[(size_t)m * d + c], acc);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) g[(size_t)m * d + o] = acc + (bias ? bias[o] : 0.f);
}

// ------------------------------------------------------------------ host side
int pick_bn(int M, int* groups) {
  const int G = (M + 255) / 256;
  const int per = (M + G - 1) / G;
  *groups = G;
  return (per + 15) / 16 * 16;
}

int pick_stages(int bn, size_t extra) {
  const size_t budget = 227 * 1024 - 1024 - extra - 256;
  const size_t stage = (size_t)kTileA + (size_t)bn * 128;
  int s = (int)(budget / stage);
  return s > kMaxStages ? kMaxStages : s;
}

size_t lm_epi_bytes(int bn, int K) { return 16 * 128 * 4 + (size_t)bn * (12 + 8 * (size_t)K); }

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_lmhead_topk_workspace_size(int M, int d, int V, int k, int dtype) {
  (void)d;
  (void)V;
  (void)dtype;
  if (M <= 0 || k <= 0) return 0;
  int G;
  const int bn = pick_bn(M, &G);
  const size_t n = (size_t)kMaxCtas * bn;
  return round_up(n * 8, 256) + 2 * round_up(n * k * 4, 256) + round_up(n * 4, 256) +
         round_up((size_t)G * 4, 256) + 1024;
}

extern "C" int eagle_lmhead_topk(const void* x, const void* w_lm, const float* bias, int M, int d,
                                 int V, int k, float temperature, int32_t* topk_ids,
                                 float* topk_logprobs, float* row_max, float* row_sumexp, int dtype,
                                 void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!x || !w_lm || !topk_ids || !topk_logprobs) return EAGLE_ERR_INVALID_ARG;
  if (M <= 0 || d <= 0 || V <= 0 || k <= 0 || !(temperature > 0.f) || isinf(temperature))
    return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (k > V) return EAGLE_ERR_INVALID_ARG;
  if (M > 2048 || k > 32 || d % 64 || V % 128) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w_lm)) return EAGLE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < eagle_lmhead_topk_workspace_size(M, d, V, k, dtype)) return EAGLE_ERR_WORKSPACE;
  const int esz = dtype == EAGLE_BF16 ? 2 : 4;
  const int bke = 128 / esz;
  int G;
  const int bn = pick_bn(M, &G);
  const int n_vtiles = V / 128;
  int sms = sm_count();
  if (sms <= 0) return EAGLE_ERR_CUDA;
  sms = sms > kMaxCtas ? kMaxCtas : sms;
  int cpg = sms / G;
  if (cpg < 1) cpg = 1;
  if (cpg > n_vtiles) cpg = n_vtiles;
  const int n_ctas = cpg * G;
  const size_t extra = lm_epi_bytes(bn, k);
  const int stages = dtype == EAGLE_BF16 ? pick_stages(bn, extra) : 2;
  if (stages < 2) return EAGLE_ERR_UNSUPPORTED;
  const size_t smem = dtype == EAGLE_BF16
                          ? 1024 + (size_t)stages * (kTileA + (size_t)bn * 128) + extra
                          : (size_t)(128 * (kF32Kc + 1) + 16 * kF32Kc) * 4 + extra;
  if (smem > 227 * 1024) return EAGLE_ERR_UNSUPPORTED;

  CUtensorMap mw, mx;
  if (dtype == EAGLE_BF16 &&
      (!make_tmap_2d(&mw, w_lm, esz, (uint64_t)V, (uint64_t)d, 128, (uint32_t)bke) ||
       !make_tmap_2d(&mx, x, esz, (uint64_t)M, (uint64_t)d, (uint32_t)bn, (uint32_t)bke)))
    return EAGLE_ERR_CUDA;

  char* cur = static_cast<char*>(ws);
  const size_t n = (size_t)kMaxCtas * bn;
  LmParams p;
  p.part_ms = static_cast<float2*>(ws_carve(cur, n * 8));
  p.part_v = static_cast<float*>(ws_carve(cur, n * k * 4));
  p.part_i = static_cast<int*>(ws_carve(cur, n * k * 4));
  p.part_cnt = static_cast<int*>(ws_carve(cur, n * 4));
  p.counters = static_cast<int*>(ws_carve(cur, (size_t)G * 4));
  p.M = M;
  p.V = V;
  p.K = k;
  p.bn = bn;
  p.groups = G;
  p.ctas_per_group = cpg;
  p.n_vtiles = n_vtiles;
  p.nk = d / bke;
  p.stages = stages;
  p.inv_t = 1.f / temperature;
  p.bias = bias;
  p.topk_ids = topk_ids;
  p.topk_lp = topk_logprobs;
  p.row_max = row_max;
  p.row_sumexp = row_sumexp;
  p.status = dev_status;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(p.counters, 0, (size_t)G * 4, s) != cudaSuccess) return EAGLE_ERR_CUDA;
  if (dtype == EAGLE_BF16) {
    cudaFuncSetAttribute(lmhead_topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    lmhead_topk_kernel<false><<<n_ctas, kThreads, smem, s>>>(mw, mx, p);
  } else {
    cudaFuncSetAttribute(lmhead_topk_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    lmhead_topk_f32_kernel<<<n_ctas, kEpiThreads, smem, s>>>((const float*)x, (const float*)w_lm, d, p);
  }
  note_launch();
  return last_launch_status();
}

namespace {
struct FpPlan {
  int bn, G, n_otiles, nk, nkd, n_tiles, n_ctas, max_contrib;
  long long W;
};
FpPlan fp_plan(int M, int d, int esz, int n_ctas_cap) {
  FpPlan f;
  f.bn = pick_bn(M, &f.G);
  const int bke = 128 / esz;
  f.n_otiles = d / 128;
  f.nkd = d / bke;
  f.nk = 3 * f.nkd;
  f.n_tiles = f.n_otiles * f.G;
  f.W = (long long)f.n_tiles * f.nk;
  f.n_ctas = (int)(f.W < n_ctas_cap ? f.W : n_ctas_cap);
  const long long per = f.W / f.n_ctas;  // minimum chunks per CTA
  f.max_contrib = (int)((f.nk + per - 1) / per) + 1;
  if (f.max_contrib > f.n_ctas) f.max_contrib = f.n_ctas;
  return f;
}
}  // namespace

extern "C" size_t eagle_fuse_proj_workspace_size(int M, int d, int dtype) {
  if (M <= 0 || d <= 0 || d % 128) return 0;
  const int esz = dtype == EAGLE_BF16 ? 2 : 4;
  // sized for the largest grid the library launches (kMaxCtas CTAs)
  size_t best = 0;
  for (int cap = 1; cap <= kMaxCtas; ++cap) {
    const FpPlan f = fp_plan(M, d, esz, cap);
    const size_t sz = round_up((size_t)f.n_tiles * 4, 256) +
                      round_up((size_t)f.n_tiles * f.max_contrib * f.bn * 128 * 4, 256) + 1024;
    best = sz > best ? sz : best;
  }
  return best;
}

extern "C" int eagle_fuse_proj(const void* h_low, const void* h_mid, const void* h_high,
                               const void* w_proj, const float* bias, void* g, int M, int d, int dtype,
                               void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!h_low || !h_mid || !h_high || !w_proj || !g) return EAGLE_ERR_INVALID_ARG;
  if (M <= 0 || d <= 0) return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (M > 4096 || d % 128 || d > 16384) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(h_low) || !aligned16(h_mid) || !aligned16(h_high) || !aligned16(w_proj))
    return EAGLE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < eagle_fuse_proj_workspace_size(M, d, dtype)) return EAGLE_ERR_WORKSPACE;
  if (dtype == EAGLE_FP32) {
    const long long outs = (long long)M * d;
    fuse_proj_f32_kernel<<<(unsigned)((outs + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        (const float*)h_low, (const float*)h_mid, (const float*)h_high, (const float*)w_proj, bias,
        (float*)g, M, d);
    note_launch();
    return last_launch_status();
  }
  const int esz = 2;
  const int bke = 64;
  int sms = sm_count();
  if (sms <= 0) return EAGLE_ERR_CUDA;
  const FpPlan f = fp_plan(M, d, esz, sms > kMaxCtas ? kMaxCtas : sms);
  const int stages = pick_stages(f.bn, 0);
  if (stages < 2) return EAGLE_ERR_UNSUPPORTED;
  const size_t smem = 1024 + (size_t)stages * (kTileA + (size_t)f.bn * 128);

  CUtensorMap mw, ml, mm, mh;
  if (!make_tmap_2d(&mw, w_proj, esz, (uint64_t)d, (uint64_t)3 * d, 128, (uint32_t)bke) ||
      !make_tmap_2d(&ml, h_low, esz, (uint64_t)M, (uint64_t)d, (uint32_t)f.bn, (uint32_t)bke) ||
      !make_tmap_2d(&mm, h_mid, esz, (uint64_t)M, (uint64_t)d, (uint32_t)f.bn, (uint32_t)bke) ||
      !make_tmap_2d(&mh, h_high, esz, (uint64_t)M, (uint64_t)d, (uint32_t)f.bn, (uint32_t)bke))
    return EAGLE_ERR_CUDA;

  char* cur = static_cast<char*>(ws);
  FpParams p;
  p.counters = static_cast<int*>(ws_carve(cur, (size_t)f.n_tiles * 4));
  p.part = static_cast<float*>(ws_carve(cur, (size_t)f.n_tiles * f.max_contrib * f.bn * 128 * 4));
  p.M = M;
  p.d = d;
  p.bn = f.bn;
  p.groups = f.G;
  p.n_otiles = f.n_otiles;
  p.nk = f.nk;
  p.nkd = f.nkd;
  p.n_tiles = f.n_tiles;
  p.n_ctas = f.n_ctas;
  p.max_contrib = f.max_contrib;
  p.stages = stages;
  p.W = f.W;
  p.bias = bias;
  p.out = g;
  p.status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(p.counters, 0, (size_t)f.n_tiles * 4, s) != cudaSuccess) return EAGLE_ERR_CUDA;
  cudaFuncSetAttribute(fuse_proj_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  fuse_proj_kernel<false><<<f.n_ctas, kThreads, smem, s>>>(mw, ml, mm, mh, p);
  note_launch();
  return last_launch_status();
}
