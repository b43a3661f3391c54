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

#include <mutex>
#include <vector>

#include "common.cuh"
#include "lm_merge.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 10;
constexpr int kMaxAcc = 4;  // TMEM accumulator buffers (as many as 512 columns hold)
constexpr int kTileA = 128 * 128;  // bytes of one A (weight) stage: 128 rows x 128 B
constexpr int kMaxCtas = 256;      // upper bound used for workspace sizing
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory ring of one GEMM: stage s holds the A tile at a0 + s*a_stride
// (a_bytes of it loaded by TMA) and the B tile at b0 + s*b_stride (b_bytes).
// The MMA always reads 128 A rows; rows past the loaded ones are don't-care
// data that only reach accumulator rows the epilogue ignores.
struct Ring {
  uint32_t a0, a_stride, a_bytes;
  uint32_t b0, b_stride, b_bytes;
  int stages;
  int n;     // MMA N (rows of the B tile)
  int nbuf;  // TMEM accumulator buffers of n columns each (2 n with DUAL)
};
// DUAL (a template flag of the pipeline below): each stage holds two 128-row
// A tiles (rows a_row .. a_row + 255, the second at a0 + kTileA) that share
// the B tile; two MMAs per K step into accumulators n columns apart.

struct Seg {
  int a_row;  // first weight row of the tile
  int b_row;  // first activation row
  int k0, k1; // K-chunk range [k0, k1)
  int tile;   // tile index (fuse_proj) / vocab tile (lmhead)
};

struct CtaShared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[kMaxAcc];
  uint64_t acc_empty[kMaxAcc];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;  // raised by any role whose bounded wait ran out
  int epi_abort;   // epilogue-wide decision, read only after a named barrier
  int flag;
};

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

__host__ __device__ inline int acc_buffers_for(int n) {
  const int b = 512 / n;
  return b > kMaxAcc ? kMaxAcc : b;
}
__host__ __device__ inline uint32_t tmem_cols_for(int n) {
  uint32_t need = (uint32_t)(acc_buffers_for(n) * n), c = 32;
  while (c < need) c <<= 1;
  return c;
}

// ------------------------------------------------------------ shared pipeline
// Weight half of the first ring stages, issued by the producer thread before
// the previous grid on the stream has finished (the weights are constants of
// the model; only the activations depend on that grid).  Each stage's full
// barrier expects both halves; the activation half follows after the wait.
// Returns the number of stages pre-issued.
template <bool TF32, bool DUAL, class Sched>
__device__ __forceinline__ int prefetch_weights(const Sched& sc, CtaShared& sh, const Ring& rg) {
  constexpr int kBke = TF32 ? 32 : 64;
  int it = 0;
  Seg sg;
  for (int si = 0; it < rg.stages && sc.seg(si, sg); ++si) {
    for (int kc = sg.k0; kc < sg.k1 && it < rg.stages; ++kc, ++it) {
      const uint32_t fb = smem_u32(&sh.full[it]);
      mbar_arrive_expect_tx(fb, rg.a_bytes + rg.b_bytes);
      if (Sched::kWeightIsA) {
        tma_load_2d(rg.a0 + it * rg.a_stride, sc.map_a(), fb, kc * kBke, sg.a_row, sc.a_policy());
        if (DUAL)
          tma_load_2d(rg.a0 + it * rg.a_stride + kTileA, sc.map_a(), fb, kc * kBke, sg.a_row + 128,
                      sc.a_policy());
      } else {
        sc.load_b(rg.b0 + it * rg.b_stride, fb, kc, sg.b_row, sc.b_policy());
      }
    }
  }
  return it;
}

// Bounded wait for the copies a producer issued into each ring stage before it
// gave up at iteration `it` (stage s last used by iteration i_s).
__device__ __forceinline__ void drain_full(CtaShared& sh, int stages, int it) {
  const int last = it - 1;
  for (int s = 0; s < stages && s <= last; ++s) {
    const int i_s = last - ((last - s) % stages);
    const uint32_t ph = (uint32_t)(i_s / stages) & 1u;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&sh.full[s]), ph) && globaltimer_ns() - t0 < 100000000ull) {
    }
  }
}

template <bool TF32, bool DUAL, class Sched>
__device__ __forceinline__ void run_producer(const Sched& sc, CtaShared& sh, const Ring& rg,
                                             int pre) {
  constexpr int kBke = TF32 ? 32 : 64;  // elements per 128-byte chunk
  const uint64_t pol_a = sc.a_policy();
  const uint64_t pol_b = sc.b_policy();
  const int stages = rg.stages;
  const uint32_t tx = rg.a_bytes + rg.b_bytes;
  int it = 0, s = 0;  // iteration, its ring stage (it % stages) and phase
  uint32_t ph = 0;
  Seg sg;
  for (int si = 0; sc.seg(si, sg); ++si) {
    for (int kc = sg.k0; kc < sg.k1; ++kc, ++it) {
      const uint32_t fb = smem_u32(&sh.full[s]);
      if (it < pre) {  // weight half already in flight: the activation half only
        if (Sched::kWeightIsA)
          sc.load_b(rg.b0 + s * rg.b_stride, fb, kc, sg.b_row, pol_b);
        else
          tma_load_2d(rg.a0 + s * rg.a_stride, sc.map_a(), fb, kc * kBke, sg.a_row, pol_a);
      } else {
        if (!mbar_wait(smem_u32(&sh.empty[s]), ph ^ 1u, &sh.abort_flag)) goto drain;
        mbar_arrive_expect_tx(fb, tx);
        tma_load_2d(rg.a0 + s * rg.a_stride, sc.map_a(), fb, kc * kBke, sg.a_row, pol_a);
        if (DUAL)
          tma_load_2d(rg.a0 + s * rg.a_stride + kTileA, sc.map_a(), fb, kc * kBke, sg.a_row + 128, pol_a);
        sc.load_b(rg.b0 + s * rg.b_stride, fb, kc, sg.b_row, pol_b);
      }
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  return;
drain:
  drain_full(sh, stages, it);
}

template <bool TF32, bool DUAL, class Sched>
__device__ __forceinline__ void run_mma(const Sched& sc, CtaShared& sh, const Ring& rg) {
  const uint32_t idesc = mma_idesc(TF32 ? 2 : 1, 128, rg.n);
  const int stages = rg.stages;
  int s = 0, buf = 0;  // ring stage and accumulator buffer, with their phases
  uint32_t ph = 0, aph = 0;
  bool ok = true;
  Seg sg;
  for (int si = 0; ok && sc.seg(si, sg); ++si) {
    if (!mbar_wait(smem_u32(&sh.acc_empty[buf]), aph ^ 1u, &sh.abort_flag)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = sh.tmem_base + (uint32_t)(buf * rg.n * (DUAL ? 2 : 1));
    for (int kc = sg.k0; kc < sg.k1; ++kc) {
      if (!mbar_wait(smem_u32(&sh.full[s]), ph, &sh.abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t da = smem_desc_sw128(rg.a0 + s * rg.a_stride);
      const uint64_t db = smem_desc_sw128(rg.b0 + s * rg.b_stride);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t accum = (kc == sg.k0 && kk == 0) ? 0u : 1u;
        // +32 bytes along K inside the 128-byte swizzle atom = +2 in the
        // descriptor's (address >> 4) field
        if (TF32)
          mma_tf32(d_tmem, da + 2u * kk, db + 2u * kk, idesc, accum);
        else
          mma_bf16(d_tmem, da + 2u * kk, db + 2u * kk, idesc, accum);
        // the second A tile: +kTileA bytes = +kTileA / 16 in the address field
        if (DUAL)
          mma_bf16(d_tmem + (uint32_t)rg.n, da + (uint64_t)(kTileA >> 4) + 2u * kk, db + 2u * kk, idesc, accum);
      }
      mma_commit(smem_u32(&sh.empty[s]));
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (ok) mma_commit(smem_u32(&sh.acc_full[buf]));
    if (++buf == rg.nbuf) {
      buf = 0;
      aph ^= 1u;
    }
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
// CTA set-up in two halves: cta_init (thread 0: barriers) and cta_start (all
// threads: wait for the previous grid, claim TMEM, then let dependents launch);
// the producer may pre-issue weight loads in between (prefetch_weights).
__device__ __forceinline__ void cta_init(CtaShared& sh, int stages) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    for (int b = 0; b < kMaxAcc; ++b) {
      mbar_init(smem_u32(&sh.acc_full[b]), 1);
      mbar_init(smem_u32(&sh.acc_empty[b]), 4);  // one arrive per epilogue warp
    }
    mbar_init(smem_u32(&sh.drain), 1);
    sh.abort_flag = 0;
    sh.epi_abort = 0;
    sh.flag = 0;
    fence_mbar_init();
  }
}
__device__ __forceinline__ void cta_start(CtaShared& sh, uint32_t tmem_cols) {
  const int warp = threadIdx.x >> 5;
  pdl_wait();  // the previous grid (and its TMEM) is gone from here on
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem_base), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
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
  int M, V, K, groups, ctas_per_group, n_vtiles, nk, stages;
  int tn;  // vocabulary rows per tile (MMA N, multiple of 16, <= 256)
  int xr;  // activation rows loaded per stage (group rows rounded up to 16)
  float inv_t;
  // exponential-race mode (verification statistics): the top-K is taken over
  // key = z/T - log(-log u_{b,y}) with u from Philox4x32-10 (key race_k0/1,
  // counter (y >> 2, b, race_c2, race_c3), word y & 3), b = row / R
  int race, R;
  uint32_t race_k0, race_k1, race_c2, race_c3;
  const float* bias;
  int32_t* topk_ids;
  float* topk_lp;     // log-probs, or the race keys in race mode
  float* row_max;
  float* row_sumexp;
  float2* part_ms;   // [M][cpg]       (max of z/T, sum exp) per row and CTA of its group
  float* part_v;     // [M][cpg][K]    sorted top-k logits (z)
  int* part_i;       // [M][cpg][K]
  int* part_cnt;     // [M][cpg]
  int32_t* status;
  const void* residual;  // [M, d] of the output dtype added to the result, or null
};

// LM head, not swapped: the (up to) 128 activation rows of a group are the
// MMA's M side (rows past M are zero-filled by TMA), 128 vocabulary rows of
// W_U the N side, so TMEM lane e holds activation row e and each epilogue
// thread scans its own row's logits with no cross-thread reduction.
struct LmSched {
  static constexpr bool kWeightIsA = false;  // W_U is the B operand
  const CUtensorMap* mx;
  const CUtensorMap* mw;
  int t0, t1, a_row, nk, tn;
  bool w_reused;  // several activation groups read the same W tiles
  __device__ bool seg(int i, Seg& s) const {
    const int t = t0 + i;
    if (t >= t1) return false;
    s.a_row = a_row;
    s.b_row = t * tn;
    s.k0 = 0;
    s.k1 = nk;
    s.tile = t;
    return true;
  }
  __device__ const CUtensorMap* map_a() const { return mx; }
  __device__ int b_x(int kc) const { return kc * 64; }
  __device__ void load_b(uint32_t dst, uint32_t fb, int kc, int b_row, uint64_t pol) const {
    tma_load_2d(dst, mw, fb, b_x(kc), b_row, pol);
  }
  __device__ uint64_t a_policy() const { return l2_policy_evict_last(); }
  __device__ uint64_t b_policy() const {
    return w_reused ? l2_policy_evict_normal() : l2_policy_evict_first();
  }
};

// Running state of one activation row, held in registers by the thread that
// owns the row: online max / sum-exp of z/T and the sorted top-K list (z
// descending, id ascending) of the ids seen so far.  KMAX >= K is a
// compile-time bound so the list lives in registers.
// The real list occupies the last K slots; the first KMAX - K slots hold +inf
// sentinels that nothing displaces, so the K-th best is always slot KMAX - 1
// (a static register index).  Insertion is a predicated compare-and-swap
// pass, executed by the whole warp only when some lane holds a candidate.
template <int KMAX>
struct RowTopK {
  float m, s;          // running max of z/T and sum of exp(z/T - m)
  float av[KMAX];      // sorted top-K values (z, or the race keys)
  int ai[KMAX];        // ... their ids
  float tv;            // K-th best so far (-inf while fewer than K)
  int ti;
  bool nan_seen;
};

template <int KMAX>
__device__ __forceinline__ void row_init(RowTopK<KMAX>& r, int K) {
  r.m = -INFINITY;
  r.s = 0.f;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const bool sentinel = j < KMAX - K;
    r.av[j] = sentinel ? INFINITY : -INFINITY;
    r.ai[j] = sentinel ? -1 : 0x7fffffff;
  }
  r.tv = -INFINITY;
  r.ti = 0x7fffffff;
  r.nan_seen = false;
}

// -log(-log u) of one Philox word (u = (2 (x >> 9) + 1) 2^-24 in (0, 1)).
__device__ __forceinline__ float gumbel_of(uint32_t x) { return -logf(-logf(bits_to_uniform(x))); }

// Race noise g[j] = -log(-log u_{b,id0+j}) for this lane's request b and the
// 16 ids id0.. (id0 a multiple of 16).  Rows of a warp are consecutive, so
// they span few requests: lane L draws the four words of request
// (first request + L / 4), ids id0 + 4 (L % 4) .., and the lanes gather their
// own request's 16 values by shuffles (each Philox word drawn once per warp).
// Must be called by all 32 lanes together.
__device__ __forceinline__ void race_gumbel16(const LmParams& p, int grow, int id0, float (&g)[16],
                                              int lane) {
  const int b = min(grow, p.M - 1) / p.R;
  const int b0 = __shfl_sync(0xffffffffu, b, 0);
  const int nreq = __shfl_sync(0xffffffffu, b, 31) - b0 + 1;
  if (nreq * 4 <= 32) {
    float gw[4] = {0.f, 0.f, 0.f, 0.f};
    if (lane < nreq * 4) {
      const uint4 w = philox4x32_10(
          make_uint4((uint32_t)(id0 >> 2) + (uint32_t)(lane & 3), (uint32_t)(b0 + (lane >> 2)),
                     p.race_c2, p.race_c3),
          p.race_k0, p.race_k1);
      gw[0] = gumbel_of(w.x);
      gw[1] = gumbel_of(w.y);
      gw[2] = gumbel_of(w.z);
      gw[3] = gumbel_of(w.w);
    }
    const int src = (b - b0) * 4;
#pragma unroll
    for (int j = 0; j < 16; ++j) g[j] = __shfl_sync(0xffffffffu, gw[j & 3], src + (j >> 2));
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = philox4x32_10(
          make_uint4((uint32_t)(id0 >> 2) + (uint32_t)q, (uint32_t)b, p.race_c2, p.race_c3),
          p.race_k0, p.race_k1);
      g[4 * q] = gumbel_of(w.x);
      g[4 * q + 1] = gumbel_of(w.y);
      g[4 * q + 2] = gumbel_of(w.z);
      g[4 * q + 3] = gumbel_of(w.w);
    }
  }
}

// Insert (z, id) into the sorted list; id is larger than every listed id.
// Slot t is beaten iff z is larger, or (unless PLAIN: no slot is empty) equal
// while the slot is empty; the beaten slots form a suffix, which shifts down
// by one with z at its head.
template <int KMAX, bool PLAIN>
__device__ __forceinline__ void list_insert(RowTopK<KMAX>& r, float z, int id) {
  float pv = 0.f;
  int pi = 0;
  bool pb = false;
#pragma unroll
  for (int t = 0; t < KMAX; ++t) {
    const float ov = r.av[t];
    const int oi = r.ai[t];
    const bool b = PLAIN ? z > ov : (z > ov || (z == ov && oi == 0x7fffffff));
    r.av[t] = b ? (pb ? pv : z) : ov;
    r.ai[t] = b ? (pb ? pi : id) : oi;
    pv = ov;
    pi = oi;
    pb = b;
  }
}

// Fold 16 consecutive vocabulary ids id0.. (values v, the first `valid` of
// them real; valid <= 0 for a lane without a row) into the row: log-sum-exp
// of z/T always; top-K of z, or with RACE of z/T + g (g from race_gumbel16).
// A row's ids arrive in strictly increasing order (its CTA's tiles, then the
// 16-column chunks, in order), so a new id loses every tie with a listed one:
// it beats a slot iff its value is larger, or equal while the slot is still
// empty (id 0x7fffffff).  Against a list sorted by (value desc, id asc) that
// test is monotone along the slots, so a candidate's insertion is one
// independent compare per slot, not a chain through the list.
// Must be called by all 32 lanes of the warp together.
template <int KMAX, bool RACE>
__device__ __forceinline__ void row_chunk(RowTopK<KMAX>& r, float (&v)[16], const float (&g)[16],
                                          int id0, int valid, float inv_t, int K) {
  // chunk maximum of z/T: multiplying by inv_t > 0 is monotone in fp32, so
  // max(z) inv_t is exactly max(z inv_t); the NaN-propagating maximum also
  // tells whether any real column is NaN
  float vm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 16; ++j) vm = fmax_nan(vm, j < valid ? v[j] : -INFINITY);
  const bool nan = isnan(vm);
  r.nan_seen |= nan;
  if (nan) {  // rare: the maximum over the real columns that are not NaN
    vm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) vm = fmaxf(vm, j < valid ? v[j] : -INFINITY);
  }
  const float nm = fmaxf(r.m, vm * inv_t);
  if (nm != -INFINITY) {
    // exp(z/T - m) = 2^(z log2e/T - m log2e): one fused multiply-add per id
    const float sl = inv_t * kLog2e, ml = nm * kLog2e;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const float e0 = ex2_approx(fmaf(v[j], sl, -ml)), e1 = ex2_approx(fmaf(v[j + 1], sl, -ml));
      a0 += j < valid ? e0 : 0.f;
      a1 += j + 1 < valid ? e1 : 0.f;
    }
    r.s = r.s * ex2_approx((r.m - nm) * kLog2e) + (a0 + a1);
    r.m = nm;
  }
  if (RACE) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = v[j] * inv_t + g[j];  // the race key replaces z below
  }
  // candidates: values that beat the current K-th slot
  const bool full = r.ti != 0x7fffffff;
  unsigned cmask = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < valid && (v[j] > r.tv || (!full && v[j] == r.tv))) cmask |= 1u << j;
  // one candidate per lane per round, the whole warp in step
  while (__any_sync(0xffffffffu, cmask != 0)) {
    const int jc = cmask ? __ffs(cmask) - 1 : -1;
    cmask &= cmask - 1;
    // v[jc] by a 4-level select on the bits of jc; a lane without a
    // candidate re-inserts an empty slot (-inf beats only empty slots)
    float z;
    {
      float h[8], q[4], w[2];
#pragma unroll
      for (int t = 0; t < 8; ++t) h[t] = (jc & 8) ? v[t + 8] : v[t];
#pragma unroll
      for (int t = 0; t < 4; ++t) q[t] = (jc & 4) ? h[t + 4] : h[t];
#pragma unroll
      for (int t = 0; t < 2; ++t) w[t] = (jc & 2) ? q[t + 2] : q[t];
      z = jc < 0 ? -INFINITY : ((jc & 1) ? w[1] : w[0]);
    }
    const int id = jc < 0 ? 0x7fffffff : id0 + jc;
    // once every candidate lane's list is full no slot is empty, and the
    // slot test is the plain value compare
    if (__all_sync(0xffffffffu, jc < 0 || r.ti != 0x7fffffff))
      list_insert<KMAX, true>(r, z, id);
    else
      list_insert<KMAX, false>(r, z, id);
    r.tv = r.av[KMAX - 1];
    r.ti = r.ai[KMAX - 1];
  }
}

// Publish every row's partial state (running max / sum-exp and its sorted
// top-K list) for lmhead_merge_kernel.
template <int KMAX>
__device__ __forceinline__ void lm_publish(const LmParams& p, const RowTopK<KMAX>& r, int nrow, int e) {
  const int K = p.K;
  const int g = blockIdx.x % p.groups, ci = blockIdx.x / p.groups;
  const size_t slot = (size_t)(g * 128 + e) * p.ctas_per_group + ci;  // [row][cta]
  if (e < nrow) {
    p.part_ms[slot] = make_float2(r.m, r.s);
    int cnt = 0;
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
      const int j = t - (KMAX - K);  // position in the reported list
      if (j >= 0 && r.ai[t] != 0x7fffffff) {
        p.part_v[slot * K + j] = r.av[t];
        p.part_i[slot * K + j] = r.ai[t];
        cnt = j + 1;
      }
    }
    p.part_cnt[slot] = cnt;
  }
}

// Merge of the per-CTA partials: one CTA per activation row.  All warps stage
// the row's contiguous lists into shared memory with independent loads; warp
// 0 then takes the log-sum-exp by max / rescale over the CTAs and the top-K by
// K rounds of "best head among the CTAs' sorted lists".
constexpr int kMergeThreads = 256;
__global__ void __launch_bounds__(kMergeThreads) lmhead_merge_kernel(const LmParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char msm[];
  const int tid = threadIdx.x;
  const int m = blockIdx.x;
  const int K = p.K, nc = p.ctas_per_group, n = nc * K;
  float* sv = reinterpret_cast<float*>(msm);
  int* si = reinterpret_cast<int*>(sv + n);
  int* sc = si + n;
  // this row's partials are contiguous: [cta][K] values / ids, [cta] counts
  const float* gv = p.part_v + (size_t)m * n;
  const int* gi = p.part_i + (size_t)m * n;
  const int* gc = p.part_cnt + (size_t)m * nc;
  LmPartials lp;
  lp.ms = p.part_ms;
  lp.v = p.part_v;
  lp.id = p.part_i;
  lp.cnt = p.part_cnt;
  lp.cpg = nc;
  lp.K = K;
  lp.inv_t = p.inv_t;
  lp.race = p.race;
  // the merging warp's (max, sum) pairs go out with the staging loads, and
  // eight loads of each kind per thread stage 152 lists of 12 in one pass
  float2 ms[kLmMergePer];
  if (tid < 32) lm_load_ms(lp, m, ms);
  constexpr int kU = 8;
  for (int f0 = tid; f0 < n; f0 += kMergeThreads * kU) {
    float v[kU];
    int id[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int f = f0 + u * kMergeThreads;
      v[u] = f < n ? __ldcg(gv + f) : 0.f;
      id[u] = f < n ? __ldcg(gi + f) : 0;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int f = f0 + u * kMergeThreads;
      if (f < n) {
        sv[f] = v[u];
        si[f] = id[u];
      }
    }
  }
  for (int c = tid; c < nc; c += kMergeThreads) sc[c] = __ldcg(gc + c);
  __syncthreads();
  if (tid >= 32) return;
  lm_merge_row_ms(lp, m, ms, sv, si, sc, p.topk_ids + (size_t)m * K, p.topk_lp + (size_t)m * K, p.row_max,
                  p.row_sumexp);
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_topk_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                       const LmParams p) {
  __shared__ CtaShared sh;
  extern __shared__ unsigned char dsmem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stages = p.stages, K = p.K;
  const int tn = p.tn;  // vocabulary rows per tile (MMA N)
  const uint32_t tmem_cols = tmem_cols_for(tn);
  const uint32_t base = align1024(smem_u32(dsmem));
  unsigned char* gbase = dsmem + (base - smem_u32(dsmem));
  // W tiles, then the activation tiles (only xr rows each are loaded), then
  // slack so that the MMA's 128-row view of the last activation tile stays
  // inside the allocation, then the per-row top-K lists
  Ring rg;
  rg.stages = stages;
  rg.n = tn;
  rg.nbuf = acc_buffers_for(tn);
  rg.b0 = base;
  rg.b_stride = (uint32_t)tn * 128u;
  rg.b_bytes = (uint32_t)tn * 128u;
  rg.a0 = base + stages * (uint32_t)tn * 128u;
  rg.a_stride = rg.a_bytes = (uint32_t)p.xr * 128u;
  (void)gbase;

  const int g = blockIdx.x % p.groups, ci = blockIdx.x / p.groups;
  LmSched sc;
  sc.mx = &map_x;
  sc.mw = &map_w;
  sc.t0 = (int)((long long)ci * p.n_vtiles / p.ctas_per_group);
  sc.t1 = (int)((long long)(ci + 1) * p.n_vtiles / p.ctas_per_group);
  sc.a_row = g * 128;
  sc.nk = p.nk;
  sc.tn = tn;
  sc.w_reused = p.groups > 1;
  const int m0 = g * 128;
  const int nrow = min(128, p.M - m0);

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_w);
  }
  cta_init(sh, stages);
  int pre = 0;
  if (threadIdx.x == 0) pre = prefetch_weights<false, false>(sc, sh, rg);
  cta_start(sh, tmem_cols);

  if (warp == 0) {
    if (lane == 0) run_producer<false, false>(sc, sh, rg, pre);
  } else if (warp == 1) {
    if (lane == 0) run_mma<false, false>(sc, sh, rg);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;       // TMEM lane quarter of this warp
    const int e = q * 32 + lane;  // activation row inside the group
    const bool valid = e < nrow;
    RowTopK<KMAX> r;
    row_init(r, K);
    int acc = 0;
    Seg sg;
    for (int si = 0; sc.seg(si, sg); ++si, ++acc) {
      const int buf = acc % rg.nbuf;
      const uint32_t aph = (uint32_t)(acc / rg.nbuf) & 1u;
      if (!epi_wait(sh, smem_u32(&sh.acc_full[buf]), aph)) break;
      tc_fence_after();
      const int v0 = sg.tile * tn;
      const int vend = min(tn, p.V - v0);  // rows past V were zero-filled
      const uint32_t taddr = sh.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * tn);
#pragma unroll 1
      for (int c16 = 0; c16 < tn / 16; ++c16) {
        float v[16];
        tmem_ld16(taddr + c16 * 16, v);
        if (p.bias) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += p.bias[min(v0 + c16 * 16 + j, p.V - 1)];
        }
        const int id0 = v0 + c16 * 16, nv = valid ? vend - c16 * 16 : 0;
        float gk[16];
        if (p.race) {
          race_gumbel16(p, m0 + e, id0, gk, lane);
          row_chunk<KMAX, true>(r, v, gk, id0, nv, p.inv_t, K);
        } else {
          row_chunk<KMAX, false>(r, v, gk, id0, nv, p.inv_t, K);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[buf]));
    }
    if (r.nan_seen) set_status(p.status, EAGLE_ERR_NONFINITE);
    named_bar(1, kEpiThreads);
    if (!*reinterpret_cast<volatile int*>(&sh.epi_abort)) lm_publish(p, r, nrow, e);
  }
  cta_teardown(sh, tmem_cols, p.status);
}

// fp32 LM head on the CUDA cores (exact fp32 products and sums), same
// schedule and epilogue: 128 threads, thread e owns activation row e of the
// group; 16 vocabulary rows at a time from shared-memory tiles of 32 K-values.
constexpr int kF32Kc = 32;
template <int KMAX>
__global__ void __launch_bounds__(kEpiThreads)
    lmhead_topk_f32_kernel(const float* __restrict__ x, const float* __restrict__ w, int d,
                           const LmParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char dsm[];
  float* Xs = reinterpret_cast<float*>(dsm);        // [128][kF32Kc + 1]
  float* Ws = Xs + 128 * (kF32Kc + 1);              // [16][kF32Kc]
  const int e = threadIdx.x, K = p.K;
  const int g = blockIdx.x % p.groups, ci = blockIdx.x / p.groups;
  const int t0 = (int)((long long)ci * p.n_vtiles / p.ctas_per_group);
  const int t1 = (int)((long long)(ci + 1) * p.n_vtiles / p.ctas_per_group);
  const int m0 = g * 128, nrow = min(128, p.M - m0);
  RowTopK<KMAX> r;
  row_init(r, K);
  for (int t = t0; t < t1; ++t) {
    for (int v16 = 0; v16 < p.tn; v16 += 16) {
      const int vb = t * p.tn + v16;
      float acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.f;
      for (int k0 = 0; k0 < d; k0 += kF32Kc) {
        __syncthreads();
        for (int i = e; i < 128 * kF32Kc; i += kEpiThreads) {
          const int rr = i / kF32Kc, c = i % kF32Kc;
          Xs[rr * (kF32Kc + 1) + c] = rr < nrow ? x[(size_t)(m0 + rr) * d + k0 + c] : 0.f;
        }
        for (int i = e; i < 16 * kF32Kc; i += kEpiThreads) {
          const int rr = i / kF32Kc, c = i % kF32Kc;
          Ws[i] = vb + rr < p.V ? w[(size_t)(vb + rr) * d + k0 + c] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < kF32Kc; ++c) {
          const float xv = Xs[e * (kF32Kc + 1) + c];
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = fmaf(xv, Ws[j * kF32Kc + c], acc[j]);
        }
      }
      if (p.bias) {
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] += p.bias[min(vb + j, p.V - 1)];
      }
      float gk[16];
      if (p.race) {
        race_gumbel16(p, m0 + e, vb, gk, e & 31);
        row_chunk<KMAX, true>(r, acc, gk, vb, e < nrow ? p.V - vb : 0, p.inv_t, K);
      } else {
        row_chunk<KMAX, false>(r, acc, gk, vb, e < nrow ? p.V - vb : 0, p.inv_t, K);
      }
    }
  }
  if (r.nan_seen) set_status(p.status, EAGLE_ERR_NONFINITE);
  __syncthreads();
  lm_publish(p, r, nrow, e);
}

// ==================================================================== fuse_proj
struct FpParams {
  int M, d, bn, groups, n_otiles, nk, nkd, n_tiles, n_ctas, max_contrib, stages;  // d: output width
  long long W;  // total chunks = n_tiles * nk
  const float* bias;
  void* out;
  float* part;    // [n_tiles][max_contrib][bn][128]
  int32_t* status;
  const void* residual;  // [M, d] of the output dtype added to the result, or null
  // Rows known only on the device (the accepted-rows fusion): with m_dev set,
  // only the first *m_dev of the M activation rows are projected -- the
  // stream-K split is re-planned on the device over the groups that hold
  // them -- and activation row i lands in output row row_map[i].
  const int32_t* m_dev;
  const int32_t* row_map;
  // tile order: output-tile-major (tile t = output tile t / groups, group
  // t % groups) when several groups share each weight tile and the rows are
  // known on the host; group-major (output tile t % n_otiles, group
  // t / n_otiles) otherwise, so that the live groups of a device row count
  // form a prefix of the tiles
  int tmajor;
  // lanes > 0 (with tmajor): CTA c computes group c % groups over lane
  // c / groups's share of the (output tile, K chunk) items of one group, so
  // the groups' CTAs of a lane stream the same weight chunks at the same time
  // (one HBM read, the others' from L2); a tile's contributors are
  // consecutive lanes
  int lanes;
  // dual (with lanes): the items are (pair of output tiles 2 t, 2 t + 1, K
  // chunk); each stage's activation tile feeds both tiles' MMAs, so the
  // activations are read from L2 once per pair instead of once per tile
  int dual;
  // view_w > 0: segment 0 is read through a row view, rows r0 .. r0 + view_w
  // - 1 of each request of a [B, Rmax, K] array (activation row b view_w + j);
  // a group then starts at a request boundary (bn a multiple of view_w)
  int view_w;
  // cs >= 1 (one activation group, all rows known on the host): output tile
  // t is computed by CTAs t * cs .. t * cs + cs - 1, each over an equal share
  // of the K chunks; with cs >= 2 they are one thread-block cluster that sums
  // the shares through distributed shared memory.  0: the stream-K split.
  int cs;
};

// The activation rows, stream-K chunk count and active CTAs of one launch:
// all M rows (W chunks over every CTA) unless the row count comes from the
// device.  The chunks are split over at most W CTAs, so that every active
// CTA holds at least one chunk and a tile's contributors are consecutive CTAs
// (the partial slot of a contributor is its distance from the tile's first
// one); CTAs past the active count do nothing.
struct FpLive {
  int m;
  long long W;
  int n;
};
__device__ __forceinline__ FpLive fp_live(const FpParams& p) {
  FpLive l{p.M, p.W, p.n_ctas};
  if (p.m_dev) {
    const int m = __ldcg(p.m_dev);
    l.m = m < 0 ? 0 : (m > p.M ? p.M : m);
    l.W = (long long)p.n_otiles * ((l.m + p.bn - 1) / p.bn) * p.nk;
    l.n = l.W < p.n_ctas ? (int)l.W : p.n_ctas;
  }
  return l;
}

__host__ __device__ inline long long sk_lo(long long c, long long W, int n) { return c * W / n; }
// CTA whose stream-K range holds chunk x
__device__ inline int sk_owner(long long x, long long W, int n) {
  int c = (int)((x * n) / W);
  while (c + 1 < n && sk_lo(c + 1, W, n) <= x) ++c;
  while (c > 0 && sk_lo(c, W, n) > x) --c;
  return c;
}

template <bool TF32, bool DUAL = false>
struct FpSched {
  static constexpr bool kWeightIsA = true;  // W_proj is the A operand
  const CUtensorMap* mw;
  const CUtensorMap* mx[3];
  long long lo, hi;
  int nk, nkd, n_otiles, bn, groups, tmajor;
  int lane_gr;  // lanes: this CTA's group (the items [lo, hi) are output tiles x K chunks), else -1
  int view_w;   // rows per request of a row view of the activations (see FpParams::view_w), else 0
  // DUAL (lanes): the items are pairs of output tiles (s.tile = pair * groups + group)
  __device__ bool seg(int i, Seg& s) const {
    if (lo >= hi) return false;
    const int t = (int)(lo / nk) + i;
    const long long a = (long long)t * nk;
    if (a >= hi) return false;
    s.k0 = (int)(max(lo, a) - a);
    s.k1 = (int)(min(hi, a + nk) - a);
    if (lane_gr >= 0) {
      s.tile = t * groups + lane_gr;
      s.a_row = t * (DUAL ? 256 : 128);
      s.b_row = lane_gr * bn;
    } else {
      s.tile = t;
      s.a_row = (tmajor ? t / groups : t % n_otiles) * 128;
      s.b_row = (tmajor ? t % groups : t / n_otiles) * bn;
    }
    return true;
  }
  __device__ const CUtensorMap* map_a() const { return mw; }
  __device__ const CUtensorMap* map_b(int kc) const { return mx[kc / nkd]; }
  __device__ int b_x(int kc) const { return (kc % nkd) * (TF32 ? 32 : 64); }
  // the activation rows b_row .. of one K chunk: a 2-D box, or with a row
  // view (view_w > 0) a 3-D box of view_w rows of bn / view_w requests
  __device__ void load_b(uint32_t dst, uint32_t fb, int kc, int b_row, uint64_t pol) const {
    if (view_w > 0)
      tma_load_3d(dst, map_b(kc), fb, b_x(kc), 0, b_row / view_w, pol);
    else
      tma_load_2d(dst, map_b(kc), fb, b_x(kc), b_row, pol);
  }
  // a weight tile that several groups read stays in L2 for their passes
  __device__ uint64_t a_policy() const { return groups > 1 ? l2_policy_evict_normal() : l2_policy_evict_first(); }
  __device__ uint64_t b_policy() const { return l2_policy_evict_last(); }
};

// Sum of the stream-K partials of every tile that several CTAs share, in
// contributor (slot) order, so the result does not depend on timing; one
// thread per 4 outputs of a tile, all SMs at once.
template <bool TF32>
__global__ void __launch_bounds__(256) fuse_proj_reduce_kernel(const FpParams p) {
  pdl_wait();
  pdl_trigger();
  const FpLive lv = fp_live(p);
  const int tile = blockIdx.y;
  int c_first, c_last;
  if (p.lanes) {  // contributors: consecutive lanes over the tile's (or its pair's) K chunks
    const int sh = p.dual ? 1 : 0;
    const long long W1 = (long long)(p.n_otiles >> sh) * p.nk, x0 = (long long)((tile / p.groups) >> sh) * p.nk;
    c_first = sk_owner(x0, W1, p.lanes);
    c_last = sk_owner(x0 + p.nk - 1, W1, p.lanes);
  } else {
    const long long x0 = (long long)tile * p.nk;
    if (x0 >= lv.W) return;  // a group past the live rows
    c_first = sk_owner(x0, lv.W, lv.n);
    c_last = sk_owner(x0 + p.nk - 1, lv.W, lv.n);
  }
  if (c_first == c_last) return;  // one CTA held the whole tile and wrote it
  const int ot = p.tmajor ? tile / p.groups : tile % p.n_otiles;
  const int gr = p.tmajor ? tile % p.groups : tile / p.n_otiles;
  const int m0 = gr * p.bn, ncol = min(p.bn, lv.m - m0);
  const int f = blockIdx.x * 256 + threadIdx.x;  // float4 index in the [ncol][128] tile
  if (f >= ncol * 32) return;
  const int ncontrib = c_last - c_first + 1;
  const float4* pbase = reinterpret_cast<const float4*>(p.part + ((size_t)tile * p.max_contrib * p.bn) * 128);
  const size_t slot4 = (size_t)p.bn * 32;  // float4s per contributor slot
  constexpr int kC = 8;  // contributors loaded per round
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < ncontrib; k0 += kC) {
    float4 x[kC];
#pragma unroll
    for (int k = 0; k < kC; ++k)
      x[k] = k0 + k < ncontrib ? __ldcg(pbase + (size_t)(k0 + k) * slot4 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kC; ++k) {
      acc.x += x[k].x;
      acc.y += x[k].y;
      acc.z += x[k].z;
      acc.w += x[k].w;
    }
  }
  const int col = f / 32, oo = ot * 128 + (f % 32) * 4;
  if (p.bias) {
    acc.x += p.bias[oo];
    acc.y += p.bias[oo + 1];
    acc.z += p.bias[oo + 2];
    acc.w += p.bias[oo + 3];
  }
  const int orow = p.row_map ? p.row_map[m0 + col] : m0 + col;
  const size_t idx = (size_t)orow * p.d + oo;
  if (p.residual) {
    if (TF32) {
      const float4 rv = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.residual) + idx);
      acc.x += rv.x;
      acc.y += rv.y;
      acc.z += rv.z;
      acc.w += rv.w;
    } else {
      const uint2 rv = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.residual) + idx);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rv.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rv.y));
      acc.x += a.x;
      acc.y += a.y;
      acc.z += b.x;
      acc.w += b.y;
    }
  }
  if (TF32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + idx) = acc;
  } else {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + idx) = pk;
  }
}

// K = nk chunks over nk / nkd segments of width d, segment i read through
// map_l, map_m, map_h in that order (two segments: map_h is unused).  DUAL:
// the lanes schedule over pairs of output tiles (FpParams::dual).
template <bool TF32, bool DUAL = false>
__global__ void __launch_bounds__(kThreads, 1)
    fuse_proj_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_l,
                     const __grid_constant__ CUtensorMap map_m, const __grid_constant__ CUtensorMap map_h,
                     const FpParams p) {
  __shared__ CtaShared sh;
  extern __shared__ unsigned char dsmem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bn = p.bn, stages = p.stages;
  const uint32_t base = align1024(smem_u32(dsmem));
  static_assert(!(TF32 && DUAL), "pairs of output tiles are a bf16 schedule");
  constexpr bool dual = DUAL;
  const int acc_cols = dual ? 2 * bn : bn;  // TMEM columns of one accumulator buffer
  const uint32_t tmem_cols = tmem_cols_for(acc_cols);
  Ring rg;
  rg.stages = stages;
  rg.n = bn;
  rg.nbuf = acc_buffers_for(acc_cols);
  rg.a0 = base;
  rg.a_stride = rg.a_bytes = (dual ? 2u : 1u) * kTileA;
  rg.b0 = base + stages * rg.a_stride;
  rg.b_stride = rg.b_bytes = (uint32_t)bn * 128u;

  FpSched<TF32, DUAL> sc;
  sc.mw = &map_w;
  sc.mx[0] = &map_l;
  sc.mx[1] = &map_m;
  sc.mx[2] = &map_h;
  sc.lo = sk_lo(blockIdx.x, p.W, p.n_ctas);
  sc.hi = sk_lo(blockIdx.x + 1, p.W, p.n_ctas);
  sc.lane_gr = -1;
  if (p.cs) {
    const long long t = blockIdx.x / p.cs, r = blockIdx.x % p.cs;
    sc.lo = t * p.nk + r * p.nk / p.cs;
    sc.hi = t * p.nk + (r + 1) * p.nk / p.cs;
  } else if (p.lanes) {
    const int j = blockIdx.x / p.groups;
    const long long W1 = (long long)(dual ? p.n_otiles / 2 : p.n_otiles) * p.nk;
    sc.lo = sk_lo(j, W1, p.lanes);
    sc.hi = sk_lo(j + 1, W1, p.lanes);
    sc.lane_gr = blockIdx.x % p.groups;
  }
  sc.nk = p.nk;
  sc.nkd = p.nkd;
  sc.n_otiles = p.n_otiles;
  sc.bn = bn;
  sc.groups = p.groups;
  sc.tmajor = p.tmajor;
  sc.view_w = p.view_w;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_l);
    tma_prefetch_desc(&map_m);
    if (p.nk > 2 * p.nkd) tma_prefetch_desc(&map_h);
  }
  cta_init(sh, stages);
  int pre = 0;
  // a device row count is only known once the previous grid is done, so the
  // weights of such a launch are not fetched early
  if (threadIdx.x == 0 && !p.m_dev) pre = prefetch_weights<TF32, DUAL>(sc, sh, rg);
  cta_start(sh, tmem_cols);
  const FpLive lv = fp_live(p);
  if (p.m_dev) {
    const bool active = (int)blockIdx.x < lv.n;
    sc.lo = active ? sk_lo(blockIdx.x, lv.W, lv.n) : 0;
    sc.hi = active ? sk_lo(blockIdx.x + 1, lv.W, lv.n) : 0;
  }

  if (warp == 0) {
    if (lane == 0) run_producer<TF32, DUAL>(sc, sh, rg, pre);
  } else if (warp == 1) {
    if (lane == 0) run_mma<TF32, DUAL>(sc, sh, rg);
  } else {
    const int q = warp & 3, e = q * 32 + lane;
    int acc = 0;
    Seg sg;
    for (int si = 0; sc.seg(si, sg); ++si, ++acc) {
      const int buf = acc % rg.nbuf;
      const uint32_t aph = (uint32_t)(acc / rg.nbuf) & 1u;
      if (!epi_wait(sh, smem_u32(&sh.acc_full[buf]), aph)) break;
      tc_fence_after();
      // dual: the segment's pair of output tiles, one after the other
      for (int h = 0; h < (dual ? 2 : 1); ++h) {
        const int ot = dual ? 2 * (sg.tile / p.groups) + h : p.tmajor ? sg.tile / p.groups : sg.tile % p.n_otiles;
        const int gr = p.tmajor ? sg.tile % p.groups : sg.tile / p.n_otiles;
        const int tile = dual ? ot * p.groups + gr : sg.tile;  // output tile (partials, reduction)
        const int o = ot * 128 + e, m0 = gr * bn, ncol = min(bn, lv.m - m0);
        const uint32_t taddr =
            sh.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * acc_cols + h * bn);
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
                const int orow = p.row_map ? p.row_map[m0 + col] : m0 + col;
                const size_t idx = (size_t)orow * p.d + o;
                float y = v[j] + bias_o;
                if (p.residual)
                  y += TF32 ? reinterpret_cast<const float*>(p.residual)[idx]
                            : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.residual)[idx]);
                if (TF32)
                  reinterpret_cast<float*>(p.out)[idx] = y;
                else
                  reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16(y);
              }
            }
          }
        } else if (p.cs) {
          // this CTA's K share of the tile: kept in shared memory (over the
          // ring, whose stages are all consumed) for the cluster's sum below
          float* xs = reinterpret_cast<float*>(dsmem + (base - smem_u32(dsmem)));
          for (int c16 = 0; c16 * 16 < ncol; ++c16) {
            float v[16];
            tmem_ld16(taddr + c16 * 16, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c16 * 16 + j;
              if (col < ncol) xs[col * 128 + e] = v[j];
            }
          }
        } else {
          // stream-K partial: write it; fuse_proj_reduce_kernel sums the
          // contributors of the tile afterwards
          int slot;
          if (p.lanes) {  // consecutive lanes contribute to a tile (or a pair)
            const long long x0 = (long long)(sg.tile / p.groups) * p.nk;
            const long long W1 = (long long)(dual ? p.n_otiles / 2 : p.n_otiles) * p.nk;
            slot = (int)(blockIdx.x / p.groups) - sk_owner(x0, W1, p.lanes);
          } else {
            const long long x0 = (long long)sg.tile * p.nk;
            slot = blockIdx.x - sk_owner(x0, lv.W, lv.n);
          }
          float* part = p.part + (((size_t)tile * p.max_contrib + slot) * bn) * 128;
          for (int c16 = 0; c16 * 16 < ncol; ++c16) {
            float v[16];
            tmem_ld16(taddr + c16 * 16, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c16 * 16 + j;
              if (col < ncol) part[(size_t)col * 128 + e] = v[j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[buf]));
    }
  }
  cta_teardown(sh, tmem_cols, p.status);
  if (!TF32 && p.cs > 1) {
    // the cluster's sum: CTA r of the cluster takes an equal share of the
    // tile's activation rows and adds the cs K shares in rank order (a fixed
    // order, so the result does not depend on timing), then bias / residual
    cluster_barrier();  // every share is in its CTA's shared memory
    const int t = blockIdx.x / p.cs, r = blockIdx.x % p.cs;
    const int ot = t % p.n_otiles, ncol = min(bn, p.M);
    const int c0 = r * ncol / p.cs, c1 = (r + 1) * ncol / p.cs;
    const float4* xs4 = reinterpret_cast<const float4*>(dsmem + (base - smem_u32(dsmem)));
    for (int f = threadIdx.x; f < (c1 - c0) * 32; f += kThreads) {
      const int col = c0 + f / 32, e4 = f % 32;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s2 = 0; s2 < p.cs; ++s2) {
        const float4 v = ld_cluster_f4(xs4 + col * 32 + e4, (uint32_t)s2);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const int oo = ot * 128 + e4 * 4;
      if (p.bias) {
        acc.x += p.bias[oo];
        acc.y += p.bias[oo + 1];
        acc.z += p.bias[oo + 2];
        acc.w += p.bias[oo + 3];
      }
      const size_t idx = (size_t)col * p.d + oo;
      if (p.residual) {
        const uint2 rv = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.residual) + idx);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rv.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rv.y));
        acc.x += a.x;
        acc.y += a.y;
        acc.z += b.x;
        acc.w += b.y;
      }
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&lo);
      pk.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + idx) = pk;
    }
    cluster_barrier();  // no CTA leaves while another reads its share
  }
}

// Accepted-rows fusion, first half: the accepted rows of every request
// (path_rows[b, 0 .. accept_len[b]], in path order) are packed, request after
// request, into three compact [cap, d] buffers that the projection reads by
// TMA; row_map[i] is the output slot b * slots + j of packed row i, *m_out the
// number of packed rows.  Output slots past a request's accepted length are
// zeroed here.  A request with accept_len outside [0, slots) or a path row
// outside [0, R) records EAGLE_ERR_BAD_TREE and contributes no row (all its
// slots are zeroed).  Every CTA scans the per-request counts itself (B <= 4096
// entries, 16 per thread), then all CTAs copy 16-byte chunks.
constexpr int kAccThreads = 256;
constexpr int kAccMaxB = 4096;
__global__ void __launch_bounds__(kAccThreads) accepted_gather_kernel(
    int B, int R, int slots, int chunks /* 16-byte chunks per row */,
    const int32_t* __restrict__ path_rows, const int32_t* __restrict__ accept_len,
    const uint4* __restrict__ hl, const uint4* __restrict__ hm, const uint4* __restrict__ hh,
    uint4* __restrict__ cl, uint4* __restrict__ cm, uint4* __restrict__ ch, int32_t* __restrict__ row_map,
    int32_t* __restrict__ m_out, uint4* __restrict__ g_out, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_off[kAccMaxB + 1];
  __shared__ int s_warp[kAccThreads / 32];
  constexpr int kPer = kAccMaxB / kAccThreads;  // requests per thread
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int n[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int b = t * kPer + i;
    n[i] = 0;
    if (b < B) {
      const int a = accept_len[b];
      bool ok = a >= 0 && a < slots;
      for (int j = 0; ok && j <= a; ++j) {
        const int r = path_rows[(size_t)b * slots + j];
        ok = r >= 0 && r < R;
      }
      if (ok)
        n[i] = a + 1;
      else if (blockIdx.x == 0)
        set_status(status, EAGLE_ERR_BAD_TREE);
    }
    sum += n[i];
  }
  // block exclusive scan of the per-thread sums
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_warp[w];
  int run = wbase + x - sum;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int b = t * kPer + i;
    if (b < B) s_off[b] = run;
    run += n[i];
  }
  if (t == kAccThreads - 1) s_off[B] = run;  // the last thread's running total is the grand total
  __syncthreads();
  const int total = s_off[B];
  if (blockIdx.x == 0 && t == 0) *m_out = total;
  // packed rows [0, total) and the zeroed output slots, chunk by chunk
  const long long cap = (long long)B * slots;
  const long long work = cap * chunks;
  for (long long w = (long long)blockIdx.x * kAccThreads + t; w < work; w += (long long)gridDim.x * kAccThreads) {
    const int i = (int)(w / chunks), c = (int)(w % chunks);
    if (i < total) {
      int lo = 0, hi = B;  // request b with s_off[b] <= i < s_off[b + 1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= i) lo = mid; else hi = mid;
      }
      const int b = lo, j = i - s_off[b];
      const size_t src = ((size_t)b * R + path_rows[(size_t)b * slots + j]) * chunks + c;
      const size_t dst = (size_t)i * chunks + c;
      cl[dst] = __ldg(hl + src);
      cm[dst] = __ldg(hm + src);
      ch[dst] = __ldg(hh + src);
      if (c == 0) row_map[i] = b * slots + j;
    }
    // output slot i = (b, j): zero past the request's accepted rows
    const int b = i / slots, j = i % slots;
    if (j >= s_off[b + 1] - s_off[b]) g_out[(size_t)i * chunks + c] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// fp32 accepted-rows fusion on the CUDA cores (exact fp32): one warp per
// output element g[b, j, o]; slots past the accepted path (or of a request
// whose path is invalid) are zero.
__global__ void __launch_bounds__(256)
    fuse_proj_accepted_f32_kernel(const float* __restrict__ hl, const float* __restrict__ hm,
                                  const float* __restrict__ hh, const float* __restrict__ w,
                                  const float* __restrict__ bias, const int32_t* __restrict__ path_rows,
                                  const int32_t* __restrict__ accept_len, float* __restrict__ g, int B, int R,
                                  int slots, int d, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)B * slots * d) return;
  const int o = (int)(gw % d);
  const int bj = (int)(gw / d), b = bj / slots, j = bj % slots;
  const int a = accept_len[b];
  bool ok = a >= 0 && a < slots;
  for (int jj = 0; ok && jj <= a; ++jj) {
    const int r = path_rows[(size_t)b * slots + jj];
    ok = r >= 0 && r < R;
  }
  if (!ok && j == 0 && o == 0 && lane == 0) set_status(status, EAGLE_ERR_BAD_TREE);
  if (!ok || j > a) {
    if (lane == 0) g[gw] = 0.f;
    return;
  }
  const size_t m = (size_t)b * R + path_rows[(size_t)b * slots + j];
  const float* wr = w + (size_t)o * 3 * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) {
    acc = fmaf(wr[c], hl[m * d + c], acc);
    acc = fmaf(wr[d + c], hm[m * d + c], acc);
    acc = fmaf(wr[2 * d + c], hh[m * d + c], acc);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) g[gw] = acc + (bias ? bias[o] : 0.f);
}

// fp32 fused projection on the CUDA cores (exact fp32): one warp per output
// element g[m, o]; lanes stride the 3d inputs of the concatenation.
__global__ void __launch_bounds__(256)
    fuse_proj_f32_kernel(const float* __restrict__ hl, const float* __restrict__ hm,
                         const float* __restrict__ hh, const float* __restrict__ w,
                         const float* __restrict__ bias, float* __restrict__ g, int M, int d) {
  pdl_wait();
  pdl_trigger();
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

// fp32 drafter input FC on the CUDA cores (exact fp32): one warp per output
// element u[m, o]; lanes stride the feature half and the embedding half of
// the concatenation [r_m; embed[token_ids[m]]].  An id outside [0, vocab)
// reads as a zero embedding and records EAGLE_ERR_BAD_TREE.
__global__ void __launch_bounds__(256)
    draft_input_f32_kernel(const float* __restrict__ r, const int32_t* __restrict__ ids,
                           const float* __restrict__ embed, int vocab, const float* __restrict__ w,
                           const float* __restrict__ bias, float* __restrict__ u, int M, int d,
                           int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)M * d) return;
  const int m = (int)(gw / d), o = (int)(gw % d);
  const int id = ids[m];
  const bool ok = id >= 0 && id < vocab;
  if (!ok && lane == 0 && o == 0) set_status(status, EAGLE_ERR_BAD_TREE);
  const float* wr = w + (size_t)o * 2 * d;
  const float* er = embed + (size_t)(ok ? id : 0) * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) {
    acc = fmaf(wr[c], r[(size_t)m * d + c], acc);
    if (ok) acc = fmaf(wr[d + c], er[c], acc);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) u[(size_t)m * d + o] = acc + (bias ? bias[o] : 0.f);
}

// Token-embedding lookup of the drafter input FC: out[m] = table[ids[m]]
// (bf16 rows of d elements), 16 bytes per thread over all SMs, so the
// projection then reads both halves of [r; e] through TMA.  An id outside
// [0, n_rows) gives a zero row and records EAGLE_ERR_BAD_TREE.
__global__ void __launch_bounds__(256)
    embed_gather_kernel(const int32_t* __restrict__ ids, const uint4* __restrict__ table, int n_rows,
                        int M, int d, uint4* __restrict__ out, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int cpr = d / 8;  // 16-byte chunks per row
  const long long n = (long long)M * cpr;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(i / cpr), c = (int)(i % cpr);
    const int id = __ldg(ids + m);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (id >= 0 && id < n_rows)
      v = __ldg(table + (size_t)id * cpr + c);
    else if (c == 0)
      set_status(status, EAGLE_ERR_BAD_TREE);
    out[i] = v;
  }
}

// fp32 linear layer on the CUDA cores (exact fp32): one warp per output
// element y[m, o] = sum_c w[o, c] x[m, c] (+ bias[o]) (+ residual[m, o]).
__global__ void __launch_bounds__(256)
    linear_f32_kernel(const float* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
                      const float* residual, float* y, int M, int n_out, int k_in) {
  pdl_wait();
  pdl_trigger();
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)M * n_out) return;
  const int m = (int)(gw / n_out), o = (int)(gw % n_out);
  const float* wr = w + (size_t)o * k_in;
  const float* xr = x + (size_t)m * k_in;
  float acc = 0.f;
  for (int c = lane; c < k_in; c += 32) acc = fmaf(wr[c], xr[c], acc);
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const size_t idx = (size_t)m * n_out + o;
    y[idx] = acc + (bias ? bias[o] : 0.f) + (residual ? residual[idx] : 0.f);
  }
}

// ------------------------------------------------------------------ host side
int pick_bn(int M, int* groups) {
  const int G = (M + 255) / 256;
  const int per = (M + G - 1) / G;
  *groups = G;
  return (per + 15) / 16 * 16;
}

int pick_stages(size_t stage, size_t extra) {
  const size_t budget = 227 * 1024 - 1024 - extra - 256;
  int s = (int)(budget / stage);
  return s > kMaxStages ? kMaxStages : s;
}


}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_lmhead_topk_workspace_size(int M, int d, int V, int k, int dtype) {
  (void)d;
  (void)V;
  (void)dtype;
  if (M <= 0 || k <= 0) return 0;
  const size_t n = (size_t)((M + 127) / 128) * 128 * kMaxCtas;  // [row][cta of its group]
  return round_up(n * 8, 256) + 2 * round_up(n * k * 4, 256) + round_up(n * 4, 256) + 1024;
}

namespace eagle {
namespace {
struct RaceCfg {
  int R;
  uint64_t seed, offset;
};

// The LM head proper: GEMM + per-CTA top-K / log-sum-exp partials, then the
// merge.  race != nullptr selects the exponential-race keys.
// phase: kBoth, or only the GEMM + per-CTA partials (kPartial, into ws), or
// only the merge of partials a kPartial call left in ws (kMerge).
enum LmPhase { kBoth = 0, kPartial = 1, kMerge = 2 };

// Activation groups (128 rows each), CTAs per group and vocabulary rows per
// tile of one LM-head call.
struct LmPlan {
  int G, cpg, tn, n_vtiles;
};
LmPlan lm_plan(int M, int V, int dtype, int sms) {
  LmPlan pl;
  pl.G = (M + 127) / 128;
  sms = sms > kMaxCtas ? kMaxCtas : sms;
  int cpg = sms / pl.G;
  if (cpg < 1) cpg = 1;
  if (cpg > kMaxCtas / pl.G) cpg = kMaxCtas / pl.G;
  // vocabulary rows per tile: 128 (fewer, larger K-chunks per byte of W_U
  // measured faster than narrower tiles with better balance); narrower only
  // when V is smaller than one tile per CTA
  int tn = 128;
  while (tn > 16 && (V + tn - 1) / tn < cpg) tn -= 16;
  // several activation groups re-read every W_U tile from L2: 256-row tiles
  // (two 256-column TMEM buffers) cut that traffic per flop by a third
  if (pl.G >= 2 && dtype == EAGLE_BF16 && (V + 255) / 256 >= 4 * cpg) tn = 256;
  pl.tn = tn;
  pl.n_vtiles = (V + tn - 1) / tn;
  if (cpg > pl.n_vtiles) cpg = pl.n_vtiles;
  pl.cpg = cpg;
  return pl;
}

int lmhead_run(const void* x, const void* w_lm, const float* bias, int M, int d, int V, int k,
               float temperature, int32_t* topk_ids, float* topk_logprobs, float* row_max,
               float* row_sumexp, int dtype, void* ws, size_t ws_bytes, int32_t* dev_status,
               void* stream, const RaceCfg* race, LmPhase phase = kBoth) {
  if (phase != kMerge && (!x || !w_lm)) return EAGLE_ERR_INVALID_ARG;
  if (phase != kPartial && (!topk_ids || !topk_logprobs)) return EAGLE_ERR_INVALID_ARG;
  if (M <= 0 || d <= 0 || V <= 0 || k <= 0 || !(temperature > 0.f) || isinf(temperature))
    return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (k > V) return EAGLE_ERR_INVALID_ARG;
  if (M > 2048 || k > 32 || d % 64 || V % 16) return EAGLE_ERR_UNSUPPORTED;
  if (phase != kMerge && (!aligned16(x) || !aligned16(w_lm))) return EAGLE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < eagle_lmhead_topk_workspace_size(M, d, V, k, dtype)) return EAGLE_ERR_WORKSPACE;
  const int sms = sm_count();
  if (sms <= 0) return EAGLE_ERR_CUDA;
  const LmPlan pl = lm_plan(M, V, dtype, sms);
  const int G = pl.G, cpg = pl.cpg, tn = pl.tn, n_vtiles = pl.n_vtiles;
  const int n_ctas = cpg * G;
  const size_t lists = 0;
  const int rows_g = M < 128 ? M : 128;           // rows of the largest group
  const int xr = (rows_g + 15) / 16 * 16;         // activation rows loaded per stage
  const size_t xbytes = (size_t)xr * 128;
  const size_t wtile = (size_t)tn * 128;  // bytes of one W_U stage
  const int stages = dtype == EAGLE_BF16 ? pick_stages(wtile + xbytes, lists + (kTileA - xbytes)) : 2;
  if (stages < 2) return EAGLE_ERR_UNSUPPORTED;
  const size_t smem = dtype == EAGLE_BF16
                          ? 1024 + (size_t)stages * (wtile + xbytes) + (kTileA - xbytes) + lists
                          : (size_t)(128 * (kF32Kc + 1) + 16 * kF32Kc) * 4 + lists;

  char* cur = static_cast<char*>(ws);
  const size_t n = (size_t)G * 128 * kMaxCtas;
  LmParams p;
  p.part_ms = static_cast<float2*>(ws_carve(cur, n * 8));
  p.part_v = static_cast<float*>(ws_carve(cur, n * k * 4));
  p.part_i = static_cast<int*>(ws_carve(cur, n * k * 4));
  p.part_cnt = static_cast<int*>(ws_carve(cur, n * 4));
  p.M = M;
  p.V = V;
  p.K = k;
  p.groups = G;
  p.ctas_per_group = cpg;
  p.n_vtiles = n_vtiles;
  p.nk = d / 64;
  p.tn = tn;
  p.stages = stages;
  p.xr = xr;
  p.inv_t = 1.f / temperature;
  p.race = race ? 1 : 0;
  p.R = race ? race->R : 1;
  p.race_k0 = race ? (uint32_t)race->seed : 0u;
  p.race_k1 = race ? (uint32_t)(race->seed >> 32) : 0u;
  p.race_c2 = race ? 2u * (uint32_t)(race->offset >> 32) + 1u : 0u;
  p.race_c3 = race ? (uint32_t)race->offset : 0u;
  p.bias = bias;
  p.topk_ids = topk_ids;
  p.topk_lp = topk_logprobs;
  p.row_max = row_max;
  p.row_sumexp = row_sumexp;
  p.status = dev_status;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (phase == kMerge) {
    // nothing to launch here but the merge below
  } else if (dtype == EAGLE_BF16) {
    CUtensorMap mx, mw;
    if (!make_tmap_2d(&mx, x, 2, (uint64_t)M, (uint64_t)d, (uint32_t)xr, 64) ||
        !make_tmap_2d(&mw, w_lm, 2, (uint64_t)V, (uint64_t)d, (uint32_t)tn, 64))
      return EAGLE_ERR_CUDA;
    auto kern = k <= 1 ? lmhead_topk_kernel<1>
                : k <= 4 ? lmhead_topk_kernel<4>
                : k <= 8 ? lmhead_topk_kernel<8>
                : k <= 12 ? lmhead_topk_kernel<12>
                : k <= 16 ? lmhead_topk_kernel<16> : lmhead_topk_kernel<32>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch(kern, n_ctas, kThreads, smem, s, mx, mw, p);
  } else {
    auto kern = k <= 1 ? lmhead_topk_f32_kernel<1>
                : k <= 4 ? lmhead_topk_f32_kernel<4>
                : k <= 8 ? lmhead_topk_f32_kernel<8>
                : k <= 12 ? lmhead_topk_f32_kernel<12>
                : k <= 16 ? lmhead_topk_f32_kernel<16> : lmhead_topk_f32_kernel<32>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch(kern, n_ctas, kEpiThreads, smem, s, (const float*)x, (const float*)w_lm, d, p);
  }
  if (phase != kMerge) note_launch();
  if (phase == kPartial) return last_launch_status();
  // merge of the per-CTA partials: one CTA per row, lists staged in shared memory
  const size_t msmem = (size_t)cpg * (k * 8 + 4);
  if (msmem > 227 * 1024) return EAGLE_ERR_UNSUPPORTED;
  if (msmem > 48 * 1024)
    cudaFuncSetAttribute(lmhead_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msmem);
  launch(lmhead_merge_kernel, M, kMergeThreads, msmem, s, p);
  note_launch();
  return last_launch_status();
}

// Target logit of each child's token at its parent row: one warp per tree
// row c of request b, z = x[b R + parent(c)] . W_U[token(c)] (+ bias), fp32
// accumulation of the exact products; 0 for the root and rows past n_rows.
template <typename T>
__global__ void __launch_bounds__(256) child_logit_kernel(
    const T* __restrict__ x, const T* __restrict__ w, const float* __restrict__ bias,
    const int32_t* __restrict__ parent_row, const int32_t* __restrict__ token,
    const int32_t* __restrict__ n_rows, int B, int R, int d, int V, float* __restrict__ out,
    int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)B * R) return;
  const int b = (int)(gw / R), c = (int)(gw % R);
  const int n = n_rows ? n_rows[b] : R;
  float acc = 0.f;
  bool ok = c > 0 && c < n && n <= R;
  int pr = 0, t = 0;
  if (ok) {
    pr = parent_row[gw];
    t = token[gw];
    ok = pr >= 0 && pr < c && t >= 0 && t < V;
    if (!ok && lane == 0) set_status(status, EAGLE_ERR_BAD_TREE);
  }
  if (ok) {
    const T* xr = x + ((size_t)b * R + pr) * d;
    const T* wr = w + (size_t)t * d;
    if (sizeof(T) == 2) {
      for (int c8 = lane; c8 < d / 8; c8 += 32) {
        const uint4 xa = *reinterpret_cast<const uint4*>(xr + c8 * 8);
        const uint4 wa = *reinterpret_cast<const uint4*>(wr + c8 * 8);
        const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(&xa);
        const __nv_bfloat162* wh = reinterpret_cast<const __nv_bfloat162*>(&wa);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 xf = __bfloat1622float2(xh[u]), wf = __bfloat1622float2(wh[u]);
          acc = fmaf(xf.x, wf.x, acc);
          acc = fmaf(xf.y, wf.y, acc);
        }
      }
    } else {
      for (int c1 = lane; c1 < d; c1 += 32) acc = fmaf((float)xr[c1], (float)wr[c1], acc);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) out[gw] = ok ? acc + (bias ? bias[t] : 0.f) : 0.f;
}
}  // namespace
}  // namespace eagle

namespace eagle {
// The partials an eagle_lmhead_topk_partial call left in ws (the carve of lmhead_run).
bool lm_partials_view(void* ws, size_t ws_bytes, int M, int d, int V, int k, int dtype, float temperature,
                      LmPartials* out) {
  if (!ws || M <= 0 || d <= 0 || V <= 0 || k <= 0 || k > 32 || k > V || M > 2048 || d % 64 || V % 16)
    return false;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return false;
  if (!(temperature > 0.f) || isinf(temperature)) return false;
  if (ws_bytes < eagle_lmhead_topk_workspace_size(M, d, V, k, dtype)) return false;
  const int sms = sm_count();
  if (sms <= 0) return false;
  const LmPlan pl = lm_plan(M, V, dtype, sms);
  char* cur = static_cast<char*>(ws);
  const size_t n = (size_t)pl.G * 128 * kMaxCtas;
  out->ms = static_cast<const float2*>(ws_carve(cur, n * 8));
  out->v = static_cast<const float*>(ws_carve(cur, n * k * 4));
  out->id = static_cast<const int*>(ws_carve(cur, n * k * 4));
  out->cnt = static_cast<const int*>(ws_carve(cur, n * 4));
  out->cpg = pl.cpg;
  out->K = k;
  out->inv_t = 1.f / temperature;
  out->race = 0;
  return true;
}
}  // namespace eagle

extern "C" int eagle_lmhead_topk(const void* x, const void* w_lm, const float* bias, int M, int d,
                                 int V, int k, float temperature, int32_t* topk_ids,
                                 float* topk_logprobs, float* row_max, float* row_sumexp, int dtype,
                                 void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return lmhead_run(x, w_lm, bias, M, d, V, k, temperature, topk_ids, topk_logprobs, row_max,
                    row_sumexp, dtype, ws, ws_bytes, dev_status, stream, nullptr);
}

extern "C" int eagle_lmhead_topk_partial(const void* x, const void* w_lm, const float* bias, int M, int d,
                                         int V, int k, float temperature, int dtype, void* ws,
                                         size_t ws_bytes, int32_t* dev_status, void* stream) {
  return lmhead_run(x, w_lm, bias, M, d, V, k, temperature, nullptr, nullptr, nullptr, nullptr, dtype, ws,
                    ws_bytes, dev_status, stream, nullptr, kPartial);
}

extern "C" int eagle_lmhead_topk_merge(int M, int d, int V, int k, float temperature, int32_t* topk_ids,
                                       float* topk_logprobs, float* row_max, float* row_sumexp, int dtype,
                                       void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return lmhead_run(nullptr, nullptr, nullptr, M, d, V, k, temperature, topk_ids, topk_logprobs, row_max,
                    row_sumexp, dtype, ws, ws_bytes, dev_status, stream, nullptr, kMerge);
}

extern "C" int eagle_lmhead_verify_stats(const void* x, const void* w_lm, const float* bias, int B,
                                         int R, int d, int V, const int32_t* parent_row,
                                         const int32_t* token, const int32_t* n_rows,
                                         float temperature, uint64_t seed, uint64_t offset,
                                         int race_k, int32_t* race_ids, float* race_keys,
                                         float* row_max, float* row_sumexp, float* child_logit,
                                         int dtype, void* ws, size_t ws_bytes,
                                         int32_t* dev_status, void* stream) {
  if (B <= 0 || R <= 0 || !parent_row || !token || !row_max || !row_sumexp || !child_logit)
    return EAGLE_ERR_INVALID_ARG;
  if ((long long)B * R > 2048) return EAGLE_ERR_UNSUPPORTED;
  if ((offset >> 63) != 0) return EAGLE_ERR_INVALID_ARG;
  const RaceCfg rc{R, seed, offset};
  const int st = lmhead_run(x, w_lm, bias, B * R, d, V, race_k, temperature, race_ids, race_keys,
                            row_max, row_sumexp, dtype, ws, ws_bytes, dev_status, stream, &rc);
  if (st != EAGLE_OK) return st;
  const long long rows = (long long)B * R;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == EAGLE_BF16)
    launch(child_logit_kernel<__nv_bfloat16>, (unsigned)((rows + 7) / 8), 256, 0, s,
           (const __nv_bfloat16*)x, (const __nv_bfloat16*)w_lm, bias, parent_row, token, n_rows, B,
           R, d, V, child_logit, dev_status);
  else
    launch(child_logit_kernel<float>, (unsigned)((rows + 7) / 8), 256, 0, s, (const float*)x,
           (const float*)w_lm, bias, parent_row, token, n_rows, B, R, d, V, child_logit,
           dev_status);
  note_launch();
  return last_launch_status();
}

namespace {
struct FpPlan {
  int bn, G, n_otiles, nk, nkd, n_tiles, n_ctas, max_contrib;
  long long W;
};
// nseg: K segments of width d (3 for the feature fusion, 2 for the drafter input)
// n_out output features (multiple of 128); nseg K segments of kseg inputs each
FpPlan fp_plan(int M, int n_out, int kseg, int esz, int n_ctas_cap, int nseg) {
  FpPlan f;
  f.bn = pick_bn(M, &f.G);
  const int bke = 128 / esz;
  f.n_otiles = n_out / 128;
  f.nkd = kseg / bke;
  f.nk = nseg * f.nkd;
  f.n_tiles = f.n_otiles * f.G;
  f.W = (long long)f.n_tiles * f.nk;
  f.n_ctas = (int)(f.W < n_ctas_cap ? f.W : n_ctas_cap);
  const long long per = f.W / f.n_ctas;  // minimum chunks per CTA
  f.max_contrib = (int)((f.nk + per - 1) / per) + 1;
  if (f.max_contrib > f.n_ctas) f.max_contrib = f.n_ctas;
  return f;
}

// Contributor slots a tile needs when only the first g of the plan's groups
// hold live rows (a row count known on the device): the same CTAs split the
// smaller chunk range, so a tile may be shared by more of them.
int fp_live_contrib(const FpPlan& f) {
  int mc = f.max_contrib;
  for (int g = 1; g < f.G; ++g) {
    const long long W = (long long)f.n_otiles * g * f.nk;
    const int n = W < f.n_ctas ? (int)W : f.n_ctas;  // the active CTAs (fp_live)
    const long long per = W / n;                       // >= 1
    long long c = (f.nk + per - 1) / per + 1;
    if (c > n) c = n;
    if (c > mc) mc = (int)c;
  }
  return mc;
}

// The lanes schedule (several groups, rows known on the host) over pairs of
// output tiles: taken when the tiles pair up and every lane still holds at
// least 4 (pair, K chunk) items.  Contributor slots a tile then needs.
bool fp_use_dual(const FpPlan& f) {
  if (f.G < 2 || f.n_otiles % 2) return false;
  const int lanes = f.n_ctas / f.G;
  return lanes >= 1 && (long long)(f.n_otiles / 2) * f.nk >= 4LL * lanes;
}
int fp_dual_contrib(const FpPlan& f) {
  const int lanes = f.n_ctas / f.G;
  const long long per = (long long)(f.n_otiles / 2) * f.nk / lanes;  // >= 4
  long long c = (f.nk + per - 1) / per + 1;
  if (c > lanes) c = lanes;
  return (int)c;
}

// gathered: room for the [M, d] looked-up embedding rows (drafter input FC);
// live: a device row count (the accepted-rows fusion), whose partials need
// fp_live_contrib slots and which packs nseg [M, kseg] segments, a row map
// and the count into the workspace
size_t fp_workspace(int M, int n_out, int kseg, int dtype, int nseg, bool gathered, bool live = false) {
  if (M <= 0 || n_out <= 0 || kseg <= 0 || n_out % 128 || kseg % 64) return 0;
  const int esz = dtype == EAGLE_BF16 ? 2 : 4;
  // sized for the largest grid the library launches (kMaxCtas CTAs)
  size_t best = 0;
  for (int cap = 1; cap <= kMaxCtas; ++cap) {
    const FpPlan f = fp_plan(M, n_out, kseg, esz, cap, nseg);
    int mc = live ? fp_live_contrib(f) : f.max_contrib;
    if (!live && fp_use_dual(f) && fp_dual_contrib(f) > mc) mc = fp_dual_contrib(f);
    size_t sz = round_up((size_t)f.n_tiles * mc * f.bn * 128 * 4, 256) + 1024 +
                (gathered ? round_up((size_t)M * kseg * esz, 256) : 0);
    if (live) sz += nseg * round_up((size_t)M * kseg * esz, 256) + round_up((size_t)M * 4, 256) + 256;
    best = sz > best ? sz : best;
  }
  return best;
}

// bf16 tensor-core launch shared by both projections: xs[0..nseg) are the
// [M, d] activation segments, read by TMA; with `ids` set the last segment is
// first looked up from `table` ([n_rows, d]) into the workspace.
// Rows of an accepted-rows fusion: the packed activation segments, their
// output rows and their count are written by a gather kernel on the device.
struct FpLiveRows {
  const int32_t* path_rows;
  const int32_t* accept_len;
  int B, R, slots;
};
// Activations read as rows r0 .. r0 + W - 1 of each of B requests of a
// [B, Rmax, K] array (one K segment), activation row b W + j.
struct FpRowView {
  int B, W, Rmax, r0;
};

// Clusters of cs CTAs of the projection kernel (with `smem` bytes of shared
// memory) that the current device runs at once; cached per (device, cs, smem).
int fp_max_clusters(int cs, size_t smem) {
  struct Entry {
    int dev, cs;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.cs == cs && e.smem == smem) return e.n;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fuse_proj_kernel<false>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache.push_back(Entry{dev, cs, smem, n});
  return n;
}

// The tile split of a projection with one activation group and a host row
// count: the largest cs in {1, 2, 4, 8} whose n_otiles * cs CTAs fit on the
// SMs in one wave (as clusters of cs) with at least kFpMinChunks K chunks
// each, provided they occupy at least 4/5 of the SMs; else 0 (stream-K over
// every SM, partial tiles summed by a second kernel).  Measured: 32 tiles in
// clusters of 4 (128 SMs) beat stream-K; 48 tiles in clusters of 2 (96 SMs)
// lose to it (16.3 against 14.2 µs for a 6144 x 4096 weight).
constexpr int kFpMinChunks = 4;
int fp_cluster_size(const FpPlan& f, int sms, size_t smem) {
  if (f.G != 1) return 0;
  int best = 0;
  for (int cs = 1; cs <= 8; cs *= 2) {
    if ((long long)f.n_otiles * cs > sms || f.nk / cs < kFpMinChunks) break;
    if (cs > 1 && fp_max_clusters(cs, smem) < f.n_otiles) break;
    best = cs;
  }
  if (best && 5LL * f.n_otiles * best < 4LL * sms) return 0;
  return best;
}

int fp_launch_bf16(const void* const* xs, int nseg, const int32_t* ids, const void* table, int n_rows,
                   const void* w, const float* bias, const void* residual, void* out, int M, int n_out,
                   int kseg, void* ws, int32_t* dev_status, cudaStream_t s,
                   const FpLiveRows* live = nullptr, const FpRowView* view = nullptr) {
  constexpr int esz = 2, bke = 64;
  int sms = sm_count();
  if (sms <= 0) return EAGLE_ERR_CUDA;
  const FpPlan f = fp_plan(M, n_out, kseg, esz, sms > kMaxCtas ? kMaxCtas : sms, nseg);
  if (view && (nseg != 1 || live || ids || view->W < 1 || view->W > 256 ||
               (view->B > 1 && (f.bn % view->W || f.bn / view->W > 256))))
    return EAGLE_ERR_UNSUPPORTED;  // nothing launched
  // several groups with a host row count: lockstep lanes, over pairs of
  // output tiles when they pair up (two A tiles per stage)
  const bool dual = !live && fp_use_dual(f);
  const size_t stage_bytes = (dual ? 2 : 1) * (size_t)kTileA + (size_t)f.bn * 128;
  const int stages = pick_stages(stage_bytes, 0);
  if (stages < 2) return EAGLE_ERR_UNSUPPORTED;
  const size_t smem = 1024 + (size_t)stages * stage_bytes;
  const int max_contrib = dual ? fp_dual_contrib(f) : live ? fp_live_contrib(f) : f.max_contrib;

  char* cur = static_cast<char*>(ws);
  float* part = static_cast<float*>(ws_carve(cur, (size_t)f.n_tiles * max_contrib * f.bn * 128 * 4));
  const void* seg[3] = {xs[0], nseg > 1 ? xs[1] : xs[0], nseg > 2 ? xs[2] : xs[0]};
  int32_t* row_map = nullptr;
  int32_t* m_dev = nullptr;
  if (live) {
    void* packed[3];
    for (int i = 0; i < 3; ++i) packed[i] = ws_carve(cur, (size_t)M * kseg * esz);
    row_map = static_cast<int32_t*>(ws_carve(cur, (size_t)M * 4));
    m_dev = static_cast<int32_t*>(ws_carve(cur, 4));
    const long long work = (long long)M * (kseg / 8);
    const long long blocks = (work + kAccThreads - 1) / kAccThreads;
    launch(accepted_gather_kernel, (unsigned)(blocks < 2LL * sms ? blocks : 2LL * sms), kAccThreads, 0, s,
           live->B, live->R, live->slots, kseg / 8, live->path_rows, live->accept_len,
           static_cast<const uint4*>(seg[0]), static_cast<const uint4*>(seg[1]),
           static_cast<const uint4*>(seg[2]), static_cast<uint4*>(packed[0]), static_cast<uint4*>(packed[1]),
           static_cast<uint4*>(packed[2]), row_map, m_dev, static_cast<uint4*>(out), dev_status);
    note_launch();
    for (int i = 0; i < 3; ++i) seg[i] = packed[i];
  }
  void* gathered = nullptr;
  if (ids) {
    gathered = ws_carve(cur, (size_t)M * kseg * esz);
    seg[nseg - 1] = gathered;
  }
  CUtensorMap mw, mx[3];
  if (!make_tmap_2d(&mw, w, esz, (uint64_t)n_out, (uint64_t)nseg * kseg, 128, (uint32_t)bke))
    return EAGLE_ERR_CUDA;
  int view_w = 0;
  if (view) {
    // one request: its W rows are contiguous; several: a 3-D box of W rows
    // of bn / W requests lands the bn rows as a 2-D box would
    const char* vb = static_cast<const char*>(seg[0]) + (size_t)view->r0 * kseg * esz;
    if (view->B == 1) {
      if (!make_tmap_2d(&mx[0], vb, esz, (uint64_t)view->W, (uint64_t)kseg, (uint32_t)f.bn, (uint32_t)bke))
        return EAGLE_ERR_CUDA;
    } else {
      if (!make_tmap_3d_bf16(&mx[0], vb, (uint64_t)kseg, (uint64_t)view->W, (uint64_t)view->B,
                             (uint64_t)kseg * esz, (uint64_t)view->Rmax * kseg * esz, (uint32_t)bke,
                             (uint32_t)view->W, (uint32_t)(f.bn / view->W)))
        return EAGLE_ERR_CUDA;
      view_w = view->W;
    }
    mx[1] = mx[2] = mx[0];
  } else {
    for (int i = 0; i < 3; ++i)
      if (!make_tmap_2d(&mx[i], seg[i], esz, (uint64_t)M, (uint64_t)kseg, (uint32_t)f.bn, (uint32_t)bke))
        return EAGLE_ERR_CUDA;
  }

  if (ids) {
    const long long chunks = (long long)M * (kseg / 8);
    const long long blocks = (chunks + 255) / 256;
    launch(embed_gather_kernel, (unsigned)(blocks < 4LL * sms ? blocks : 4LL * sms), 256, 0, s, ids,
           static_cast<const uint4*>(table), n_rows, M, kseg, static_cast<uint4*>(gathered), dev_status);
    note_launch();
  }
  FpParams p;
  p.part = part;
  p.M = M;
  p.d = n_out;
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
  p.residual = residual;
  p.out = out;
  p.status = dev_status;
  p.m_dev = m_dev;
  p.row_map = row_map;
  p.max_contrib = max_contrib;
  p.tmajor = (!live && f.G > 1) ? 1 : 0;
  p.lanes = 0;
  p.dual = 0;
  p.view_w = view_w;
  cudaFuncSetAttribute(fuse_proj_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (dual)
    cudaFuncSetAttribute(fuse_proj_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  p.cs = live ? 0 : fp_cluster_size(f, sms, smem);
  if (p.cs) {
    // one wave of n_otiles * cs CTAs, no partials in the workspace
    const unsigned grid = (unsigned)(f.n_otiles * p.cs);
    p.n_ctas = (int)grid;
    if (p.cs > 1)
      launch_cluster(fuse_proj_kernel<false>, grid, kThreads, dim3((unsigned)p.cs), smem, s, mw, mx[0], mx[1],
                     mx[2], p);
    else
      launch(fuse_proj_kernel<false>, grid, kThreads, smem, s, mw, mx[0], mx[1], mx[2], p);
    note_launch();
    return last_launch_status();
  }
  if (p.tmajor) {
    // groups in lockstep: lanes of `groups` CTAs (n_ctas is at most W, so a
    // lane holds at least one chunk of its group when W >= n_ctas)
    p.lanes = f.n_ctas / f.G;
    p.n_ctas = p.lanes * f.G;
    p.dual = dual ? 1 : 0;
  }
  if (p.dual)
    launch(fuse_proj_kernel<false, true>, p.n_ctas, kThreads, smem, s, mw, mx[0], mx[1], mx[2], p);
  else
    launch(fuse_proj_kernel<false>, p.n_ctas, kThreads, smem, s, mw, mx[0], mx[1], mx[2], p);
  launch(fuse_proj_reduce_kernel<false>, dim3((unsigned)((f.bn * 32 + 255) / 256), (unsigned)f.n_tiles),
         256, 0, s, p);
  note_launch(2);
  return last_launch_status();
}
}  // namespace

extern "C" size_t eagle_fuse_proj_workspace_size(int M, int d, int dtype) {
  return fp_workspace(M, d, d, dtype, 3, false);
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
    launch(fuse_proj_f32_kernel, (unsigned)((outs + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream),
        (const float*)h_low, (const float*)h_mid, (const float*)h_high, (const float*)w_proj, bias,
        (float*)g, M, d);
    note_launch();
    return last_launch_status();
  }
  const void* xs[3] = {h_low, h_mid, h_high};
  return fp_launch_bf16(xs, 3, nullptr, nullptr, 0, w_proj, bias, nullptr, g, M, d, d, ws, dev_status,
                        static_cast<cudaStream_t>(stream));
}

extern "C" size_t eagle_fuse_proj_accepted_workspace_size(int B, int max_depth, int d, int dtype) {
  if (B <= 0 || max_depth < 0 || (long long)B * (max_depth + 1) > 4096) return 0;
  if (dtype == EAGLE_FP32) return 256;
  return fp_workspace(B * (max_depth + 1), d, d, dtype, 3, false, true);
}

extern "C" int eagle_fuse_proj_accepted(const void* h_low, const void* h_mid, const void* h_high,
                                        const void* w_proj, const float* bias, const int32_t* path_rows,
                                        const int32_t* accept_len, int B, int R, int max_depth, int d,
                                        int dtype, void* g, void* ws, size_t ws_bytes, int32_t* dev_status,
                                        void* stream) {
  if (!h_low || !h_mid || !h_high || !w_proj || !g || !path_rows || !accept_len) return EAGLE_ERR_INVALID_ARG;
  if (B <= 0 || R <= 0 || max_depth < 0 || d <= 0) return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  const long long cap = (long long)B * (max_depth + 1);
  if (cap > 4096 || B > kAccMaxB || d % 128 || d > 16384 || (long long)B * R > 2147483647LL / d)
    return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(h_low) || !aligned16(h_mid) || !aligned16(h_high) || !aligned16(w_proj) || !aligned16(g))
    return EAGLE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < eagle_fuse_proj_accepted_workspace_size(B, max_depth, d, dtype))
    return EAGLE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == EAGLE_FP32) {
    const long long outs = cap * d;
    launch(fuse_proj_accepted_f32_kernel, (unsigned)((outs + 7) / 8), 256, 0, s, (const float*)h_low,
           (const float*)h_mid, (const float*)h_high, (const float*)w_proj, bias, path_rows, accept_len,
           (float*)g, B, R, max_depth + 1, d, dev_status);
    note_launch();
    return last_launch_status();
  }
  const void* xs[3] = {h_low, h_mid, h_high};
  const FpLiveRows live{path_rows, accept_len, B, R, max_depth + 1};
  return fp_launch_bf16(xs, 3, nullptr, nullptr, 0, w_proj, bias, nullptr, g, (int)cap, d, d, ws, dev_status, s,
                        &live);
}

extern "C" size_t eagle_draft_input_workspace_size(int M, int d, int dtype) {
  return fp_workspace(M, d, d, dtype, 2, true);
}

extern "C" int eagle_draft_input(const void* r, const int32_t* token_ids, const void* embed, int vocab,
                                 const void* w_in, const float* bias, void* u, int M, int d, int dtype,
                                 void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!r || !token_ids || !embed || !w_in || !u) return EAGLE_ERR_INVALID_ARG;
  if (M <= 0 || d <= 0 || vocab <= 0) return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (M > 4096 || d % 128 || d > 16384) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(r) || !aligned16(embed) || !aligned16(w_in)) return EAGLE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < eagle_draft_input_workspace_size(M, d, dtype)) return EAGLE_ERR_WORKSPACE;
  if (dtype == EAGLE_FP32) {
    const long long outs = (long long)M * d;
    launch(draft_input_f32_kernel, (unsigned)((outs + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream),
           (const float*)r, token_ids, (const float*)embed, vocab, (const float*)w_in, bias, (float*)u, M, d,
           dev_status);
    note_launch();
    return last_launch_status();
  }
  const void* xs[2] = {r, nullptr};
  return fp_launch_bf16(xs, 2, token_ids, embed, vocab, w_in, bias, nullptr, u, M, d, d, ws, dev_status,
                        static_cast<cudaStream_t>(stream));
}

namespace eagle {
int linear_rows_bf16(const void* x, int B, int W, int Rmax, int r0, const void* w, const float* bias,
                     const void* residual, void* y, int n_out, int k_in, void* ws, size_t ws_bytes,
                     int32_t* dev_status, cudaStream_t s) {
  if (!x || !w || !y || B <= 0 || W <= 0 || r0 < 0 || r0 + W > Rmax) return EAGLE_ERR_INVALID_ARG;
  const long long M = (long long)B * W;
  if (M > 4096 || n_out % 128 || k_in % 64 || n_out > 65536 || k_in > 65536) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (residual && !aligned16(residual)))
    return EAGLE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < eagle_linear_workspace_size((int)M, n_out, k_in, EAGLE_BF16)) return EAGLE_ERR_WORKSPACE;
  const void* xs[1] = {x};
  const FpRowView v{B, W, Rmax, r0};
  return fp_launch_bf16(xs, 1, nullptr, nullptr, 0, w, bias, residual, y, (int)M, n_out, k_in, ws, dev_status, s,
                        nullptr, &v);
}
}  // namespace eagle

extern "C" size_t eagle_linear_workspace_size(int M, int n_out, int k_in, int dtype) {
  return fp_workspace(M, n_out, k_in, dtype, 1, false);
}

extern "C" int eagle_linear(const void* x, const void* w, const float* bias, const void* residual, void* y,
                            int M, int n_out, int k_in, int dtype, void* ws, size_t ws_bytes,
                            int32_t* dev_status, void* stream) {
  if (!x || !w || !y) return EAGLE_ERR_INVALID_ARG;
  if (M <= 0 || n_out <= 0 || k_in <= 0) return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (x == y) return EAGLE_ERR_INVALID_ARG;
  if (M > 4096 || n_out % 128 || k_in % 64 || n_out > 65536 || k_in > 65536) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (residual && !aligned16(residual)))
    return EAGLE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < eagle_linear_workspace_size(M, n_out, k_in, dtype)) return EAGLE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == EAGLE_FP32) {
    const long long outs = (long long)M * n_out;
    launch(linear_f32_kernel, (unsigned)((outs + 7) / 8), 256, 0, s, (const float*)x, (const float*)w, bias,
           (const float*)residual, (float*)y, M, n_out, k_in);
    note_launch();
    return last_launch_status();
  }
  const void* xs[1] = {x};
  return fp_launch_bf16(xs, 1, nullptr, nullptr, 0, w, bias, residual, y, M, n_out, k_in, ws, dev_status, s);
}
