// Tree-masked attention of draft-tree rows against a paged KV cache plus the
// tree's own K/V rows.
//
// Source: "M7.5 - EAGLE Feature Drafting: Uncertainty, Dynamic Trees, HASS, and
// EAGLE-3", section 0x08C "Training-Time Test" (visibility: A(u, v) = 1 iff v
// in TargetPrefix(u) u DraftAncestors(u) u {u}); "EAGLE: Speculative Sampling
// Requires Rethinking Feature Uncertainty", "Tree-Structured Draft
// Generation" (each node attends only to its ancestors); "EAGLE-3: Scaling up
// Inference Acceleration ...", "The Attention Mechanism Modifications".
//
// bf16 path: tcgen05 tensor-core kernels.  The work is a set of units, one per
// (request, kv head, group of one or two query tiles): all query rows of one
// kv head (R tree rows x G grouped heads) share every K/V byte the CTA stages,
// so each prefix byte leaves HBM once per query-tile group.  A unit's key
// blocks are its 64-key prefix blocks, then one block of the tree's own rows
// (masked by the u64 ancestry bits).  Two schedules:
//   stream (many key blocks per SM): a persistent kernel, one CTA per SM.  The
//     CTAs form groups of Hkv, one CTA per kv head, so that the heads of one
//     page are read together; a group's blocks -- those of every (request,
//     query-tile group) laid end to end -- are split evenly over the groups,
//     planned on the device from the real ctx_lens.  Every SM streams the same
//     number of blocks whatever the mix of context lengths and pays its
//     set-up once.  A CTA walks its range as segments (a unit, or the part of
//     one in the range); the K/V ring runs on across segments.  A whole unit
//     writes the output; a piece of a unit split between CTAs writes its
//     normalised (O, lse) to a workspace slot, merged by a second kernel.
//   split (few key blocks per SM): one CTA per (query-tile group, KV range,
//     request x kv head); the KV ranges' (O, lse) partials are merged by a
//     second kernel.
// fp32 path (small shapes): a warp per query row.
#include <math.h>

#include "common.cuh"

namespace eagle {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ----------------------------------------------------------------------------
// tcgen05 path (bf16).  128 + 128 * TPC threads per CTA:
//   warp 0     producer of Q (split schedule; the stream schedule's S issuer
//              loads each segment's Q itself once the previous segment's S
//              MMAs are complete, so the K loads never stop at a segment's
//              end) and of the K blocks (4 paged 16-key boxes per
//              64-column half: a 3-D map over the pool viewed as
//              [pages*16][Hkv][D], or the tree's own K rows), into a ring of
//              kv_stages(TPC) stages; a K stage is free once S of its block is
//              complete
//   warp 1     allocates the tensor memory, then issues O += P V (M 128, N D,
//              K 64, V read MN-major) as soon as P of a block is ready; its
//              commit frees the block's V stage
//   warp 2     producer of the V blocks (same boxes as K)
//   warp 3     S issuer (one thread): S = Q K^T (M 128, N 64, K D) into one of
//              two TMEM S buffers per tile, up to two blocks ahead.  Two
//              issuing threads, because one thread issues an MMA only every
//              ~50 cycles
//   warps 4.. (4 per query tile): softmax, one thread per query row (TMEM
//              lane; a quarter or tile without query rows only keeps the
//              barrier protocol): the block's 64 scores loaded once, masked
//              row max, P = exp2(S - m) rounded to bf16 into a double-buffered
//              128-byte-swizzled shared tile (the A operand of P V), and O
//              rescaled in TMEM only when the row max grows by more than 2^8;
//              at the end of a segment, O / l (and the lse) to the output or
//              to the segment's partial slot
// Masked keys read as -inf through a select, so nothing a masked K row holds
// reaches the softmax; V rows of a partly filled page or of the padded tree
// block are zeroed in shared memory before P V reads them.
namespace tc {
constexpr int kBlk = 64;           // keys per block (4 pages)
constexpr int kBlkBytesHalf = kBlk * 128;  // one 64-column half of a K or V block
constexpr int kMaxStages = 8;
// K/V ring depth: what the shared memory left by the Q tiles and the double
// buffered P tiles holds
template <int D>
__host__ __device__ constexpr int kv_stages(int tpc) {
  return D == 128 ? (tpc == 2 ? 3 : 5) : 8;
}
constexpr float kRescaleLog2 = 8.f;        // O / l reference moves when the max grows by > 2^8
struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kMaxStages], v_full[kMaxStages], k_empty[kMaxStages], kv_empty[kMaxStages];
  uint64_t s_full[2], s_empty[2], p_full[2];
  uint64_t drain, drain_pv;
  uint32_t tmem_base;
  int abort_flag;
  // the CTA's range of blocks [lo, hi); the requests holding lo and hi - 1
  // and their first blocks
  long long lo, hi, off, off_last;
  int b, b_last;
  long long tot;  // blocks of one head over all requests
  int n_groups;   // active head groups
  long long warp_sum[32];
  int stop;          // a uniform leave decision of the softmax warps
  float xlse[64];    // two-copy tiles: the second copy's row lse at a segment's end
};
struct Params {
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const uint64_t* tree_mask;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;    // [n_ctas * 2 slots][TPC][128 rows][D]: normalised O of a piece
  float* part_lse;  // [n_ctas * 2 slots][TPC][128 rows]
  int4* merge;      // [n_ctas]: the split unit a CTA's merge column handles, or x = -1
  int32_t* status;
  int B, R, Hq, Hkv, G, max_pages, num_pages;
  int nr;         // tree rows per query tile (rows per tile = nr * G <= 128)
  int qtiles;     // query tiles of a (request, kv head)
  int ncq;        // query-tile groups (units) per (request, kv head)
  int tr;         // tree keys loaded: R rounded up to 16
  int q_box_rows; // tree rows per Q box: nr, or the rows of one copy of a two-copy tile
  int n_ctas;     // stream schedule: the grid, groups of Hkv CTAs, one per kv head
  int splits;     // split schedule: KV ranges per (query-tile group, request x kv head)
  float scale_log2;
};

// A request's context length, clamped to its block table (an out-of-range
// value is reported as EAGLE_ERR_BAD_KV when `report`).
__device__ __forceinline__ int req_ctx(const Params& p, int b, bool report) {
  int ctx = p.ctx_lens[b];
  if (ctx < 0 || ctx > p.max_pages * 16) {
    if (report) set_status(p.status, EAGLE_ERR_BAD_KV);
    ctx = ctx < 0 ? 0 : p.max_pages * 16;
  }
  return ctx;
}
// key blocks of one unit of a request: its prefix blocks and the tree block
__device__ __forceinline__ int unit_len(int ctx) { return (ctx + kBlk - 1) / kBlk + 1; }

__host__ __device__ __forceinline__ long long share_lo(long long c, long long T, long long n) {
  return c * T / n;
}
__device__ __forceinline__ int share_owner(long long x, long long T, int n) {
  int c = (int)((x * n) / T);
  while (c + 1 < n && share_lo(c + 1, T, n) <= x) ++c;
  while (c > 0 && share_lo(c, T, n) > x) --c;
  return c;
}

// The plan (all threads of the block call it).  The CTAs form groups of Hkv,
// CTA c serving kv head c % Hkv in group c / Hkv, so that the Hkv CTAs that
// read the heads of one page do so at the same time.  A group's work is the
// key blocks of every (request, query-tile group) unit of its head laid end
// to end: T = sum_b unit_len(ctx_b) * ncq.  Group g of n = min(groups, T)
// active groups takes the blocks [g T / n, (g + 1) T / n) (every active group
// holds at least one).  Also located: the requests holding the range's first
// and last blocks.  Returns false when group g has no work.  Block-wide: two
// chunked scans of the requests' block counts.
__device__ bool plan_range(const Params& p, int g, Bars& sb) {
  const int nthr = blockDim.x, t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = nthr >> 5;
  const long long per_req = p.ncq;
  // pass 1: T
  long long mine = 0;
  for (int b = t; b < p.B; b += nthr) mine += unit_len(req_ctx(p, b, g == 0)) * per_req;
#pragma unroll
  for (int o = 16; o; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) sb.warp_sum[warp] = mine;
  __syncthreads();
  if (t == 0) {
    long long T = 0;
    for (int w = 0; w < nw; ++w) T += sb.warp_sum[w];
    sb.tot = T;
    const long long groups = p.n_ctas / p.Hkv;
    const int n = (int)(T < groups ? T : groups);
    sb.n_groups = n;
    sb.lo = g < n ? share_lo(g, T, n) : 0;
    sb.hi = g < n ? share_lo(g + 1, T, n) : 0;
    sb.b = -1;
    sb.b_last = -1;
  }
  __syncthreads();
  const long long lo = sb.lo, hi = sb.hi;
  if (lo >= hi) return false;
  const long long x0 = lo, x1 = hi - 1;
  // pass 2: the requests holding x0 and x1 (chunks of nthr requests,
  // exclusive scan across the chunk, carried over chunks)
  long long carry = 0;
  for (int base = 0; base < p.B; base += nthr) {
    const int b = base + t;
    const long long u = b < p.B ? unit_len(req_ctx(p, b, false)) * per_req : 0;
    long long inc = u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    __syncthreads();  // warp_sum of the previous chunk is read
    if (lane == 31) sb.warp_sum[warp] = inc;
    __syncthreads();
    long long wb = carry;
    for (int w = 0; w < warp; ++w) wb += sb.warp_sum[w];
    const long long excl = wb + inc - u;
    if (b < p.B && excl <= x0 && x0 < excl + u) {
      sb.b = b;
      sb.off = excl;
    }
    if (b < p.B && excl <= x1 && x1 < excl + u) {
      sb.b_last = b;
      sb.off_last = excl;
    }
    for (int w = 0; w < nw; ++w) carry += sb.warp_sum[w];
  }
  __syncthreads();
  return sb.b >= 0 && sb.b_last >= 0;
}

// One segment: the part [u0, u1) of a unit's L key blocks that lies in the
// CTA's range (block L - 1 is the tree block).
struct Seg {
  int b, kvh, cq, ctx, L, u0, u1;
};
// Walks the CTA's range segment by segment; every role runs its own copy over
// the same range, so all roles see the same sequence.
struct SegWalk {
  long long pos, hi, off;
  int b, ctx, L, kvh;
  __device__ void init(const Params& p, const Bars& sb) {
    kvh = (int)(blockIdx.x % p.Hkv);
    pos = sb.lo;
    hi = sb.hi;
    off = sb.off;
    b = sb.b;
    ctx = req_ctx(p, b, false);
    L = unit_len(ctx);
  }
  __device__ bool next(const Params& p, Seg& s) {
    while (pos < hi) {
      const long long U = (long long)L * p.ncq;
      if (pos >= off + U) {
        off += U;
        ++b;
        ctx = req_ctx(p, b, false);
        L = unit_len(ctx);
        continue;
      }
      const long long r = pos - off;
      const int unit = (int)(r / L);
      s.b = b;
      s.kvh = kvh;
      s.cq = unit;
      s.ctx = ctx;
      s.L = L;
      s.u0 = (int)(r % L);
      const long long left = hi - pos;
      s.u1 = (int)((long long)(L - s.u0) < left ? L : s.u0 + left);
      pos += s.u1 - s.u0;
      return true;
    }
    return false;
  }
};
}  // namespace tc

// COPIES = 2 (one query tile of at most 64 rows): the tile's rows are loaded
// twice, at TMEM lanes 0.. and 64.., so one S MMA gives each row's scores
// twice; the first copy takes keys 0-31 of every block and the second keys
// 32-63 (each writes zeros into its P row for the other half), each with its
// own m, l and O rows, and the copies are merged at the end of a segment.
// Each softmax warp thus handles half the keys of a block, and the four warps
// of the tile (four sub-partitions) all have rows.
template <int D, int TPC, int COPIES>
__global__ void __launch_bounds__(128 + 128 * TPC, 1)
    tree_attn_stream_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_kt,
                        const __grid_constant__ CUtensorMap map_vt, const tc::Params p) {
  using namespace tc;
  static_assert(COPIES == 1 || (COPIES == 2 && TPC == 1), "two copies of a single query tile");
  constexpr int NH = D / 64;                         // 128-byte column halves of a row
  constexpr uint32_t kTileQ = 128u * 128u * NH;      // 128 rows x D
  constexpr uint32_t kTileKV = (uint32_t)kBlk * 128u * NH;
  constexpr uint32_t kTileP = 128u * kBlk * 2u;      // 128 rows x 64 keys
  constexpr int kSt = kv_stages<D>(TPC);
  // TMEM columns: S of tile t, buffer x at t * 2 kBlk + x kBlk; O of tile t at
  // tpc * 2 kBlk + t D
  constexpr uint32_t kColO = (uint32_t)(TPC * 2 * kBlk);
  constexpr uint32_t tmem_cols = TPC == 2 ? 512u : 256u;
  __shared__ Bars sb;
  extern __shared__ unsigned char dsm[];
  const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
  // P of tile t, buffer x at sP + (2 t + x) kTileP
  const uint32_t sQ = base, sK = sQ + TPC * kTileQ, sV = sK + kSt * kTileKV,
                 sP = sV + kSt * kTileKV;
  unsigned char* gbase = dsm + (base - smem_u32(dsm));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &sb.abort_flag;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    sb.stop = 0;
    mbar_init(smem_u32(&sb.q_full), 1);
    mbar_init(smem_u32(&sb.q_empty), 1);
    for (int x = 0; x < kSt; ++x) {
      mbar_init(smem_u32(&sb.k_full[x]), 1);
      mbar_init(smem_u32(&sb.v_full[x]), 1);
      mbar_init(smem_u32(&sb.k_empty[x]), 1);
      mbar_init(smem_u32(&sb.kv_empty[x]), 1);
    }
    // every softmax warp arrives, also those of a tile a segment leaves empty
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sb.s_full[x]), 1);
      mbar_init(smem_u32(&sb.s_empty[x]), 4 * TPC);
      mbar_init(smem_u32(&sb.p_full[x]), 4 * TPC);
    }
    mbar_init(smem_u32(&sb.drain), 1);
    mbar_init(smem_u32(&sb.drain_pv), 1);
    sb.abort_flag = 0;
    fence_mbar_init();
  }
  pdl_wait();  // the previous grid (its ctx_lens, and its TMEM) is complete from here on
  if (warp == 1) {
    tmem_alloc(smem_u32(&sb.tmem_base), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool has_work = plan_range(p, (int)(blockIdx.x / p.Hkv), sb);
  pdl_trigger();
  if (threadIdx.x == 0) {
    // merge descriptor of this CTA's column: the unit its range ends in, when
    // that unit starts inside the range and goes on past it
    int4 md = make_int4(-1, 0, 0, 0);
    if (has_work) {
      const int L = unit_len(req_ctx(p, sb.b_last, false));
      const int unit = (int)((sb.hi - 1 - sb.off_last) / L);
      const long long ps = sb.off_last + (long long)unit * L, pe = ps + L;
      if (pe > sb.hi && ps >= sb.lo) {
        const int g_last = share_owner(pe - 1, sb.tot, sb.n_groups);
        md = make_int4(sb.b_last, unit, g_last - (int)(blockIdx.x / p.Hkv) + 1, ps > sb.lo ? 1 : 0);
      }
    }
    p.merge[blockIdx.x] = md;
  }
  const uint32_t tmem = sb.tmem_base;
  const int rows_tile = p.nr * p.G, rows_total = p.R * p.G;

  if (!has_work) {
    // nothing to run: fall through to the teardown
  } else if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers
    // warp 0: the K blocks, a K stage released as soon as S of its block is
    // complete; warp 2: the V blocks, a V stage released after P V.  The K
    // loads thus run ahead of the V loads by the softmax of a block.  Q is
    // loaded by the S issuer, so neither producer stops at a segment's end.
    const bool kload = warp == 0;
    const uint64_t pol_kv = l2_policy_evict_normal();  // other units of the request re-read it
    const uint64_t pol_tree = l2_policy_evict_first();
    const uint32_t oob_row = (uint32_t)p.num_pages * 16u;  // a row past the pool: reads zeros
    constexpr int kGrp = 32 / (kBlk / 16);  // blocks per group of 32 page ids
    SegWalk wk;
    wk.init(p, sb);
    Seg sg;
    bool ok = true;
    int st = 0;
    uint32_t ph = 0;
    long long issued = 0;
    while (ok && wk.next(p, sg)) {
      const int nctx = sg.L - 1;  // prefix blocks of the unit
      // page ids, 32 at a time (8 blocks of 4 pages) from block u0: lane q
      // holds page slot q of the group; the next group is loaded one ahead
      auto page_group = [&](int g) -> int {
        const int blk = sg.u0 + g * kGrp + lane / (kBlk / 16);
        const int key0 = blk * kBlk + (lane % (kBlk / 16)) * 16;
        if (blk >= min(sg.u1, nctx) || key0 >= sg.ctx) return -1;
        const int pg = p.block_table[(size_t)sg.b * p.max_pages + key0 / 16];
        if (pg < 0 || pg >= p.num_pages) {
          set_status(p.status, EAGLE_ERR_BAD_KV);
          return -1;
        }
        return pg;
      };
      const int nblk = sg.u1 - sg.u0;
      int pg_cur = page_group(0), pg_next = kGrp < nblk ? page_group(1) : -1;
      for (int i = 0; i < nblk; ++i) {
        const int u = sg.u0 + i;
        if (i > 0 && i % kGrp == 0) {
          pg_cur = pg_next;
          pg_next = i + kGrp < nblk ? page_group(i / kGrp + 1) : -1;
        }
        if (lane == 0)
          ok = mbar_wait(smem_u32(kload ? &sb.k_empty[st] : &sb.kv_empty[st]), ph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const uint32_t dst = (kload ? sK : sV) + st * kTileKV;
        const uint32_t fb = smem_u32(kload ? &sb.k_full[st] : &sb.v_full[st]);
        if (u < nctx) {
          int rows[kBlk / 16];
#pragma unroll
          for (int q = 0; q < kBlk / 16; ++q) {
            const int pq = __shfl_sync(0xffffffffu, pg_cur, (i % kGrp) * (kBlk / 16) + q);
            rows[q] = pq >= 0 ? pq * 16 : (int)oob_row;
          }
          if (lane == 0) {
            const CUtensorMap* map = kload ? &map_k : &map_v;
            mbar_arrive_expect_tx(fb, kTileKV);
#pragma unroll
            for (int q = 0; q < kBlk / 16; ++q)
#pragma unroll
              for (int h = 0; h < NH; ++h)
                tma_load_3d(dst + h * kBlkBytesHalf + q * 2048u, map, fb, h * 64, sg.kvh, rows[q], pol_kv);
          }
        } else if (lane == 0) {  // the tree block: rows of this request's tree K / V
          const uint32_t bytes = (uint32_t)NH * p.tr * 128u;
          const CUtensorMap* map = kload ? &map_kt : &map_vt;
          mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tma_load_3d(dst + h * kBlkBytesHalf, map, fb, h * 64, sg.kvh, sg.b * p.R, pol_tree);
        }
        if (++st == kSt) {
          st = 0;
          ph ^= 1u;
        }
        ++issued;
      }
    }
    if (!ok && lane == 0) {
      // wait (bounded) for the copies already issued into each stage
      for (long long j = issued > kSt ? issued - kSt : 0; j < issued; ++j) {
        const uint32_t ph2 = (uint32_t)(j / kSt) & 1u;
        const uint32_t bar = smem_u32(kload ? &sb.k_full[j % kSt] : &sb.v_full[j % kSt]);
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, ph2) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ S issuer
    SegWalk wk;
    wk.init(p, sb);
    Seg sg;
    bool ok = true;
    long long j = 0;
    int nq = 0, q_issued = 0;
    const uint64_t dq0 = smem_desc_sw128(sQ);
    const uint64_t pol_q = l2_policy_evict_first();
    while (ok && wk.next(p, sg)) {
      const int nt = min(TPC, p.qtiles - TPC * sg.cq);
      if (lane == 0) {
        // the Q tile is free once S of the previous segment's last block is
        // complete (this thread's own commit)
        if (nq > 0) ok = mbar_wait(smem_u32(&sb.q_empty), (uint32_t)(nq - 1) & 1u, abort_flag);
        if (ok) {
          const uint32_t box_rows = (uint32_t)(p.q_box_rows * p.G);
          mbar_arrive_expect_tx(smem_u32(&sb.q_full), (uint32_t)(nt * NH * COPIES) * box_rows * 128u);
          for (int t = 0; t < nt; ++t)
#pragma unroll
            for (int c = 0; c < COPIES; ++c)
#pragma unroll
              for (int h = 0; h < NH; ++h)
                tma_load_3d(sQ + t * kTileQ + h * 16384u + (uint32_t)c * (128u / COPIES) * 128u, &map_q,
                            smem_u32(&sb.q_full), h * 64, sg.kvh * p.G, sg.b * p.R + (TPC * sg.cq + t) * p.nr,
                            pol_q);
          q_issued = nq + 1;
          ok = mbar_wait(smem_u32(&sb.q_full), (uint32_t)nq & 1u, abort_flag);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      ++nq;
      for (int u = sg.u0; u < sg.u1; ++u, ++j) {
        // S(j) = Q_t K_j^T for each query tile t into S buffer j & 1
        const int x = (int)(j & 1), st = (int)(j % kSt);
        const uint32_t sph = (uint32_t)(j >> 1) & 1u, kph = (uint32_t)(j / kSt) & 1u;
        if (lane == 0)
          ok = mbar_wait(smem_u32(&sb.k_full[st]), kph, abort_flag) &&
               mbar_wait(smem_u32(&sb.s_empty[x]), sph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        tc_fence_after();
        const int n = u < sg.L - 1 ? kBlk : p.tr;
        const uint32_t idesc = mma_idesc(1, 128, n);
        if (lane == 0) {
          // The MMA thread shares its issue slots with a busy softmax warp, so
          // the loop is kept to a few instructions per MMA: base descriptors
          // once, then constant offsets in the descriptors' address field
          // (bytes >> 4): +32 bytes per 16 columns inside a 128-byte row, the
          // next 64 columns in the next half tile
          const uint64_t dk = smem_desc_sw128(sK + st * kTileKV);
          for (int t = 0; t < nt; ++t) {
            const uint64_t dq = dq0 + (uint64_t)((t * kTileQ) >> 4);
            const uint32_t dt = tmem + (uint32_t)(t * 2 * kBlk + x * kBlk);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t qoff = ((uint32_t)(k >> 2) * 16384u + (uint32_t)(k & 3) * 32u) >> 4;
              const uint32_t koff = ((uint32_t)(k >> 2) * kBlkBytesHalf + (uint32_t)(k & 3) * 32u) >> 4;
              mma_bf16(dt, dq + qoff, dk + koff, idesc, k > 0 ? 1u : 0u);
            }
          }
          mma_commit(smem_u32(&sb.s_full[x]));
          mma_commit(smem_u32(&sb.k_empty[st]));  // the K stage is free once S is complete
          if (u == sg.u1 - 1) mma_commit(smem_u32(&sb.q_empty));  // and Q after the segment's last S
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      // a Q load issued but not seen complete (abort): wait for it, bounded
      if (q_issued > nq) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&sb.q_full), (uint32_t)(q_issued - 1) & 1u) &&
               globaltimer_ns() - t0 < 100000000ull) {
        }
      }
      // drain (always: after an abort elsewhere no consumer may have waited
      // for the last S): every S MMA completes before tensor memory is freed
      mma_commit(smem_u32(&sb.drain));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&sb.drain), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ P V issuer
    // A second MMA-issuing thread: O += P V of block j goes out as soon as P
    // of block j is ready, without queuing behind the S MMAs of later blocks
    // (S(j) is complete before P(j) exists)
    SegWalk wk;
    wk.init(p, sb);
    Seg sg;
    bool ok = true;
    long long j = 0;
    const uint32_t idesc_pv = mma_idesc_bmn(1, 128, D);
    const uint64_t dp0 = smem_desc_sw128(sP);
    while (ok && wk.next(p, sg)) {
      const int nt = min(TPC, p.qtiles - TPC * sg.cq);
      for (int u = sg.u0; u < sg.u1; ++u, ++j) {
        const int x = (int)(j & 1), st = (int)(j % kSt);
        const uint32_t pph = (uint32_t)(j >> 1) & 1u, kph = (uint32_t)(j / kSt) & 1u;
        if (lane == 0) ok = mbar_wait(smem_u32(&sb.v_full[st]), kph, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // zero V rows [z0, z1) that hold no key: the unused tail of a partly
        // filled page, or the padding of the tree block
        int z0 = 0, z1 = 0, nk = kBlk;
        if (u < sg.L - 1) {
          const int valid = sg.ctx - u * kBlk;  // >= 1
          if (valid < kBlk) {
            z0 = valid;
            z1 = min(kBlk, (valid + 15) / 16 * 16);
          }
        } else {
          z0 = p.R;
          z1 = p.tr;
          nk = p.tr;
        }
        if (z0 < z1) {
          const uint32_t vd = sV + st * kTileKV;
          for (int c = lane; c < (z1 - z0) * NH * 8; c += 32) {
            const int row = z0 + c / (NH * 8), h = (c / 8) % NH, ch = c % 8;
            *reinterpret_cast<uint4*>(gbase + (vd - base) + h * kBlkBytesHalf + row * 128 + ch * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) ok = mbar_wait(smem_u32(&sb.p_full[x]), pph, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dv = smem_desc_sw128_mn(sV + st * kTileKV, kBlkBytesHalf);
          for (int t = 0; t < nt; ++t) {
            const uint64_t dp = dp0 + (uint64_t)(((2 * t + x) * kTileP) >> 4);
            const uint32_t dt = tmem + kColO + (uint32_t)(t * D);
            // 64 keys = one 128-byte row of P: +32 bytes of P and 16 rows
            // (2048 bytes) of V per MMA; a segment's first block starts O afresh
            for (int k = 0; k < nk / 16; ++k)
              mma_bf16(dt, dp + (uint32_t)k * 2u, dv + (uint32_t)k * 128u, idesc_pv,
                       (u > sg.u0 || k > 0) ? 1u : 0u);
          }
          // one commit per block for P V: its completion frees the V stage
          // and is what the softmax warps wait for before touching O
          mma_commit(smem_u32(&sb.kv_empty[st]));
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      // drain: every P V MMA completes before tensor memory is freed
      mma_commit(smem_u32(&sb.drain_pv));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&sb.drain_pv), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    constexpr int KC = kBlk / COPIES;   // keys of a block this warp's copy takes
    constexpr int LC = 128 / COPIES;    // TMEM lanes per copy
    const int tq = (warp - 4) / 4;      // query tile of this warp group
    const int q4 = warp & 3;            // TMEM lane quarter of this warp
    const int i = q4 * 32 + lane;       // TMEM lane
    const int cpy = COPIES == 1 ? 0 : (q4 * 32) / LC;  // the copy this lane belongs to
    const int il = i - cpy * LC;        // query row of the tile
    const int kc0 = cpy * KC;           // first key of a block this copy takes
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const uint32_t o_addr = tmem + lane_addr + kColO + (uint32_t)(tq * D);
    unsigned char* prow0 = gbase + (sP - base) + 2 * tq * kTileP + i * 128;
    bool ok = true;
    long long j = 0;
    int seg_i = 0;
    auto wait_pv = [&](long long jp) -> bool {  // P V of block jp complete
      bool w = true;
      // P V(jp) completes the phase jp / kSt of its stage's kv_empty barrier;
      // the next phase needs P V(jp + kSt), hence P(jp + kSt), which this
      // warp writes only after every wait on jp (jp >= j - 2, kSt >= 3), so
      // the parity is unambiguous
      if (lane == 0)
        w = mbar_wait(smem_u32(&sb.kv_empty[jp % kSt]), (uint32_t)(jp / kSt) & 1u, abort_flag);
      w = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      if (w) tc_fence_after();
      return w;
    };
    SegWalk wk;
    wk.init(p, sb);
    Seg sg;
    while (wk.next(p, sg)) {
      const int nt = min(TPC, p.qtiles - TPC * sg.cq);
      const int gi = (TPC * sg.cq + tq) * rows_tile + il;
      const bool row_ok = tq < nt && il < rows_tile && gi < rows_total;
      // a quarter with no query row keeps only the barrier protocol: its P rows
      // and O rows feed nothing that is written out
      const int tile_rows = tq < nt ? min(rows_tile, rows_total - (TPC * sg.cq + tq) * rows_tile) : 0;
      const bool quad_live = q4 * 32 - cpy * LC < tile_rows;
      const int r_i = row_ok ? gi / p.G : 0;
      const uint64_t mrow = row_ok ? p.tree_mask[(size_t)sg.b * p.R + r_i] : 0ull;
      float m = -INFINITY, l = 0.f;
      for (int u = sg.u0; ok && u < sg.u1; ++u, ++j) {
        const int x = (int)(j & 1);
        const uint32_t sph = (uint32_t)(j >> 1) & 1u;
        if (lane == 0) ok = mbar_wait(smem_u32(&sb.s_full[x]), sph, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        tc_fence_after();
        if (!quad_live) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sb.s_empty[x]));
          // p_full of block j only after P V(j - 2): the S thread runs up to
          // two blocks ahead of P V, so without this wait the arrivals of a
          // warp with no rows for block j + 2 could complete block j's phase
          // before the warps with rows have written P(j)
          if (j >= 2 && !(ok = wait_pv(j - 2))) break;
          if (lane == 0) mbar_arrive(smem_u32(&sb.p_full[x]));
          continue;
        }
        const bool tree = u == sg.L - 1;
        // visible keys of this block as a 64-bit mask, then this copy's KC
        // of them; a masked score reads as -inf through a select
        uint64_t vis;
        if (tree) {
          vis = p.R >= 64 ? mrow : (mrow & ((1ull << p.R) - 1ull));
        } else {
          const int lim = sg.ctx - u * kBlk;  // >= 1
          vis = lim >= 64 ? ~0ull : ((1ull << lim) - 1ull);
        }
        const uint64_t myvis = KC == 64 ? vis : ((vis >> kc0) & ((1ull << KC) - 1ull));
        const bool full = KC == 64 ? vis == ~0ull : myvis == ((1ull << KC) - 1ull);
        // this copy's KC scores of the row, loaded once; the S buffer is free
        // for S(j + 2) as soon as they are in registers
        const uint32_t sa = tmem + lane_addr + (uint32_t)(tq * 2 * kBlk + x * kBlk + kc0);
        uint32_t sr[KC];
#pragma unroll
        for (int c = 0; c < KC / 32; ++c) tmem_ld32_issue(sa + 32u * c, sr + 32 * c);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sb.s_empty[x]));
        // pass 1: block max of the raw scores (scale > 0 commutes with max)
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
        if (full) {
#pragma unroll
          for (int k = 0; k < KC; ++k) mx[k & 7] = fmaxf(mx[k & 7], __uint_as_float(sr[k]));
        } else {
#pragma unroll
          for (int k = 0; k < KC; ++k)
            mx[k & 7] = fmaxf(mx[k & 7], ((myvis >> k) & 1ull) ? __uint_as_float(sr[k]) : -INFINITY);
        }
        const float bm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
        // m is the reference of O and l; it moves only when a block's max
        // exceeds it by more than 2^8 (or when it is still -inf), and then O
        // and l are rescaled by 2^(m_old - m_new).  (TMEM loads and stores are
        // warp-wide: a warp rescales when any of its rows needs it, with
        // factor 1 for the others.)  The segment's first block starts O afresh.
        const bool need = bm > m + kRescaleLog2;
        const bool resc = need && m != -INFINITY && u > sg.u0;
        if (__ballot_sync(0xffffffffu, resc)) {
          // O must be stable: every earlier P V complete
          if (!(ok = wait_pv(j - 1))) break;
          const float alpha = resc ? ex2_approx(m - bm) : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32_issue(o_addr + (uint32_t)(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
            tmem_st32(o_addr + (uint32_t)(c * 32), r);
          }
          tmem_wait_st();
          l *= alpha;
        }
        if (need) m = bm;
        // pass 2: P = 2^(S * scale_log2 - m) as bf16 into the swizzled P tile
        // (zeros in the other copy's key chunks), once P V(j - 2) has read
        // this buffer (the P V thread commits it separately from the S MMAs,
        // so S(j) being complete says nothing about it)
        if (j >= 2 && !(ok = wait_pv(j - 2))) break;
        const float neg_m = m == -INFINITY ? 0.f : -m;
        unsigned char* prow = prow0 + x * kTileP;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < KC / 32; ++c) {
          const uint32_t* r = sr + c * 32;
          const uint32_t w = (uint32_t)(myvis >> (c * 32));
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float e0 = ex2_approx(fmaf(__uint_as_float(r[2 * k]), p.scale_log2, neg_m));
            float e1 = ex2_approx(fmaf(__uint_as_float(r[2 * k + 1]), p.scale_log2, neg_m));
            if (!full) {
              e0 = ((w >> (2 * k)) & 1u) ? e0 : 0.f;
              e1 = ((w >> (2 * k + 1)) & 1u) ? e1 : 0.f;
            }
            ls[k & 3] += e0 + e1;
            pk[k] = pack_bf16(e0, e1);
          }
          // 32 keys = half of the row's 128 bytes: chunks kc0 / 8 + 4 c .. + 3
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            const int ch = kc0 / 8 + c * 4 + uu;
            *reinterpret_cast<uint4*>(prow + ((ch ^ (i & 7)) << 4)) =
                make_uint4(pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]);
          }
        }
        if (COPIES == 2) {  // the other copy's keys contribute nothing to these rows
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            const int ch = (kc0 == 0 ? 4 : 0) + uu;
            *reinterpret_cast<uint4*>(prow + ((ch ^ (i & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sb.p_full[x]));
      }
      // O of the segment is final once its last P V completes
      if (ok && quad_live) ok = wait_pv(j - 1);
      const bool whole = sg.u0 == 0 && sg.u1 == sg.L;
      // a piece of a unit split between CTAs: slot 0 holds the CTA's first
      // segment, slot 1 its last (any other segment is a whole unit)
      const size_t slot = (size_t)blockIdx.x * 2 + (seg_i == 0 ? 0 : 1);
      const size_t prow_i = (slot * TPC + tq) * 128 + il;
      const int h = sg.kvh * p.G + gi % p.G;
      const size_t row = ((size_t)sg.b * p.R + r_i) * p.Hq + h;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      if (COPIES == 1) {
        if (!ok) break;
        if (quad_live) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32_issue(o_addr + (uint32_t)(c * 32), o);
            tmem_wait_ld();
            if (!row_ok) continue;
            if (whole) {
              uint4* dst = reinterpret_cast<uint4*>(p.out + row * D + c * 32);
#pragma unroll
              for (int uu = 0; uu < 4; ++uu) {
                const float* f = reinterpret_cast<const float*>(o + 8 * uu);
                dst[uu] = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                                     pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
              }
            } else {
              float4* po = reinterpret_cast<float4*>(p.part_o + prow_i * D + c * 32);
#pragma unroll
              for (int uu = 0; uu < 8; ++uu) {
                const float* f = reinterpret_cast<const float*>(o + 4 * uu);
                po[uu] = make_float4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
              }
            }
          }
          if (row_ok) {
            if (whole) {
              if (p.lse) p.lse[row] = lse;
            } else {
              p.part_lse[prow_i] = lse;
            }
          }
          // O is read out before this warp's next arrival on p_full lets the
          // next segment's first P V overwrite it
          tc_fence_before();
        }
      } else {
        // Two copies: the second copy's O / l and lse go through the P tiles
        // (every P V of the segment is complete, and no P of the next segment
        // is written before the last barrier below); the first copy merges
        // them with its own and writes the rows.  All four softmax warps pass
        // the three barriers of every segment, also after an abort, and leave
        // together on one decision.
        float* xo = reinterpret_cast<float*>(gbase + (sP - base));
        if (ok && quad_live && cpy == 1) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32_issue(o_addr + (uint32_t)(c * 32), o);
            tmem_wait_ld();
            if (!row_ok) continue;
            float4* xr = reinterpret_cast<float4*>(xo + (size_t)il * D + c * 32);
#pragma unroll
            for (int uu = 0; uu < 8; ++uu) {
              const float* f = reinterpret_cast<const float*>(o + 4 * uu);
              xr[uu] = make_float4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
            }
          }
          if (row_ok) sb.xlse[il] = lse;
        }
        tc_fence_before();
        named_bar(1, 128);
        if (threadIdx.x == 128) sb.stop = *abort_flag ? 1 : 0;
        named_bar(2, 128);
        const bool stop = *reinterpret_cast<volatile int*>(&sb.stop) != 0;
        if (!stop && quad_live && cpy == 0) {
          const float lse1 = row_ok ? sb.xlse[il] : -INFINITY;
          const float Lm = fmaxf(lse, lse1);
          const float w0 = Lm == -INFINITY || lse == -INFINITY ? 0.f : exp2f((lse - Lm) * kLog2e);
          const float w1 = Lm == -INFINITY || lse1 == -INFINITY ? 0.f : exp2f((lse1 - Lm) * kLog2e);
          const float ws = w0 + w1;
          const float iw = ws > 0.f ? 1.f / ws : 0.f;
          const float a0 = w0 * inv * iw, a1 = w1 * iw;
          lse = ws > 0.f ? Lm + logf(ws) : -INFINITY;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32_issue(o_addr + (uint32_t)(c * 32), o);
            tmem_wait_ld();
            if (!row_ok) continue;
            const float* xr = xo + (size_t)il * D + c * 32;
            float f[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) f[k] = a0 * __uint_as_float(o[k]) + (w1 > 0.f ? a1 * xr[k] : 0.f);
            if (whole) {
              uint4* dst = reinterpret_cast<uint4*>(p.out + row * D + c * 32);
#pragma unroll
              for (int uu = 0; uu < 4; ++uu)
                dst[uu] = make_uint4(pack_bf16(f[8 * uu], f[8 * uu + 1]), pack_bf16(f[8 * uu + 2], f[8 * uu + 3]),
                                     pack_bf16(f[8 * uu + 4], f[8 * uu + 5]), pack_bf16(f[8 * uu + 6], f[8 * uu + 7]));
            } else {
              float4* po = reinterpret_cast<float4*>(p.part_o + prow_i * D + c * 32);
#pragma unroll
              for (int uu = 0; uu < 8; ++uu)
                po[uu] = make_float4(f[4 * uu], f[4 * uu + 1], f[4 * uu + 2], f[4 * uu + 3]);
            }
          }
          if (row_ok) {
            if (whole) {
              if (p.lse) p.lse[row] = lse;
            } else {
              p.part_lse[prow_i] = lse;
            }
          }
        }
        tc_fence_before();
        named_bar(3, 128);  // the exchange is read before any P of the next segment
        if (stop) break;
        ok = true;
      }
      ++seg_i;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (sb.abort_flag && threadIdx.x == 0) set_status(p.status, EAGLE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// Merge of the pieces of every unit split between CTAs.  Each attention CTA
// left a descriptor for its column: the unit its range ends in when that unit
// started inside the range and goes on past it, so that each split unit is
// merged from the column of the CTA holding its first block.  The pieces are
// that CTA (slot 0 if the unit is its first segment, else slot 1) and the
// CTAs of the same head in the next groups (slot 0: their range starts inside
// the unit).  The gridDim.y CTAs of a column share the unit's rows, one warp
// per row:
//   out = sum_s w_s O_s / sum_s w_s, w_s = exp(lse_s - max lse), lse = max + log sum w.
// A row's pieces are read with independent loads: their lse across the
// lanes, their O rows four pieces at a time.
constexpr int kCombWarps = 8;
template <int D, int TPC>
__global__ void __launch_bounds__(kCombWarps * 32) tree_attn_stream_merge_kernel(const tc::Params p) {
  using namespace tc;
  pdl_wait();
  pdl_trigger();
  const int4 md = p.merge[blockIdx.x];
  if (md.x < 0) return;
  const int b = md.x, cq = md.y, np = md.z, slot0 = md.w;
  const int c0 = blockIdx.x, kvh = c0 % p.Hkv;
  const int nt = min(TPC, p.qtiles - TPC * cq);
  const int rows_tile = p.nr * p.G, rows_total = p.R * p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // piece q of a row: the CTA of this head q groups on, its slot and row
  auto prow = [&](int q, int t, int i) -> size_t {
    const size_t slot = (size_t)(c0 + q * p.Hkv) * 2 + (q == 0 ? slot0 : 0);
    return (slot * TPC + t) * 128 + i;
  };
  for (int rr = blockIdx.y * kCombWarps + warp; rr < nt * 128; rr += gridDim.y * kCombWarps) {
    const int t = rr / 128, i = rr % 128;
    const int gi = (TPC * cq + t) * rows_tile + i;
    if (i >= rows_tile || gi >= rows_total) continue;
    float Lm = -INFINITY;
    for (int q = lane; q < np; q += 32) Lm = fmaxf(Lm, p.part_lse[prow(q, t, i)]);
#pragma unroll
    for (int o = 16; o; o >>= 1) Lm = fmaxf(Lm, __shfl_xor_sync(0xffffffffu, Lm, o));
    float acc[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) acc[k] = 0.f;
    float wpart = 0.f;
    for (int q0 = 0; q0 < np; q0 += 32) {
      const int q = q0 + lane;
      const float ls = q < np ? p.part_lse[prow(q, t, i)] : -INFINITY;
      const float wq = ls == -INFINITY ? 0.f : exp2f((ls - Lm) * kLog2e);
      wpart += wq;
      const int cnt = min(32, np - q0);
      for (int k0 = 0; k0 < cnt; k0 += 4) {
        float v[4][D / 32], w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wq, (k0 + u) & 31);
          const bool on = k0 + u < cnt && w[u] > 0.f;
          const float* po = p.part_o + prow(on ? q0 + k0 + u : 0, t, i) * D;
#pragma unroll
          for (int k = 0; k < D / 32; ++k) v[u][k] = on ? po[lane + 32 * k] : 0.f;
          if (!on) w[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int k = 0; k < D / 32; ++k) acc[k] = fmaf(w[u], v[u][k], acc[k]);
      }
    }
    float wsum = wpart;
#pragma unroll
    for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int r = gi / p.G, h = kvh * p.G + gi % p.G;
    const size_t row = ((size_t)b * p.R + r) * p.Hq + h;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) p.out[row * D + lane + 32 * k] = __float2bfloat16(acc[k] * inv);
    if (p.lse && lane == 0) p.lse[row] = wsum > 0.f ? Lm + logf(wsum) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Split schedule (few key blocks per SM): one CTA per (one or two query tiles,
// KV split, request x kv head), each split's (O, lse) merged by a second kernel.
template <int D, int TPC>
__global__ void __launch_bounds__(128 + 128 * TPC, 1)
    tree_attn_split_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_kt,
                        const __grid_constant__ CUtensorMap map_vt, const tc::Params p) {
  using namespace tc;
  constexpr int NH = D / 64;                         // 128-byte column halves of a row
  constexpr uint32_t kTileQ = 128u * 128u * NH;      // 128 rows x D
  constexpr uint32_t kTileKV = (uint32_t)kBlk * 128u * NH;
  constexpr uint32_t kTileP = 128u * kBlk * 2u;      // 128 rows x 64 keys
  constexpr int kSt = kv_stages<D>(TPC);
  constexpr bool kSplitLoad = TPC == 2;  // separate K and V producers (see the producers)
  // TMEM columns: S of tile t, buffer x at t * 2 kBlk + x kBlk; O of tile t at
  // tpc * 2 kBlk + t D
  constexpr uint32_t kColO = (uint32_t)(TPC * 2 * kBlk);
  constexpr uint32_t tmem_cols = TPC == 2 ? 512u : 256u;
  __shared__ Bars sb;
  extern __shared__ unsigned char dsm[];
  const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
  // P of tile t, buffer x at sP + (2 t + x) kTileP
  const uint32_t sQ = base, sK = sQ + TPC * kTileQ, sV = sK + kSt * kTileKV,
                 sP = sV + kSt * kTileKV;
  unsigned char* gbase = dsm + (base - smem_u32(dsm));

  const int cq = blockIdx.x, split = blockIdx.y;
  const int b = blockIdx.z / p.Hkv, kvh = blockIdx.z % p.Hkv;
  const int nt = min(TPC, p.qtiles - TPC * cq);  // query tiles of this CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &sb.abort_flag;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    mbar_init(smem_u32(&sb.q_full), 1);
    for (int x = 0; x < kSt; ++x) {
      mbar_init(smem_u32(&sb.k_full[x]), 1);
      mbar_init(smem_u32(&sb.v_full[x]), 1);
      mbar_init(smem_u32(&sb.k_empty[x]), 1);
      mbar_init(smem_u32(&sb.kv_empty[x]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sb.s_full[x]), 1);
      mbar_init(smem_u32(&sb.s_empty[x]), 4 * nt);
      mbar_init(smem_u32(&sb.p_full[x]), 4 * nt);
    }
    mbar_init(smem_u32(&sb.drain), 1);
    mbar_init(smem_u32(&sb.drain_pv), 1);
    sb.abort_flag = 0;
    fence_mbar_init();
  }
  pdl_wait();  // the previous grid (and its TMEM) is gone from here on
  if (warp == 1) {
    tmem_alloc(smem_u32(&sb.tmem_base), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = sb.tmem_base;

  // this CTA's key blocks: [blk_lo, blk_hi) of the prefix, then the tree block
  int ctx = p.ctx_lens[b];
  if (ctx < 0 || ctx > p.max_pages * 16) {
    if (threadIdx.x == 0) set_status(p.status, EAGLE_ERR_BAD_KV);
    ctx = ctx < 0 ? 0 : p.max_pages * 16;
  }
  const int nblk = (ctx + kBlk - 1) / kBlk;
  const int bps = (nblk + p.splits - 1) / p.splits;
  const int blk_lo = min(nblk, split * bps), blk_hi = min(nblk, blk_lo + bps);
  const int n_ctx = blk_hi - blk_lo;
  const int n_iter = n_ctx + (split == 0 ? 1 : 0);
  const int rows_tile = p.nr * p.G, rows_total = p.R * p.G;

  if (warp == 2 || (kSplitLoad && warp == 0)) {
    // ------------------------------------------------------------ producers
    // With two query tiles (a 3-stage ring) warp 0 loads Q and the K blocks
    // and warp 2 the V blocks: a K stage is released as soon as S of its
    // block is complete, a V stage only after P V, so the K loads run ahead
    // of the V loads by the softmax of a block.  With one tile (5 stages)
    // warp 2 loads everything and a stage is released after P V.
    const bool kload = !kSplitLoad || warp == 0, vload = !kSplitLoad || warp == 2;
    const uint64_t pol_kv = l2_policy_evict_normal();  // other CTAs of the request re-read it
    const uint64_t pol_q = l2_policy_evict_first();
    const uint32_t oob_row = (uint32_t)p.num_pages * 16u;  // a row past the pool: reads zeros
    // page ids, 32 at a time (8 blocks of 4 pages): lane q holds page slot
    // q of the group; the next group is loaded one group ahead
    constexpr int kGrp = 32 / (kBlk / 16);  // blocks per group of 32 page ids
    auto page_group = [&](int g) -> int {
      const int key0 = (blk_lo + g * kGrp) * kBlk + lane * 16;
      if (g * kGrp + lane / (kBlk / 16) >= n_ctx || key0 >= ctx) return -1;
      const int pg = p.block_table[(size_t)b * p.max_pages + key0 / 16];
      if (pg < 0 || pg >= p.num_pages) {
        set_status(p.status, EAGLE_ERR_BAD_KV);
        return -1;
      }
      return pg;
    };
    int issued = 0;
    if (kload && lane == 0 && n_iter > 0) {
      mbar_arrive_expect_tx(smem_u32(&sb.q_full), (uint32_t)(nt * NH * rows_tile) * 128u);
      for (int t = 0; t < nt; ++t)
#pragma unroll
        for (int h = 0; h < NH; ++h)
          tma_load_3d(sQ + t * kTileQ + h * 16384u, &map_q, smem_u32(&sb.q_full), h * 64,
                      kvh * p.G, b * p.R + (TPC * cq + t) * p.nr, pol_q);
    }
    int pg_cur = page_group(0), pg_next = kGrp < n_ctx ? page_group(1) : -1;
    bool ok = true;
    int st = 0;
    uint32_t ph = 0;
    for (int j = 0; j < n_iter && ok; ++j) {
      if (j > 0 && j % kGrp == 0) {
        pg_cur = pg_next;
        pg_next = j + kGrp < n_ctx ? page_group(j / kGrp + 1) : -1;
      }
      if (lane == 0)
        ok = mbar_wait(smem_u32(vload ? &sb.kv_empty[st] : &sb.k_empty[st]), ph ^ 1u, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const uint32_t kd = sK + st * kTileKV, vd = sV + st * kTileKV;
      const uint32_t kf = smem_u32(&sb.k_full[st]), vf = smem_u32(&sb.v_full[st]);
      if (j < n_ctx) {
        int rows[kBlk / 16];
#pragma unroll
        for (int q = 0; q < kBlk / 16; ++q) {
          const int pq = __shfl_sync(0xffffffffu, pg_cur, (j % kGrp) * (kBlk / 16) + q);
          rows[q] = pq >= 0 ? pq * 16 : (int)oob_row;
        }
        if (lane == 0) {
#pragma unroll
          for (int o = 0; o < 2; ++o) {
            if (!(o == 0 ? kload : vload)) continue;
            const uint32_t dst = o == 0 ? kd : vd, fb = o == 0 ? kf : vf;
            const CUtensorMap* map = o == 0 ? &map_k : &map_v;
            mbar_arrive_expect_tx(fb, kTileKV);
#pragma unroll
            for (int q = 0; q < kBlk / 16; ++q)
#pragma unroll
              for (int h = 0; h < NH; ++h)
                tma_load_3d(dst + h * kBlkBytesHalf + q * 2048u, map, fb, h * 64, kvh, rows[q], pol_kv);
          }
        }
      } else if (lane == 0) {  // the tree block: rows of this request's tree K / V
        const uint32_t bytes = (uint32_t)NH * p.tr * 128u;
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          if (!(o == 0 ? kload : vload)) continue;
          const uint32_t dst = o == 0 ? kd : vd, fb = o == 0 ? kf : vf;
          const CUtensorMap* map = o == 0 ? &map_kt : &map_vt;
          mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tma_load_3d(dst + h * kBlkBytesHalf, map, fb, h * 64, kvh, b * p.R, pol_q);
        }
      }
      if (++st == kSt) {
        st = 0;
        ph ^= 1u;
      }
      issued = j + 1;
    }
    if (!ok && lane == 0) {
      // wait (bounded) for the copies already issued into each stage
      for (int j = max(0, issued - kSt); j < issued; ++j) {
        const uint32_t ph2 = (uint32_t)(j / kSt) & 1u;
        const unsigned long long t0 = globaltimer_ns();
        while (!((!kload || mbar_try_wait(smem_u32(&sb.k_full[j % kSt]), ph2)) &&
                 (!vload || mbar_try_wait(smem_u32(&sb.v_full[j % kSt]), ph2))) &&
               globaltimer_ns() - t0 < 100000000ull) {
        }
      }
      if (kload && n_iter > 0 && !mbar_try_wait(smem_u32(&sb.q_full), 0)) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&sb.q_full), 0) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ S issuer
    bool ok = true;
    if (n_iter > 0) {
      if (lane == 0) ok = mbar_wait(smem_u32(&sb.q_full), 0, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    const uint64_t dq0 = smem_desc_sw128(sQ);
    // S(j) = Q_t K_j^T for each query tile t into S buffer j & 1
    auto issue_s = [&](int j) -> bool {
      const int x = j & 1, st = j % kSt;  // kSt is a compile-time constant
      const uint32_t ph = (uint32_t)(j >> 1) & 1u, kph = (uint32_t)(j / kSt) & 1u;
      bool w = true;
      if (lane == 0)
        w = mbar_wait(smem_u32(&sb.k_full[st]), kph, abort_flag) &&
            mbar_wait(smem_u32(&sb.s_empty[x]), ph ^ 1u, abort_flag);
      w = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      if (!w) return false;
      tc_fence_after();
      const int n = j < n_ctx ? kBlk : p.tr;
      const uint32_t idesc = mma_idesc(1, 128, n);
      if (lane == 0) {
        // The MMA thread shares its issue slots with a busy softmax warp, so
        // the loop is kept to a few instructions per MMA: base descriptors
        // once, then constant offsets in the descriptors' address field
        // (bytes >> 4): +32 bytes per 16 columns inside a 128-byte row, the
        // next 64 columns in the next half tile
        const uint64_t dk = smem_desc_sw128(sK + st * kTileKV);
        for (int t = 0; t < nt; ++t) {
          const uint64_t dq = dq0 + (uint64_t)((t * kTileQ) >> 4);
          const uint32_t dt = tmem + (uint32_t)(t * 2 * kBlk + x * kBlk);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t qoff = ((uint32_t)(k >> 2) * 16384u + (uint32_t)(k & 3) * 32u) >> 4;
            const uint32_t koff = ((uint32_t)(k >> 2) * kBlkBytesHalf + (uint32_t)(k & 3) * 32u) >> 4;
            mma_bf16(dt, dq + qoff, dk + koff, idesc, k > 0 ? 1u : 0u);
          }
        }
        mma_commit(smem_u32(&sb.s_full[x]));
        if (kSplitLoad) mma_commit(smem_u32(&sb.k_empty[st]));  // the K stage is free once S is complete
      }
      __syncwarp();
      return true;
    };
    for (int j = 0; ok && j < n_iter; ++j) ok = issue_s(j);
    if (lane == 0) {
      // drain (always: after an abort elsewhere no consumer may have waited
      // for the last S): every S MMA completes before tensor memory is freed
      mma_commit(smem_u32(&sb.drain));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&sb.drain), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ P V issuer
    // A second MMA-issuing thread: O += P V of block j goes out as soon as P
    // of block j is ready, without queuing behind the S MMAs of later blocks
    // (S(j) is complete before P(j) exists, so the K/V stage that P V's
    // commit frees holds nothing an S MMA still reads)
    bool ok = true;
    const uint32_t idesc_pv = mma_idesc_bmn(1, 128, D);
    const uint64_t dp0 = smem_desc_sw128(sP);
    for (int j = 0; ok && j < n_iter; ++j) {
      const int x = j & 1, st = j % kSt;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u, kph = (uint32_t)(j / kSt) & 1u;
      if (lane == 0) ok = mbar_wait(smem_u32(&sb.v_full[st]), kph, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      // zero V rows [z0, z1) that hold no key: the unused tail of a partly
      // filled page, or the padding of the tree block
      int z0 = 0, z1 = 0, nk = kBlk;
      if (j < n_ctx) {
        const int valid = ctx - (blk_lo + j) * kBlk;
        if (valid < kBlk) {
          z0 = valid;
          z1 = min(kBlk, (valid + 15) / 16 * 16);
        }
      } else {
        z0 = p.R;
        z1 = p.tr;
        nk = p.tr;
      }
      if (z0 < z1) {
        const uint32_t vd = sV + st * kTileKV;
        for (int c = lane; c < (z1 - z0) * NH * 8; c += 32) {
          const int row = z0 + c / (NH * 8), h = (c / 8) % NH, ch = c % 8;
          *reinterpret_cast<uint4*>(gbase + (vd - base) + h * kBlkBytesHalf + row * 128 + ch * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) ok = mbar_wait(smem_u32(&sb.p_full[x]), ph, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t dv = smem_desc_sw128_mn(sV + st * kTileKV, kBlkBytesHalf);
        for (int t = 0; t < nt; ++t) {
          const uint64_t dp = dp0 + (uint64_t)(((2 * t + x) * kTileP) >> 4);
          const uint32_t dt = tmem + kColO + (uint32_t)(t * D);
          // 64 keys = one 128-byte row of P: +32 bytes of P and 16 rows
          // (2048 bytes) of V per MMA
          for (int k = 0; k < nk / 16; ++k)
            mma_bf16(dt, dp + (uint32_t)k * 2u, dv + (uint32_t)k * 128u, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
        }
        // one commit per block for P V: its completion frees the K/V stage
        // and is what the softmax warps wait for before touching O
        mma_commit(smem_u32(&sb.kv_empty[st]));
      }
      __syncwarp();
    }
    if (lane == 0) {
      // drain: every P V MMA completes before tensor memory is freed
      mma_commit(smem_u32(&sb.drain_pv));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&sb.drain_pv), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp >= 4 && (warp - 4) / 4 < nt) {
    // ------------------------------------------------------------ softmax
    const int tq = (warp - 4) / 4;      // query tile of this warp group
    const int q4 = warp & 3;            // TMEM lane quarter of this warp
    const int i = q4 * 32 + lane;       // query row of the tile = TMEM lane
    const int gi = (TPC * cq + tq) * rows_tile + i;
    const bool row_ok = i < rows_tile && gi < rows_total;
    // a quarter with no query row keeps only the barrier protocol: its P rows
    // and O rows feed nothing that is written out
    const int tile_rows = min(rows_tile, rows_total - (TPC * cq + tq) * rows_tile);
    const bool quad_live = q4 * 32 < tile_rows;
    const int r_i = row_ok ? gi / p.G : 0;
    const uint64_t mrow = row_ok ? p.tree_mask[(size_t)b * p.R + r_i] : 0ull;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const uint32_t o_addr = tmem + lane_addr + kColO + (uint32_t)(tq * D);
    unsigned char* prow0 = gbase + (sP - base) + 2 * tq * kTileP + i * 128;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    auto wait_pv = [&](int jp) -> bool {  // P V of block jp complete
      bool w = true;
      // P V(jp) completes the phase jp / kSt of its stage's kv_empty barrier;
      // the next phase needs P V(jp + kSt), hence P(jp + kSt), which this
      // warp writes only after every wait on jp (jp >= j - 2, kSt >= 3), so
      // the parity is unambiguous
      if (lane == 0)
        w = mbar_wait(smem_u32(&sb.kv_empty[jp % kSt]), (uint32_t)(jp / kSt) & 1u, abort_flag);
      w = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
      if (w) tc_fence_after();
      return w;
    };
    for (int j = 0; j < n_iter; ++j) {
      const int x = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (lane == 0) ok = mbar_wait(smem_u32(&sb.s_full[x]), ph, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      if (!quad_live) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sb.s_empty[x]));
        // p_full of block j only after P V(j - 2): the S thread runs up to
        // two blocks ahead of P V, so without this wait the arrivals of a
        // warp with no rows for block j + 2 could complete block j's phase
        // before the warps with rows have written P(j)
        if (j >= 2 && !(ok = wait_pv(j - 2))) break;
        if (lane == 0) mbar_arrive(smem_u32(&sb.p_full[x]));
        continue;
      }
      const bool tree = j >= n_ctx;
      const int kb = (blk_lo + j) * kBlk;
      // visible keys of this block as a 64-bit mask (all set for a full
      // prefix block); a masked score reads as -inf through a select
      uint64_t vis;
      bool full = false;
      if (tree) {
        vis = p.R >= 64 ? mrow : (mrow & ((1ull << p.R) - 1ull));
      } else {
        const int lim = ctx - kb;  // >= 1
        full = lim >= kBlk;
        vis = lim >= 64 ? ~0ull : ((1ull << lim) - 1ull);
      }
      // the block's 64 scores of this row, loaded once; the S buffer is free
      // for S(j + 2) as soon as they are in registers
      const uint32_t sa = tmem + lane_addr + (uint32_t)(tq * 2 * kBlk + x * kBlk);
      uint32_t sr[kBlk];
      tmem_ld32_issue(sa, sr);
      tmem_ld32_issue(sa + 32u, sr + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sb.s_empty[x]));
      // pass 1: block max of the raw scores (scale > 0 commutes with max)
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
      if (full) {
#pragma unroll
        for (int k = 0; k < kBlk; ++k) mx[k & 7] = fmaxf(mx[k & 7], __uint_as_float(sr[k]));
      } else {
#pragma unroll
        for (int k = 0; k < kBlk; ++k)
          mx[k & 7] = fmaxf(mx[k & 7], ((vis >> k) & 1ull) ? __uint_as_float(sr[k]) : -INFINITY);
      }
      const float bm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
      // m is the reference of O and l; it moves only when a block's max
      // exceeds it by more than 2^8 (or when it is still -inf), and then O
      // and l are rescaled by 2^(m_old - m_new).  (TMEM loads and stores are
      // warp-wide: a warp rescales when any of its rows needs it, with
      // factor 1 for the others.)
      const bool need = bm > m + kRescaleLog2;
      const bool resc = need && m != -INFINITY && j > 0;
      if (__ballot_sync(0xffffffffu, resc)) {
        // O must be stable: every earlier P V complete
        if (!(ok = wait_pv(j - 1))) break;
        const float alpha = resc ? ex2_approx(m - bm) : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_issue(o_addr + (uint32_t)(c * 32), r);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
          tmem_st32(o_addr + (uint32_t)(c * 32), r);
        }
        tmem_wait_st();
        l *= alpha;
      }
      if (need) m = bm;
      // pass 2: P = 2^(S * scale_log2 - m) as bf16 into the swizzled P tile,
      // once P V(j - 2) has read this buffer (the P V thread commits it
      // separately from the S MMAs, so S(j) being complete says nothing
      // about it)
      if (j >= 2 && !(ok = wait_pv(j - 2))) break;
      const float neg_m = m == -INFINITY ? 0.f : -m;
      unsigned char* prow = prow0 + x * kTileP;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kBlk / 32; ++c) {
        const uint32_t* r = sr + c * 32;
        const uint32_t w = (uint32_t)(vis >> (c * 32));
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float e0 = ex2_approx(fmaf(__uint_as_float(r[2 * k]), p.scale_log2, neg_m));
          float e1 = ex2_approx(fmaf(__uint_as_float(r[2 * k + 1]), p.scale_log2, neg_m));
          if (!full) {
            e0 = ((w >> (2 * k)) & 1u) ? e0 : 0.f;
            e1 = ((w >> (2 * k + 1)) & 1u) ? e1 : 0.f;
          }
          ls[k & 3] += e0 + e1;
          pk[k] = pack_bf16(e0, e1);
        }
        // 32 keys = half of the row's 128 bytes: chunks 4 c .. 4 c + 3
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ch = c * 4 + u;
          *reinterpret_cast<uint4*>(prow + ((ch ^ (i & 7)) << 4)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sb.p_full[x]));
    }
    // O is final once the last P V completes
    if (ok && quad_live && n_iter > 0) ok = wait_pv(n_iter - 1);
    if (ok && quad_live) {
      const int r = r_i, h = kvh * p.G + gi % p.G;
      const size_t row = ((size_t)b * p.R + r) * p.Hq + h;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (n_iter > 0) {
          tmem_ld32_issue(o_addr + (uint32_t)(c * 32), o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        if (!row_ok) continue;
        if (p.splits == 1) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + row * D + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float* f = reinterpret_cast<const float*>(o + 8 * u);
            dst[u] = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                                pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
          }
        } else {
          float4* po = reinterpret_cast<float4*>(p.part_o + (row * p.splits + split) * D + c * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float* f = reinterpret_cast<const float*>(o + 4 * u);
            po[u] = make_float4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
          }
        }
      }
      if (row_ok) {
        if (p.splits == 1) {
          if (p.lse) p.lse[row] = lse;
        } else {
          p.part_lse[row * p.splits + split] = lse;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (sb.abort_flag && threadIdx.x == 0) set_status(p.status, EAGLE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// Merge of the split schedule's partials: out = sum_s exp(lse_s - L) O_s,
// L = log sum_s exp(lse_s).
template <int D>
__global__ void __launch_bounds__(256) tree_attn_split_combine_kernel(const float* __restrict__ part_o,
                                                                const float* __restrict__ part_lse,
                                                                int nrows, int splits,
                                                                __nv_bfloat16* __restrict__ out,
                                                                float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= nrows) return;
  const float* pl = part_lse + (size_t)row * splits;
  // the splits' lse across the lanes (one load each, a warp max), then the O
  // rows four splits at a time with every load issued before the first is
  // used; the sums run in split order
  float L = -INFINITY;
  for (int s0 = 0; s0 < splits; s0 += 32) L = fmaxf(L, s0 + lane < splits ? pl[s0 + lane] : -INFINITY);
#pragma unroll
  for (int o = 16; o; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, o));
  float acc[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j) acc[j] = 0.f;
  float wsum = 0.f;
  constexpr int kS = 4;
  for (int s0 = 0; s0 < splits; s0 += kS) {
    float ls[kS], ov[kS][D / 32];
#pragma unroll
    for (int u = 0; u < kS; ++u) {
      const int s = s0 + u;
      ls[u] = s < splits ? pl[s] : -INFINITY;
      const float* po = part_o + ((size_t)row * splits + (s < splits ? s : 0)) * D;
#pragma unroll
      for (int j = 0; j < D / 32; ++j) ov[u][j] = s < splits ? po[lane + 32 * j] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kS; ++u) {
      if (ls[u] == -INFINITY) continue;
      const float w = exp2f((ls[u] - L) * kLog2e);
      wsum += w;
#pragma unroll
      for (int j = 0; j < D / 32; ++j) acc[j] += w * ov[u][j];
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int j = 0; j < D / 32; ++j) out[(size_t)row * D + lane + 32 * j] = __float2bfloat16(acc[j] * inv);
  if (lse && lane == 0) lse[row] = L + logf(wsum);
}

// fp32 path: one warp per (request, row, head); lanes split the head dim.
__global__ void __launch_bounds__(256) tree_attn_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k_tree, const float* __restrict__ v_tree,
    const float* __restrict__ k_cache, const float* __restrict__ v_cache,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ ctx_lens,
    const uint64_t* __restrict__ tree_mask, float* __restrict__ out, float* __restrict__ lse,
    int B, int R, int Hq, int Hkv, int D, int max_pages, int num_pages, float scale,
    int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (gw >= B * R * Hq) return;
  const int h = gw % Hq, r = (gw / Hq) % R, b = gw / (Hq * R);
  const int G = Hq / Hkv, kvh = h / G;
  const float* qp = q + (size_t)gw * D;
  float qv[4], acc[4];
  const int nd = (D + 31) / 32;
  for (int j = 0; j < 4; ++j) {
    qv[j] = (j < nd && lane + 32 * j < D) ? qp[lane + 32 * j] : 0.f;
    acc[j] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int ctx = ctx_lens[b];
  const uint64_t mask = tree_mask[(size_t)b * R + r];
  const int nkeys = ctx + R;
  for (int key = 0; key < nkeys; ++key) {
    const float *kp, *vp;
    if (key < ctx) {
      const int page = block_table[(size_t)b * max_pages + key / 16];
      if (page < 0 || page >= num_pages) {
        set_status(status, EAGLE_ERR_BAD_KV);
        continue;
      }
      const size_t off = (((size_t)page * 16 + key % 16) * Hkv + kvh) * D;
      kp = k_cache + off;
      vp = v_cache + off;
    } else {
      const int j = key - ctx;
      if (!((mask >> j) & 1ull)) continue;
      const size_t off = (((size_t)b * R + j) * Hkv + kvh) * D;
      kp = k_tree + off;
      vp = v_tree + off;
    }
    float dot = 0.f;
    for (int j = 0; j < nd; ++j)
      if (lane + 32 * j < D) dot += qv[j] * kp[lane + 32 * j];
#pragma unroll
    for (int o2 = 16; o2; o2 >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o2);
    const float sc = dot * scale;
    const float mn = fmaxf(m, sc);
    const float a = m == -INFINITY ? 0.f : expf(m - mn);
    const float w = expf(sc - mn);
    l = l * a + w;
    for (int j = 0; j < nd; ++j)
      if (lane + 32 * j < D) acc[j] = acc[j] * a + w * vp[lane + 32 * j];
    m = mn;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  for (int j = 0; j < nd; ++j)
    if (lane + 32 * j < D) out[(size_t)gw * D + lane + 32 * j] = acc[j] * inv;
  if (lse && lane == 0) lse[gw] = m + logf(l);
}


struct Plan {
  int nr, qtiles, tpc, ncq;
  int copies;   // stream schedule: 2 when one query tile of at most 64 rows is replicated
  bool stream;  // the persistent stream schedule (else the split schedule)
  int n_ctas;   // stream: the grid
  int splits;   // split: KV ranges per (query-tile group, request x kv head)
};

template <int D>
size_t tc_smem(int tpc) {
  return 1024 + (size_t)tpc * 128 * 128 * (D / 64) +
         2 * (size_t)tc::kv_stages<D>(tpc) * tc::kBlk * 128 * (D / 64) +
         (size_t)tpc * 2 * 128 * tc::kBlk * 2;
}

// Query tiles of nr tree rows x G heads (nr * G <= 128 MMA rows), query-tile
// groups per (request, kv head), and the schedule.  The stream schedule pays
// its set-up, its plan and a merge launch once, so it is taken when there are
// many key blocks per SM (at least 16, counted with the block table's width);
// below that the split schedule's short CTAs finish sooner.  num_splits < 0
// asks for the stream schedule, > 0 for the split schedule with that many KV
// ranges.  Auto splits: the count minimising (waves of CTAs, one per SM) x
// (64-key blocks per CTA + the tree block + 5 blocks' worth of set-up), plus
// a small charge per split for the (O, lse) partials and their merge.
Plan make_plan(int B, int R, int Hq, int Hkv, int max_pages, int num_splits) {
  Plan pl;
  const int G = Hq / Hkv;
  pl.nr = 128 / G;
  pl.qtiles = (R + pl.nr - 1) / pl.nr;
  const int max_blocks = max(1, (max_pages * 16 + tc::kBlk - 1) / tc::kBlk);
  // two query tiles share each K/V block when the prefix is long enough
  // (>= 4096 keys) that the blocks, not the tiles, are the work to spread
  pl.tpc = (pl.qtiles >= 2 && max_blocks >= 64) ? 2 : 1;
  pl.ncq = (pl.qtiles + pl.tpc - 1) / pl.tpc;
  const int sms = max(1, sm_count());
  const long long work = (long long)B * Hkv * pl.ncq * (max_blocks + 1);
  pl.stream = num_splits < 0 || (num_splits == 0 && work >= 16LL * sms);
  pl.n_ctas = 0;
  pl.splits = 1;
  // a single query tile whose rows fit in 64 TMEM lanes is loaded twice so
  // that each softmax warp takes half the keys of a block
  pl.copies = (pl.stream && pl.qtiles == 1 && pl.tpc == 1 && R <= 64 / G) ? 2 : 1;
  if (pl.stream) {
    // groups of Hkv CTAs (one per kv head), as many as fit on the SMs
    const long long groups = min((long long)max(1, sms / Hkv), 65535LL / Hkv);
    pl.n_ctas = (int)(groups * Hkv);
  } else if (num_splits > 0) {
    pl.splits = min(num_splits, max_blocks);
  } else {
    const long long base = (long long)pl.ncq * B * Hkv;
    double best = 1e300;
    for (int sp = 1; sp <= min(max_blocks, 256); ++sp) {
      const long long waves = (base * sp + sms - 1) / sms;
      const int bps = (max_blocks + sp - 1) / sp;
      const double cost = (double)waves * (bps + 6) * pl.tpc + (sp > 1 ? 0.1 * sp : 0.0);
      if (cost < best - 1e-9) {
        best = cost;
        pl.splits = sp;
      }
    }
  }
  return pl;
}

size_t ws_bytes_for(const Plan& pl, int B, int R, int Hq, int D) {
  if (pl.stream) {
    const size_t slots = (size_t)pl.n_ctas * 2 * pl.tpc * 128;  // rows of the pieces' slots
    return round_up(slots * D * 4, 256) + round_up(slots * 4, 256) + round_up((size_t)pl.n_ctas * 16, 256) +
           512;
  }
  if (pl.splits == 1) return 0;
  const size_t rows = (size_t)B * R * Hq;
  return round_up(rows * pl.splits * D * 4, 256) + round_up(rows * pl.splits * 4, 256) + 512;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_attn_workspace_size(int B, int R, int Hq, int Hkv, int D, int max_pages,
                                                 int page_size, int num_splits, int dtype) {
  (void)page_size;
  if (B <= 0 || R <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_pages <= 0) return 0;
  if (dtype != EAGLE_BF16 || Hq % Hkv || num_splits < -1) return 0;
  return ws_bytes_for(make_plan(B, R, Hq, Hkv, max_pages, num_splits), B, R, Hq, D);
}

extern "C" int eagle_tree_attn(const void* q, const void* k_tree, const void* v_tree,
                               const void* k_cache, const void* v_cache, int num_pages,
                               const int32_t* block_table, int max_pages, const int32_t* ctx_lens,
                               const uint64_t* tree_mask, void* out, float* lse, int B, int R,
                               int Hq, int Hkv, int D, int page_size, float scale, int num_splits,
                               int dtype, void* ws, size_t ws_bytes, int32_t* dev_status,
                               void* stream) {
  if (!q || !k_tree || !v_tree || !k_cache || !v_cache || !block_table || !ctx_lens || !tree_mask ||
      !out)
    return EAGLE_ERR_INVALID_ARG;
  if (B <= 0 || R <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_pages <= 0 || num_pages <= 0 ||
      num_splits < -1 || !(scale > 0.f) || isinf(scale))
    return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (Hq % Hkv) return EAGLE_ERR_INVALID_ARG;
  if (R > 64 || (D != 64 && D != 128) || page_size != 16 || Hq / Hkv > 16 || B * Hkv > 65535)
    return EAGLE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == EAGLE_FP32) {
    const int rows = B * R * Hq;
    launch(tree_attn_f32_kernel, (rows + 7) / 8, 256, 0, s,
        (const float*)q, (const float*)k_tree, (const float*)v_tree, (const float*)k_cache,
        (const float*)v_cache, block_table, ctx_lens, tree_mask, (float*)out, lse, B, R, Hq, Hkv, D,
        max_pages, num_pages, scale, dev_status);
    note_launch();
    return last_launch_status();
  }
  if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out))
    return EAGLE_ERR_INVALID_ARG;
  if (num_pages > (1 << 26) || (long long)B * R > (1LL << 30) || max_pages > (1 << 24))
    return EAGLE_ERR_UNSUPPORTED;
  const Plan pl = make_plan(B, R, Hq, Hkv, max_pages, num_splits);
  if (!pl.stream && pl.splits > 65535) return EAGLE_ERR_UNSUPPORTED;
  const size_t need = ws_bytes_for(pl, B, R, Hq, D);
  if (need > 0 && (!ws || ws_bytes < need)) return EAGLE_ERR_WORKSPACE;
  const int G = Hq / Hkv;
  tc::Params p;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.tree_mask = tree_mask;
  p.out = (__nv_bfloat16*)out;
  p.lse = lse;
  p.part_o = nullptr;
  p.part_lse = nullptr;
  p.merge = nullptr;
  p.status = dev_status;
  p.B = B;
  p.R = R;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.nr = pl.nr;
  p.tr = (R + 15) / 16 * 16;
  p.q_box_rows = pl.copies == 2 ? 64 / G : pl.nr;
  p.qtiles = pl.qtiles;
  p.ncq = pl.ncq;
  p.n_ctas = pl.n_ctas;
  p.splits = pl.splits;
  p.scale_log2 = scale * kLog2e;
  char* cur = static_cast<char*>(ws);
  if (pl.stream) {
    const size_t slots = (size_t)pl.n_ctas * 2 * pl.tpc * 128;
    p.part_o = static_cast<float*>(ws_carve(cur, slots * D * 4));
    p.part_lse = static_cast<float*>(ws_carve(cur, slots * 4));
    p.merge = static_cast<int4*>(ws_carve(cur, (size_t)pl.n_ctas * 16));
  } else if (pl.splits > 1) {
    const size_t rows = (size_t)B * R * Hq;
    p.part_o = static_cast<float*>(ws_carve(cur, rows * pl.splits * D * 4));
    p.part_lse = static_cast<float*>(ws_carve(cur, rows * pl.splits * 4));
  }
  // tensor maps: q as [B*R][Hq][D], the pools as [pages*16][Hkv][D], the
  // tree K/V as [B*R][Hkv][D]; boxes of 64 columns (128 bytes)
  CUtensorMap mq, mk, mv, mkt, mvt;
  const uint64_t hb = (uint64_t)D * 2;
  if (!make_tmap_3d_bf16(&mq, q, D, Hq, (uint64_t)B * R, hb, hb * Hq, 64, G, (uint32_t)p.q_box_rows) ||
      !make_tmap_3d_bf16(&mk, k_cache, D, Hkv, (uint64_t)num_pages * 16, hb, hb * Hkv, 64, 1, 16) ||
      !make_tmap_3d_bf16(&mv, v_cache, D, Hkv, (uint64_t)num_pages * 16, hb, hb * Hkv, 64, 1, 16) ||
      !make_tmap_3d_bf16(&mkt, k_tree, D, Hkv, (uint64_t)B * R, hb, hb * Hkv, 64, 1, p.tr) ||
      !make_tmap_3d_bf16(&mvt, v_tree, D, Hkv, (uint64_t)B * R, hb, hb * Hkv, 64, 1, p.tr))
    return EAGLE_ERR_CUDA;
  auto run_stream = [&](auto kern, auto merge, size_t sm, int threads) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    launch(kern, pl.n_ctas, threads, sm, s, mq, mk, mv, mkt, mvt, p);
    // the merge: the rows of a split unit over 16 CTAs per query tile of its column
    launch(merge, dim3((unsigned)pl.n_ctas, 16u * (unsigned)pl.tpc), kCombWarps * 32, 0, s, p);
    note_launch(2);
  };
  auto run_split = [&](auto kern, size_t sm, int threads) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    const dim3 grid((pl.qtiles + pl.tpc - 1) / pl.tpc, pl.splits, B * Hkv);
    launch(kern, grid, threads, sm, s, mq, mk, mv, mkt, mvt, p);
    note_launch();
    if (pl.splits > 1) {
      const int rows = B * R * Hq;
      if (D == 128)
        launch(tree_attn_split_combine_kernel<128>, (rows + 7) / 8, 256, 0, s, p.part_o, p.part_lse, rows,
               pl.splits, p.out, lse);
      else
        launch(tree_attn_split_combine_kernel<64>, (rows + 7) / 8, 256, 0, s, p.part_o, p.part_lse, rows,
               pl.splits, p.out, lse);
      note_launch();
    }
  };
  if (pl.stream) {
    if (D == 128) {
      if (pl.tpc == 2)
        run_stream(tree_attn_stream_kernel<128, 2, 1>, tree_attn_stream_merge_kernel<128, 2>, tc_smem<128>(2), 384);
      else if (pl.copies == 2)
        run_stream(tree_attn_stream_kernel<128, 1, 2>, tree_attn_stream_merge_kernel<128, 1>, tc_smem<128>(1), 256);
      else
        run_stream(tree_attn_stream_kernel<128, 1, 1>, tree_attn_stream_merge_kernel<128, 1>, tc_smem<128>(1), 256);
    } else {
      if (pl.tpc == 2)
        run_stream(tree_attn_stream_kernel<64, 2, 1>, tree_attn_stream_merge_kernel<64, 2>, tc_smem<64>(2), 384);
      else if (pl.copies == 2)
        run_stream(tree_attn_stream_kernel<64, 1, 2>, tree_attn_stream_merge_kernel<64, 1>, tc_smem<64>(1), 256);
      else
        run_stream(tree_attn_stream_kernel<64, 1, 1>, tree_attn_stream_merge_kernel<64, 1>, tc_smem<64>(1), 256);
    }
  } else {
    if (D == 128) {
      if (pl.tpc == 2)
        run_split(tree_attn_split_kernel<128, 2>, tc_smem<128>(2), 384);
      else
        run_split(tree_attn_split_kernel<128, 1>, tc_smem<128>(1), 256);
    } else {
      if (pl.tpc == 2)
        run_split(tree_attn_split_kernel<64, 2>, tc_smem<64>(2), 384);
      else
        run_split(tree_attn_split_kernel<64, 1>, tc_smem<64>(1), 256);
    }
  }
  return last_launch_status();
}
