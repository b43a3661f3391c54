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
// bf16 path: tcgen05 tensor-core kernel, one CTA per (query tile, KV split,
// request x kv head).  All query rows of one kv head (R tree rows x G grouped
// heads) share every K/V byte the CTA stages, so each prefix byte leaves HBM
// once per query tile.  The tree's own rows form one extra key block masked by
// the u64 ancestry bits.  KV splits write (O, lse) partials that a second
// kernel merges.  fp32 path (small shapes): a warp per query row.
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
// tcgen05 path (bf16).  One CTA per (one or two query tiles of up to 128
// rows, KV split, request x kv head); 128 + 128 * TPC threads:
//   warp 1     allocates the tensor memory, then issues the P V MMAs (one
//              thread); with one query tile warp 0 has no role, so that the
//              producer and the S issuer sit on the sub-partitions of lane
//              quarters 2 and 3, the quarters that have no query rows when a
//              tile holds 64 rows or fewer (short trees, batch 64)
//   warp 2     TMA producer: the Q tiles once (3-D box [rows of r][G heads]
//              [64]), then per 64-key block 4 paged K boxes and 4 V boxes of
//              16 keys per 64-column half (3-D map over the pool viewed as
//              [pages*16][Hkv][D]) or the tree's own K/V rows, into a ring of
//              kv_stages(TPC) stages; with two query tiles warp 0 loads Q and
//              K (its stages freed by S) and warp 2 only V (freed by P V)
//   warp 3     S issuer (one thread): S = Q K^T (M 128, N 64, K D) into one
//              of two TMEM S buffers per tile, up to two blocks ahead; warp 1
//              issues O += P V (M 128, N D, K 64, V read MN-major) into the
//              tile's TMEM O accumulator as soon as P is ready.  Two issuing
//              threads, because one thread issues an MMA only every ≈ 50
//              cycles; the commits: S ready, and P V done (which also frees
//              the K/V stage)
//   warps 4.. (4 per query tile): softmax, one thread per query row (TMEM lane;
//              a quarter without query rows only keeps the barrier protocol):
//              the block's 64 scores loaded once, masked row max, P =
//              exp2(S - m) rounded to bf16 into a double-buffered
//              128-byte-swizzled shared tile (the A operand of P V), and O
//              rescaled in TMEM only when the row max grows by more than 2^8
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
  uint64_t q_full;
  uint64_t k_full[kMaxStages], v_full[kMaxStages], k_empty[kMaxStages], kv_empty[kMaxStages];
  uint64_t s_full[2], s_empty[2], p_full[2];
  uint64_t drain, drain_pv;
  uint32_t tmem_base;
  int abort_flag;
};
struct Params {
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const uint64_t* tree_mask;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int32_t* status;
  int B, R, Hq, Hkv, G, max_pages, num_pages, splits;
  int nr;         // tree rows per query tile (rows per tile = nr * G <= 128)
  int qtiles;     // query tiles of a (request, kv head)
  int tr;         // tree keys loaded: R rounded up to 16
  float scale_log2;
};
}  // namespace tc

template <int D, int TPC>
__global__ void __launch_bounds__(128 + 128 * TPC, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap map_q,
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

// Merge split partials: out = sum_s exp(lse_s - L) O_s, L = log sum_s exp(lse_s).
template <int D>
__global__ void __launch_bounds__(256) tree_attn_combine_kernel(const float* __restrict__ part_o,
                                                                const float* __restrict__ part_lse,
                                                                int nrows, int splits,
                                                                __nv_bfloat16* __restrict__ out,
                                                                float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= nrows) return;
  const float* pl = part_lse + (size_t)row * splits;
  float L = -INFINITY;
  for (int s = 0; s < splits; ++s) L = fmaxf(L, pl[s]);
  float acc[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j) acc[j] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ls = pl[s];
    if (ls == -INFINITY) continue;
    const float w = exp2f((ls - L) * kLog2e);
    wsum += w;
    const float* po = part_o + ((size_t)row * splits + s) * D;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) acc[j] += w * po[lane + 32 * j];
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
  int nr, qtiles, tpc, splits;
};

template <int D>
size_t tc_smem(int tpc) {
  return 1024 + (size_t)tpc * 128 * 128 * (D / 64) +
         2 * (size_t)tc::kv_stages<D>(tpc) * tc::kBlk * 128 * (D / 64) +
         (size_t)tpc * 2 * 128 * tc::kBlk * 2;
}

// Query tiles of nr tree rows x G heads (nr * G <= 128 MMA rows) and the KV
// split count.  Auto splits: the count minimising (waves of CTAs, one per SM)
// x (64-key blocks per CTA + the tree block + 5 blocks' worth of set-up),
// plus a small charge per split for the (O, lse) partials and their merge.
Plan make_plan(int B, int R, int Hq, int Hkv, int max_pages, int num_splits) {
  Plan pl;
  const int G = Hq / Hkv;
  pl.nr = 128 / G;
  pl.qtiles = (R + pl.nr - 1) / pl.nr;
  const int max_blocks = max(1, (max_pages * 16 + tc::kBlk - 1) / tc::kBlk);
  // two query tiles share each K/V block when the prefix is long enough
  // (>= 4096 keys) for the splits to keep every SM busy anyway
  pl.tpc = (pl.qtiles >= 2 && max_blocks >= 64) ? 2 : 1;
  if (num_splits > 0) {
    pl.splits = min(num_splits, max_blocks);
  } else {
    const long long base = (long long)((pl.qtiles + pl.tpc - 1) / pl.tpc) * B * Hkv;
    const long long slots = max(1, sm_count());
    double best = 1e300;
    pl.splits = 1;
    for (int sp = 1; sp <= min(max_blocks, 256); ++sp) {
      const long long waves = (base * sp + slots - 1) / slots;
      const int bps = (max_blocks + sp - 1) / sp;
      const double cost = (double)waves * (bps + 6) * pl.tpc + (sp > 1 ? 0.1 * sp : 0.0);
      if (cost < best - 1e-9) {
        best = cost;
        pl.splits = sp;
      }
    }
  }
  pl.splits = max(1, pl.splits);
  return pl;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_attn_workspace_size(int B, int R, int Hq, int Hkv, int D, int max_pages,
                                                 int page_size, int num_splits, int dtype) {
  (void)page_size;
  if (B <= 0 || R <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_pages <= 0) return 0;
  if (dtype != EAGLE_BF16 || Hq % Hkv) return 0;
  const Plan pl = make_plan(B, R, Hq, Hkv, max_pages, num_splits);
  if (pl.splits == 1) return 0;
  const size_t rows = (size_t)B * R * Hq;
  return round_up(rows * pl.splits * D * 4, 256) + round_up(rows * pl.splits * 4, 256) + 512;
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
      num_splits < 0 || !(scale > 0.f) || isinf(scale))
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
  const Plan pl = make_plan(B, R, Hq, Hkv, max_pages, num_splits);
  if (pl.splits > 65535 || num_pages > (1 << 26) || (long long)B * R > (1LL << 30))
    return EAGLE_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  tc::Params p;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.tree_mask = tree_mask;
  p.out = (__nv_bfloat16*)out;
  p.lse = lse;
  p.part_o = nullptr;
  p.part_lse = nullptr;
  p.status = dev_status;
  p.B = B;
  p.R = R;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.splits = pl.splits;
  p.nr = pl.nr;
  p.tr = (R + 15) / 16 * 16;
  p.qtiles = pl.qtiles;
  p.scale_log2 = scale * kLog2e;
  if (pl.splits > 1) {
    if (!ws || ws_bytes < eagle_tree_attn_workspace_size(B, R, Hq, Hkv, D, max_pages, page_size,
                                                         num_splits, dtype))
      return EAGLE_ERR_WORKSPACE;
    char* cur = static_cast<char*>(ws);
    const size_t rows = (size_t)B * R * Hq;
    p.part_o = static_cast<float*>(ws_carve(cur, rows * pl.splits * D * 4));
    p.part_lse = static_cast<float*>(ws_carve(cur, rows * pl.splits * 4));
  }
  // tensor maps: q as [B*R][Hq][D], the pools as [pages*16][Hkv][D], the
  // tree K/V as [B*R][Hkv][D]; boxes of 64 columns (128 bytes)
  CUtensorMap mq, mk, mv, mkt, mvt;
  const uint64_t hb = (uint64_t)D * 2;
  if (!make_tmap_3d_bf16(&mq, q, D, Hq, (uint64_t)B * R, hb, hb * Hq, 64, G, pl.nr) ||
      !make_tmap_3d_bf16(&mk, k_cache, D, Hkv, (uint64_t)num_pages * 16, hb, hb * Hkv, 64, 1, 16) ||
      !make_tmap_3d_bf16(&mv, v_cache, D, Hkv, (uint64_t)num_pages * 16, hb, hb * Hkv, 64, 1, 16) ||
      !make_tmap_3d_bf16(&mkt, k_tree, D, Hkv, (uint64_t)B * R, hb, hb * Hkv, 64, 1, p.tr) ||
      !make_tmap_3d_bf16(&mvt, v_tree, D, Hkv, (uint64_t)B * R, hb, hb * Hkv, 64, 1, p.tr))
    return EAGLE_ERR_CUDA;
  const dim3 grid((pl.qtiles + pl.tpc - 1) / pl.tpc, pl.splits, B * Hkv);
  auto run = [&](auto kern, size_t sm, int threads) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    launch(kern, grid, threads, sm, s, mq, mk, mv, mkt, mvt, p);
  };
  if (D == 128) {
    if (pl.tpc == 2)
      run(tree_attn_tc_kernel<128, 2>, tc_smem<128>(2), 384);
    else
      run(tree_attn_tc_kernel<128, 1>, tc_smem<128>(1), 256);
  } else {
    if (pl.tpc == 2)
      run(tree_attn_tc_kernel<64, 2>, tc_smem<64>(2), 384);
    else
      run(tree_attn_tc_kernel<64, 1>, tc_smem<64>(1), 256);
  }
  note_launch();
  if (pl.splits > 1) {
    const int rows = B * R * Hq;
    if (D == 128)
      launch(tree_attn_combine_kernel<128>, (rows + 7) / 8, 256, 0, s, p.part_o, p.part_lse, rows,
                                                                  pl.splits, p.out, lse);
    else
      launch(tree_attn_combine_kernel<64>, (rows + 7) / 8, 256, 0, s, p.part_o, p.part_lse, rows,
                                                                 pl.splits, p.out, lse);
    note_launch();
  }
  return last_launch_status();
}
