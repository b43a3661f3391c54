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
// bf16 path: one CTA per (query tile, KV split, request x kv head).  All
// query rows of one kv head (R tree rows x G grouped heads) share every K/V
// byte the CTA stages, so each prefix byte leaves HBM once per query tile.
// K/V pages are gathered through the block table with cp.async into a
// 3-stage ring of XOR-swizzled shared tiles; warps run m16n8k16 bf16 MMAs with
// an fp32 online softmax; the tree's own rows form one extra 64-key block
// masked by the u64 ancestry bits.  KV splits write (O, lse) partials that a
// second kernel merges.  fp32 path (small shapes): a warp per query row.
#include <math.h>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int kBlkKeys = 64;
constexpr int kStages = 3;
constexpr int kMaxWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_tree;
  const __nv_bfloat16* v_tree;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const uint64_t* tree_mask;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;    // [B*R*Hq, splits, D] (splits > 1)
  float* part_lse;  // [B*R*Hq, splits]
  int32_t* status;
  int B, R, Hq, Hkv, G, max_pages, num_pages, splits, rows_per_cta;
  float scale_log2;  // scale * log2(e)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of 16-byte chunk `c` of row `row` in a swizzled [64][D] bf16 tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return (uint32_t)(row * (D * 2) + ((c ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kMaxWarps * 32) tree_attn_bf16_kernel(const AttnParams p) {
  pdl_wait();
  pdl_trigger();
  constexpr int kChunks = D / 8;            // 16-byte chunks per key row
  constexpr int kTile = kBlkKeys * D * 2;   // bytes of one K (or V) tile
  extern __shared__ __align__(1024) unsigned char smem[];
  const int qtile = blockIdx.x, split = blockIdx.y;
  const int b = blockIdx.z / p.Hkv, kvh = blockIdx.z % p.Hkv;
  const int nthreads = blockDim.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int rows_total = p.R * p.G;
  const uint32_t sbase = smem_u32(smem);

  const int ctx = p.ctx_lens[b];
  const int nblk = (ctx + kBlkKeys - 1) / kBlkKeys;
  const int bps = (nblk + p.splits - 1) / p.splits;
  const int blk_lo = min(nblk, split * bps), blk_hi = min(nblk, blk_lo + bps);
  const bool has_tree = split == 0;
  const int n_iter = (blk_hi - blk_lo) + (has_tree ? 1 : 0);

  // ---- K/V block loader (iteration it -> stage it % kStages)
  auto load_block = [&](int it) {
    const int st = it % kStages;
    const uint32_t kdst = sbase + st * 2 * kTile, vdst = kdst + kTile;
    const bool tree_blk = it == (blk_hi - blk_lo);
    const int kb = (blk_lo + it) * kBlkKeys;
    for (int c = tid; c < kBlkKeys * kChunks; c += nthreads) {
      const int row = c / kChunks, ch = c % kChunks;
      const __nv_bfloat16 *ks = p.k_cache, *vs = p.v_cache;
      int bytes = 0;
      if (tree_blk) {
        if (row < p.R) {
          const size_t off = (((size_t)b * p.R + row) * p.Hkv + kvh) * D + ch * 8;
          ks = p.k_tree + off;
          vs = p.v_tree + off;
          bytes = 16;
        }
      } else {
        const int key = kb + row;
        if (key < ctx) {
          int page = p.block_table[(size_t)b * p.max_pages + key / 16];
          if (page < 0 || page >= p.num_pages) {
            set_status(p.status, EAGLE_ERR_BAD_KV);
          } else {
            const size_t off = (((size_t)page * 16 + key % 16) * p.Hkv + kvh) * D + ch * 8;
            ks = p.k_cache + off;
            vs = p.v_cache + off;
            bytes = 16;
          }
        }
      }
      cp_async16(kdst + swz<D>(row, ch), ks, bytes);
      cp_async16(vdst + swz<D>(row, ch), vs, bytes);
    }
  };

  // ---- per-warp query rows and their tree masks
  const int qrow0 = qtile * p.rows_per_cta + warp * 16;
  const int i0 = qrow0 + gid, i1 = i0 + 8;
  const uint64_t m_row0 = i0 < rows_total ? p.tree_mask[(size_t)b * p.R + i0 / p.G] : 0ull;
  const uint64_t m_row1 = i1 < rows_total ? p.tree_mask[(size_t)b * p.R + i1 / p.G] : 0ull;
  uint32_t qa[D / 16][4];
  {
    auto qptr = [&](int i) -> const uint32_t* {
      const int r = i / p.G, g = i % p.G;
      return reinterpret_cast<const uint32_t*>(p.q + (((size_t)b * p.R + r) * p.Hq + kvh * p.G + g) * D);
    };
    const uint32_t* q0 = i0 < rows_total ? qptr(i0) : nullptr;
    const uint32_t* q1 = i1 < rows_total ? qptr(i1) : nullptr;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int w0 = kk * 8 + tig, w1 = w0 + 4;  // 32-bit words (2 bf16)
      qa[kk][0] = q0 ? q0[w0] : 0u;
      qa[kk][1] = q1 ? q1[w0] : 0u;
      qa[kk][2] = q0 ? q0[w1] : 0u;
      qa[kk][3] = q1 ? q1[w1] : 0u;
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  // prologue
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < n_iter) load_block(s);
    cp_async_commit();
  }
  for (int it = 0; it < n_iter; ++it) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    if (it + kStages - 1 < n_iter) load_block(it + kStages - 1);
    cp_async_commit();
    if (qrow0 >= rows_total) continue;

    const int st = it % kStages;
    const uint32_t ks = sbase + st * 2 * kTile, vs = ks + kTile;
    const bool tree_blk = it == (blk_hi - blk_lo);
    const int kb = (blk_lo + it) * kBlkKeys;

    // S = Q K^T for 64 keys (8 n-tiles of 8 keys)
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int k2 = 0; k2 < D / 32; ++k2) {
        const int key = nt * 8 + (lane & 7);
        const int ch = k2 * 4 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks + swz<D>(key, ch), b0, b1, b2, b3);
        mma16816(s[nt], qa[2 * k2][0], qa[2 * k2][1], qa[2 * k2][2], qa[2 * k2][3], b0, b1);
        mma16816(s[nt], qa[2 * k2 + 1][0], qa[2 * k2 + 1][1], qa[2 * k2 + 1][2], qa[2 * k2 + 1][3],
                 b2, b3);
      }
    }
    // mask, scale and block max
    float bmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = nt * 8 + tig * 2 + (e & 1);
        const int hr = e >> 1;  // 0: row gid, 1: row gid+8
        bool valid;
        if (tree_blk) {
          const uint64_t m = hr ? m_row1 : m_row0;
          valid = key < p.R && ((m >> key) & 1ull);
        } else {
          valid = kb + key < ctx;
        }
        const float v = valid ? s[nt][e] * p.scale_log2 : -INFINITY;
        s[nt][e] = v;
        bmax[hr] = fmaxf(bmax[hr], v);
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      bmax[hr] = fmaxf(bmax[hr], __shfl_xor_sync(0xffffffffu, bmax[hr], 1));
      bmax[hr] = fmaxf(bmax[hr], __shfl_xor_sync(0xffffffffu, bmax[hr], 2));
    }
    float alpha[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const float mnew = fmaxf(mrow[hr], bmax[hr]);
      alpha[hr] = (mrow[hr] == -INFINITY) ? 0.f : exp2f(mrow[hr] - mnew);
      mrow[hr] = mnew;
      lrow[hr] *= alpha[hr];
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      o[dn][0] *= alpha[0];
      o[dn][1] *= alpha[0];
      o[dn][2] *= alpha[1];
      o[dn][3] *= alpha[1];
    }
    // P = exp2(S - m) -> bf16 A fragments; l accumulates the rounded P
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = mrow[e >> 1];
        pv[e] = (m == -INFINITY || s[nt][e] == -INFINITY) ? 0.f : exp2f(s[nt][e] - m);
      }
      const uint32_t lo = pack_bf16(pv[0], pv[1]), hi = pack_bf16(pv[2], pv[3]);
      const __nv_bfloat162 blo = *reinterpret_cast<const __nv_bfloat162*>(&lo);
      const __nv_bfloat162 bhi = *reinterpret_cast<const __nv_bfloat162*>(&hi);
      lrow[0] += __low2float(blo) + __high2float(blo);
      lrow[1] += __low2float(bhi) + __high2float(bhi);
      const int kk = nt >> 1;
      if ((nt & 1) == 0) {
        pa[kk][0] = lo;
        pa[kk][1] = hi;
      } else {
        pa[kk][2] = lo;
        pa[kk][3] = hi;
      }
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        const int i = lane >> 3;
        const int key = kk * 16 + (i & 1) * 8 + (lane & 7);
        const int ch = dn * 2 + (i >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vs + swz<D>(key, ch), b0, b1, b2, b3);
        mma16816(o[2 * dn], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
        mma16816(o[2 * dn + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
      }
    }
  }
  cp_async_wait<0>();
  if (qrow0 >= rows_total) return;

  // finish: quad-reduce l, normalise, write
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = hr ? i1 : i0;
    if (i >= rows_total) continue;
    const int r = i / p.G, h = kvh * p.G + i % p.G;
    const size_t row = ((size_t)b * p.R + r) * p.Hq + h;
    const float l = lrow[hr];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (mrow[hr] + log2f(l)) * kLn2 : -INFINITY;
    if (p.splits == 1) {
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const int d = dn * 8 + tig * 2;
        *reinterpret_cast<uint32_t*>(p.out + row * D + d) =
            pack_bf16(o[dn][hr * 2] * inv, o[dn][hr * 2 + 1] * inv);
      }
      if (p.lse && tig == 0) p.lse[row] = lse;
    } else {
      float* po = p.part_o + (row * p.splits + split) * D;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const int d = dn * 8 + tig * 2;
        *reinterpret_cast<float2*>(po + d) = make_float2(o[dn][hr * 2] * inv, o[dn][hr * 2 + 1] * inv);
      }
      if (tig == 0) p.part_lse[row * p.splits + split] = lse;
    }
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
  int nwarps, rows_per_cta, qtiles, splits;
};

template <int D>
size_t attn_smem() {
  return (size_t)kStages * 2 * kBlkKeys * D * 2;
}

// CTAs of the bf16 kernel that fit on one SM at once.
int resident_per_sm(int D, int threads) {
  const size_t sm = D == 128 ? attn_smem<128>() : attn_smem<64>();
  auto kern = D == 128 ? tree_attn_bf16_kernel<128> : tree_attn_bf16_kernel<64>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, sm) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

Plan make_plan(int B, int R, int Hq, int Hkv, int D, int max_pages, int num_splits) {
  Plan pl;
  const int rows = R * (Hq / Hkv);
  pl.nwarps = min(kMaxWarps, (rows + 15) / 16);
  pl.rows_per_cta = pl.nwarps * 16;
  pl.qtiles = (rows + pl.rows_per_cta - 1) / pl.rows_per_cta;
  const int max_blocks = max(1, (max_pages * 16 + kBlkKeys - 1) / kBlkKeys);
  if (num_splits > 0) {
    pl.splits = min(num_splits, max_blocks);
  } else {
    // The split count that minimises waves x key blocks per CTA (the tree
    // block included), plus a small charge per split for the (O, lse)
    // partials and their merge.
    const long long base = (long long)pl.qtiles * B * Hkv;
    const long long slots = (long long)max(1, sm_count()) * resident_per_sm(D, pl.nwarps * 32);
    double best = 1e300;
    pl.splits = 1;
    for (int sp = 1; sp <= min(max_blocks, 256); ++sp) {
      const long long waves = (base * sp + slots - 1) / slots;
      const int bps = (max_blocks + sp - 1) / sp;
      const double cost = (double)waves * (bps + 1) + (sp > 1 ? 0.1 * sp : 0.0);
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
  const Plan pl = make_plan(B, R, Hq, Hkv, D, max_pages, num_splits);
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
  const Plan pl = make_plan(B, R, Hq, Hkv, D, max_pages, num_splits);
  if (pl.splits > 65535) return EAGLE_ERR_UNSUPPORTED;
  AttnParams p;
  p.q = (const __nv_bfloat16*)q;
  p.k_tree = (const __nv_bfloat16*)k_tree;
  p.v_tree = (const __nv_bfloat16*)v_tree;
  p.k_cache = (const __nv_bfloat16*)k_cache;
  p.v_cache = (const __nv_bfloat16*)v_cache;
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
  p.G = Hq / Hkv;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.splits = pl.splits;
  p.rows_per_cta = pl.rows_per_cta;
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
  const dim3 grid(pl.qtiles, pl.splits, B * Hkv);
  const int threads = pl.nwarps * 32;
  if (D == 128) {
    const size_t sm = attn_smem<128>();
    cudaFuncSetAttribute(tree_attn_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    launch(tree_attn_bf16_kernel<128>, grid, threads, sm, s, p);
  } else {
    const size_t sm = attn_smem<64>();
    cudaFuncSetAttribute(tree_attn_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    launch(tree_attn_bf16_kernel<64>, grid, threads, sm, s, p);
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
