// The drafter's decoder layer over the new tree nodes of one depth, and the
// small kernels it is made of.
//
// Source: "EAGLE-3: Scaling up Inference Acceleration of Large Language
// Models via Training-Time Test", section 3.4 "The transformer decoder
// layer" (one standard layer: self-attention and feed-forward sublayers with
// residual connections and normalisation) and section 6, Limitation 6 (the
// targets are LLaMA-family: pre-normalisation, SwiGLU, rotary position
// embeddings, grouped-query attention), which fixes the form taken here;
// "M7.5 - EAGLE Feature Drafting ...", sections 0x03C (the drafter keeps its
// own K/V) and 0x05B (the nodes of one depth are expanded in one pass with
// tree attention, each with its position and draft-KV row).
//
// Layer = RMSNorm -> QKV projection -> RoPE (K/V rows written into the
// drafter's tree arrays) -> tree attention -> output projection + residual
// -> RMSNorm -> gate/up projection -> SwiGLU -> down projection + residual.
// The projections are eagle_linear (tcgen05 weight stream), the attention is
// eagle_tree_attn; the kernels below are the element-wise steps between them.
#include <math.h>

#include <algorithm>

#include "common.cuh"

namespace eagle {
namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16(x);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

// y[m] = x[m] / sqrt(mean(x[m]^2) + eps) * w; one CTA per row, fp32 sums.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    rmsnorm_kernel(const T* __restrict__ x, const T* __restrict__ w, float eps, T* __restrict__ y, int d) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kRowThreads / 32];
  const T* xr = x + (size_t)blockIdx.x * d;
  T* yr = y + (size_t)blockIdx.x * d;
  float ss = 0.f;
  for (int c = threadIdx.x; c < d; c += kRowThreads) {
    const float v = to_f(xr[c]);
    ss = fmaf(v, v, ss);
  }
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + eps);
  for (int c = threadIdx.x; c < d; c += kRowThreads) yr[c] = from_f<T>(to_f(xr[c]) * inv * to_f(w[c]));
}

// RoPE (rotate-half: pair (i, i + D/2) turned by pos * theta^(-2i/D)) of the
// q and k heads of one QKV row, written with the v heads into the drafter's
// tree arrays at row r0 + j of request b (row m = b * W + j).  The angle is
// formed in double precision so that large positions lose nothing: the
// frequency theta^(-2i/D) = ratio^i by binary powering of ratio =
// theta^(-2/D) (from the host), the product with the position, and its
// reduction to [-pi, pi]; only the sine and cosine of the reduced angle are
// taken in fp32.  (Double-precision transcendentals and division are slow
// on this part.)  Each thread moves 16-byte vectors: a chunk of the first
// half of a head and its partner chunk of the second half.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    rope_scatter_kernel(const T* __restrict__ qkv, const int32_t* __restrict__ positions, int W, int r0,
                        int Rmax, int Hq, int Hkv, int D, double ratio, T* __restrict__ q_tree,
                        T* __restrict__ k_tree, T* __restrict__ v_tree) {
  pdl_wait();
  pdl_trigger();
  constexpr int kV = 16 / sizeof(T);  // elements per 16-byte vector
  __shared__ float cs[64], sn[64];
  const int m = blockIdx.x, b = m / W, j = m % W, half = D / 2;
  const double pos = (double)positions[m];
  constexpr double kTwoPi = 6.283185307179586, kInvTwoPi = 0.15915494309189535;
  for (int i = threadIdx.x; i < half; i += kRowThreads) {
    double f = 1.0, base = ratio;
    for (int e = i; e; e >>= 1, base *= base)
      if (e & 1) f *= base;
    const double ang = pos * f;
    const double red = fma(-rint(ang * kInvTwoPi), kTwoPi, ang);
    float s, c;
    sincosf((float)red, &s, &c);
    cs[i] = c;
    sn[i] = s;
  }
  __syncthreads();
  const T* row = qkv + (size_t)m * (Hq + 2 * Hkv) * D;
  const size_t trow = (size_t)b * Rmax + r0 + j;
  // 16-byte vectors of the first half of each q / k head with their partners
  const int vph = half / kV;  // vectors per half head
  for (int t = threadIdx.x; t < (Hq + Hkv) * vph; t += kRowThreads) {
    const int h = t / vph, i0 = (t % vph) * kV;
    const T* src = row + (size_t)h * D + i0;
    uint4 a = *reinterpret_cast<const uint4*>(src), bb = *reinterpret_cast<const uint4*>(src + half);
    const T* x1 = reinterpret_cast<const T*>(&a);
    const T* x2 = reinterpret_cast<const T*>(&bb);
    uint4 ya, yb;
    T* y1 = reinterpret_cast<T*>(&ya);
    T* y2 = reinterpret_cast<T*>(&yb);
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      const float u = to_f(x1[e]), w = to_f(x2[e]), c = cs[i0 + e], sv = sn[i0 + e];
      y1[e] = from_f<T>(u * c - w * sv);
      y2[e] = from_f<T>(w * c + u * sv);
    }
    T* dst = h < Hq ? q_tree + (trow * Hq + h) * D : k_tree + (trow * Hkv + (h - Hq)) * D;
    *reinterpret_cast<uint4*>(dst + i0) = ya;
    *reinterpret_cast<uint4*>(dst + i0 + half) = yb;
  }
  const uint4* vsrc = reinterpret_cast<const uint4*>(row + (size_t)(Hq + Hkv) * D);
  uint4* vdst = reinterpret_cast<uint4*>(v_tree + trow * Hkv * D);
  for (int t = threadIdx.x; t < Hkv * D / kV; t += kRowThreads) vdst[t] = vsrc[t];
}

// a[m] = attn[b, r0 + j] (Hq * D values), m = b * W + j.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    rows_gather_kernel(const T* __restrict__ attn, int W, int r0, int Rmax, int width, T* __restrict__ a) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x, b = m / W, j = m % W;
  const T* src = attn + ((size_t)b * Rmax + r0 + j) * width;
  T* dst = a + (size_t)m * width;
  for (int c = threadIdx.x; c < width; c += kRowThreads) dst[c] = src[c];
}

// act[m, i] = silu(gu[m, i]) * gu[m, I + i], silu(g) = g / (1 + e^-g).
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    swiglu_kernel(const T* __restrict__ gu, int I, long long n, T* __restrict__ act) {
  pdl_wait();
  pdl_trigger();
  for (long long t = (long long)blockIdx.x * kRowThreads + threadIdx.x; t < n;
       t += (long long)gridDim.x * kRowThreads) {
    const long long m = t / I, i = t % I;
    const float g = to_f(gu[m * 2 * I + i]), u = to_f(gu[m * 2 * I + I + i]);
    act[t] = from_f<T>(g / (1.f + expf(-g)) * u);
  }
}

// Bookkeeping of one drafter pass (one CTA per request): which draft-KV row
// each node of the depth takes, the rows it sees, its position, token and
// feature input.  Step 0 is the root: row 0, position ctx, the seed token and
// the target feature prev[b].  At step s >= 1, frontier slot j takes row
// r0 = 1 + (s - 1) * width + j, sees its parent's row and what that row sees,
// sits at ctx + depth, and reads the drafter output of its parent's slot of
// the previous pass, prev[b * W_prev + (row(parent) - r0_prev)].  Empty
// slots get token 0, position ctx, zero features and a row that sees only
// itself.  A parent that the previous pass did not process, or a node id out
// of range, records EAGLE_ERR_BAD_TREE and reads as an empty slot.
constexpr int kRowsMaxWidth = 64;
__global__ void __launch_bounds__(kRowThreads)
    draft_rows_kernel(int step, int width, int Rmax, int max_nodes, int vec_per_row,
                      const int32_t* __restrict__ root_token, const int32_t* __restrict__ frontier,
                      const int32_t* __restrict__ n_frontier, const int32_t* __restrict__ node_parent,
                      const int32_t* __restrict__ node_token, const int32_t* __restrict__ node_depth,
                      const int32_t* __restrict__ ctx_lens, int32_t* __restrict__ node_row,
                      uint64_t* __restrict__ row_mask, const uint4* __restrict__ prev, uint4* __restrict__ r_in,
                      int32_t* __restrict__ tokens, int32_t* __restrict__ positions, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_src[kRowsMaxWidth];  // feature row of prev per slot, -1: zeros
  const int b = blockIdx.x;
  const int W = step == 0 ? 1 : width;
  const int ctx = ctx_lens[b];
  int32_t* nrow = node_row + (size_t)b * max_nodes;
  uint64_t* rmask = row_mask + (size_t)b * Rmax;
  if (step == 0) {
    // a new round: no node has a row yet; unused rows see only themselves
    for (int n = threadIdx.x; n < max_nodes; n += kRowThreads) nrow[n] = n == 0 ? 0 : -1;
    for (int r = threadIdx.x; r < Rmax; r += kRowThreads) rmask[r] = 1ull << r;
    if (threadIdx.x == 0) {
      tokens[b] = root_token[b];
      positions[b] = ctx;
      s_src[0] = b;
    }
  } else if (threadIdx.x < W) {
    const int j = threadIdx.x;
    const int W_prev = step == 1 ? 1 : width;
    const int r0_prev = step == 1 ? 0 : 1 + (step - 2) * width;
    const int row = 1 + (step - 1) * width + j;
    const int nf = n_frontier[b];
    int src = -1, tok = 0, pos = ctx;
    uint64_t m = 1ull << row;
    if (j < nf) {
      const int n = frontier[(size_t)b * width + j];
      const int p = (n > 0 && n < max_nodes) ? node_parent[(size_t)b * max_nodes + n] : -1;
      const int prow = (p >= 0 && p < max_nodes) ? nrow[p] : -1;
      if (prow >= r0_prev && prow < r0_prev + W_prev) {
        nrow[n] = row;
        m |= rmask[prow];
        tok = node_token[(size_t)b * max_nodes + n];
        pos = ctx + node_depth[(size_t)b * max_nodes + n];
        src = b * W_prev + (prow - r0_prev);
      } else {
        set_status(status, EAGLE_ERR_BAD_TREE);
      }
    }
    rmask[row] = m;
    tokens[(size_t)b * width + j] = tok;
    positions[(size_t)b * width + j] = pos;
    s_src[j] = src;
  }
  __syncthreads();
  // feature inputs, 16-byte vectors
  for (int t = threadIdx.x; t < W * vec_per_row; t += kRowThreads) {
    const int j = t / vec_per_row, v = t % vec_per_row;
    const int src = s_src[j];
    r_in[((size_t)b * W + j) * vec_per_row + v] =
        src >= 0 ? prev[(size_t)src * vec_per_row + v] : make_uint4(0u, 0u, 0u, 0u);
  }
}

struct LayerWs {
  size_t h, qkv, attn, a, x1, h2, gu, act, lin, att, total;
};

LayerWs layer_ws(int B, int W, int d, int Hq, int Hkv, int D, int I, int Rmax, int max_pages, int dtype) {
  const size_t es = dtype == EAGLE_BF16 ? 2 : 4;
  const size_t M = (size_t)B * W;
  LayerWs L;
  L.h = round_up(M * d * es, 256);
  L.qkv = round_up(M * (Hq + 2 * Hkv) * D * es, 256);
  L.attn = round_up((size_t)B * Rmax * Hq * D * es, 256);
  L.a = round_up(M * Hq * D * es, 256);
  L.x1 = L.h;
  L.h2 = L.h;
  L.gu = round_up(M * 2 * I * es, 256);
  L.act = round_up(M * I * es, 256);
  size_t lin = eagle_linear_workspace_size((int)M, (Hq + 2 * Hkv) * D, d, dtype);
  lin = std::max(lin, eagle_linear_workspace_size((int)M, d, Hq * D, dtype));
  lin = std::max(lin, eagle_linear_workspace_size((int)M, 2 * I, d, dtype));
  lin = std::max(lin, eagle_linear_workspace_size((int)M, d, I, dtype));
  L.lin = round_up(lin, 256);
  L.att = round_up(eagle_tree_attn_workspace_size(B, Rmax, Hq, Hkv, D, max_pages, 16, 0, dtype), 256);
  L.total = L.h + L.qkv + L.attn + L.a + L.x1 + L.h2 + L.gu + L.act + L.lin + L.att + 11 * 256;
  return L;
}

bool layer_shape_ok(int B, int W, int d, int Hq, int Hkv, int D, int I, int Rmax, int r0) {
  if (B <= 0 || W <= 0 || d <= 0 || Hq <= 0 || Hkv <= 0 || I <= 0 || Rmax <= 0 || r0 < 0) return false;
  if ((long long)B * W > 4096 || r0 + W > Rmax || Rmax > 64) return false;
  if (D != 64 && D != 128) return false;
  if (Hq % Hkv || d % 128 || ((Hq + 2 * Hkv) * D) % 128 || (Hq * D) % 128 || I % 64) return false;
  return true;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_draft_layer_workspace_size(int B, int W, int d, int Hq, int Hkv, int D, int I, int Rmax,
                                                   int max_pages, int dtype) {
  if (!layer_shape_ok(B, W, d, Hq, Hkv, D, I, Rmax, 0) || max_pages <= 0) return 0;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return 0;
  return layer_ws(B, W, d, Hq, Hkv, D, I, Rmax, max_pages, dtype).total;
}

extern "C" int eagle_draft_layer(const void* x, const void* w_norm1, const void* w_qkv, const void* w_o,
                                 const void* w_norm2, const void* w_gu, const void* w_down, float eps,
                                 float theta, const int32_t* positions, const void* k_cache,
                                 const void* v_cache, int num_pages, const int32_t* block_table, int max_pages,
                                 const int32_t* ctx_lens, void* q_tree, void* k_tree, void* v_tree,
                                 const uint64_t* tree_mask, int r0, int Rmax, void* out, int B, int W, int d,
                                 int Hq, int Hkv, int D, int I, int dtype, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, void* stream) {
  if (!x || !w_norm1 || !w_qkv || !w_o || !w_norm2 || !w_gu || !w_down || !positions || !k_cache ||
      !v_cache || !block_table || !ctx_lens || !q_tree || !k_tree || !v_tree || !tree_mask || !out)
    return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !(theta > 0.f) || x == out) return EAGLE_ERR_INVALID_ARG;
  if (B <= 0 || W <= 0 || r0 < 0 || num_pages <= 0 || max_pages <= 0) return EAGLE_ERR_INVALID_ARG;
  if (!layer_shape_ok(B, W, d, Hq, Hkv, D, I, Rmax, r0)) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(q_tree) || !aligned16(k_tree) || !aligned16(v_tree)) return EAGLE_ERR_INVALID_ARG;
  const LayerWs L = layer_ws(B, W, d, Hq, Hkv, D, I, Rmax, max_pages, dtype);
  if (!ws || ws_bytes < L.total) return EAGLE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int M = B * W;
  char* cur = static_cast<char*>(ws);
  void* h = ws_carve(cur, L.h);
  void* qkv = ws_carve(cur, L.qkv);
  void* attn = ws_carve(cur, L.attn);
  void* a = ws_carve(cur, L.a);
  void* x1 = ws_carve(cur, L.x1);
  void* h2 = ws_carve(cur, L.h2);
  void* gu = ws_carve(cur, L.gu);
  void* act = ws_carve(cur, L.act);
  void* lin_ws = ws_carve(cur, L.lin);
  void* att_ws = ws_carve(cur, L.att);
  const bool bf = dtype == EAGLE_BF16;
  const int nqkv = (Hq + 2 * Hkv) * D;
  int rc;
#define EAGLE_TRY(call)              \
  do {                               \
    rc = (call);                     \
    if (rc != EAGLE_OK) return rc;   \
  } while (0)
  // 1. h = RMSNorm(x) * w_norm1
  if (bf)
    launch(rmsnorm_kernel<__nv_bfloat16>, M, kRowThreads, 0, s, (const __nv_bfloat16*)x,
           (const __nv_bfloat16*)w_norm1, eps, (__nv_bfloat16*)h, d);
  else
    launch(rmsnorm_kernel<float>, M, kRowThreads, 0, s, (const float*)x, (const float*)w_norm1, eps, (float*)h, d);
  note_launch();
  // 2. qkv = h W_qkv^T;  3. RoPE, rows into the tree arrays
  const double ratio = pow((double)theta, -2.0 / D);
  EAGLE_TRY(eagle_linear(h, w_qkv, nullptr, nullptr, qkv, M, nqkv, d, dtype, lin_ws, L.lin, dev_status, stream));
  if (bf)
    launch(rope_scatter_kernel<__nv_bfloat16>, M, kRowThreads, 0, s, (const __nv_bfloat16*)qkv, positions, W,
           r0, Rmax, Hq, Hkv, D, ratio, (__nv_bfloat16*)q_tree, (__nv_bfloat16*)k_tree,
           (__nv_bfloat16*)v_tree);
  else
    launch(rope_scatter_kernel<float>, M, kRowThreads, 0, s, (const float*)qkv, positions, W, r0, Rmax, Hq, Hkv,
           D, ratio, (float*)q_tree, (float*)k_tree, (float*)v_tree);
  note_launch();
  // 4. tree attention over the drafter's prefix and its tree rows
  EAGLE_TRY(eagle_tree_attn(q_tree, k_tree, v_tree, k_cache, v_cache, num_pages, block_table, max_pages,
                            ctx_lens, tree_mask, attn, nullptr, B, Rmax, Hq, Hkv, D, 16,
                            1.f / sqrtf((float)D), 0, dtype, att_ws, L.att, dev_status, stream));
  // 5. x1 = x + a W_o^T, a = the new rows r0 .. r0 + W - 1 of each request's
  // attention output, read in place by the projection (gathered first where
  // that row view is not one TMA box per stage)
  rc = bf ? linear_rows_bf16(attn, B, W, Rmax, r0, w_o, nullptr, x, x1, d, Hq * D, lin_ws, L.lin, dev_status, s)
          : (int)EAGLE_ERR_UNSUPPORTED;
  if (rc == EAGLE_ERR_UNSUPPORTED) {
    if (bf)
      launch(rows_gather_kernel<__nv_bfloat16>, M, kRowThreads, 0, s, (const __nv_bfloat16*)attn, W, r0, Rmax,
             Hq * D, (__nv_bfloat16*)a);
    else
      launch(rows_gather_kernel<float>, M, kRowThreads, 0, s, (const float*)attn, W, r0, Rmax, Hq * D, (float*)a);
    note_launch();
    EAGLE_TRY(eagle_linear(a, w_o, nullptr, x, x1, M, d, Hq * D, dtype, lin_ws, L.lin, dev_status, stream));
  } else if (rc != EAGLE_OK) {
    return rc;
  }
  // 6. h2 = RMSNorm(x1) * w_norm2
  if (bf)
    launch(rmsnorm_kernel<__nv_bfloat16>, M, kRowThreads, 0, s, (const __nv_bfloat16*)x1,
           (const __nv_bfloat16*)w_norm2, eps, (__nv_bfloat16*)h2, d);
  else
    launch(rmsnorm_kernel<float>, M, kRowThreads, 0, s, (const float*)x1, (const float*)w_norm2, eps, (float*)h2,
           d);
  note_launch();
  // 7. gu = h2 W_gu^T;  8. act = silu(gate) * up;  9. out = x1 + act W_down^T
  EAGLE_TRY(eagle_linear(h2, w_gu, nullptr, nullptr, gu, M, 2 * I, d, dtype, lin_ws, L.lin, dev_status, stream));
  const long long n = (long long)M * I;
  const int sms = sm_count();
  const long long blocks = std::min((n + kRowThreads - 1) / kRowThreads, 4LL * (sms > 0 ? sms : 1));
  if (bf)
    launch(swiglu_kernel<__nv_bfloat16>, (unsigned)blocks, kRowThreads, 0, s, (const __nv_bfloat16*)gu, I, n,
           (__nv_bfloat16*)act);
  else
    launch(swiglu_kernel<float>, (unsigned)blocks, kRowThreads, 0, s, (const float*)gu, I, n, (float*)act);
  note_launch();
  EAGLE_TRY(eagle_linear(act, w_down, nullptr, x1, out, M, d, I, dtype, lin_ws, L.lin, dev_status, stream));
#undef EAGLE_TRY
  return last_launch_status();
}

extern "C" int eagle_draft_rows(int B, int step, int width, int Rmax, int max_nodes, int d, int dtype,
                                const int32_t* root_token, const int32_t* frontier, const int32_t* n_frontier,
                                const int32_t* node_parent, const int32_t* node_token,
                                const int32_t* node_depth, const int32_t* ctx_lens, int32_t* node_row,
                                uint64_t* row_mask, const void* prev, void* r_in, int32_t* tokens,
                                int32_t* positions, int32_t* dev_status, void* stream) {
  if (B <= 0 || step < 0 || width < 1 || Rmax < 1 || max_nodes < 1 || d <= 0) return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (!ctx_lens || !node_row || !row_mask || !prev || !r_in || !tokens || !positions)
    return EAGLE_ERR_INVALID_ARG;
  if (step == 0 && !root_token) return EAGLE_ERR_INVALID_ARG;
  if (step > 0 && (!frontier || !n_frontier || !node_parent || !node_token || !node_depth))
    return EAGLE_ERR_INVALID_ARG;
  const int es = dtype == EAGLE_BF16 ? 2 : 4;
  if (width > kRowsMaxWidth || Rmax > 64 || (d * es) % 16 || B > 65535) return EAGLE_ERR_UNSUPPORTED;
  if (step > 0 && 1LL + (long long)step * width > Rmax) return EAGLE_ERR_INVALID_ARG;
  if (!aligned16(prev) || !aligned16(r_in)) return EAGLE_ERR_INVALID_ARG;
  launch(draft_rows_kernel, B, kRowThreads, 0, static_cast<cudaStream_t>(stream), step, width, Rmax, max_nodes,
         d * es / 16, root_token, frontier, n_frontier, node_parent, node_token, node_depth, ctx_lens, node_row,
         row_mask, static_cast<const uint4*>(prev), static_cast<uint4*>(r_in), tokens, positions, dev_status);
  note_launch();
  return last_launch_status();
}
