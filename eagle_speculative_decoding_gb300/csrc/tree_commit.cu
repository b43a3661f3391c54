// Publish the verified path: the accepted rows' target K/V go into the paged
// cache after the committed prefix, their target features are gathered for
// the next draft round, and the prefix length advances.
//
// Source: "M7.5 - EAGLE Feature Drafting: Uncertainty, Dynamic Trees, HASS, and
// EAGLE-3", section 0x05D "Feature And KV Commit" (the publication is one
// transaction; rows are taken by the flat row map from verification, never
// by token id; the new frontier token needs a later target append).
//
// One CTA per request: thread 0 validates the whole request first (path rows,
// room in the block table, page ids); if anything is wrong nothing of that
// request is written and its prefix length is unchanged.  Then every thread
// copies 16-byte chunks of the accepted rows and, last, thread 0 advances
// ctx_lens[b] (only this CTA reads it).
#include "common.cuh"

namespace eagle {
namespace {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) tree_commit_kernel(
    int R, int max_depth, int row_chunks, const uint4* __restrict__ k_tree,
    const uint4* __restrict__ v_tree, const int32_t* __restrict__ path_rows,
    const int32_t* __restrict__ accept_len, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    int num_pages, const int32_t* __restrict__ block_table, int max_pages,
    int32_t* __restrict__ ctx_lens, const uint4* __restrict__ feat, int feat_chunks,
    uint4* __restrict__ feat_out, int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  __shared__ int s_ok, s_n, s_ctx;
  __shared__ int s_row[65], s_slot[65];  // tree row and cache row (page * 16 + slot)
  if (threadIdx.x == 0) {
    const int n = accept_len[b] + 1;
    const int ctx = ctx_lens[b];
    int ok = (n >= 1 && n <= max_depth + 1) ? 1 : EAGLE_ERR_BAD_TREE;
    if (ok == 1 && (ctx < 0 || (long long)ctx + n > (long long)max_pages * 16)) ok = EAGLE_ERR_BAD_KV;
    for (int i = 0; ok == 1 && i < n; ++i) {
      const int row = path_rows[(size_t)b * (max_depth + 1) + i];
      if (row < 0 || row >= R) {
        ok = EAGLE_ERR_BAD_TREE;
        break;
      }
      const int pos = ctx + i;
      const int page = block_table[(size_t)b * max_pages + pos / 16];
      if (page < 0 || page >= num_pages) {
        ok = EAGLE_ERR_BAD_KV;
        break;
      }
      s_row[i] = row;
      s_slot[i] = page * 16 + pos % 16;
    }
    if (ok != 1) set_status(dev_status, ok);
    s_ok = ok == 1;
    s_n = n;
    s_ctx = ctx;
  }
  __syncthreads();
  if (!s_ok) return;
  const int n = s_n;
  constexpr int kU = 4;  // independent 16-byte loads in flight per thread
  for (int c0 = threadIdx.x; c0 < n * row_chunks; c0 += kCommitThreads * kU) {
    uint4 kv[kU], vv[kU];
    size_t dst[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * kCommitThreads;
      if (c < n * row_chunks) {
        const int i = c / row_chunks, ch = c % row_chunks;
        const size_t src = ((size_t)b * R + s_row[i]) * row_chunks + ch;
        dst[u] = (size_t)s_slot[i] * row_chunks + ch;
        kv[u] = k_tree[src];
        vv[u] = v_tree[src];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (c0 + u * kCommitThreads < n * row_chunks) {
        k_cache[dst[u]] = kv[u];
        v_cache[dst[u]] = vv[u];
      }
    }
  }
  if (feat_out) {
    const int total = (max_depth + 1) * feat_chunks;
    for (int c0 = threadIdx.x; c0 < total; c0 += kCommitThreads * kU) {
      uint4 fv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + u * kCommitThreads;
        const int i = c / feat_chunks, ch = c % feat_chunks;
        fv[u] = (c < total && i < n) ? feat[((size_t)b * R + s_row[i]) * feat_chunks + ch]
                                     : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + u * kCommitThreads;
        if (c < total) feat_out[(size_t)b * total + c] = fv[u];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) ctx_lens[b] = s_ctx + n;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" int eagle_tree_commit(int B, int R, int Hkv, int D, int max_depth, int dtype,
                                 const void* k_tree, const void* v_tree, const int32_t* path_rows,
                                 const int32_t* accept_len, void* k_cache, void* v_cache,
                                 int num_pages, const int32_t* block_table, int max_pages,
                                 int32_t* ctx_lens, const void* features, int F, void* features_out,
                                 int32_t* dev_status, void* stream) {
  if (B <= 0 || R <= 0 || Hkv <= 0 || D <= 0 || max_depth < 0 || num_pages <= 0 || max_pages <= 0)
    return EAGLE_ERR_INVALID_ARG;
  if (dtype != EAGLE_BF16 && dtype != EAGLE_FP32) return EAGLE_ERR_INVALID_ARG;
  if (!k_tree || !v_tree || !path_rows || !accept_len || !k_cache || !v_cache || !block_table ||
      !ctx_lens)
    return EAGLE_ERR_INVALID_ARG;
  if ((features == nullptr) != (features_out == nullptr) || (features && F <= 0))
    return EAGLE_ERR_INVALID_ARG;
  const size_t es = dtype == EAGLE_BF16 ? 2 : 4;
  const size_t row_bytes = (size_t)Hkv * D * es, feat_bytes = features ? (size_t)F * es : 16;
  if (max_depth > 64 || row_bytes % 16 || feat_bytes % 16 || B > 65535 || num_pages > (1 << 26))
    return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (features && (!aligned16(features) || !aligned16(features_out))))
    return EAGLE_ERR_INVALID_ARG;
  launch(tree_commit_kernel, B, kCommitThreads, 0, static_cast<cudaStream_t>(stream), R, max_depth,
         (int)(row_bytes / 16), (const uint4*)k_tree, (const uint4*)v_tree, path_rows, accept_len,
         (uint4*)k_cache, (uint4*)v_cache, num_pages, block_table, max_pages, ctx_lens,
         (const uint4*)features, (int)(feat_bytes / 16), (uint4*)features_out, dev_status);
  note_launch();
  return last_launch_status();
}
