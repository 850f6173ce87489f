// spec_kv_commit: the processed length after acceptance and, for a draft
// tree, the accepted path's K/V rows compacted into the next logical prefix.
// "Speculative Decoding" (atlas), sections "Committed tokens versus cached
// states" and "Chains, trees and visibility".
//
// One CTA per (sequence, KV head).  Thread 0 checks the sequence (accepted
// length, that every path node is a later node than the one before it -- and
// its child when the parent array is given --, every page index it will
// touch); then the CTA reads every 16-byte chunk of its head's moving rows
// (K and V) into shared memory and writes them at their new positions: a row
// may move into the slot of a later path node, so no write starts before all
// reads are done.  The path is the tree sampler's output as it stands: the
// accepted nodes in order, node 0 (the anchor, which stays at position ctx)
// implied, so the sampler's outputs feed this call with no host step.
#include "common.cuh"

namespace {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(
    char* __restrict__ k_cache, char* __restrict__ v_cache, int esz, int num_pages, int P,
    int Hkv, int D, const int32_t* __restrict__ block_table, int max_pages,
    const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ accepted_len,
    const int32_t* __restrict__ path, const int32_t* __restrict__ parent, int R,
    int32_t* __restrict__ new_len, int32_t* __restrict__ keep_pages,
    int32_t* __restrict__ status) {
  extern __shared__ __align__(16) uint4 rows[];
  __shared__ int ok;
  const int b = blockIdx.x / Hkv, h = blockIdx.x % Hkv;
  const int c = ctx_len[b];
  const int a = accepted_len[b];
  const int32_t* bt = block_table + (size_t)b * max_pages;
  const int32_t* pth = path ? path + (size_t)b * R : nullptr;
  const int32_t* par = parent ? parent + (size_t)b * R : nullptr;
  if (threadIdx.x == 0) {
    bool good = c >= 0 && a >= 0 && a < R && (long long)c + R <= (long long)max_pages * P;
    if (good && pth) {
      int prev = 0;  // the anchor
      for (int k = 0; k < a && good; ++k) {
        const int v = pth[k];
        good = v > prev && v < R && (!par || par[v] == prev);
        prev = v;
        if (good) {  // the source row (position c + v) and the destination (c + k + 1)
          const int ps = bt[(c + v) / P], pd = bt[(c + k + 1) / P];
          good = ps >= 0 && ps < num_pages && pd >= 0 && pd < num_pages;
        }
      }
    }
    ok = good ? 1 : 0;
    if (h == 0) {
      const int n = good ? c + 1 + a : c;
      new_len[b] = n;
      if (keep_pages) keep_pages[b] = (n + P - 1) / P;
      if (status) status[b] = good ? 0 : SPEC_SEQ_BAD_TREE;
    }
  }
  __syncthreads();
  if (!ok || !pth) return;
  const int cpr = D * esz / 16;  // 16-byte chunks per row of one head
  const int n = a * 2 * cpr;     // path nodes 1..a move; node 0 stays
  auto addr = [&](int kv, int pos, int ch) {
    const size_t row = ((size_t)bt[pos / P] * P + pos % P) * Hkv + h;
    return (kv ? v_cache : k_cache) + row * (size_t)D * esz + (size_t)ch * 16;
  };
  for (int i = threadIdx.x; i < n; i += kCommitThreads) {
    const int k = i / (2 * cpr), r = i % (2 * cpr);
    rows[i] = *reinterpret_cast<const uint4*>(addr(r / cpr, c + pth[k], r % cpr));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kCommitThreads) {
    const int k = i / (2 * cpr), r = i % (2 * cpr);
    *reinterpret_cast<uint4*>(addr(r / cpr, c + k + 1, r % cpr)) = rows[i];
  }
}

}  // namespace

extern "C" spec_status spec_kv_commit(void* k_cache, void* v_cache, int elem_bytes, int num_pages,
                                      int page_size, int Hkv, int D, const int32_t* block_table,
                                      int max_pages, const int32_t* ctx_len,
                                      const int32_t* accepted_len, const int32_t* path,
                                      const int32_t* parent, int B, int R, int32_t* new_len,
                                      int32_t* keep_pages,
                                      int32_t* status_per_seq, void* stream) {
  if (B < 0 || R < 1 || R > 64 || !ctx_len || !accepted_len || !new_len || !block_table)
    return SPEC_EINVAL;
  if (parent && !path) return SPEC_EINVAL;
  if (!k_cache || !v_cache || num_pages < 1 || page_size < 1 || Hkv < 1 || max_pages < 1)
    return SPEC_EINVAL;
  if ((elem_bytes != 2 && elem_bytes != 4) || (D != 64 && D != 128)) return SPEC_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  const size_t smem = (size_t)(R - 1) * 2 * (D * elem_bytes / 16) * 16;  // < 64 KB
  static PerDeviceOnce<int> smem_once;  // once per device, at the largest size
  const spec_status ra =
      ensure_smem_limit(smem_once, (const void*)kv_commit_kernel, 64 * 2 * (128 * 4 / 16) * 16);
  if (ra != SPEC_OK) return ra;
  kv_commit_kernel<<<B * Hkv, kCommitThreads, smem, (cudaStream_t)stream>>>(
      static_cast<char*>(k_cache), static_cast<char*>(v_cache), elem_bytes, num_pages, page_size,
      Hkv, D, block_table, max_pages, ctx_len, accepted_len, path, parent, R, new_len, keep_pages,
      status_per_seq);
  return launch_status();
}
