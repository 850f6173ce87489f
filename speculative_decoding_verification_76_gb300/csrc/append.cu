// The two steps in front of the verify calls that the pages require of the
// block's inputs (row f3 of the hot path):
//
//  spec_append_block -- the proposed block's K/V rows written into the paged
//    cache, row j at position ctx_len + j (where the verify attention reads
//    it), the key rotated for the row's position id: "Speculative Decoding"
//    (atlas), "Chains, trees and visibility": position ids follow depth, not
//    flattened storage order.  The rotation is the split-half rotary form
//    (pair (x_i, x_{i + D/2}) rotated by pos * base^(-2i/D)); the block's
//    queries may be rotated in place at the same positions.  One CTA per block
//    row: the row's D/2 angles are computed once in double precision (a
//    position past 10^5 times an fp32 frequency would lose 10^-2 rad) and
//    reduced before the fp32 sine/cosine; every head then rotates in fp32.
//
//  spec_logits_penalize -- the target logits as served: "Greedy, sampling and
//    the real sampler": p must include token bans and repetition penalties.
//    A repetition penalty theta on every distinct token of the row's prefix
//    (the sequence history plus the block tokens in front of the row: a
//    chain's earlier drafts, a tree node's ancestors and itself): l / theta if
//    l > 0, else l * theta; then -inf on banned ids.  Only those tokens are
//    touched (one CTA per row; a shared-memory bitmap of the vocabulary keeps
//    each distinct id to one update).
#include "common.cuh"

namespace {

constexpr int kAppendThreads = 128;
constexpr int kPenaltyThreads = 256;
constexpr int kMaxVocabWords = 172032 / 32;  // the sampler's largest vocabulary

template <typename T>
SPEC_DEV float ld_el(const T* p) {
  if constexpr (sizeof(T) == 2)
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
  else
    return *reinterpret_cast<const float*>(p);
}

template <typename T>
SPEC_DEV void st_el(T* p, float v) {
  if constexpr (sizeof(T) == 2)
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
  else
    *reinterpret_cast<float*>(p) = v;
}

// rows [nh, D] of one block row: rotate pairs (i, i + D/2) by the row's angles
template <typename T>
SPEC_DEV void rotate_rows(const T* src, T* dst, int nh, int D, const float* cs, const float* sn) {
  const int half = D / 2;
  for (int k = threadIdx.x; k < nh * half; k += kAppendThreads) {
    const int h = k / half, i = k % half;
    const T* x = src + (size_t)h * D;
    const float a = ld_el(x + i), b = ld_el(x + i + half);
    const float c = cs[i], s = sn[i];
    T* y = dst + (size_t)h * D;
    st_el(y + i, a * c - b * s);
    st_el(y + i + half, a * s + b * c);
  }
}

template <typename T>
__global__ void __launch_bounds__(kAppendThreads) append_block_kernel(
    const T* __restrict__ k_new, const T* __restrict__ v_new, T* __restrict__ q, T* k_cache,
    T* v_cache, int num_pages, int P, const int32_t* __restrict__ block_table, int max_pages,
    const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ pos_ids, int R, int Hq,
    int Hkv, int D, double log2_base, int32_t* __restrict__ status) {
  __shared__ float cs[64], sn[64];
  __shared__ int row_ok;
  const int b = blockIdx.x / R, j = blockIdx.x % R;
  const int c = ctx_len[b];
  const int32_t* bt = block_table + (size_t)b * max_pages;
  auto row_valid = [&](int jj) {
    if (c < 0 || (long long)c + R > (long long)max_pages * P) return false;
    const int pg = bt[(c + jj) / P];
    const int pos = pos_ids ? pos_ids[(size_t)b * R + jj] : c + jj;
    return pg >= 0 && pg < num_pages && pos >= 0;
  };
  if (threadIdx.x == 0) {
    // a sequence with any row it cannot write is left untouched as a whole
    bool all = true;
    for (int jj = 0; jj < R; ++jj) all = all && row_valid(jj);
    row_ok = all ? 1 : 0;
    if (j == 0 && status) status[b] = all ? 0 : SPEC_SEQ_BAD_TREE;
  }
  const int half = D / 2;
  if (threadIdx.x < half) {
    const int i = threadIdx.x;
    const int pos = row_valid(j) ? (pos_ids ? pos_ids[(size_t)b * R + j] : c + j) : 0;
    const double theta = exp2(-(2.0 * i / D) * log2_base);
    const double ang = (double)pos * theta;
    const double two_pi = 6.283185307179586476925286766559;
    const double r = ang - two_pi * rint(ang / two_pi);  // |r| <= pi
    double sd, cd;
    sincos(r, &sd, &cd);
    cs[i] = (float)cd;
    sn[i] = (float)sd;
  }
  __syncthreads();
  if (!row_ok) return;
  const int pos_slot = c + j;
  const size_t crow = ((size_t)bt[pos_slot / P] * P + pos_slot % P) * Hkv * D;
  const size_t brow = ((size_t)b * R + j) * (size_t)Hkv * D;
  rotate_rows(k_new + brow, k_cache + crow, Hkv, D, cs, sn);
  for (int k = threadIdx.x; k < Hkv * D; k += kAppendThreads) v_cache[crow + k] = v_new[brow + k];
  if (q) {  // in place: each pair is read and written by the same thread
    T* qr = q + ((size_t)b * R + j) * (size_t)Hq * D;
    rotate_rows(qr, qr, Hq, D, cs, sn);
  }
}

__global__ void __launch_bounds__(kPenaltyThreads) penalize_kernel(
    float* __restrict__ logits, int R, int V, const int32_t* __restrict__ history, int H,
    const int32_t* __restrict__ block_tokens, const int32_t* __restrict__ parent, float penalty,
    const int32_t* __restrict__ banned, int n_banned) {
  __shared__ uint32_t seen[kMaxVocabWords];
  __shared__ int32_t pre[64];
  __shared__ int npre;
  const int b = blockIdx.x / R, i = blockIdx.x % R;
  float* row = logits + ((size_t)b * R + i) * V;
  const int words = (V + 31) / 32;
  for (int k = threadIdx.x; k < words; k += kPenaltyThreads) seen[k] = 0u;
  if (threadIdx.x == 0) {  // the block tokens in front of this row
    int n = 0;
    if (!parent) {
      for (int k = 0; k < i; ++k) pre[n++] = block_tokens[(size_t)b * (R - 1) + k];
    } else {
      const int32_t* par = parent + (size_t)b * R;
      int v = i;
      while (v > 0 && n < 64) {  // a parent that does not precede its node ends the walk
        pre[n++] = block_tokens[(size_t)b * R + v];
        const int pv = par[v];
        v = (pv >= 0 && pv < v) ? pv : 0;
      }
    }
    npre = n;
  }
  __syncthreads();
  if (penalty != 1.f) {
    const int total = H + npre;
    for (int k = threadIdx.x; k < total; k += kPenaltyThreads) {
      const int t = k < H ? history[(size_t)b * H + k] : pre[k - H];
      if (t < 0 || t >= V) continue;
      const uint32_t bit = 1u << (t & 31);
      if (atomicOr(&seen[t >> 5], bit) & bit) continue;  // already penalised
      const float l = row[t];
      row[t] = l > 0.f ? l / penalty : l * penalty;
    }
    __syncthreads();  // bans land after the penalties on the same tokens
  }
  for (int k = threadIdx.x; k < n_banned; k += kPenaltyThreads) {
    const int t = banned[k];
    if (t >= 0 && t < V) row[t] = -INFINITY;
  }
}

}  // namespace

extern "C" spec_status spec_append_block(const void* k_new, const void* v_new, void* q,
                                         spec_dtype dtype, void* k_cache, void* v_cache,
                                         int num_pages, int page_size, const int32_t* block_table,
                                         int max_pages, const int32_t* ctx_len,
                                         const int32_t* pos_ids, int B, int R, int Hq, int Hkv,
                                         int D, float rope_base, int32_t* status_per_seq,
                                         void* stream) {
  if (B < 0 || R < 1 || R > 64 || Hkv < 1 || (q && (Hq < 1 || Hq % Hkv)) || num_pages < 1 ||
      page_size < 1 || max_pages < 1)
    return SPEC_EINVAL;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !ctx_len) return SPEC_EINVAL;
  if (!(rope_base > 1.f)) return SPEC_EINVAL;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_EINVAL;
  if (D != 64 && D != 128) return SPEC_EUNSUPPORTED;
  if (B == 0) return SPEC_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const double lb = log2((double)rope_base);
  if (dtype == SPEC_BF16) {
    using T = __nv_bfloat16;
    append_block_kernel<T><<<B * R, kAppendThreads, 0, st>>>(
        static_cast<const T*>(k_new), static_cast<const T*>(v_new), static_cast<T*>(q),
        static_cast<T*>(k_cache), static_cast<T*>(v_cache), num_pages, page_size, block_table,
        max_pages, ctx_len, pos_ids, R, Hq, Hkv, D, lb, status_per_seq);
  } else {
    append_block_kernel<float><<<B * R, kAppendThreads, 0, st>>>(
        static_cast<const float*>(k_new), static_cast<const float*>(v_new),
        static_cast<float*>(q), static_cast<float*>(k_cache), static_cast<float*>(v_cache),
        num_pages, page_size, block_table, max_pages, ctx_len, pos_ids, R, Hq, Hkv, D, lb,
        status_per_seq);
  }
  return launch_status();
}

extern "C" spec_status spec_logits_penalize(float* logits, int B, int R, int V,
                                            const int32_t* history, int H,
                                            const int32_t* block_tokens, const int32_t* parent,
                                            float penalty, const int32_t* banned, int n_banned,
                                            void* stream) {
  if (B < 0 || R < 1 || R > 64 || V < 1 || H < 0 || n_banned < 0) return SPEC_EINVAL;
  if (!logits || (H > 0 && !history) || (n_banned > 0 && !banned)) return SPEC_EINVAL;
  if (R > 1 && !block_tokens) return SPEC_EINVAL;
  if (!(penalty > 0.f) || penalty != penalty) return SPEC_EINVAL;
  if (V > kMaxVocabWords * 32) return SPEC_EUNSUPPORTED;
  if (B == 0 || (penalty == 1.f && n_banned == 0)) return SPEC_OK;
  penalize_kernel<<<B * R, kPenaltyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      logits, R, V, history, H, block_tokens, parent, penalty, banned, n_banned);
  return launch_status();
}
