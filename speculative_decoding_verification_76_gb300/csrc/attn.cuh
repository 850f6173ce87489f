// Definitions shared by the verify-attention kernels (attn.cu: the warp-MMA
// partial pass, the fp32 path, the combine and the host entry points;
// attn_tc.cu: the tcgen05 partial pass).
#pragma once
#include "common.cuh"

namespace attn {

constexpr int kStageTokens = 64;  // granularity of chunks
constexpr int kMaxChunk = 4096;   // longest chunk: the page-table slice one CTA stages
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const __nv_bfloat16* q;  // [B,R,Hq,D]
  const float* qf;         // fp32 path
  const float* kf;
  const float* vf;
  const void* k;  // bf16 caches
  const void* v;
  const int32_t* block_table;
  const int32_t* ctx_len;
  const uint64_t* anc_mask;
  float* o_part;    // [B,Hkv,RGpad,S,D]
  float* lse_part;  // [B,Hkv,RGpad,S]   (log2 domain)
  int32_t* err;
  int B, R, Hq, Hkv, G, D, page_size, max_pages, num_pages;
  int RG, RGpad, row_tiles, chunk, S;
  float scale_log2;
  uint64_t wait_ns;    // bound of every device wait (SPEC_WAIT_NS unless a test lowers it)
  int withhold_stage;  // -1; a test sets a K/V stage whose arrival the copy warps withhold
};

// The visibility word of block row i of sequence b: the caller's ancestor mask,
// or for a chain (no mask given) rows 0 .. i.
SPEC_DEV uint64_t row_mask(const AttnParams& p, int b, int i) {
  if (p.anc_mask) return p.anc_mask[(size_t)b * p.R + i];
  return i >= 63 ? ~0ull : ((2ull << i) - 1ull);
}

// The tcgen05 partial pass: rows_per_cta (128 or 256) query rows of one KV head
// per CTA, 128-token stages, grid (Hkv * row_tiles, S, B).  Defined in
// attn_tc.cu.
constexpr int kTcRows = 128;
constexpr int kTcStageTokens = 128;
spec_status launch_partial_tc(const AttnParams& prm, int rows_per_cta, cudaStream_t st);

}  // namespace attn
