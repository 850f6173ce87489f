// spec_verify_attn: multi-row, tree-masked, paged GQA attention of the
// verify step, as split-K flash-decoding partials plus a log-sum-exp combine.
//
// What is computed ("Drafters and Speculative Decoding", section "From a
// proposed block to a causal target pass"; "Speculative Decoding" (atlas),
// "Chains, trees and visibility"): for sequence b, query head h and block row
// i, attention over the cache positions visible to row i: all committed
// positions [0, ctx) and block position ctx + j iff bit j of anc_mask[b,i].
// "Speculative Token Decoupling: Asynchronous Verification via
// Flash-Decoding" (section 03) names split-K attention for this pass: every
// (sequence, KV head) splits its keys into chunks, each chunk yields an
// unnormalised softmax partial with its log-sum-exp, and a combine rescales
// the partials by exp(lse_s - max lse).
//
// GB300 design.  One CTA per (chunk, KV head x row tile, sequence).  All
// R*G query rows of a KV head (G = Hq/Hkv) share each K/V tile, so the KV
// stream -- the bytes that bound this step -- is read once.  A producer warp
// streams 64-token K/V stages with TMA (128-byte swizzle, one 16-token box
// per page segment) through a 4-deep mbarrier ring; eight consumer warps run
// QK^T and PV on the tensor cores (bf16 in, fp32 accumulate) with the
// online softmax in registers.  Warps are (row group of 16) x (token group);
// token groups take alternate stages and merge through shared memory at
// the end.  An fp32 CUDA-core kernel serves fp32 caches.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kStageTokens = 64;
constexpr int kStageBytes = 4 * 8192;  // K lo/hi + V lo/hi, 64 tokens x 128 B each
constexpr int kNumStages = 4;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kQStride = 136;  // bf16 per Q row in shared memory (272 B: conflict-free ldmatrix)
constexpr int kMaxChunk = 4096;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const __nv_bfloat16* q;  // [B,R,Hq,D]
  const float* qf;         // fp32 path
  const float* kf;
  const float* vf;
  const int32_t* block_table;
  const int32_t* ctx_len;
  const uint64_t* anc_mask;
  float* o_part;    // [B,Hkv,RGpad,S,D]
  float* lse_part;  // [B,Hkv,RGpad,S]   (log2 domain)
  int32_t* err;
  int B, R, Hq, Hkv, G, D, page_size, max_pages, num_pages;
  int RG, RGpad, row_tiles, chunk, S;
  float scale_log2;
};

// ------------------------------------------------------------------ bf16 tensor-core kernel
template <int NRG>
__global__ void __launch_bounds__(kThreads, 1)
    attn_partial_bf16(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  constexpr int NTG = kConsumerWarps / NRG;
  constexpr int RT = 16 * NRG;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;                                                  // kNumStages * 32 KB
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + kNumStages * kStageBytes);
  int32_t* bt_s = reinterpret_cast<int32_t*>(qs + RT * kQStride);          // chunk/16 + 1
  uint64_t* full = reinterpret_cast<uint64_t*>(bt_s + kMaxChunk / 16 + 8);
  uint64_t* empty = full + kNumStages;

  const int s = blockIdx.x;
  const int kvh = blockIdx.y % p.Hkv;
  const int rt = blockIdx.y / p.Hkv;
  const int b = blockIdx.z;
  const int ctx = p.ctx_len[b];
  const int kv_len = ctx + p.R;
  const int c0 = s * p.chunk;
  if (c0 >= kv_len) return;  // this sequence needs fewer chunks
  const int c1 = min(c0 + p.chunk, kv_len);
  const int nst = (c1 - c0 + kStageTokens - 1) / kStageTokens;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NRG);
    }
    fence_mbar_init();
  }
  // Q tile: row rho = i*G + g of this KV head -> q[b, i, kvh*G + g, :]
  for (int idx = threadIdx.x; idx < RT * 16; idx += kThreads) {
    const int r = idx >> 4, c = idx & 15;
    const int rho = rt * RT + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (rho < p.RG) {
      const int i = rho / p.G, g = rho % p.G;
      const size_t off = (((size_t)b * p.R + i) * p.Hq + (size_t)kvh * p.G + g) * 128 + c * 8;
      v = *reinterpret_cast<const uint4*>(p.q + off);
    }
    *reinterpret_cast<uint4*>(qs + r * kQStride + c * 8) = v;
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp: block-table slice, then TMA stages
    const int P = p.page_size;
    const int pg0 = c0 / P;
    const int npg = (c1 - 1) / P - pg0 + 1;
    // entries past the table width (a caller error) read as -1: such tokens
    // load as TMA out-of-bounds zeros instead of touching foreign memory
    for (int i = lane; i < npg; i += 32)
      bt_s[i] = (pg0 + i < p.max_pages) ? p.block_table[(size_t)b * p.max_pages + pg0 + i] : -1;
    __syncwarp();
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      for (int k = 0; k < nst; ++k) {
        const int slot = k % kNumStages;
        if (k >= kNumStages) {
          if (!mbar_wait(&empty[slot], ((k / kNumStages) - 1) & 1, p.err)) break;
        }
        uint8_t* st = stages + slot * kStageBytes;
        mbar_arrive_expect_tx(&full[slot], kStageBytes);
        const int t0 = c0 + k * kStageTokens;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int t = t0 + 16 * g;
          int y = -16;  // fully out of bounds: TMA fills zeros
          if (t < kv_len) {
            const int pg = bt_s[t / P - pg0];
            if (pg >= 0 && pg < p.num_pages) y = pg * P + (t % P);
          }
          tma_load_3d(st + 0 * 8192 + g * 2048, &kmap, &full[slot], 0, kvh, y);
          tma_load_3d(st + 1 * 8192 + g * 2048, &kmap, &full[slot], 64, kvh, y);
          tma_load_3d(st + 2 * 8192 + g * 2048, &vmap, &full[slot], 0, kvh, y);
          tma_load_3d(st + 3 * 8192 + g * 2048, &vmap, &full[slot], 64, kvh, y);
        }
      }
    }
    return;
  }

  // ---------------- consumer warps
  const int rg = warp % NRG;
  const int tg = warp / NRG;
  const int r0 = lane >> 2;           // accumulator rows r0 and r0 + 8
  const int cq = 2 * (lane & 3);      // accumulator column pair
  const int rho0 = rt * RT + rg * 16 + r0;
  const int rho1 = rho0 + 8;
  const bool v0 = rho0 < p.RG, v1 = rho1 < p.RG;
  const uint64_t w0 = v0 ? p.anc_mask[(size_t)b * p.R + rho0 / p.G] : 0ull;
  const uint64_t w1 = v1 ? p.anc_mask[(size_t)b * p.R + rho1 / p.G] : 0ull;

  const uint32_t q_base = smem_u32(qs);
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  bool ok = true;

  for (int k = tg; k < nst && ok; k += NTG) {
    const int slot = k % kNumStages;
    if (!mbar_wait(&full[slot], (k / kNumStages) & 1, p.err)) {
      ok = false;
      break;
    }
    const uint32_t st = smem_u32(stages + slot * kStageBytes);
    const int tb = c0 + k * kStageTokens;

    // ---- S = Q K^T for 16 rows x 64 tokens
    float sacc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      {
        const int m = lane >> 3, r = lane & 7;
        const int row = rg * 16 + r + 8 * (m & 1);
        const int chunk = 2 * ks + (m >> 1);
        ldmatrix_x4(a[0], a[1], a[2], a[3], q_base + row * (kQStride * 2) + chunk * 16);
      }
      const uint32_t kb = st + (ks >> 2) * 8192;
      const int cbase = (2 * ks) & 7;
#pragma unroll
      for (int ntp = 0; ntp < 4; ++ntp) {
        const int m = lane >> 3, r = lane & 7;
        const int tok = 8 * (2 * ntp + (m >> 1)) + r;
        const int chunk = cbase + (m & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3, kb + tok * 128 + ((chunk ^ (tok & 7)) << 4));
        mma_bf16_16816(sacc[2 * ntp], a, b0, b1);
        mma_bf16_16816(sacc[2 * ntp + 1], a, b2, b3);
      }
    }

    // ---- scale, visibility mask, online softmax (log2 domain)
    const bool need_mask = tb + kStageTokens > ctx;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = sacc[nt][e] * p.scale_log2;
        if (need_mask) {
          const int pos = tb + nt * 8 + cq + (e & 1);
          const uint64_t w = (e < 2) ? w0 : w1;
          const int j = pos - ctx;
          const bool vis = (pos < ctx) || (j < p.R && ((w >> j) & 1ull));
          if (!vis) x = -INFINITY;
        }
        sacc[nt][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    }
    float base[2], alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mnew = fmaxf(m_run[h], mx[h]);
      base[h] = (mnew == -INFINITY) ? 0.f : mnew;
      alpha[h] = fast_exp2(m_run[h] - base[h]);  // exp2(-inf) = 0 on the first stage
      m_run[h] = mnew;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pe = fast_exp2(sacc[nt][e] - base[e >> 1]);
        sacc[nt][e] = pe;
        rs[e >> 1] += pe;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + rs[h];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }

    // ---- rows of V past the end of the sequence may hold stale cache
    // contents; zero them so that 0 * garbage cannot produce NaN.
    const uint32_t vb = st + 2 * 8192;
    if (tb + kStageTokens > kv_len) {
      const int first = max(kv_len - tb, 0);
      for (int idx = lane; idx < (kStageTokens - first) * 16; idx += 32) {
        const int tok = first + (idx >> 4), ch = idx & 15;
        const uint32_t addr = vb + (ch >> 3) * 8192 + tok * 128 + ((ch & 7) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
      }
      __syncwarp();
    }

    // ---- O += P V
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t a[4];
      a[0] = pack_bf16(sacc[2 * j][0], sacc[2 * j][1]);
      a[1] = pack_bf16(sacc[2 * j][2], sacc[2 * j][3]);
      a[2] = pack_bf16(sacc[2 * j + 1][0], sacc[2 * j + 1][1]);
      a[3] = pack_bf16(sacc[2 * j + 1][2], sacc[2 * j + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int c = 2 * dp;
        const int m = lane >> 3, r = lane & 7;
        const int tok = 16 * j + 8 * (m & 1) + r;
        const int chunk = (c & 7) + (m >> 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(b0, b1, b2, b3,
                          vb + (c >> 3) * 8192 + tok * 128 + ((chunk ^ (tok & 7)) << 4));
        mma_bf16_16816(o[c], a, b0, b1);
        mma_bf16_16816(o[c + 1], a, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  // ---------------- merge token groups through shared memory, write partials
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");  // stages are free
  float* scr = reinterpret_cast<float*>(stages);        // [NTG][RT][128]
  float* ml = scr + NTG * RT * 128;                     // [NTG][RT][2]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  {
    const int ra = rg * 16 + r0;
    float* dst = scr + (size_t)(tg * RT) * 128;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      *reinterpret_cast<float2*>(dst + ra * 128 + 8 * c + cq) = make_float2(o[c][0], o[c][1]);
      *reinterpret_cast<float2*>(dst + (ra + 8) * 128 + 8 * c + cq) = make_float2(o[c][2], o[c][3]);
    }
    if ((lane & 3) == 0) {
      ml[(tg * RT + ra) * 2 + 0] = m_run[0];
      ml[(tg * RT + ra) * 2 + 1] = l_run[0];
      ml[(tg * RT + ra + 8) * 2 + 0] = m_run[1];
      ml[(tg * RT + ra + 8) * 2 + 1] = l_run[1];
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
  for (int r = warp; r < RT; r += kConsumerWarps) {
    const int rho = rt * RT + r;
    if (rho >= p.RG) break;
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < NTG; ++t) M = fmaxf(M, ml[(t * RT + r) * 2]);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < NTG; ++t) {
      const float mt = ml[(t * RT + r) * 2];
      const float e = (mt == -INFINITY) ? 0.f : fast_exp2(mt - M);
      L += e * ml[(t * RT + r) * 2 + 1];
      const float4 v = *reinterpret_cast<const float4*>(scr + (size_t)(t * RT + r) * 128 + 4 * lane);
      acc.x += e * v.x;
      acc.y += e * v.y;
      acc.z += e * v.z;
      acc.w += e * v.w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    const size_t prow = (((size_t)b * p.Hkv + kvh) * p.RGpad + rho) * p.S + s;
    *reinterpret_cast<float4*>(p.o_part + prow * 128 + 4 * lane) = acc;
    if (lane == 0) p.lse_part[prow] = L > 0.f ? M + __log2f(L) : -INFINITY;
  }
}

// ------------------------------------------------------------------ fp32 CUDA-core kernel
// One warp per query row; lanes split the keys 32 at a time, each lane owns
// D/32 output dimensions.  Used for fp32 caches (small shapes).
__global__ void __launch_bounds__(128) attn_partial_f32(const AttnParams p) {
  const int s = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int ctx = p.ctx_len[b];
  const int kv_len = ctx + p.R;
  const int c0 = s * p.chunk;
  if (c0 >= kv_len) return;
  const int c1 = min(c0 + p.chunk, kv_len);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = p.D;
  const int nd = D / 32;
  const int P = p.page_size;
  for (int rho = warp; rho < p.RG; rho += 4) {
    const int i = rho / p.G, g = rho % p.G;
    const float* qrow = p.qf + (((size_t)b * p.R + i) * p.Hq + (size_t)kvh * p.G + g) * D;
    const uint64_t w = p.anc_mask[(size_t)b * p.R + i];
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    float m_run = -INFINITY, l_run = 0.f;
    for (int t0 = c0; t0 < c1; t0 += 32) {
      const int t = t0 + lane;
      float x = -INFINITY;
      size_t roff = 0;
      if (t < c1) {
        const int j = t - ctx;
        const bool vis = (t < ctx) || (j < p.R && ((w >> j) & 1ull));
        const int page = (t / P < p.max_pages) ? p.block_table[(size_t)b * p.max_pages + t / P] : -1;
        const bool pg_ok = page >= 0 && page < p.num_pages;
        roff = pg_ok ? (((size_t)page * P + (t % P)) * p.Hkv + kvh) * D : 0;
        if (vis && pg_ok) {
          float dot = 0.f;
          for (int d = 0; d < D; ++d) dot = fmaf(qrow[d], p.kf[roff + d], dot);
          x = dot * p.scale_log2;
        }
      }
      const float mx = warp_max(x);
      const float mnew = fmaxf(m_run, mx);
      const float base = (mnew == -INFINITY) ? 0.f : mnew;
      const float alpha = fast_exp2(m_run - base);
      const float pe = fast_exp2(x - base);
      l_run = l_run * alpha + warp_sum(pe);
      m_run = mnew;
      for (int c = 0; c < nd; ++c) o[c] *= alpha;
      const int nvalid = min(32, c1 - t0);
      for (int jj = 0; jj < nvalid; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, pe, jj);
        const size_t rj = __shfl_sync(0xffffffffu, roff, jj);
        if (pj != 0.f)
          for (int c = 0; c < nd; ++c) o[c] = fmaf(pj, p.vf[rj + lane + 32 * c], o[c]);
      }
    }
    const size_t prow = (((size_t)b * p.Hkv + kvh) * p.RGpad + rho) * p.S + s;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    for (int c = 0; c < nd; ++c) p.o_part[prow * D + lane + 32 * c] = o[c] * inv;
    if (lane == 0) p.lse_part[prow] = l_run > 0.f ? m_run + __log2f(l_run) : -INFINITY;
  }
}

// ------------------------------------------------------------------ LSE combine
// out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M), one warp per output row.
template <typename OutT>
__global__ void __launch_bounds__(128) attn_combine(const AttnParams p, OutT* __restrict__ out,
                                                   float* __restrict__ lse_out) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int total = p.B * p.R * p.Hq;
  if (gw >= total) return;
  const int hq = gw % p.Hq;
  const int i = (gw / p.Hq) % p.R;
  const int b = gw / (p.Hq * p.R);
  const int kvh = hq / p.G, g = hq % p.G;
  const int rho = i * p.G + g;
  const int kv_len = p.ctx_len[b] + p.R;
  const int ns = min(p.S, (kv_len + p.chunk - 1) / p.chunk);
  const size_t prow0 = (((size_t)b * p.Hkv + kvh) * p.RGpad + rho) * p.S;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, p.lse_part[prow0 + s]);
  M = warp_max(M);
  const int D = p.D;
  const int nv = D / 128 == 1 ? 1 : 0;  // D == 128: float4 per lane; D == 64: float2
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float L = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float ls = p.lse_part[prow0 + s];
    const float e = (ls == -INFINITY) ? 0.f : fast_exp2(ls - M);
    L += e;
    const float* src = p.o_part + (prow0 + s) * D;
    if (nv) {
      const float4 v = *reinterpret_cast<const float4*>(src + 4 * lane);
      acc[0] += e * v.x;
      acc[1] += e * v.y;
      acc[2] += e * v.z;
      acc[3] += e * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src + 2 * lane);
      acc[0] += e * v.x;
      acc[1] += e * v.y;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  OutT* dst = out + (((size_t)b * p.R + i) * p.Hq + hq) * D;
  const int per = nv ? 4 : 2;
  for (int c = 0; c < per; ++c) {
    const float v = acc[c] * inv;
    if constexpr (sizeof(OutT) == 2)
      dst[per * lane + c] = __float2bfloat16_rn(v);
    else
      dst[per * lane + c] = v;
  }
  if (lse_out && lane == 0)
    lse_out[((size_t)b * p.R + i) * p.Hq + hq] =
        (L > 0.f) ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

struct Plan {
  int G, RG, NRG, RT, row_tiles, RGpad, chunk, S;
  bool tc;  // tensor-core path
};

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

bool make_plan(int B, int R, int Hq, int Hkv, int D, int page_size, int max_pages, int num_splits,
               bool bf16, Plan* pl) {
  if (B < 1 || R < 1 || R > 64 || Hq < 1 || Hkv < 1 || Hq % Hkv || page_size < 1 || max_pages < 1)
    return false;
  pl->tc = bf16;
  pl->G = Hq / Hkv;
  pl->RG = R * pl->G;
  if (bf16) {
    pl->NRG = pl->RG <= 16 ? 1 : pl->RG <= 32 ? 2 : pl->RG <= 64 ? 4 : 8;
    pl->RT = 16 * pl->NRG;
    pl->row_tiles = (pl->RG + pl->RT - 1) / pl->RT;
    pl->RGpad = pl->row_tiles * pl->RT;
  } else {
    pl->NRG = 0;
    pl->RT = pl->RG;
    pl->row_tiles = 1;
    pl->RGpad = pl->RG;
  }
  const long long max_kv = (long long)max_pages * page_size;
  const int units = B * Hkv * pl->row_tiles;
  int chunk;
  if (num_splits > 0) {
    chunk = (int)((max_kv + num_splits - 1) / num_splits);
    chunk = chunk >= 128 ? chunk / kStageTokens * kStageTokens : round_up(chunk, kStageTokens);
  } else {
    const int sms = num_sms();
    if (units >= sms) {
      chunk = 2048;
    } else {
      const int S = std::max(1, sms / units);
      chunk = round_up((int)((max_kv + S - 1) / S), kStageTokens);
      if (chunk > 2048) chunk = 2048;
    }
  }
  chunk = std::max(kStageTokens, std::min(chunk, kMaxChunk));
  pl->chunk = chunk;
  pl->S = (int)((max_kv + chunk - 1) / chunk);
  return true;
}

size_t ws_layout(const Plan& pl, int B, int Hkv, int D, size_t* off_o, size_t* off_lse) {
  const size_t rows = (size_t)B * Hkv * pl.RGpad * pl.S;
  size_t off = sizeof(WsHeader);
  *off_o = off;
  off += (rows * D * sizeof(float) + 255) / 256 * 256;
  *off_lse = off;
  off += (rows * sizeof(float) + 255) / 256 * 256;
  return off;
}

size_t smem_bytes_bf16(int NRG) {
  return 1024 + (size_t)kNumStages * kStageBytes + (size_t)16 * NRG * kQStride * 2 +
         (kMaxChunk / 16 + 8) * 4 + 2 * kNumStages * 8;
}

template <int NRG>
spec_status launch_bf16(const CUtensorMap& km, const CUtensorMap& vm, const AttnParams& prm,
                        const Plan& pl, cudaStream_t st) {
  const size_t smem = smem_bytes_bf16(NRG);
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_partial_bf16<NRG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return SPEC_ECUDA;
    attr_set = true;
  }
  dim3 grid(pl.S, prm.Hkv * pl.row_tiles, prm.B);
  attn_partial_bf16<NRG><<<grid, kThreads, smem, st>>>(km, vm, prm);
  return launch_status();
}

}  // namespace

extern "C" size_t spec_verify_attn_workspace_size(int B, int R, int Hq, int Hkv, int D,
                                                  int page_size, int max_pages, int num_splits) {
  Plan pl;
  // size for the larger of the two layouts so one workspace serves both dtypes
  size_t best = 0;
  for (int bf = 0; bf < 2; ++bf) {
    if (!make_plan(B, R, Hq, Hkv, D, page_size, max_pages, num_splits, bf != 0, &pl)) return 0;
    size_t a, c;
    best = std::max(best, ws_layout(pl, B, Hkv, D, &a, &c));
  }
  return best;
}

extern "C" int spec_verify_attn_num_splits(int B, int R, int Hq, int Hkv, int D, int page_size,
                                           int max_pages, int num_splits) {
  Plan pl;
  if (!make_plan(B, R, Hq, Hkv, D, page_size, max_pages, num_splits, true, &pl)) return 0;
  return pl.S;
}

namespace {

enum Phase { kPartials = 1, kCombine = 2, kBoth = 3 };

spec_status verify_attn_impl(const void* q, const void* k_cache, const void* v_cache,
                             spec_dtype dtype, int page_size, int num_pages,
                             const int32_t* block_table, int max_pages, const int32_t* ctx_len,
                             const uint64_t* anc_mask, int B, int R, int Hq, int Hkv, int D,
                             float scale, int num_splits, void* workspace, size_t workspace_bytes,
                             void* out, float* lse_out, void* stream, int phase) {
  if (!ctx_len || !workspace) return SPEC_EINVAL;
  if ((phase & kPartials) && (!q || !k_cache || !v_cache || !block_table || !anc_mask))
    return SPEC_EINVAL;
  if ((phase & kCombine) && !out) return SPEC_EINVAL;
  if (B < 0 || R < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || page_size < 1 || num_pages < 1 ||
      max_pages < 1 || num_splits < 0)
    return SPEC_EINVAL;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (R > 64 || (D != 64 && D != 128)) return SPEC_EUNSUPPORTED;
  const bool bf16 = dtype == SPEC_BF16;
  if (bf16 && (D != 128 || page_size % 16 != 0 || R * (Hq / Hkv) > 512)) return SPEC_EUNSUPPORTED;
  if ((phase & kPartials) && bf16 &&
      ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
        reinterpret_cast<uintptr_t>(q)) & 15))
    return SPEC_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return SPEC_EINVAL;
  Plan pl;
  if (!make_plan(B, R, Hq, Hkv, D, page_size, max_pages, num_splits, bf16, &pl)) return SPEC_EINVAL;
  size_t off_o, off_lse;
  const size_t need = ws_layout(pl, B, Hkv, D, &off_o, &off_lse);
  if (workspace_bytes < need) return SPEC_EINVAL;

  AttnParams prm{};
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.qf = static_cast<const float*>(q);
  prm.kf = static_cast<const float*>(k_cache);
  prm.vf = static_cast<const float*>(v_cache);
  prm.block_table = block_table;
  prm.ctx_len = ctx_len;
  prm.anc_mask = anc_mask;
  prm.o_part = reinterpret_cast<float*>(ws + off_o);
  prm.lse_part = reinterpret_cast<float*>(ws + off_lse);
  prm.err = reinterpret_cast<int32_t*>(ws);
  prm.B = B;
  prm.R = R;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = pl.G;
  prm.D = D;
  prm.page_size = page_size;
  prm.max_pages = max_pages;
  prm.num_pages = num_pages;
  prm.RG = pl.RG;
  prm.RGpad = pl.RGpad;
  prm.row_tiles = pl.row_tiles;
  prm.chunk = pl.chunk;
  prm.S = pl.S;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  prm.scale_log2 = sc * kLog2e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (phase & kPartials) {
    spec_status rc;
    if (bf16) {
      EncodeTiledFn enc = get_encode();
      if (!enc) return SPEC_ECUDA;
      CUtensorMap km, vm;
      const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv,
                                  (cuuint64_t)num_pages * page_size};
      const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
      const cuuint32_t box[3] = {64, 1, 16};
      const cuuint32_t estr[3] = {1, 1, 1};
      if (enc(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k_cache), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SPEC_ECUDA;
      if (enc(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v_cache), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SPEC_ECUDA;
      switch (pl.NRG) {
        case 1: rc = launch_bf16<1>(km, vm, prm, pl, st); break;
        case 2: rc = launch_bf16<2>(km, vm, prm, pl, st); break;
        case 4: rc = launch_bf16<4>(km, vm, prm, pl, st); break;
        default: rc = launch_bf16<8>(km, vm, prm, pl, st); break;
      }
    } else {
      dim3 grid(pl.S, Hkv, B);
      attn_partial_f32<<<grid, 128, 0, st>>>(prm);
      rc = launch_status();
    }
    if (rc != SPEC_OK) return rc;
  }
  if (phase & kCombine) {
    const int rows = B * R * Hq;
    const int blocks = (rows * 32 + 127) / 128;
    if (bf16)
      attn_combine<__nv_bfloat16><<<blocks, 128, 0, st>>>(prm, static_cast<__nv_bfloat16*>(out),
                                                          lse_out);
    else
      attn_combine<float><<<blocks, 128, 0, st>>>(prm, static_cast<float*>(out), lse_out);
    return launch_status();
  }
  return SPEC_OK;
}

}  // namespace

#define SPEC_ATTN_ARGS                                                                          \
  const void *q, const void *k_cache, const void *v_cache, spec_dtype dtype, int page_size,     \
      int num_pages, const int32_t *block_table, int max_pages, const int32_t *ctx_len,         \
      const uint64_t *anc_mask, int B, int R, int Hq, int Hkv, int D, float scale,              \
      int num_splits, void *workspace, size_t workspace_bytes
#define SPEC_ATTN_FWD                                                                        \
  q, k_cache, v_cache, dtype, page_size, num_pages, block_table, max_pages, ctx_len, anc_mask, \
      B, R, Hq, Hkv, D, scale, num_splits, workspace, workspace_bytes

extern "C" spec_status spec_verify_attn(SPEC_ATTN_ARGS, void* out, float* lse_out, void* stream) {
  return verify_attn_impl(SPEC_ATTN_FWD, out, lse_out, stream, kBoth);
}

extern "C" spec_status spec_verify_attn_partials(SPEC_ATTN_ARGS, void* stream) {
  return verify_attn_impl(SPEC_ATTN_FWD, nullptr, nullptr, stream, kPartials);
}

extern "C" spec_status spec_verify_attn_combine(SPEC_ATTN_ARGS, void* out, float* lse_out,
                                                void* stream) {
  return verify_attn_impl(SPEC_ATTN_FWD, out, lse_out, stream, kCombine);
}

// ------------------------------------------------------------------ allocation-free variant
// spec_verify_attn_noalloc runs exactly the work of spec_verify_attn, but its
// split-K partials live in a fixed array compiled into this library instead
// of a caller-provided workspace.  It exists for callers that cannot make a
// device allocation at the point where they call us -- for example a host
// that only hands a plugin its input and output buffers, or a serving loop
// whose memory budget is frozen after start-up.  The array is reserved on
// every GPU that loads the library and stays there until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress, with that device current);
// later calls reuse the cached address.  No memory is allocated.
spec_status noalloc_scratch(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ECUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SPEC_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ECUDA;
    g_noalloc_addr[dev] = p;
  }
  *addr = g_noalloc_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_verify_attn_noalloc(const void* q, const void* k_cache,
                                                const void* v_cache, spec_dtype dtype,
                                                int page_size, int num_pages,
                                                const int32_t* block_table, int max_pages,
                                                const int32_t* ctx_len, const uint64_t* anc_mask,
                                                int B, int R, int Hq, int Hkv, int D, float scale,
                                                int num_splits, void* out, float* lse_out,
                                                void* stream) {
  if (B < 0) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  const size_t need = spec_verify_attn_workspace_size(B, R, Hq, Hkv, D, page_size, max_pages,
                                                      num_splits);
  if (need == 0) return SPEC_EINVAL;
  if (need > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_EUNSUPPORTED;  // too big for the array
  void* scratch = nullptr;
  const spec_status rs = noalloc_scratch(&scratch);
  if (rs != SPEC_OK) return rs;
  // the error word at the head of the scratch must start at zero on every call
  if (cudaMemsetAsync(scratch, 0, sizeof(WsHeader), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return SPEC_ECUDA;
  return verify_attn_impl(q, k_cache, v_cache, dtype, page_size, num_pages, block_table,
                          max_pages, ctx_len, anc_mask, B, R, Hq, Hkv, D, scale, num_splits,
                          scratch, SPEC_NOALLOC_SCRATCH_BYTES, out, lse_out, stream, kBoth);
}
