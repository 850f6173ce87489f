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
// GB300 design.  Two partial passes share the split plan and the partial
// layout [B, Hkv, RGpad, S, D] (+ log2-domain LSE):
//  * up to 64 query rows per KV head (the chain shapes: R * G = 20 .. 64):
//    attn_partial_bf16 below.  One CTA per (chunk, KV head x row tile,
//    sequence); all R*G rows of a KV head share each K/V tile, so the KV
//    stream -- the bytes that bound these shapes -- is read once.  Four copy
//    warps stream K/V stages with 16-byte cp.async (64 contiguous bytes per
//    thread, one page lookup per token, 128-byte swizzle) into a 3-stage
//    (128-token) or 6-stage (64-token) mbarrier ring; eight MMA warps run
//    QK^T and PV with mma.sync m16n8k16 (bf16 in, fp32 accumulate) and the
//    online softmax in registers.  Warps are (row group of 16) x (token group)
//    and the token groups merge through shared memory at the end.
//  * more than 64 rows per KV head (draft trees, long chains): the tcgen05
//    pass in attn_tc.cu (128-row MMAs, tensor-memory accumulators).
// An fp32 CUDA-core kernel serves fp32 caches.
#include <algorithm>
#include <atomic>

#include "attn.cuh"

namespace {

using attn::AttnParams;
using attn::kLog2e;
using attn::kMaxChunk;
using attn::kStageTokens;

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarps = 4;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kQStride = 136;  // bf16 per Q row in shared memory (272 B: conflict-free ldmatrix)

// ------------------------------------------------------------------ bf16 tensor-core kernel
// Stages in the K/V ring: as many as fit beside the Q tile (<= 227 KB).
// Tokens per ring stage: 128 for 32-row tiles (more independent MMA tiles per
// warp per stage), 64 when the accumulators of larger row tiles leave no room.
template <int NRG>
__host__ __device__ constexpr int stage_tokens() {
  return NRG == 2 ? 128 : 64;
}
// Stages in the ring: as many as fit beside the Q tile (<= 227 KB).
template <int NRG>
__host__ __device__ constexpr int stages_for() {
  return NRG == 2 ? 3 : 6;
}

template <int NRG>
__global__ void __launch_bounds__(kThreads, 1) attn_partial_bf16(const AttnParams p) {
  static_assert(NRG >= 2, "a warp needs at least 16 tokens of every stage");
  constexpr int NTG = kConsumerWarps / NRG;   // token sub-blocks of each stage
  constexpr int ST = stage_tokens<NRG>();    // tokens per stage
  constexpr int H = ST * 128;                // bytes of one K or V half-row block (64 dims)
  constexpr int kStageBytes = 4 * H;         // K lo/hi + V lo/hi
  constexpr int TS = ST / NTG;               // tokens of a stage handled by one warp
  constexpr int NT = TS / 8;                  // 8-token MMA n-tiles per warp per stage
  constexpr int RT = 16 * NRG;
  constexpr int kNumStages = stages_for<NRG>();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;                                                  // kNumStages * 32 KB
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + kNumStages * kStageBytes);
  int32_t* bt_s = reinterpret_cast<int32_t*>(qs + RT * kQStride);          // chunk/16 + 1
  uint64_t* full = reinterpret_cast<uint64_t*>(bt_s + kMaxChunk / 16 + 8);
  uint64_t* empty = full + kNumStages;
  static_assert(kNumStages * kStageBytes >= kConsumerWarps * 16 * (128 + 2) * 4,
                "epilogue scratch must fit in the stage ring");

  // KV heads are fastest in the grid: CTAs of all heads of the same tokens run
  // together and use whole 2 KB token rows of the cache between them
  const int kvh = blockIdx.x % p.Hkv;
  const int rt = blockIdx.x / p.Hkv;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int ctx = p.ctx_len[b];
  const int kv_len = ctx + p.R;
  const int c0 = s * p.chunk;
  if (c0 >= kv_len) return;  // this sequence needs fewer chunks
  const int c1 = min(c0 + p.chunk, kv_len);
  const int nst = (c1 - c0 + ST - 1) / ST;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // let a dependent grid (the LSE combine) start launching; it waits for
  // this grid's completion before it reads any partial
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumStages; ++i) {
      mbar_init(&full[i], kProducerThreads);   // one arrive per producer thread per stage
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();  // barriers initialised before anyone waits on them

  if (warp >= kConsumerWarps) {
    // ---------------- producer warps: the block-table slice, then K/V stages
    // through 16-byte cp.async (L2 -> shared, L1 bypassed) into the swizzled
    // stage layout; each thread's copies complete on the stage's mbarrier.
    const int pt = threadIdx.x - 32 * kConsumerWarps;   // 0 .. 127
    static_assert(kProducerThreads == 128, "4 column groups x 32 token lanes");
    const int P = p.page_size;
    const int pg0 = c0 / P;
    const int npg = (c1 - 1) / P - pg0 + 1;
    // entries past the table width (a caller error) read as -1 and are
    // zero-filled below instead of touching foreign memory
    for (int i = pt; i < npg; i += kProducerThreads)
      bt_s[i] = (pg0 + i < p.max_pages) ? p.block_table[(size_t)b * p.max_pages + pg0 + i] : -1;
    asm volatile("bar.sync 2, %0;" ::"n"(kProducerThreads) : "memory");
    // Thread pt copies 64 contiguous bytes (16-byte columns 4 c4 .. 4 c4 + 3)
    // of token lanes tl, tl + 32, ... of every stage, K and V: one page lookup
    // per token, and the four swizzled column offsets are fixed per thread (a
    // token's swizzle depends only on tl & 7).  A warp covers 8 whole 256-byte
    // rows per instruction.
    const int c4 = pt & 3, tl = pt >> 2;
    uint32_t col[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ch = 4 * c4 + u;
      col[u] = (uint32_t)((ch >> 3) * H + (((ch & 7) ^ (tl & 7)) << 4));
    }
    const size_t tok_stride = (size_t)p.Hkv * 256;   // bytes between consecutive cache rows
    const uint8_t* kcol = reinterpret_cast<const uint8_t*>(p.k) + (size_t)kvh * 256 + c4 * 64;
    const uint8_t* vcol = reinterpret_cast<const uint8_t*>(p.v) + (size_t)kvh * 256 + c4 * 64;
    const bool pow2 = (P & (P - 1)) == 0;
    const int pshift = __ffs(P) - 1;
    // K/V rows are read once (the CTAs of one chunk are its only readers):
    // first out of L2, so that the partials and the block tables stay
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    for (int k = 0; k < nst; ++k) {
      const int slot = k % kNumStages;
      if (k >= kNumStages && !mbar_wait(&empty[slot], ((k / kNumStages) - 1) & 1, p.err, p.wait_ns)) break;
      const uint32_t sbase = smem_u32(stages + slot * kStageBytes);
#pragma unroll
      for (int j = 0; j < ST / 32; ++j) {
        const int tok = tl + 32 * j;   // token within the stage
        const int t = c0 + k * ST + tok;
        int pg = -1, slotp = 0;
        if (t < kv_len) {
          const int pi = pow2 ? (t >> pshift) : (t / P);
          slotp = t - pi * P;
          pg = bt_s[pi - pg0];
        }
        const bool ok = pg >= 0 && pg < p.num_pages;
        const size_t row = ok ? ((size_t)pg * P + slotp) * tok_stride : 0;
        const uint32_t n = ok ? 16u : 0u;   // positions past the sequence / bad pages: zeros
        const uint32_t drow = sbase + tok * 128;
        const uint8_t* ks = kcol + row;
        const uint8_t* vs = vcol + row;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
                           drow + col[u]),
                       "l"(ks + 16 * u), "r"(n), "l"(pol)
                       : "memory");
          asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
                           drow + col[u] + 2 * H),
                       "l"(vs + 16 * u), "r"(n), "l"(pol)
                       : "memory");
        }
      }
      if (k != p.withhold_stage)  // (a test can withhold one stage: its waiters time out)
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                         smem_u32(&full[slot]))
                     : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // Q tile (consumer warps): row rho = i*G + g of this KV head -> q[b, i, kvh*G + g, :]
  for (int idx = threadIdx.x; idx < RT * 16; idx += 32 * kConsumerWarps) {
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
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");

  // ---------------- consumer warps: every warp takes its 16-row group and its
  // TS-token sub-block of EVERY stage, so a stage is released as soon as the
  // eight warps finish their short slices of it
  const int rg = warp % NRG;
  const int tg = warp / NRG;
  const int r0 = lane >> 2;           // accumulator rows r0 and r0 + 8
  const int cq = 2 * (lane & 3);      // accumulator column pair
  const int rho0 = rt * RT + rg * 16 + r0;
  const int rho1 = rho0 + 8;
  const bool v0 = rho0 < p.RG, v1 = rho1 < p.RG;
  const uint64_t w0 = v0 ? attn::row_mask(p, b, rho0 / p.G) : 0ull;
  const uint64_t w1 = v1 ? attn::row_mask(p, b, rho1 / p.G) : 0ull;
  const int tsb = tg * TS;            // first token of this warp's sub-block

  const uint32_t q_base = smem_u32(qs);
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  for (int k = 0; k < nst; ++k) {
    const int slot = k % kNumStages;
    if (!mbar_wait(&full[slot], (k / kNumStages) & 1, p.err, p.wait_ns)) break;
    const uint32_t st = smem_u32(stages + slot * kStageBytes);
    const int tb = c0 + k * ST + tsb;   // first cache position of the sub-block

    // ---- S = Q K^T for 16 rows x TS tokens
    float sacc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      {
        const int m = lane >> 3, r = lane & 7;
        const int row = rg * 16 + r + 8 * (m & 1);
        const int chunk = 2 * ks + (m >> 1);
        ldmatrix_x4(a[0], a[1], a[2], a[3], q_base + row * (kQStride * 2) + chunk * 16);
      }
      const uint32_t kb = st + (ks >> 2) * H;
      const int cbase = (2 * ks) & 7;
#pragma unroll
      for (int ntp = 0; ntp < NT / 2; ++ntp) {
        const int m = lane >> 3, r = lane & 7;
        const int tok = tsb + 8 * (2 * ntp + (m >> 1)) + r;
        const int chunk = cbase + (m & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3, kb + tok * 128 + ((chunk ^ (tok & 7)) << 4));
        mma_bf16_16816(sacc[2 * ntp], a, b0, b1);
        mma_bf16_16816(sacc[2 * ntp + 1], a, b2, b3);
      }
    }

    // ---- scale, visibility mask, online softmax (log2 domain)
    // (pairs e = 0, 1 and 2, 3 share a row: packed f32x2 arithmetic)
    const bool need_mask = tb + TS > ctx;
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float x[4];
      f2_unpack(f2_mul(f2_pack(sacc[nt][0], sacc[nt][1]), sc2), x[0], x[1]);
      f2_unpack(f2_mul(f2_pack(sacc[nt][2], sacc[nt][3]), sc2), x[2], x[3]);
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = tb + nt * 8 + cq + (e & 1);
          const uint64_t w = (e < 2) ? w0 : w1;
          const int j = pos - ctx;
          const bool vis = (pos < ctx) || (j < p.R && ((w >> j) & 1ull));
          if (!vis) x[e] = -INFINITY;
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = x[e];
      mx[0] = fmax3(mx[0], x[0], x[1]);
      mx[1] = fmax3(mx[1], x[2], x[3]);
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
    const uint64_t nb0 = f2_pack(-base[0], -base[0]), nb1 = f2_pack(-base[1], -base[1]);
    uint64_t rs2[2] = {0ull, 0ull};  // +0.0f pairs, one per row
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float d[4];
      f2_unpack(f2_add(f2_pack(sacc[nt][0], sacc[nt][1]), nb0), d[0], d[1]);
      f2_unpack(f2_add(f2_pack(sacc[nt][2], sacc[nt][3]), nb1), d[2], d[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = fast_exp2(d[e]);
      rs2[0] = f2_add(rs2[0], f2_pack(sacc[nt][0], sacc[nt][1]));
      rs2[1] = f2_add(rs2[1], f2_pack(sacc[nt][2], sacc[nt][3]));
    }
    float rs[2], r2a, r2b;
    f2_unpack(rs2[0], r2a, r2b);
    rs[0] = r2a + r2b;
    f2_unpack(rs2[1], r2a, r2b);
    rs[1] = r2a + r2b;
#pragma unroll
    for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + rs[h];
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {  // a row maximum moved
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
    }

    const uint32_t vb = st + 2 * H;

    // ---- O += P V over the sub-block
#pragma unroll
    for (int j = 0; j < TS / 16; ++j) {
      uint32_t a[4];
      a[0] = pack_bf16(sacc[2 * j][0], sacc[2 * j][1]);
      a[1] = pack_bf16(sacc[2 * j][2], sacc[2 * j][3]);
      a[2] = pack_bf16(sacc[2 * j + 1][0], sacc[2 * j + 1][1]);
      a[3] = pack_bf16(sacc[2 * j + 1][2], sacc[2 * j + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int c = 2 * dp;
        const int m = lane >> 3, r = lane & 7;
        const int tok = tsb + 16 * j + 8 * (m & 1) + r;
        const int chunk = (c & 7) + (m >> 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(b0, b1, b2, b3,
                          vb + (c >> 3) * H + tok * 128 + ((chunk ^ (tok & 7)) << 4));
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
// fp32 caches: 32-token K/V tiles staged through shared memory (coalesced
// row loads through the block table, padded rows for conflict-free dot
// products); one warp per query row, lane j scores token j of the tile,
// lanes own D/32 output dimensions each.
constexpr int kF32Tile = 32;

__global__ void __launch_bounds__(128) attn_partial_f32(const AttnParams p) {
  __shared__ float ks[kF32Tile][128 + 1];
  __shared__ float vs[kF32Tile][128 + 1];
  __shared__ float qsh[4][128];
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
  // rows are processed four at a time (one per warp); every warp walks every tile
  for (int rbase = 0; rbase < p.RG; rbase += 4) {
    const int rho = rbase + warp;
    const bool live = rho < p.RG;
    const int i = live ? rho / p.G : 0, g = live ? rho % p.G : 0;
    const uint64_t w = live ? attn::row_mask(p, b, i) : 0ull;
    if (live)
      for (int d = lane; d < D; d += 32)
        qsh[warp][d] = p.qf[(((size_t)b * p.R + i) * p.Hq + (size_t)kvh * p.G + g) * D + d];
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    float m_run = -INFINITY, l_run = 0.f;
    for (int t0 = c0; t0 < c1; t0 += kF32Tile) {
      __syncthreads();  // previous tile consumed
      for (int idx = threadIdx.x; idx < kF32Tile * D; idx += 128) {
        const int j = idx / D, d = idx % D;
        const int t = t0 + j;
        float kv = 0.f, vv = 0.f;
        if (t < c1) {
          const int page = (t / P < p.max_pages) ? p.block_table[(size_t)b * p.max_pages + t / P] : -1;
          if (page >= 0 && page < p.num_pages) {
            const size_t roff = (((size_t)page * P + (t % P)) * p.Hkv + kvh) * D + d;
            kv = p.kf[roff];
            vv = p.vf[roff];
          }
        }
        ks[j][d] = kv;
        vs[j][d] = vv;
      }
      __syncthreads();
      const int t = t0 + lane;
      float x = -INFINITY;
      if (live && t < c1) {
        const int jb = t - ctx;
        const bool vis = (t < ctx) || (jb < p.R && ((w >> jb) & 1ull));
        if (vis) {
          float dot = 0.f;
          for (int d = 0; d < D; ++d) dot = fmaf(qsh[warp][d], ks[lane][d], dot);
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
      const int nvalid = min(kF32Tile, c1 - t0);
      for (int jj = 0; jj < nvalid; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, pe, jj);
        for (int c = 0; c < nd; ++c) o[c] = fmaf(pj, vs[jj][lane + 32 * c], o[c]);
      }
    }
    if (live) {
      const size_t prow = (((size_t)b * p.Hkv + kvh) * p.RGpad + rho) * p.S + s;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      for (int c = 0; c < nd; ++c) p.o_part[prow * D + lane + 32 * c] = o[c] * inv;
      if (lane == 0) p.lse_part[prow] = l_run > 0.f ? m_run + __log2f(l_run) : -INFINITY;
    }
  }
}

// ------------------------------------------------------------------ LSE combine
// out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M), one warp per output row.
// Launched as a programmatic dependent of the partial pass: everything up to
// griddepcontrol.wait overlaps the partial pass's tail.
template <typename OutT, int kBatch>
__global__ void __launch_bounds__(128) attn_combine(const AttnParams p, OutT* __restrict__ out,
                                                   float* __restrict__ lse_out) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int total = p.B * p.R * p.Hq;
  const bool live = gw < total;
  const int hq = live ? gw % p.Hq : 0;
  const int i = live ? (gw / p.Hq) % p.R : 0;
  const int b = live ? gw / (p.Hq * p.R) : 0;
  const int kvh = hq / p.G, g = hq % p.G;
  const int rho = i * p.G + g;
  const int kv_len = live ? p.ctx_len[b] + p.R : 0;
  const int ns = min(p.S, (kv_len + p.chunk - 1) / p.chunk);
  const size_t prow0 = (((size_t)b * p.Hkv + kvh) * p.RGpad + rho) * p.S;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!live) return;
  const int D = p.D;
  const int per = D / 32;  // 4 (D = 128) or 2 (D = 64) floats per lane
  // one pass, kBatch partials in flight at a time; the running maximum M
  // rescales the sums when a later batch raises it (one batch: no rescale)
  float M = -INFINITY;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float L = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kBatch) {
    float ls[kBatch];
    float4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {  // independent loads, all in flight together
      const int s = s0 + j;
      ls[j] = s < ns ? __ldcg(&p.lse_part[prow0 + s]) : -INFINITY;
      const float* src = p.o_part + (prow0 + s) * D + per * lane;
      v[j] = s >= ns     ? make_float4(0.f, 0.f, 0.f, 0.f)
             : per == 4 ? __ldcg(reinterpret_cast<const float4*>(src))
                        : make_float4(__ldcg(src), __ldcg(src + 1), 0.f, 0.f);
    }
    float bm = ls[0];
#pragma unroll
    for (int j = 1; j < kBatch; ++j) bm = fmaxf(bm, ls[j]);
    if (bm > M) {
      const float sc = (M == -INFINITY) ? 0.f : fast_exp2(M - bm);
      L *= sc;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] *= sc;
      M = bm;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float e = (ls[j] == -INFINITY) ? 0.f : fast_exp2(ls[j] - M);
      L += e;
      acc[0] += e * v[j].x;
      acc[1] += e * v[j].y;
      acc[2] += e * v[j].z;
      acc[3] += e * v[j].w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  OutT* dst = out + (((size_t)b * p.R + i) * p.Hq + hq) * D;
  for (int c = 0; c < per; ++c) {
    const float val = acc[c] * inv;
    if constexpr (sizeof(OutT) == 2)
      dst[per * lane + c] = __float2bfloat16_rn(val);
    else
      dst[per * lane + c] = val;
  }
  if (lse_out && lane == 0)
    lse_out[((size_t)b * p.R + i) * p.Hq + hq] =
        (L > 0.f) ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
}

template <typename OutT>
spec_status launch_combine(const AttnParams& prm, OutT* out, float* lse_out, cudaStream_t st) {
  const int rows = prm.B * prm.R * prm.Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows * 32 + 127) / 128, 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // few splits: eight partials a pass (fewer registers, more warps resident)
  const cudaError_t e =
      prm.S <= 8 ? cudaLaunchKernelEx(&cfg, attn_combine<OutT, 8>, prm, out, lse_out)
                 : cudaLaunchKernelEx(&cfg, attn_combine<OutT, 16>, prm, out, lse_out);
  if (e != cudaSuccess) return SPEC_ECUDA;
  return launch_status();
}

// ------------------------------------------------------------------ host side
int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

struct Plan {
  int G, RG, NRG, RT, row_tiles, RGpad, chunk, S;
  bool tc;   // warp-MMA tensor-core path (bf16, at most 64 rows per KV head)
  int NM;    // > 0: the tcgen05 path with NM 128-row tiles per CTA (bf16, > 64 rows)
};

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Rows per KV head above which the partial pass runs on tcgen05 (tensor-memory
// accumulators, 128-row MMAs): the draft-tree and long-chain shapes.
constexpr int kTcgen05MinRows = 65;

bool make_plan(int B, int R, int Hq, int Hkv, int D, int page_size, int max_pages, int num_splits,
               bool bf16, Plan* pl) {
  if (B < 1 || R < 1 || R > 64 || Hq < 1 || Hkv < 1 || Hq % Hkv || page_size < 1 || max_pages < 1)
    return false;
  pl->tc = bf16;
  pl->G = Hq / Hkv;
  pl->RG = R * pl->G;
  pl->NM = 0;
  if (bf16 && pl->RG >= kTcgen05MinRows) {
    // two 128-row tiles per CTA (sharing each K/V stage) beyond 128 rows
    pl->NM = pl->RG > attn::kTcRows ? 2 : 1;
    pl->NRG = 0;
    pl->RT = attn::kTcRows * pl->NM;
    pl->row_tiles = (pl->RG + pl->RT - 1) / pl->RT;
    pl->RGpad = pl->row_tiles * pl->RT;
  } else if (bf16) {
    pl->NRG = pl->RG <= 32 ? 2 : 4;
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
  // stage size of the kernel
  const int g = pl->NM > 0 ? attn::kTcStageTokens : (bf16 && pl->NRG == 2) ? 128 : kStageTokens;
  int chunk;
  if (num_splits > 0) {
    chunk = (int)((max_kv + num_splits - 1) / num_splits);
    chunk = chunk >= 2 * g ? chunk / g * g : round_up(chunk, g);
  } else {
    const int sms = num_sms();
    if (units >= sms) {
      chunk = kMaxChunk;  // measured faster than 2048-token splits on batched serving
    } else {
      // about one wave of CTAs; long contexts take the longest chunk the page
      // table slice holds (fewer, longer splits measured faster than 2048-token ones)
      const int S = std::max(1, sms / units);
      chunk = round_up((int)((max_kv + S - 1) / S), g);
    }
  }
  chunk = std::max(g, std::min(chunk, kMaxChunk));
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

size_t smem_bytes_bf16(int NRG, int stages, int stage_tok) {
  return 1024 + (size_t)stages * stage_tok * 512 + (size_t)16 * NRG * kQStride * 2 +
         (kMaxChunk / 16 + 8) * 4 + 2 * stages * 8;
}

template <int NRG>
spec_status launch_bf16(const AttnParams& prm, const Plan& pl, cudaStream_t st) {
  const size_t smem = smem_bytes_bf16(NRG, stages_for<NRG>(), stage_tokens<NRG>());
  static PerDeviceOnce<int> smem_once;  // once per device
  const spec_status ra = ensure_smem_limit(smem_once, (const void*)attn_partial_bf16<NRG>, (int)smem);
  if (ra != SPEC_OK) return ra;
  dim3 grid(prm.Hkv * pl.row_tiles, pl.S, prm.B);
  attn_partial_bf16<NRG><<<grid, kThreads, smem, st>>>(prm);
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

// Test-only fault setting of the partial passes (spec_debug_attn_fault): a
// stage whose arrival the copy warps withhold, and the bound of every wait.
std::atomic<int> g_withhold_stage{-1};
std::atomic<unsigned long long> g_wait_ns{SPEC_WAIT_NS};

spec_status verify_attn_impl(const void* q, const void* k_cache, const void* v_cache,
                             spec_dtype dtype, int page_size, int num_pages,
                             const int32_t* block_table, int max_pages, const int32_t* ctx_len,
                             const uint64_t* anc_mask, int B, int R, int Hq, int Hkv, int D,
                             float scale, int num_splits, void* workspace, size_t workspace_bytes,
                             void* out, float* lse_out, void* stream, int phase) {
  if (!ctx_len || !workspace) return SPEC_EINVAL;
  if ((phase & kPartials) && (!q || !k_cache || !v_cache || !block_table))
    return SPEC_EINVAL;
  if ((phase & kCombine) && !out) return SPEC_EINVAL;
  if (B < 0 || R < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || page_size < 1 || num_pages < 1 ||
      max_pages < 1 || num_splits < 0)
    return SPEC_EINVAL;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (R > 64 || (D != 64 && D != 128)) return SPEC_EUNSUPPORTED;
  if (B > 65535) return SPEC_EUNSUPPORTED;  // sequences index the grid's z dimension
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
  prm.k = k_cache;
  prm.v = v_cache;
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
  prm.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  prm.withhold_stage = g_withhold_stage.load(std::memory_order_relaxed);

  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (phase & kPartials) {
    spec_status rc;
    if (bf16 && pl.NM > 0) {
      rc = attn::launch_partial_tc(prm, pl.RT, st);
    } else if (bf16) {
      rc = pl.NRG == 2 ? launch_bf16<2>(prm, pl, st) : launch_bf16<4>(prm, pl, st);
    } else {
      dim3 grid(pl.S, Hkv, B);
      attn_partial_f32<<<grid, 128, 0, st>>>(prm);
      rc = launch_status();
    }
    if (rc != SPEC_OK) return rc;
  }
  if (phase & kCombine) {
    if (bf16) return launch_combine<__nv_bfloat16>(prm, static_cast<__nv_bfloat16*>(out), lse_out, st);
    return launch_combine<float>(prm, static_cast<float*>(out), lse_out, st);
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

extern "C" spec_status spec_debug_attn_fault(int withhold_stage, unsigned long long wait_limit_ns) {
  if (withhold_stage < -1) return SPEC_EINVAL;
  g_withhold_stage.store(withhold_stage);
  g_wait_ns.store(wait_limit_ns ? wait_limit_ns : SPEC_WAIT_NS);
  return SPEC_OK;
}

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

PerDeviceOnce<void*> g_noalloc_addr;

// Device address of g_noalloc_scratch on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress, with that device current);
// later calls reuse the cached address.  No memory is allocated.  The cache
// is keyed by device ordinal, so calls must not span a reset of the device
// (cudaDeviceReset), after which the cached address is stale.
spec_status noalloc_scratch(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ECUDA;
  const int rc = g_noalloc_addr.run(
      dev,
      [](void** p) {
        return (cudaGetSymbolAddress(p, g_noalloc_scratch) == cudaSuccess && *p) ? 0 : 1;
      },
      addr);
  if (rc == -1) return SPEC_EUNSUPPORTED;
  return rc == 0 ? SPEC_OK : SPEC_ECUDA;
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

// The error word of the allocation-free call's scratch (the head of the
// fixed array), for callers that cannot address that array themselves.
// Reads it with a copy from the symbol on `stream`, then waits for the
// stream; allocates nothing.
extern "C" spec_status spec_verify_attn_noalloc_error(int32_t* host_err, void* stream) {
  if (!host_err) return SPEC_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_noalloc_scratch, sizeof(int32_t), 0, cudaMemcpyDeviceToHost,
                                st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SPEC_ECUDA;
  *host_err = v;
  return SPEC_OK;
}
