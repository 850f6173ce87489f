// Verify-attention partial pass on the 5th-generation tensor cores (tcgen05,
// operands and accumulators in tensor memory) for shapes with many query rows
// per KV head: a draft tree (R = 64 nodes x 8 query heads per KV head = 512
// rows) or a long chain (16 x 8 = 128 rows).  Same contract and partial layout
// as the warp-MMA pass in attn.cu: per (sequence, KV head, chunk) a normalised
// softmax partial O_s and its log2-domain log-sum-exp, merged by the combine
// ("Speculative Token Decoupling: Asynchronous Verification via
// Flash-Decoding", section 03: split-K attention).  Visibility is the same:
// every committed position, and block position ctx + j for row i iff bit j of
// its ancestor mask ("Speculative Decoding" (atlas), "Chains, trees and
// visibility").
//
// One CTA per (KV head x 128-row tile, chunk, sequence); warp roles:
//   * 2 copy warps stream 128-token K/V stages (16-byte cp.async through the
//     block table, one page lookup per token) into a ring of 3 stages, laid
//     out as the 128-byte-swizzled operands the tensor cores read: K as a
//     K-major B operand, V as an MN-major B operand.  Each copy thread's
//     copies arrive on the stage's barrier when they land; the MMA thread
//     fences the stage into the async proxy after its wait.
//   * 1 MMA warp (one thread issues): S = Q K^T (M = 128 rows, N = 128 tokens,
//     K = 128 dims: 8 MMAs) with Q in tensor memory, into one of two score
//     buffers, so the next tile's scores are computed while the softmax works
//     on this one; then O += P V (K = 128 tokens: 8 MMAs, N = 128 dims) with P
//     read from tensor memory and V from shared memory, into a tensor-memory
//     accumulator.  A tcgen05.mma costs a roughly fixed issue time, so each
//     instruction covers the widest tile the tensor memory holds.
//   * 4 softmax warps (a thread owns one row): write the row's Q into tensor
//     memory once; per tile load the row's 128 scores from tensor memory in
//     one batch (mask, maximum, exp2 on the SFU, sum, bf16 pack in registers)
//     and write P back over them.  The running maximum is raised lazily: O is
//     rescaled only when a row's maximum grows by more than 2^8 (p stays <=
//     256, exact in the final O / l), so the O read-modify-write is rare.
// Tensor memory (512 columns allocated): Q [0, 64), score buffers [64, 192)
// and [192, 320) (P in the first 64 columns of its buffer), O [320, 448).
// Every wait is bounded (an error word in the workspace); tensor memory is
// freed on every exit path after the last MMA has completed.
#include "attn.cuh"
#include "tc_ptx.cuh"

namespace {

using attn::AttnParams;
using attn::kMaxChunk;

constexpr int kST = 128;                // tokens per stage and per score tile
constexpr int kHalf = kST * 128;        // one 64-dim half of K or V: 128 rows x 128 B
constexpr int kStageBytes = 4 * kHalf;  // K lo, K hi, V lo, V hi (64 KB)
constexpr int kStages = 3;
constexpr int kCopyWarps = 2;
constexpr int kCopyThreads = 32 * kCopyWarps;
constexpr int kSoftWarps = 4;
constexpr int kMmaWarp = kSoftWarps;
constexpr int kCopyWarp0 = kSoftWarps + 1;
constexpr int kThreads = 32 * (kSoftWarps + 1 + kCopyWarps);
constexpr float kRescaleLog2 = 8.0f;  // rescale O when a row maximum grows by > 2^8
constexpr int kColQ = 0, kColS = 64, kColO = 320;
constexpr uint32_t kTmemCols = 512;
constexpr int kOffBt = kStages * kStageBytes;             // block-table slice
constexpr int kOffBar = kOffBt + (kMaxChunk / 16 + 8) * 4;
// kv_full[3], kv_empty[3], s_full[2], p_full, o_done, q_full, mma_done
constexpr int kNumBars = 2 * kStages + 2 + 4;
constexpr int kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
static_assert(kSmem <= 232448, "shared memory per CTA");
static_assert(kOffBar % 8 == 0, "barrier alignment");

__global__ void __launch_bounds__(kThreads, 1) attn_partial_tc(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  int32_t* bt_s = reinterpret_cast<int32_t*>(smem + kOffBt);
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* q_full = o_done + 1;
  uint64_t* mma_done = q_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int kvh = blockIdx.x % p.Hkv;
  const int rt = blockIdx.x / p.Hkv;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int ctx = p.ctx_len[b];
  const int kv_len = ctx + p.R;
  const int c0 = s * p.chunk;
  if (c0 >= kv_len) return;  // this sequence needs fewer chunks (uniform over the CTA)
  const int c1 = min(c0 + p.chunk, kv_len);
  const int nst = (c1 - c0 + kST - 1) / kST;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // let the combine (a programmatic dependent) start launching
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], kCopyThreads);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, kSoftWarps);
    mbar_init(o_done, 1);
    mbar_init(q_full, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kCopyWarp0) {
    // ---------------- copy warps: block-table slice, then the K/V stages
    const int pt = threadIdx.x - 32 * kCopyWarp0;  // 0 .. kCopyThreads - 1
    const int P = p.page_size;
    const int pg0 = c0 / P;
    const int npg = (c1 - 1) / P - pg0 + 1;
    for (int i = pt; i < npg; i += kCopyThreads)
      bt_s[i] = (pg0 + i < p.max_pages) ? p.block_table[(size_t)b * p.max_pages + pg0 + i] : -1;
    asm volatile("bar.sync 2, %0;" ::"n"(kCopyThreads) : "memory");
    // thread pt copies 64 contiguous bytes (16-byte chunks 4 c4 .. 4 c4 + 3) of
    // token lanes tl, tl + 16, ..., tl + 112 of every stage, for K and for V; a
    // token's swizzle depends only on tl & 7, so the four column offsets are fixed
    constexpr int kTokLanes = kCopyThreads / 4;
    static_assert(kST % kTokLanes == 0, "token lanes cover a stage");
    const int c4 = pt & 3, tl = pt >> 2;
    uint32_t col[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ch = 4 * c4 + u;
      col[u] = (uint32_t)((ch >> 3) * kHalf + (((ch & 7) ^ (tl & 7)) << 4));
    }
    const size_t tok_stride = (size_t)p.Hkv * 256;
    const uint8_t* kcol = reinterpret_cast<const uint8_t*>(p.k) + (size_t)kvh * 256 + c4 * 64;
    const uint8_t* vcol = reinterpret_cast<const uint8_t*>(p.v) + (size_t)kvh * 256 + c4 * 64;
    const bool pow2 = (P & (P - 1)) == 0;
    const int pshift = __ffs(P) - 1;
    for (int k = 0; k < nst; ++k) {
      const int slot = k % kStages;
      if (k >= kStages && !mbar_wait(&kv_empty[slot], ((k / kStages) - 1) & 1, p.err)) break;
      const uint32_t sbase = smem_u32(stages + slot * kStageBytes);
#pragma unroll 4
      for (int jt = 0; jt < kST / kTokLanes; ++jt) {
        const int tok = tl + kTokLanes * jt;
        const int t = c0 + k * kST + tok;
        int pg = -1, slotp = 0;
        if (t < kv_len) {
          const int pi = pow2 ? (t >> pshift) : (t / P);
          slotp = t - pi * P;
          pg = bt_s[pi - pg0];
        }
        const bool ok = pg >= 0 && pg < p.num_pages;
        const size_t row = ok ? ((size_t)pg * P + slotp) * tok_stride : 0;
        const uint32_t n = ok ? 16u : 0u;  // past the sequence / bad page: zeros
        const uint32_t drow = sbase + tok * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(drow + col[u]),
                       "l"(kcol + row + 16 * u), "r"(n)
                       : "memory");
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                           drow + col[u] + 2 * kHalf),
                       "l"(vcol + row + 16 * u), "r"(n)
                       : "memory");
        }
      }
      // the stage's barrier counts this thread once its copies have landed
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                       smem_u32(&kv_full[slot]))
                   : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA warp: one thread issues every tensor-core operation
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kST, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
      bool ok = mbar_wait(q_full, 0, p.err);
      tc_fence_after();
      for (int j = 0; ok && j <= nst; ++j) {
        if (j < nst) {  // S(j) = Q K_j^T into score buffer j & 1
          const int slot = j % kStages;
          if (!mbar_wait(&kv_full[slot], (j / kStages) & 1, p.err)) break;
          fence_proxy_async();  // the copy warps' generic-proxy writes, seen by the tensor cores
          // the buffer held P(j - 2): PV(j - 2) must have read it
          if (j >= 2 && !mbar_wait(o_done, (j - 2) & 1, p.err)) break;
          tc_fence_after();
          const uint32_t kb = smem_u32(stages + slot * kStageBytes);
          const uint32_t d = tmem + kColS + (j & 1) * kST;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // 16 dims = 8 columns of Q; 32 bytes inside K's 64-dim atom
            const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
            tc_mma_ts(d, tmem + kColQ + kk * 8, bd, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[j & 1]);
        }
        if (j >= 1) {  // O += P(j-1) V_{j-1}
          const int jj = j - 1;
          const int slot = jj % kStages;
          if (!mbar_wait(p_full, jj & 1, p.err)) break;
          tc_fence_after();
          const uint32_t vb = smem_u32(stages + slot * kStageBytes) + 2 * kHalf;
          const uint32_t pa = tmem + kColS + (jj & 1) * kST;
#pragma unroll
          for (int kk = 0; kk < kST / 16; ++kk) {
            // 16 tokens = 8 columns of P; 2 swizzle atoms (2 KB) of V
            const uint64_t bd = smem_desc_sw128(vb + kk * 2048, kHalf, 1024);
            tc_mma_ts(tmem + kColO, pa + kk * 8, bd, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(o_done);
          tc_commit(&kv_empty[slot]);  // the stage is free once these MMAs complete
        }
      }
      // every issued MMA has completed before tensor memory can be freed
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, p.err);
    }
    __syncwarp();
  } else {
    // ---------------- softmax warps: warp w owns rows 32 w .. 32 w + 31 of the tile
    const int r = warp * 32 + lane;
    const int rho = rt * 128 + r;  // row rho = i * G + g of this KV head
    const bool valid = rho < p.RG;
    const bool warp_live = rt * 128 + warp * 32 < p.RG;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    {  // this thread's Q row into tensor memory (the A operand of S = Q K^T)
      uint32_t qa[32], qb[32];
      if (valid) {
        const int i = rho / p.G, g = rho % p.G;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (((size_t)b * p.R + i) * p.Hq + (size_t)kvh * p.G + g) * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 lo = src[c], hi = src[8 + c];
          qa[4 * c] = lo.x; qa[4 * c + 1] = lo.y; qa[4 * c + 2] = lo.z; qa[4 * c + 3] = lo.w;
          qb[4 * c] = hi.x; qb[4 * c + 1] = hi.y; qb[4 * c + 2] = hi.z; qb[4 * c + 3] = hi.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) qa[c] = qb[c] = 0u;
      }
      tmem_st32(lane_base + kColQ, qa);
      tmem_st32(lane_base + kColQ + 32, qb);
      tmem_wait_st();
    }
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");
    if (threadIdx.x == 0) mbar_arrive(q_full);

    const uint64_t w = valid ? p.anc_mask[(size_t)b * p.R + rho / p.G] : 0ull;
    const uint32_t o_addr = lane_base + kColO;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nst; ++j) {
      const int bi = j & 1;
      if (!mbar_wait(&s_full[bi], (j >> 1) & 1, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = lane_base + kColS + bi * kST;
      const int t0 = c0 + j * kST;
      const bool masked = t0 + kST > ctx;  // block positions (or past the sequence) in the tile
      // this row's visibility of tile column c (only the block part can be hidden)
      auto visible = [&](int c) {
        const int jb = t0 + c - ctx;
        return jb < 0 || (jb < p.R && ((w >> jb) & 1ull));
      };
      if (warp_live) {
        // the row's 128 scores in one batch of loads (a wait after every load
        // measured ~20x slower than one wait for all four)
        uint32_t sv[4][32];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tmem_ld32(s_addr + cb * 32, sv[cb]);
        tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int cb = 0; cb < 4; ++cb)
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (!visible(cb * 32 + c)) sv[cb][c] = __float_as_uint(-INFINITY);
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
          for (int c = 0; c < 32; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sv[cb][c]));
        const float mnew = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
        const bool need = mnew > m_run + kRescaleLog2;
        float alpha = 1.f;
        if (need) {
          alpha = fast_exp2(m_run - mnew);  // 0 on the first visible tile
          l_run *= alpha;
          m_run = mnew;
        }
        // p = exp2(s * scale - m) and the row sum; P packed as bf16 pairs in place
        // (pair c of a 32-score block into word c), then written over the scores
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float e0 = fast_exp2(fmaf(__uint_as_float(sv[cb][2 * c]), p.scale_log2, -base));
            const float e1 =
                fast_exp2(fmaf(__uint_as_float(sv[cb][2 * c + 1]), p.scale_log2, -base));
            rs[c & 3] += e0 + e1;
            sv[cb][c] = pack_bf16(e0, e1);
          }
        }
        if (j >= 1 && __any_sync(0xffffffffu, need)) {
          // rescale this warp's rows of O once PV(j-1) has completed (after the
          // packing, so that only the 64 packed words of P stay live)
          if (!mbar_wait(o_done, (j - 1) & 1, p.err)) {
            ok = false;
          } else {
            tc_fence_after();
            const float a = need ? alpha : 1.f;
            uint32_t o[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(o_addr + cc * 32, o[cc]);
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[cc][i] = __float_as_uint(__uint_as_float(o[cc][i]) * a);
              tmem_st32(o_addr + cc * 32, o[cc]);
            }
          }
        }
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = sv[cb][c];
          tmem_st16(s_addr + cb * 16, pk);
        }
        l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        tmem_wait_st();
      }
      // (rows no output needs have a zero Q, so their scores -- read as P by the
      // PV MMA -- are zero)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      if (!ok) break;
    }
    // ---------------- epilogue: O / l and the log2-domain LSE of this chunk
    if (ok && mbar_wait(o_done, (nst - 1) & 1, p.err)) {
      tc_fence_after();
      if (warp_live) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const size_t prow_o = (((size_t)b * p.Hkv + kvh) * p.RGpad + rho) * p.S + s;
        uint32_t o[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(o_addr + cc * 32, o[cc]);
        tmem_wait_ld();
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow_o * 128);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[cc * 8 + i] = make_float4(
                  __uint_as_float(o[cc][4 * i]) * inv, __uint_as_float(o[cc][4 * i + 1]) * inv,
                  __uint_as_float(o[cc][4 * i + 2]) * inv, __uint_as_float(o[cc][4 * i + 3]) * inv);
        }
        if (valid) p.lse_part[prow_o] = l_run > 0.f ? m_run + __log2f(l_run) : -INFINITY;
      }
    }
    __syncwarp();
  }

  // ---------------- tensor memory is freed after every role is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace attn {

spec_status launch_partial_tc(const AttnParams& prm, cudaStream_t st) {
  static PerDeviceOnce<int> smem_once;
  const spec_status ra = ensure_smem_limit(smem_once, (const void*)attn_partial_tc, kSmem);
  if (ra != SPEC_OK) return ra;
  dim3 grid(prm.Hkv * prm.row_tiles, prm.S, prm.B);
  attn_partial_tc<<<grid, kThreads, kSmem, st>>>(prm);
  return launch_status();
}

}  // namespace attn
