// Verify-attention partial pass on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory) for shapes with many query rows per KV head:
// a draft tree (R = 64 nodes x 8 query heads per KV head = 512 rows) or a long
// chain (16 x 8 = 128 rows).  Same contract and partial layout as the warp-MMA
// pass in attn.cu: per (sequence, KV head, chunk) an unnormalised-then-
// normalised softmax partial O_s and its log2-domain log-sum-exp, merged by the
// combine ("Speculative Token Decoupling: Asynchronous Verification via
// Flash-Decoding", section 03: split-K attention).  Visibility is the same:
// every committed position, and block position ctx + j for row i iff bit j of
// its ancestor mask ("Speculative Decoding" (atlas), "Chains, trees and
// visibility").
//
// One CTA per (KV head x 128*NM-row tile, chunk, sequence); warp roles:
//   * 2 copy warps stream 64-token K/V stages (16-byte cp.async through the
//     block table, one page lookup per token) into a ring of 6 stages, laid
//     out as the 128-byte-swizzled operands the tensor cores read: K as a
//     K-major B operand, V as an MN-major B operand.  Each copy thread's
//     copies arrive on the stage's barrier when they land (so every stage of
//     the ring can be in flight); the MMA thread fences the stage into the
//     async proxy after its wait, before the tensor cores read it.
//   * 1 MMA warp (one thread issues): S = Q K^T into tensor memory (M = 128
//     rows, N = 64 tokens, K = 128 dims: 8 MMAs) with Q itself held in tensor
//     memory (the A operand), so each score MMA reads only K's 2 KB from
//     shared memory; then O += P V (K = 64 tokens, N = 128 dims: 4 MMAs, P and
//     V from shared memory) into a tensor-memory accumulator; completions are
//     committed to mbarriers.  One tile's scores are computed while the softmax
//     works on the other tile's (two 128-row tiles) or on the previous scores
//     (one tile, two score buffers).
//   * 4 softmax warps per 128-row tile (a thread owns one row): write the row's
//     Q into tensor memory once; per tile load its 64 scores, mask,
//     exponentiate (exp2 on the SFU), sum, write P as bf16 into shared memory
//     (K-major A operand).  The running maximum is raised lazily: O in tensor
//     memory is rescaled only when a row's maximum grows by more than 2^8 (p
//     stays <= 256, exact in the final O / l), so the O read-modify-write is
//     rare after the first tiles.
// Tensor memory (512 columns): Q (64 columns per row tile), the score buffers
// (64 each), O (128 per row tile).
// Every wait is bounded (an error word in the workspace); tensor memory is
// freed on every exit path after the last MMA has completed.
#include "attn.cuh"
#include "tc_ptx.cuh"

namespace {

using attn::AttnParams;
using attn::kMaxChunk;

constexpr int kST = 64;                 // tokens per stage and per score tile
constexpr int kHalf = kST * 128;        // one 64-dim half of K or V: 64 rows x 128 B
constexpr int kStageBytes = 4 * kHalf;  // K lo, K hi, V lo, V hi
constexpr int kCopyWarps = 2;
constexpr int kCopyThreads = 32 * kCopyWarps;
constexpr float kRescaleLog2 = 8.0f;    // rescale O when a row maximum grows by > 2^8

template <int NM>
struct TcCfg {
  static constexpr int kStages = 6;
  static constexpr int kSB = NM == 2 ? 1 : 2;  // score buffers per row tile (tensor-memory budget)
  static constexpr int kSoftWarps = 4 * NM;
  static constexpr int kMmaWarp = kSoftWarps;
  static constexpr int kCopyWarp0 = kSoftWarps + 1;
  // 8 softmax + 1 MMA + 2 copy warps: at most 3 warps on each of the 4 scheduler
  // partitions, whose 16K-register files then allow 168 registers per thread
  static constexpr int kThreads = 32 * (kSoftWarps + 1 + kCopyWarps);
  static constexpr int kRows = 128 * NM;
  static constexpr int kOffP = kStages * kStageBytes;            // NM x 16 KB (128 rows x 64 tokens)
  static constexpr int kOffBt = kOffP + NM * 16384;              // block-table slice
  static constexpr int kOffBar = kOffBt + (kMaxChunk / 16 + 8) * 4;
  // kv_full[S], kv_empty[S], s_full[NM SB], s_empty[NM SB], p_full[NM], o_done[NM], q_full, mma_done
  static constexpr int kNumBars = 2 * kStages + 2 * NM * kSB + 2 * NM + 2;
  static constexpr int kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
  // tensor-memory columns: Q of each row tile (128 rows x 128 bf16 = 64 columns),
  // the score buffers (64 columns each), the O accumulators (128 columns each)
  static constexpr int kColQ = 0;
  static constexpr int kColS = 64 * NM;
  static constexpr int kColO = kColS + 64 * NM * kSB;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColO + 128 * NM <= (int)kTmemCols, "tensor memory columns");
  static_assert(kSmem <= 232448, "shared memory per CTA");
  static_assert(kOffBar % 8 == 0, "barrier alignment");
};

template <int NM>
__global__ void __launch_bounds__(TcCfg<NM>::kThreads, 1) attn_partial_tc(const AttnParams p) {
  using C = TcCfg<NM>;
  constexpr int NS = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* ps = smem + C::kOffP;
  int32_t* bt_s = reinterpret_cast<int32_t*>(smem + C::kOffBt);
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_empty = kv_full + NS;
  constexpr int SB = C::kSB;
  uint64_t* s_full = kv_empty + NS;
  uint64_t* s_empty = s_full + NM * SB;
  uint64_t* p_full = s_empty + NM * SB;
  uint64_t* o_done = p_full + NM;
  uint64_t* q_full = o_done + NM;
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
    for (int i = 0; i < NS; ++i) {
      mbar_init(&kv_full[i], kCopyThreads);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < NM * SB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
    }
    for (int i = 0; i < NM; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= C::kCopyWarp0) {
    // ---------------- copy warps: block-table slice, then the K/V stages
    const int pt = threadIdx.x - 32 * C::kCopyWarp0;  // 0 .. kCopyThreads - 1
    const int P = p.page_size;
    const int pg0 = c0 / P;
    const int npg = (c1 - 1) / P - pg0 + 1;
    for (int i = pt; i < npg; i += kCopyThreads)
      bt_s[i] = (pg0 + i < p.max_pages) ? p.block_table[(size_t)b * p.max_pages + pg0 + i] : -1;
    asm volatile("bar.sync 2, %0;" ::"n"(kCopyThreads) : "memory");
    // thread pt copies 64 contiguous bytes (16-byte chunks 4 c4 .. 4 c4 + 3) of
    // token lanes tl, tl + 16, tl + 32 and tl + 48 of every stage, for K and for
    // V; a token's swizzle depends only on tl & 7, so the four column offsets are
    // fixed
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
      const int slot = k % NS;
      if (k >= NS && !mbar_wait(&kv_empty[slot], ((k / NS) - 1) & 1, p.err)) break;
      const uint32_t sbase = smem_u32(stages + slot * kStageBytes);
#pragma unroll
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
      // the stage's barrier counts this thread once its copies have landed; the
      // MMA thread fences them into the async proxy after its wait
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                       smem_u32(&kv_full[slot]))
                   : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ---------------- MMA warp: one thread issues every tensor-core operation
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kST, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
      bool ok = mbar_wait(q_full, 0, p.err);
      tc_fence_after();
      const uint32_t p0 = smem_u32(ps);
      for (int j = 0; ok && j <= nst; ++j) {
        if (j < nst) {  // S(j) = Q K_j^T for every row tile; Q is read from tensor memory
          const int slot = j % NS;
          if (!mbar_wait(&kv_full[slot], (j / NS) & 1, p.err)) break;
          fence_proxy_async();  // the copy warps' generic-proxy writes, seen by the tensor cores
          tc_fence_after();
          const uint32_t kb = smem_u32(stages + slot * kStageBytes);
          const int bi = j % SB, u = j / SB;
#pragma unroll
          for (int m = 0; m < NM; ++m) {
            if (u >= 1 && !mbar_wait(&s_empty[m * SB + bi], (u - 1) & 1, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + C::kColS + (m * SB + bi) * kST;
            const uint32_t qa = tmem + C::kColQ + m * 64;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // 16 dims = 8 columns of Q; 32 bytes inside K's 64-dim atom
              const uint64_t bd =
                  smem_desc_sw128(kb + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
              tc_mma_ts(d, qa + kk * 8, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[m * SB + bi]);
          }
          if (!ok) break;
        }
        if (j >= 1) {  // O += P(j-1) V_{j-1} for every row tile
          const int jj = j - 1;
          const int slot = jj % NS;
          const uint32_t vb = smem_u32(stages + slot * kStageBytes) + 2 * kHalf;
#pragma unroll
          for (int m = 0; m < NM; ++m) {
            if (!mbar_wait(&p_full[m], jj & 1, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + C::kColO + m * 128;
            const uint32_t pa = p0 + m * 16384;
#pragma unroll
            for (int kk = 0; kk < kST / 16; ++kk) {
              const uint64_t a = smem_desc_sw128(pa + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(vb + kk * 2048, kHalf, 1024);
              tc_mma_ss(d, a, bd, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&o_done[m]);
          }
          if (!ok) break;
          tc_commit(&kv_empty[slot]);  // the stage is free once these MMAs complete
        }
      }
      // every issued MMA has completed before tensor memory can be freed
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, p.err);
    }
    __syncwarp();
  } else {
    // ---------------- softmax warps: warp w owns rows 32 (w % 4) .. + 31 of tile w / 4
    const int m = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // row within the 128-row tile
    const int rho = rt * C::kRows + m * 128 + r;       // row rho = i * G + g of this KV head
    const bool valid = rho < p.RG;
    const bool warp_live = rt * C::kRows + m * 128 + quarter * 32 < p.RG;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
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
      tmem_st32(lane_base + C::kColQ + m * 64, qa);
      tmem_st32(lane_base + C::kColQ + m * 64 + 32, qb);
      tmem_wait_st();
    }
    uint8_t* prow = ps + m * 16384 + r * 128;
    if (!warp_live)  // rows no output needs: P stays zero
      for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(prow + c * 16) = make_uint4(0, 0, 0, 0);
    fence_proxy_async();
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(32 * C::kSoftWarps) : "memory");
    if (threadIdx.x == 0) mbar_arrive(q_full);

    const uint64_t w = valid ? p.anc_mask[(size_t)b * p.R + rho / p.G] : 0ull;
    const uint32_t s_addr = lane_base + C::kColS + m * SB * kST;
    const uint32_t o_addr = lane_base + C::kColO + m * 128;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nst; ++j) {
      const int bi = j % SB;
      if (!mbar_wait(&s_full[m * SB + bi], (j / SB) & 1, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pk[32];  // P of this row as bf16 pairs
      bool need = false;
      float alpha = 1.f;
      if (warp_live) {
        uint32_t sa[32], sb[32];
        tmem_ld32(s_addr + bi * kST, sa);
        tmem_ld32(s_addr + bi * kST + 32, sb);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[m * SB + bi]);
        float x[64];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(sa[c]);
          x[32 + c] = __uint_as_float(sb[c]);
        }
        const int t0 = c0 + j * kST;
        if (t0 + kST > ctx) {  // block positions (or past the sequence) in this tile
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int jb = t0 + c - ctx;
            const bool vis = jb < 0 || (jb < p.R && ((w >> jb) & 1ull));
            if (!vis) x[c] = -INFINITY;
          }
        }
        float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int c = 4; c < 64; ++c) m4[c & 3] = fmaxf(m4[c & 3], x[c]);
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float mnew = mx * p.scale_log2;
        need = mnew > m_run + kRescaleLog2;
        if (need) {
          alpha = fast_exp2(m_run - mnew);  // 0 on the first visible tile
          l_run *= alpha;
          m_run = mnew;
        }
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float e0 = fast_exp2(fmaf(x[2 * c], p.scale_log2, -base));
          const float e1 = fast_exp2(fmaf(x[2 * c + 1], p.scale_log2, -base));
          rs[c & 3] += e0 + e1;
          pk[c] = pack_bf16(e0, e1);
        }
        l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[m * SB + bi]);
      }
      // P(j-1) has been consumed and O holds P(j-1) V: the P buffer and O are free
      if (j >= 1 && !mbar_wait(&o_done[m], (j - 1) & 1, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (warp_live) {
        if (j >= 1 && __any_sync(0xffffffffu, need)) {  // rescale this warp's rows of O
          const float a = need ? alpha : 1.f;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(o_addr + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
            tmem_st32(o_addr + cc * 32, o);
          }
          tmem_wait_st();
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + ((c ^ (lane & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        fence_proxy_async();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[m]);
    }
    // ---------------- epilogue: O / l and the log2-domain LSE of this chunk
    if (ok && mbar_wait(&o_done[m], (nst - 1) & 1, p.err)) {
      tc_fence_after();
      if (warp_live) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const size_t prow_o = (((size_t)b * p.Hkv + kvh) * p.RGpad + rho) * p.S + s;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(o_addr + cc * 32, o);
          tmem_wait_ld();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow_o * 128 + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                   __uint_as_float(o[4 * i + 2]) * inv,
                                   __uint_as_float(o[4 * i + 3]) * inv);
          }
        }
        if (valid) p.lse_part[prow_o] = l_run > 0.f ? m_run + __log2f(l_run) : -INFINITY;
      }
    }
    __syncwarp();
  }

  // ---------------- tensor memory is freed after every role is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NM>
spec_status launch_nm(const AttnParams& prm, cudaStream_t st) {
  using C = TcCfg<NM>;
  static PerDeviceOnce<int> smem_once;
  const spec_status ra = ensure_smem_limit(smem_once, (const void*)attn_partial_tc<NM>, C::kSmem);
  if (ra != SPEC_OK) return ra;
  dim3 grid(prm.Hkv * prm.row_tiles, prm.S, prm.B);
  attn_partial_tc<NM><<<grid, C::kThreads, C::kSmem, st>>>(prm);
  return launch_status();
}

}  // namespace

namespace attn {

spec_status launch_partial_tc(const AttnParams& prm, int NM, cudaStream_t st) {
  return NM == 2 ? launch_nm<2>(prm, st) : launch_nm<1>(prm, st);
}

}  // namespace attn
