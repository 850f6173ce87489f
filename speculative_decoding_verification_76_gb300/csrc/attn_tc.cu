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
// Two kernels share the pieces below.  A CTA owns one chunk of one KV head
// and NM 128-row tiles of its R * G query rows:
//   * NM = 1 (up to 128 rows: the long chain): Q in tensor memory, two score
//     buffers (the next tile's scores computed while the softmax works).
//   * NM = 2 (more rows: the draft tree): two 128-row tiles share every K/V
//     stage, halving the K/V traffic into shared memory; Q in shared memory,
//     one score buffer per tile, the two tiles' softmax and MMAs ping-pong.
// Warp roles:
//   * 2 copy warps stream 128-token K/V stages (16-byte cp.async through the
//     block table, one page lookup per token) into a ring, laid out as the
//     128-byte-swizzled operands the tensor cores read: K as a K-major B
//     operand, V as an MN-major B operand.  Each copy thread's copies arrive
//     on the stage's barrier when they land; the MMA thread fences the stage
//     into the async proxy after its wait.
//   * 1 MMA warp (one thread issues): S = Q K^T (M = 128 rows, N = 128 tokens,
//     K = 128 dims: 8 MMAs per tile), then O += P V (K = 128 tokens: 8 MMAs,
//     N = 128 dims) with P read from tensor memory.  A tcgen05.mma costs a
//     roughly fixed issue time, so each instruction covers 128 tokens.
//   * 4 softmax warps per tile (a thread owns one row): per tile load the
//     row's 128 scores from tensor memory in one batch (a wait after every
//     load measured ~20x slower than one wait for all four), mask, maximum,
//     exp2 on the SFU, sum, pack P as bf16 pairs and store it over the scores.
//     (A cubic 2^x on the FMA pipe for half of the elements measured slower:
//     537 vs 375 us on the draft-tree shape.)
//     The running maximum is raised lazily: O is rescaled only when a row's
//     maximum grows by more than 2^8 (p stays <= 256, exact in the final
//     O / l), so the O read-modify-write is rare.
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
constexpr int kCopyWarps = 2;
constexpr int kCopyThreads = 32 * kCopyWarps;
constexpr float kRescaleLog2 = 8.0f;    // rescale O when a row maximum grows by > 2^8
constexpr uint32_t kTmemCols = 512;
constexpr int kBtBytes = (kMaxChunk / 16 + 8) * 4;

// The chunk a CTA owns.
struct Chunk {
  int kvh, rt, s, b, ctx, kv_len, c0, c1, nst;
};

SPEC_DEV Chunk chunk_of(const AttnParams& p) {
  Chunk c;
  c.kvh = blockIdx.x % p.Hkv;
  c.rt = blockIdx.x / p.Hkv;
  c.s = blockIdx.y;
  c.b = blockIdx.z;
  c.ctx = p.ctx_len[c.b];
  c.kv_len = c.ctx + p.R;
  c.c0 = c.s * p.chunk;
  c.c1 = min(c.c0 + p.chunk, c.kv_len);
  c.nst = (c.c1 - c.c0 + kST - 1) / kST;
  return c;
}

// Copy warps: the chunk's block-table slice, then its K/V stages into a ring
// of NS stages.  pt = thread index among the copy threads.  FIRST: the K/V
// rows leave L2 first (a pass whose only reader of a chunk is this CTA).
template <int NS, bool FIRST>
SPEC_DEV void copy_stages(const AttnParams& p, const Chunk& ch, uint8_t* stages, int32_t* bt_s,
                          uint64_t* kv_full, uint64_t* kv_empty, int pt) {
  const int P = p.page_size;
  const int pg0 = ch.c0 / P;
  const int npg = (ch.c1 - 1) / P - pg0 + 1;
  for (int i = pt; i < npg; i += kCopyThreads)
    bt_s[i] = (pg0 + i < p.max_pages) ? p.block_table[(size_t)ch.b * p.max_pages + pg0 + i] : -1;
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
    const int chn = 4 * c4 + u;
    col[u] = (uint32_t)((chn >> 3) * kHalf + (((chn & 7) ^ (tl & 7)) << 4));
  }
  const size_t tok_stride = (size_t)p.Hkv * 256;
  const uint8_t* kcol = reinterpret_cast<const uint8_t*>(p.k) + (size_t)ch.kvh * 256 + c4 * 64;
  const uint8_t* vcol = reinterpret_cast<const uint8_t*>(p.v) + (size_t)ch.kvh * 256 + c4 * 64;
  const bool pow2 = (P & (P - 1)) == 0;
  const int pshift = __ffs(P) - 1;
  uint64_t pol;
  if (FIRST)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  for (int k = 0; k < ch.nst; ++k) {
    const int slot = k % NS;
    if (k >= NS && !mbar_wait(&kv_empty[slot], ((k / NS) - 1) & 1, p.err, p.wait_ns)) break;
    const uint32_t sbase = smem_u32(stages + slot * kStageBytes);
#pragma unroll 4
    for (int jt = 0; jt < kST / kTokLanes; ++jt) {
      const int tok = tl + kTokLanes * jt;
      const int t = ch.c0 + k * kST + tok;
      int pg = -1, slotp = 0;
      if (t < ch.kv_len) {
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
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
                         drow + col[u]),
                     "l"(kcol + row + 16 * u), "r"(n), "l"(pol)
                     : "memory");
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
                         drow + col[u] + 2 * kHalf),
                     "l"(vcol + row + 16 * u), "r"(n), "l"(pol)
                     : "memory");
      }
    }
    // the stage's barrier counts this thread once its copies have landed
    if (k != p.withhold_stage)  // (a test can withhold one stage: its waiters time out)
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                       smem_u32(&kv_full[slot]))
                   : "memory");
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncwarp();
}

// The 8 MMAs of S = Q K^T (128 rows x 128 tokens) with A = Q from tensor
// memory (a_tq) or from shared memory (a_sq: 128-byte-swizzled K-major Q,
// 64-dim halves 16 KB apart).
SPEC_DEV void mma_scores(uint32_t d, bool q_in_tmem, uint32_t a_tq, uint32_t a_sq, uint32_t kb) {
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, kST, false, false);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    // 16 dims: 8 columns of Q in tensor memory, or 32 bytes inside a 64-dim atom
    const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
    if (q_in_tmem) {
      tc_mma_ts(d, a_tq + kk * 8, bd, idesc_s, kk > 0 ? 1u : 0u);
    } else {
      const uint64_t ad = smem_desc_sw128(a_sq + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
      tc_mma_ss(d, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
    }
  }
}

// The 8 MMAs of O (+)= P V: P (128 rows x 128 tokens, bf16 pairs) in tensor
// memory at pa, V of the stage at vb (MN-major: 64-dim blocks kHalf apart).
SPEC_DEV void mma_pv(uint32_t o, uint32_t pa, uint32_t vb, bool first) {
  constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
  for (int kk = 0; kk < kST / 16; ++kk) {
    // 16 tokens = 8 columns of P; 2 swizzle atoms (2 KB) of V
    const uint64_t bd = smem_desc_sw128(vb + kk * 2048, kHalf, 1024);
    tc_mma_ts(o, pa + kk * 8, bd, idesc_o, (!first || kk > 0) ? 1u : 0u);
  }
}

// Row state of one softmax thread.
struct RowState {
  float m_run = -INFINITY;  // running maximum (log2 domain, scaled)
  float l_run = 0.f;        // running sum of p
};

// One tile of one row (a softmax thread; whole warps call it): scores at
// s_addr (128 columns) -> P at s_addr (64 columns); a rescale of O (o_addr)
// waits for the previous PV through o_wait().  Returns false if a wait ran out.
template <class OWait>
SPEC_DEV bool softmax_tile(const AttnParams& p, RowState& st, uint32_t s_addr, uint32_t o_addr,
                           int t0, int ctx, uint64_t w, bool first, OWait&& o_wait) {
  const bool masked = t0 + kST > ctx;  // block positions (or past the sequence) in the tile
  uint32_t sv[4][32];
#pragma unroll
  for (int cb = 0; cb < 4; ++cb) tmem_ld32(s_addr + cb * 32, sv[cb]);
  tmem_wait_ld();
  if (masked) {
#pragma unroll
    for (int cb = 0; cb < 4; ++cb)
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int jb = t0 + cb * 32 + c - ctx;
        const bool vis = jb < 0 || (jb < p.R && ((w >> jb) & 1ull));
        if (!vis) sv[cb][c] = __float_as_uint(-INFINITY);
      }
  }
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int cb = 0; cb < 4; ++cb)
#pragma unroll
    for (int c = 0; c < 16; ++c)
      m4[c & 3] = fmax3(m4[c & 3], __uint_as_float(sv[cb][2 * c]),
                        __uint_as_float(sv[cb][2 * c + 1]));
  const float mnew = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
  const bool need = mnew > st.m_run + kRescaleLog2;
  float alpha = 1.f;
  if (need) {
    alpha = fast_exp2(st.m_run - mnew);  // 0 on the first visible tile
    st.l_run *= alpha;
    st.m_run = mnew;
  }
  // p = exp2(s * scale - m) and the row sum; P packed as bf16 pairs in place
  // (pair c of a 32-score block into word c), then written over the scores
  const float base = (st.m_run == -INFINITY) ? 0.f : st.m_run;
  // the scaling of a score pair and the running sums in packed f32x2
  const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nb2 = f2_pack(-base, -base);
  uint64_t rs2[2] = {0ull, 0ull};  // +0.0f pairs
#pragma unroll
  for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[cb][2 * c]), __uint_as_float(sv[cb][2 * c + 1])),
                       sc2, nb2),
                x0, x1);
      const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
      rs2[c & 1] = f2_add(rs2[c & 1], f2_pack(e0, e1));
      sv[cb][c] = pack_bf16(e0, e1);
    }
  }
  float rs[4];
  f2_unpack(rs2[0], rs[0], rs[1]);
  f2_unpack(rs2[1], rs[2], rs[3]);
  bool ok = true;
  if (!first && __any_sync(0xffffffffu, need)) {
    // rescale this warp's rows of O once the previous PV has completed (after
    // the packing, so that only the 64 packed words of P stay live)
    ok = o_wait();
    if (ok) {
      tc_fence_after();
      const float a = need ? alpha : 1.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[2][32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) tmem_ld32(o_addr + (2 * half + cc) * 32, o[cc]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[cc][i] = __float_as_uint(__uint_as_float(o[cc][i]) * a);
          tmem_st32(o_addr + (2 * half + cc) * 32, o[cc]);
        }
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
  st.l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
  tmem_wait_st();
  return ok;
}

// O / l and the log2-domain LSE of this chunk for one row (whole warps call it).
SPEC_DEV void write_partial(const AttnParams& p, const Chunk& ch, const RowState& st,
                            uint32_t o_addr, int rho, bool valid) {
  const float inv = st.l_run > 0.f ? 1.f / st.l_run : 0.f;
  const size_t prow = (((size_t)ch.b * p.Hkv + ch.kvh) * p.RGpad + rho) * p.S + ch.s;
  float4* dst = reinterpret_cast<float4*>(p.o_part + prow * 128);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t o[2][32];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) tmem_ld32(o_addr + (2 * half + cc) * 32, o[cc]);
    tmem_wait_ld();
    if (valid) {
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[(2 * half + cc) * 8 + i] = make_float4(
              __uint_as_float(o[cc][4 * i]) * inv, __uint_as_float(o[cc][4 * i + 1]) * inv,
              __uint_as_float(o[cc][4 * i + 2]) * inv, __uint_as_float(o[cc][4 * i + 3]) * inv);
    }
  }
  if (valid) p.lse_part[prow] = st.l_run > 0.f ? st.m_run + __log2f(st.l_run) : -INFINITY;
}

// One Q row (256 bytes) as 64 32-bit words (zeros for a row no output needs).
SPEC_DEV void load_q_row(const AttnParams& p, const Chunk& ch, int rho, bool valid,
                         uint32_t (&qa)[32], uint32_t (&qb)[32]) {
  if (valid) {
    const int i = rho / p.G, g = rho % p.G;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + (((size_t)ch.b * p.R + i) * p.Hq + (size_t)ch.kvh * p.G + g) * 128);
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
}

// ============================================================== NM = 1
namespace one {
constexpr int kStages = 3;
constexpr int kSoftWarps = 4, kMmaWarp = 4, kCopyWarp0 = 5;
constexpr int kThreads = 32 * (kSoftWarps + 1 + kCopyWarps);
constexpr int kColQ = 0, kColS = 64, kColO = 320;  // Q, score buffers x2, O
constexpr int kOffBt = kStages * kStageBytes;
constexpr int kOffBar = kOffBt + kBtBytes;
// kv_full[S], kv_empty[S], s_full[2], p_full, o_done, q_full, mma_done
constexpr int kNumBars = 2 * kStages + 6;
constexpr int kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
static_assert(kSmem <= 232448, "shared memory per CTA");
}  // namespace one

__global__ void __launch_bounds__(one::kThreads, 1) attn_partial_tc1(const AttnParams p) {
  using namespace one;
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

  const Chunk ch = chunk_of(p);
  if (ch.c0 >= ch.kv_len) return;  // this sequence needs fewer chunks (uniform over the CTA)
  const int nst = ch.nst;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], kCopyThreads);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 1);  // one arrival per tile, after the tile's named barrier
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
    copy_stages<kStages, true>(p, ch, stages, bt_s, kv_full, kv_empty, threadIdx.x - 32 * kCopyWarp0);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, p.err, p.wait_ns);
      tc_fence_after();
      for (int j = 0; ok && j <= nst; ++j) {
        if (j < nst) {  // S(j) = Q K_j^T into score buffer j & 1
          const int slot = j % kStages;
          if (!mbar_wait(&kv_full[slot], (j / kStages) & 1, p.err, p.wait_ns)) break;
          fence_proxy_async();  // the copy warps' generic-proxy writes, seen by the tensor cores
          // the buffer held P(j - 2): PV(j - 2) must have read it
          if (j >= 2 && !mbar_wait(o_done, (j - 2) & 1, p.err, p.wait_ns)) break;
          tc_fence_after();
          mma_scores(tmem + kColS + (j & 1) * kST, true, tmem + kColQ, 0,
                     smem_u32(stages + slot * kStageBytes));
          tc_commit(&s_full[j & 1]);
        }
        if (j >= 1) {  // O += P(j-1) V_{j-1}
          const int jj = j - 1;
          const int slot = jj % kStages;
          if (!mbar_wait(p_full, jj & 1, p.err, p.wait_ns)) break;
          tc_fence_after();
          mma_pv(tmem + kColO, tmem + kColS + (jj & 1) * kST,
                 smem_u32(stages + slot * kStageBytes) + 2 * kHalf, jj == 0);
          tc_commit(o_done);
          tc_commit(&kv_empty[slot]);  // the stage is free once these MMAs complete
        }
      }
      tc_commit(mma_done);  // every issued MMA completes before tensor memory is freed
      mbar_wait(mma_done, 0, nullptr);  // never cut short: TMEM is freed next
    }
    __syncwarp();
  } else {
    // softmax warps: warp w owns rows 32 w .. 32 w + 31 of the tile
    const int r = warp * 32 + lane;
    const int rho = ch.rt * 128 + r;  // row rho = i * G + g of this KV head
    const bool valid = rho < p.RG;
    const bool warp_live = ch.rt * 128 + warp * 32 < p.RG;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    {  // this thread's Q row into tensor memory (the A operand of S = Q K^T)
      uint32_t qa[32], qb[32];
      load_q_row(p, ch, rho, valid, qa, qb);
      tmem_st32(lane_base + kColQ, qa);
      tmem_st32(lane_base + kColQ + 32, qb);
      tmem_wait_st();
    }
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");
    if (threadIdx.x == 0) mbar_arrive(q_full);

    const uint64_t w = valid ? attn::row_mask(p, ch.b, rho / p.G) : 0ull;
    const uint32_t o_addr = lane_base + kColO;
    RowState st;
    bool ok = true;
    for (int j = 0; j < nst; ++j) {
      if (ok && !mbar_wait(&s_full[j & 1], (j >> 1) & 1, p.err, p.wait_ns)) ok = false;
      tc_fence_after();
      // (rows no output needs have a zero Q, so their scores -- read as P by the
      // PV MMA -- are zero)
      if (ok && warp_live)
        ok = softmax_tile(p, st, lane_base + kColS + (j & 1) * kST, o_addr, ch.c0 + j * kST,
                          ch.ctx, w, j == 0,
                          [&]() { return mbar_wait(o_done, (j - 1) & 1, p.err, p.wait_ns); });
      // all four warps have stored P(j) before it is signalled: a warp that is
      // done early must not start tile j + 1 (whose scores may be ready) and
      // signal again.  Every thread passes here on every tile, even after a
      // wait ran out, so the barrier cannot strand the others.
      tc_fence_before();
      asm volatile("bar.sync 3, %0;" ::"n"(32 * kSoftWarps) : "memory");
      if (threadIdx.x == 0) mbar_arrive(p_full);
    }
    if (ok && mbar_wait(o_done, (nst - 1) & 1, p.err, p.wait_ns)) {
      tc_fence_after();
      if (warp_live) write_partial(p, ch, st, o_addr, rho, valid);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================== NM = 2
namespace two {
constexpr int kStages = 2;
constexpr int kSoftWarps = 8, kMmaWarp = 8, kCopyWarp0 = 9;
constexpr int kThreads = 32 * (kSoftWarps + 1 + kCopyWarps);
// tensor memory: score / P buffer of tile m at 128 m, O of tile m at 256 + 128 m
constexpr int kColS = 0, kColO = 256;
constexpr int kOffQ = kStages * kStageBytes;  // 2 x (Q lo 16 KB + Q hi 16 KB)
constexpr int kOffBt = kOffQ + 2 * 32768;
constexpr int kOffBar = kOffBt + kBtBytes;
// kv_full[S], kv_empty[S], s_full[2], p_full[2], o_done[2], q_full, mma_done
constexpr int kNumBars = 2 * kStages + 8;
constexpr int kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
static_assert(kSmem <= 232448, "shared memory per CTA");
}  // namespace two

__global__ void __launch_bounds__(two::kThreads, 1) attn_partial_tc2(const AttnParams p) {
  using namespace two;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* qs = smem + kOffQ;
  int32_t* bt_s = reinterpret_cast<int32_t*>(smem + kOffBt);
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* q_full = o_done + 2;
  uint64_t* mma_done = q_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const Chunk ch = chunk_of(p);
  if (ch.c0 >= ch.kv_len) return;
  const int nst = ch.nst;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], kCopyThreads);
      mbar_init(&kv_empty[i], 1);
    }
    for (int m = 0; m < 2; ++m) {
      mbar_init(&s_full[m], 1);
      mbar_init(&p_full[m], 1);  // one arrival per tile, after the tile's named barrier
      mbar_init(&o_done[m], 1);
    }
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
    copy_stages<kStages, false>(p, ch, stages, bt_s, kv_full, kv_empty, threadIdx.x - 32 * kCopyWarp0);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, p.err, p.wait_ns);
      tc_fence_after();
      const uint32_t q0 = smem_u32(qs);
      for (int j = 0; ok && j < nst; ++j) {
        const int slot = j % kStages;
        if (!mbar_wait(&kv_full[slot], (j / kStages) & 1, p.err, p.wait_ns)) break;
        fence_proxy_async();  // the copy warps' generic-proxy writes, seen by the tensor cores
        const uint32_t kb = smem_u32(stages + slot * kStageBytes);
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // S_m(j) once PV_m(j-1) has read P_m(j-1)
          if (j >= 1 && !mbar_wait(&o_done[m], (j - 1) & 1, p.err, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_scores(tmem + kColS + m * kST, false, 0, q0 + m * 32768, kb);
          tc_commit(&s_full[m]);
        }
        if (!ok) break;
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // O_m += P_m(j) V_j
          if (!mbar_wait(&p_full[m], j & 1, p.err, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_pv(tmem + kColO + m * 128, tmem + kColS + m * kST, kb + 2 * kHalf, j == 0);
          tc_commit(&o_done[m]);
        }
        if (!ok) break;
        tc_commit(&kv_empty[slot]);  // the stage is free once these MMAs complete
      }
      tc_commit(mma_done);  // every issued MMA completes before tensor memory is freed
      mbar_wait(mma_done, 0, nullptr);  // never cut short: TMEM is freed next
    }
    __syncwarp();
  } else {
    // softmax warps: warp w owns rows 32 (w % 4) .. + 31 of row tile w / 4
    const int m = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int rho = ch.rt * 256 + m * 128 + r;
    const bool valid = rho < p.RG;
    const bool warp_live = ch.rt * 256 + m * 128 + quarter * 32 < p.RG;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    {  // this thread's Q row into shared memory (128-byte swizzle, K-major)
      uint32_t qa[32], qb[32];
      load_q_row(p, ch, rho, valid, qa, qb);
      uint8_t* qrow = qs + m * 32768 + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int sw = (c ^ (r & 7)) << 4;
        *reinterpret_cast<uint4*>(qrow + sw) =
            make_uint4(qa[4 * c], qa[4 * c + 1], qa[4 * c + 2], qa[4 * c + 3]);
        *reinterpret_cast<uint4*>(qrow + 16384 + sw) =
            make_uint4(qb[4 * c], qb[4 * c + 1], qb[4 * c + 2], qb[4 * c + 3]);
      }
    }
    fence_proxy_async();
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");
    if (threadIdx.x == 0) mbar_arrive(q_full);

    const uint64_t w = valid ? attn::row_mask(p, ch.b, rho / p.G) : 0ull;
    const uint32_t s_addr = lane_base + kColS + m * kST;
    const uint32_t o_addr = lane_base + kColO + m * 128;
    RowState st;
    bool ok = true;
    for (int j = 0; j < nst; ++j) {
      if (ok && !mbar_wait(&s_full[m], j & 1, p.err, p.wait_ns)) ok = false;
      tc_fence_after();
      if (ok && warp_live)
        ok = softmax_tile(p, st, s_addr, o_addr, ch.c0 + j * kST, ch.ctx, w, j == 0,
                          [&]() { return mbar_wait(&o_done[m], (j - 1) & 1, p.err, p.wait_ns); });
      // the tile's four warps have stored P_m(j) before it is signalled (see the
      // one-tile kernel); every thread passes here on every tile
      tc_fence_before();
      if (m == 0)
        asm volatile("bar.sync 3, 128;" ::: "memory");
      else
        asm volatile("bar.sync 4, 128;" ::: "memory");
      if (quarter == 0 && lane == 0) mbar_arrive(&p_full[m]);
    }
    if (ok && mbar_wait(&o_done[m], (nst - 1) & 1, p.err, p.wait_ns)) {
      tc_fence_after();
      if (warp_live) write_partial(p, ch, st, o_addr, rho, valid);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace attn {

spec_status launch_partial_tc(const AttnParams& prm, int rows_per_cta, cudaStream_t st) {
  dim3 grid(prm.Hkv * prm.row_tiles, prm.S, prm.B);
  if (rows_per_cta == 256) {
    static PerDeviceOnce<int> smem_once;
    const spec_status ra =
        ensure_smem_limit(smem_once, (const void*)attn_partial_tc2, two::kSmem);
    if (ra != SPEC_OK) return ra;
    attn_partial_tc2<<<grid, two::kThreads, two::kSmem, st>>>(prm);
  } else {
    static PerDeviceOnce<int> smem_once;
    const spec_status ra =
        ensure_smem_limit(smem_once, (const void*)attn_partial_tc1, one::kSmem);
    if (ra != SPEC_OK) return ra;
    attn_partial_tc1<<<grid, one::kThreads, one::kSmem, st>>>(prm);
  }
  return launch_status();
}

}  // namespace attn
