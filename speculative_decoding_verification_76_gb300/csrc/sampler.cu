// spec_accept_sample / spec_accept_sample_tree: the lossless acceptance
// sampler of the verify step.
//
// Method ("Speculative Decoding" (atlas), sections "One round and shifted
// logits", "Exact sampling: account for every probability", "Greedy,
// sampling and the real sampler"; "Drafters and Speculative Decoding",
// "Sampling needs a correction rule"):
//   p_i = softmax over the kept set of logits_i / T (top-k, then top-p);
//   draft x_{i+1} is accepted iff u_i * q_i(x_{i+1}) < p_i(x_{i+1});
//   at the first rejection r the correction is drawn from
//   norm(max(0, p_r - q_r)); if every draft survives the bonus is drawn
//   from p_gamma; greedy mode accepts while the draft equals the argmax.
//
// GB300 design.  One thread-block cluster (up to 8 CTAs) per target row
// holds that row in distributed shared memory: each CTA bulk-copies (TMA)
// one slice of the vocabulary once and replaces it in place by
// E = exp((l - max)/T).  Every row computes its own outcome (its draft test,
// and its correction draw if it rejects; the last row's bonus draw; for a
// tree node the first accepted child under the running residual, or its
// final draw), so all B*R rows run at once; the cluster that finishes a
// sequence's last row assembles the outcomes.
//
// The normaliser, the top-k / top-p cut and the draws need at most four
// cluster exchanges per row:
//   1. row maximum (and argmax, greedy);
//   2. Z, and (truncation only) a histogram of E: 32 bins per octave of E
//      (all E of a bin share one exponent), each holding its element count
//      and the sum of its rounded 16-bit significands, which locates the
//      bins the cut can fall in;
//   3. (truncation only) the members of those bins, gathered and sorted by
//      (logit desc, id asc) in every CTA, and the exact mass above them; the
//      cut is found on exact integer masses (units of 2^-44);
//   4. per-CTA sums of the draw weights; the CTA holding the crossing finds
//      the token with one warp scan.
// Values another CTA needs (E at a draft token, the residual at the next
// child's token) travel in the exchange posts, so no CTA reads another's
// vocabulary slice.  A crossing range too populous to sort (or a cut the
// rounded bin masses placed one bin off) falls back to an exact radix
// selection over the logit keys.  Shared-memory atomics are 32-bit only:
// 64-bit and float atomics on shared memory are many times slower on sm_103.
//
// Many truncated rows at once (more cluster CTAs than twice the SMs) take the
// streaming kernel further below instead: one 1024-thread CTA per row, one
// sweep of the row into per-warp candidate lists, no cluster exchanges.
//
// Numerics: exp((l - m)/T) = 2^x with x = (l - m) * (1/(T ln 2)) carried as
// a float pair (Knuth's TwoSum for l - m, an FMA for the product error, the
// constant split in two floats) and 2^x_hi * (1 + x_lo ln 2) on the
// special-function unit; p matches a float64 evaluation to a few 1e-7.  When
// p is not returned (FAST), 2^x is one SFU exp2 of a single FMA: the
// decisions it feeds are compared with the oracle's, and the draws and tests
// within 1e-5 of a threshold are the ones flagged.
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"

namespace {

constexpr int kMaxCS = 8;
constexpr int kMaxN = 64;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kBins = 1024;                 // 32 per octave of E over 32 octaves; bin kBins: the rest
constexpr int kHist = kBins + 1;
constexpr int kHistPad = 1032;
constexpr int kCandMax = 512;               // members of the crossing bins, whole cluster
constexpr int kListPerCTA = 2048;           // kept positions listed per CTA (split over warps)
constexpr size_t kMaxSliceBytes = 84 * 1024;
constexpr float kLn2 = 0.6931471805599453f;

// Outcome of one target row, written by rank 0 of its cluster.
struct Outcome {
  int32_t accept;  // chain: 1 if the row's draft is accepted; tree: accepted child or -1
  int32_t token;   // correction / bonus / final token of this row (-1 if none)
  int32_t status;  // SPEC_SEQ_* bits raised by this row
  int32_t flags;   // 1 if the row's logits are not finite
};

// Per warp range of a row, from the streaming pre-pass (many-row sampling).
struct RangeStat {
  float m;       // maximum of the range's logits (NaN-propagating; -inf if all are -inf)
  float zh, zl;  // Z of the range relative to its finite maximum, as a float pair
  int32_t cnt;   // ids at or above the row's candidate floor (> kSWCap: not all stored)
};

struct SP {
  const float* logits;
  const float* q;
  const int32_t* tokens;
  const int32_t* parent;
  const float* u;
  int B, R, V, slice;
  float T, c_hi, c_lo;  // 1/(T ln 2) = c_hi + c_lo
  int top_k;
  float top_p;
  int greedy, eos, tree, bulk, qbulk, qsm;
  Outcome* outcomes;
  int32_t* seq_count;
  int32_t* err;
  int32_t* acc_len;
  int32_t* emitted;
  int32_t* path;
  float* p_out;
  int32_t* status;
  // streaming pre-pass results (nullptr: the row kernel sweeps the row itself)
  RangeStat* stats;   // [rows][32]
  float* lfloor;      // [rows][2]: candidate floor as a logit (+inf: no lists), samples' maximum
  int32_t* lid_g;     // [rows][32][kSwW][kSegCap] listed ids per range segment, ascending
  float* lval_g;      // [rows][32][kSwW][kSegCap] their logits
  int32_t* segcnt;    // [rows][32][kSwW] ids listed per segment
};

// One CTA's contribution to a cluster exchange (32 bytes).
struct alignas(16) Post {
  unsigned long long w[4];
};

SPEC_DEV unsigned long long f2w(float f) { return (unsigned long long)__float_as_uint(f); }
SPEC_DEV float w2f(unsigned long long w) { return __uint_as_float((uint32_t)w); }

// The top-k / top-p cut.  Kept: key(l) > tau, or key == tau and id <= tie.
// mode 0: no truncation; 1: decided through E (E > etau kept, E < etau not,
// ties through the logit key); 2: through the logit key only.
struct Cut {
  int mode;
  float etau;
  uint32_t tau;
  int tie;
};

template <int NW>
struct Sh {
  Post posts[2];
  Post gath[kMaxCS];
  float red_f[NW];
  int red_i[NW];
  float wsum[NW];
  unsigned long long red_u[NW];
  unsigned long long zk, zcut;
  uint32_t oct[64];  // this CTA's per-octave counts [0, 32) and m16 sums [32, 64)
  uint32_t octc[32];            // one-CTA rows: per-octave counts
  unsigned long long octm[32];  // and m16 sums
  int list_n[NW];
  int bi[8];
  Cut cut;
  int par[kMaxN];
  int tok[kMaxN];
  float invw_used[kMaxN];
  Outcome outs[kMaxN];
  int cpos[kMaxN];  // list position of each child's token (-1: not kept)
  float zpre[2];    // Z as a float pair, from the streaming pre-pass
  float eprobe;
  int token_in;
  uint64_t bar;
};

// ---------------------------------------------------------------- scalar helpers
// order-preserving key: larger float -> larger key; -0 and +0 share a key
SPEC_DEV uint32_t okey(float x) {
  uint32_t u = __float_as_uint(x);
  if (x == 0.f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

SPEC_DEV bool is_kept(uint32_t key, int id, uint32_t tau, int tie) {
  return key > tau || (key == tau && id <= tie);
}

// global loads that ask L2 to keep the line (the row is swept several times):
// an L2 cache policy with evict-last priority
SPEC_DEV uint64_t l2_keep_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// L2 policy for data read once
SPEC_DEV uint64_t l2_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
SPEC_DEV float4 ldg_keep4(const float4* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
SPEC_DEV float ldg_keep(const float* p, uint64_t pol) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
  return v;
}

SPEC_DEV float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// three-input maximum, NaN-propagating (sm_100+)
SPEC_DEV float fmax3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

SPEC_DEV float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

SPEC_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp((l - m) / T) with nm = -m, lfloor = m - 150 T (below it E is 0 in float).
SPEC_DEV float texp(float l, float nm, float lfloor, float c_hi, float c_lo) {
  const float lc = fmaxf(l, lfloor);
  const float s = __fadd_rn(lc, nm);
  const float bv = __fsub_rn(s, lc);
  const float av = __fsub_rn(s, bv);
  const float e = __fadd_rn(__fsub_rn(lc, av), __fsub_rn(nm, bv));
  const float xh = __fmul_rn(s, c_hi);
  float xl = __fmaf_rn(s, c_hi, -xh);
  xl = __fmaf_rn(s, c_lo, xl);
  xl = __fmaf_rn(e, c_hi, xl);
  const float y = ex2_approx(xh);
  return __fmaf_rn(y, __fmul_rn(xl, kLn2), y);
}

// exp((l - m) / T) with one FMA and the special-function unit: nmc = -m * c_hi.
// Used when p itself is not returned: the decisions only need p to a few
// 1e-6 relative (the error grows with the distance below the maximum, where
// p is tiny); the exact float-pair form above serves p_out.
SPEC_DEV float fexp(float l, float c_hi, float nmc) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(__fmaf_rn(l, c_hi, nmc)));
  return y;  // results below 2^-126 flush to 0: such p cannot decide anything
}

// Histogram bin of E in [0, 1]: bins 0..1023 hold 32 per octave, all E of a
// bin share one exponent (126 - b/32); bin 1024 holds the rest (E < 2^-32).
SPEC_DEV int ebin(uint32_t bits) {
  return min((0x3F7FFFFF - (int)min(bits, 0x3F7FFFFFu)) >> 18, kBins);  // E >= 1: bin 0
}

// E rounded to a 16-bit significand, in units of 2^(-16 - b/32) of its bin b
SPEC_DEV uint32_t m16(uint32_t bits) {
  // E >= 1 clamps to the largest significand below 1, which rounds to 65536 = 1.0
  return ((((min(bits, 0x3F7FFFFFu) & 0x7FFFFFu) | 0x800000u) + 128u) >> 8);
}

// a bin's sum of m16 in units of 2^-44
SPEC_DEV unsigned long long bin_fx(unsigned long long m, int b) {
  const int o = b >> 5;
  return o <= 28 ? m << (28 - o) : m >> (o - 28);
}

// E (normal, <= 1) in units of 2^-44, exact for E >= 2^-20
SPEC_DEV unsigned long long fx44(uint32_t bits) {
  const int f = (int)(bits >> 23);
  if (f == 0) return 0ull;
  const unsigned long long sig = (bits & 0x7FFFFFu) | 0x800000u;
  const int sh = f - 106;
  return sh >= 0 ? sig << sh : (sh > -24 ? sig >> (-sh) : 0ull);
}

// x * 2^44 truncated toward zero, from the float's fields (|x| < 2^19)
SPEC_DEV long long fx44_signed(float x) {
  const uint32_t b = __float_as_uint(x);
  const int f = (int)((b >> 23) & 0xFFu);
  if (f == 0) return 0ll;
  const unsigned long long sig = (b & 0x7FFFFFu) | 0x800000u;
  const int sh = f - 106;
  const unsigned long long v = sh >= 0 ? sig << min(sh, 39) : (sh > -24 ? sig >> (-sh) : 0ull);
  return (b >> 31) ? -(long long)v : (long long)v;
}

// a float pair's sum in units of 2^-44 (a non-negative total)
SPEC_DEV unsigned long long fx44_pair(float hi, float lo) {
  return (unsigned long long)(fx44_signed(hi) + fx44_signed(lo));
}

// floor(z * f) for a float f in (0, 1): exact, on the 128-bit product
SPEC_DEV unsigned long long mul_frac(unsigned long long z, float f) {
  const uint32_t b = __float_as_uint(f);
  const int ex = (int)((b >> 23) & 0xFFu);
  if (ex == 0) return 0ull;
  const unsigned long long sig = (b & 0x7FFFFFu) | 0x800000u;
  const int sh = 150 - ex;  // f = sig * 2^-sh; sh >= 24 for f < 1
  if (sh <= 0) return z;
  const unsigned long long lo = z * sig, hi = __umul64hi(z, sig);
  if (sh >= 128) return 0ull;
  if (sh >= 64) return hi >> (sh - 64);
  return (hi << (64 - sh)) | (lo >> sh);
}

SPEC_DEV float residual_w(float v, float invw, float qv) {
  return fmaxf(__fmaf_rn(v, invw, -qv), 0.f);
}

// (h, l) += (ah, al) in float pairs (TwoSum), fixed order
SPEC_DEV void df_acc(float& h, float& l, float ah, float al) {
  const float s = __fadd_rn(h, ah);
  const float bb = __fsub_rn(s, h);
  const float e = __fadd_rn(__fadd_rn(__fsub_rn(h, __fsub_rn(s, bb)), __fsub_rn(ah, bb)),
                            __fadd_rn(l, al));
  h = __fadd_rn(s, e);
  l = __fsub_rn(e, __fsub_rn(h, s));
}

// ---------------------------------------------------------------- block / cluster plumbing
template <int NT>
SPEC_DEV float block_sum_f(float v, Sh<NT / 32>& sh) {  // fixed order
  constexpr int NW = NT / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if ((threadIdx.x & 31) == 0) sh.red_f[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < NW; ++i) t += sh.red_f[i];
  __syncthreads();
  return t;
}

template <int NT>
SPEC_DEV unsigned long long block_sum_u64(unsigned long long v, Sh<NT / 32>& sh) {
  constexpr int NW = NT / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if ((threadIdx.x & 31) == 0) sh.red_u[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int i = 0; i < NW; ++i) t += sh.red_u[i];
  __syncthreads();
  return t;
}

// inclusive scan over the CTA's threads (thread order), exact
template <int NT>
SPEC_DEV unsigned long long block_incl_scan_u64(unsigned long long v, Sh<NT / 32>& sh) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) sh.red_u[w] = v;
  __syncthreads();
  unsigned long long base = 0;
  for (int i = 0; i < w && i < NW; ++i) base += sh.red_u[i];
  __syncthreads();
  return base + v;
}

template <int NT>
SPEC_DEV int block_min_i(int v, Sh<NT / 32>& sh) {
  constexpr int NW = NT / 32;
  v = __reduce_min_sync(kFull, v);
  if ((threadIdx.x & 31) == 0) sh.red_i[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = INT_MAX;
  for (int i = 0; i < NW; ++i) t = min(t, sh.red_i[i]);
  __syncthreads();
  return t;
}

template <int NT>
SPEC_DEV int block_excl_scan_i(int v, int* total, Sh<NT / 32>& sh) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh.red_i[w] = incl;
  __syncthreads();
  int base = 0, all = 0;
  for (int i = 0; i < NW; ++i) {
    if (i < w) base += sh.red_i[i];
    all += sh.red_i[i];
  }
  __syncthreads();
  *total = all;
  return base + incl - v;
}

// Every CTA posts one Post; afterwards sh.gath[r] holds rank r's post in
// every CTA.  Two post buffers alternate: a buffer is rewritten only two
// exchanges later, after every reader has passed the cluster barrier between.
template <int NW>
SPEC_DEV void exchange(const Post& mine, int CS, int& ph, Sh<NW>& sh) {
  Post* s = &sh.posts[ph & 1];
  if (threadIdx.x == 0) *s = mine;
  cluster_sync();
  if ((int)threadIdx.x < CS) {
    Post r;
#pragma unroll
    for (int j = 0; j < 4; ++j) r.w[j] = dsmem_ld_u64(&s->w[j], threadIdx.x);
    sh.gath[threadIdx.x] = r;
  }
  __syncthreads();
  ++ph;
}

SPEC_DEV bool cut_keeps(const Cut& c, float e, int id, const float* lrow_full) {
  if (c.mode == 0) return true;
  if (c.mode == 1) {  // E decides only well away from the cut's E (2^-20 relative)
    if (e > c.etau * (1.0f + 9.5367431640625e-07f)) return true;
    if (e < c.etau * (1.0f - 9.5367431640625e-07f)) return false;
  }
  return is_kept(okey(__ldg(lrow_full + id)), id, c.tau, c.tie);
}

// ---------------------------------------------------------------- kept-set iteration
// Each warp owns one contiguous range of the slice; its kept positions are
// either listed (per-warp list, ascending) or the whole range is walked.
template <int NW>
struct Items {
  bool listed;
  const uint16_t* lists;  // NW x (kListPerCTA / NW)
  int r0, r1;             // this warp's range [r0, r1)
  int rw, n;              // every warp's range: [min(w rw, n), min((w + 1) rw, n))
  SPEC_DEV int count(const Sh<NW>& sh) const { return count_of(threadIdx.x >> 5, sh); }
  SPEC_DEV int at(int j) const { return at_of(threadIdx.x >> 5, j); }
  SPEC_DEV int count_of(int w, const Sh<NW>& sh) const {
    return listed ? sh.list_n[w] : min((w + 1) * rw, n) - min(w * rw, n);
  }
  SPEC_DEV int at_of(int w, int j) const {
    return listed ? (int)lists[w * (kListPerCTA / NW) + j] : min(w * rw, n) + j;
  }
};

// Weights of the draw over this CTA's items: mode 0 uses buf as is, mode 1
// replaces buf by max(0, buf * invw - q) first.  Leaves per-warp sums in
// sh.wsum and returns the CTA total (fixed order).
template <int NT>
SPEC_DEV float weight_pass(float* buf, const Items<NT / 32>& it, int mode, float invw,
                           const float* qlo, bool q_shared, Sh<NT / 32>& sh) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31;
  const int cnt = it.count(sh);
  float acc = 0.f;
  int j = lane;
  if (mode == 1) {
    for (; j + 96 < cnt; j += 128) {  // four independent q loads in flight
      int k[4];
      float v[4], qv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        k[u] = it.at(j + 32 * u);
        v[u] = buf[k[u]];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        qv[u] = v[u] > 0.f ? (q_shared ? qlo[k[u]] : __ldg(qlo + k[u])) : 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        v[u] = residual_w(v[u], invw, qv[u]);
        buf[k[u]] = v[u];
        acc += v[u];
      }
    }
  }
  for (; j < cnt; j += 32) {
    const int k = it.at(j);
    float v = buf[k];
    if (mode == 1) {
      const float qv = v > 0.f ? (q_shared ? qlo[k] : __ldg(qlo + k)) : 0.f;
      v = residual_w(v, invw, qv);
      buf[k] = v;
    }
    acc += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
  if (lane == 0) sh.wsum[threadIdx.x >> 5] = acc;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < NW; ++w) t += sh.wsum[w];
  return t;
}

// Weights of a chain draw over this warp's whole range [r0, r1) with the cut
// applied inline: w = kept ? (mode 1: max(0, E * invw - q); mode 0: E) : 0,
// written back to buf for the walk.  Per-warp sums in sh.wsum, CTA total
// returned (fixed order).  r0 is a multiple of 4.
template <int NT>
SPEC_DEV float weight_full(float* buf, int r0, int r1, const Cut& cut, int lo,
                           const float* lrow_full, int mode, float invw, const float* qlo,
                           bool q_shared, bool q_vec, Sh<NT / 32>& sh) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31;
  const int r1v = r0 + ((r1 - r0) & ~3);
  float acc = 0.f;
  for (int k = r0 + 4 * lane; k < r1v; k += 128) {
    float4 e4 = *reinterpret_cast<const float4*>(buf + k);
    float ev[4] = {e4.x, e4.y, e4.z, e4.w};
    bool kp[4];
    bool all = true, any = false;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      kp[u] = ev[u] > 0.f && cut_keeps(cut, ev[u], lo + k + u, lrow_full);
      all &= kp[u];
      any |= kp[u];
    }
    float qv[4] = {0.f, 0.f, 0.f, 0.f};
    if (mode == 1 && any) {
      if (q_shared || (all && q_vec)) {
        const float4 q4 = q_shared ? *reinterpret_cast<const float4*>(qlo + k)
                                   : __ldg(reinterpret_cast<const float4*>(qlo + k));
        qv[0] = q4.x;
        qv[1] = q4.y;
        qv[2] = q4.z;
        qv[3] = q4.w;
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) qv[u] = kp[u] ? __ldg(qlo + k + u) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = kp[u] ? (mode == 1 ? residual_w(ev[u], invw, qv[u]) : ev[u]) : 0.f;
      ev[u] = w;
      acc += w;
    }
    *reinterpret_cast<float4*>(buf + k) = make_float4(ev[0], ev[1], ev[2], ev[3]);
  }
  for (int k = r1v + lane; k < r1; k += 32) {
    const float e = buf[k];
    const bool kp = e > 0.f && cut_keeps(cut, e, lo + k, lrow_full);
    float w = 0.f;
    if (kp) w = mode == 1 ? residual_w(e, invw, q_shared ? qlo[k] : __ldg(qlo + k)) : e;
    buf[k] = w;
    acc += w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
  if (lane == 0) sh.wsum[threadIdx.x >> 5] = acc;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < NW; ++w) t += sh.wsum[w];
  return t;
}

// After the exchange of CTA totals (post word 0): the draw's owner CTA finds
// the first item whose running weight (ascending id over the cluster)
// exceeds u * W and returns its id; other CTAs return -1; -2 if W == 0
// (same in every CTA).  The owner warp splits its items into one contiguous
// chunk per lane, scans the chunk sums and walks the one chunk that crosses.
template <int NT>
SPEC_DEV int locate(const float* buf, const Items<NT / 32>& it, int lo, float u, int rank, int CS,
                    Sh<NT / 32>& sh) {
  constexpr int NW = NT / 32;
  float W = 0.f;
  for (int r = 0; r < CS; ++r) W += w2f(sh.gath[r].w[0]);
  if (!(W > 0.f)) return -2;
  const float target = u * W;
  int owner = -1, last_nz = -1;
  float pre = 0.f, pre_owner = 0.f, pre_last = 0.f;
  for (int r = 0; r < CS; ++r) {
    const float t = w2f(sh.gath[r].w[0]);
    if (t > 0.f) {
      if (owner < 0 && pre + t > target) {
        owner = r;
        pre_owner = pre;
      }
      last_nz = r;
      pre_last = pre;
    }
    pre += t;
  }
  if (owner < 0) {
    owner = last_nz;
    pre_owner = pre_last;
  }
  if (owner != rank) return -1;
  int ow = -1, lw = -1;
  float wpre = pre_owner, base_ow = 0.f, base_lw = 0.f;
  for (int w = 0; w < NW; ++w) {
    const float t = sh.wsum[w];
    if (t > 0.f) {
      if (ow < 0 && wpre + t > target) {
        ow = w;
        base_ow = wpre;
      }
      lw = w;
      base_lw = wpre;
    }
    wpre += t;
  }
  if (ow < 0) {
    ow = lw;
    base_ow = base_lw;
  }
  if (ow < 0) return -1;  // unreachable: the owner CTA has positive weight
  // every warp walks the owning warp's items (a lone warp whose siblings wait
  // at a barrier runs its shuffles far slower)
  const int lane = threadIdx.x & 31;
  const int cnt = it.count_of(ow, sh);
  const int c = ((cnt + 31) / 32) | 1;  // odd chunk length: conflict-free shared reads
  const int j0 = min(lane * c, cnt), j1 = min(j0 + c, cnt);
  float ls = 0.f;
  for (int j = j0; j < j1; ++j) ls += buf[it.at_of(ow, j)];
  const float tw = target - base_ow;  // the crossing, relative to the warp's start
  float incl = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned hit = __ballot_sync(kFull, ls > 0.f && incl > tw);
  const unsigned nz = __ballot_sync(kFull, ls > 0.f);
  const int L = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : -1);
  int found = -1;
  if (lane == L) {
    const float tl = tw - (incl - ls);  // relative to this lane's chunk
    float run = 0.f;
    int lastk = -1;
    for (int j = j0; j < j1; ++j) {
      const int k = it.at_of(ow, j);
      const float v = buf[k];
      if (v > 0.f) {
        lastk = k;
        run += v;
        if (run > tl) {
          found = k;
          break;
        }
      }
    }
    if (found < 0) found = lastk;  // rounding left the crossing just past the end
  }
  found = __shfl_sync(kFull, found, L < 0 ? 0 : L);
  __syncthreads();  // callers may rewrite buf
  return (L < 0 || found < 0) ? -1 : lo + found;
}

// ---------------------------------------------------------------- exact radix fallback
// Radix selection over the logit keys (read from global memory), most
// significant digit first, of the position in (key desc, id asc) order where
// the running weight reaches the target.  Weight = 1 per element (top-k) or
// its 2^-40 fixed-point E (top-p).  Scratch: rcnt[2][256] u32,
// rmass[2][256] u64, rtmass[256] u64, rtcnt[256] u32.
struct RadixScratch {
  uint32_t* rcnt;
  unsigned long long* rmass;
  unsigned long long* rtmass;
  uint32_t* rtcnt;
};

struct Sel {
  uint32_t tau;
  unsigned long long above, at_weight, target;
  uint32_t at_count;
};

template <int NT, class Keep, class Weight>
SPEC_DEV Sel radix_select(const float* lrow, int n, bool target_is_fraction, double frac,
                          unsigned long long target_abs, Keep keep, Weight weight,
                          const RadixScratch& rs, int CS) {
  uint32_t prefix = 0, pmask = 0;
  unsigned long long above = 0, target = target_abs;
  Sel out{};
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int h = pass & 1;
    for (int i = threadIdx.x; i < 256; i += NT) {
      rs.rmass[h * 256 + i] = 0ull;
      rs.rcnt[h * 256 + i] = 0u;
    }
    __syncthreads();
    // the lanes of a warp that share a digit add their counts and weights
    // first (weights < 2^41: two 32-bit partial sums), one shared atomic per
    // digit and warp: the keys of a row crowd into a few digits
    const int lane = threadIdx.x & 31;
    constexpr int U = 8;  // logits in flight per thread
    for (int k0 = threadIdx.x - lane; k0 < n; k0 += U * NT) {  // warp-uniform
      float lv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * NT + lane;
        lv[u] = k < n ? __ldg(lrow + k) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * NT + lane;
        uint32_t label = 0xFFFFFFFFu;
        unsigned long long wt = 0;
        if (k < n) {
          const uint32_t key = okey(lv[u]);
          if ((key & pmask) == prefix && keep(k, key)) {
            label = (key >> shift) & 255u;
            wt = weight(k);
          }
        }
        const unsigned grp = __match_any_sync(kFull, label);
        if (label != 0xFFFFFFFFu) {
          const uint32_t hi = __reduce_add_sync(grp, (uint32_t)(wt >> 24));
          const uint32_t lo = __reduce_add_sync(grp, (uint32_t)(wt & 0xFFFFFFull));
          if (lane == __ffs(grp) - 1) {
            atomicAdd(&rs.rcnt[h * 256 + label], (uint32_t)__popc(grp));
            atomicAdd(&rs.rmass[h * 256 + label], ((unsigned long long)hi << 24) + lo);
          }
        }
      }
    }
    __syncthreads();
    cluster_sync();
    for (int d = threadIdx.x; d < 256; d += NT) {
      unsigned long long mm = 0;
      uint32_t c = 0;
      for (int r = 0; r < CS; ++r) {
        mm += dsmem_ld_u64(&rs.rmass[h * 256 + d], r);
        c += dsmem_ld_u32(&rs.rcnt[h * 256 + d], r);
      }
      rs.rtmass[255 - d] = mm;  // descending digit order
      rs.rtcnt[255 - d] = c;
    }
    __syncthreads();
    if (pass == 0 && target_is_fraction) {
      unsigned long long tot = 0;
      for (int d = 0; d < 256; ++d) tot += rs.rtmass[d];
      const double thr = ceil(frac * (double)tot);
      target = thr < 1.0 ? 1ull : (unsigned long long)thr;
      if (target > tot) target = tot;
    }
    const unsigned long long need = target - above;
    unsigned long long cum = 0;
    int sel = 255;
    for (int d = 0; d < 256; ++d) {  // every thread, identical result
      if (cum + rs.rtmass[d] >= need) {
        sel = d;
        break;
      }
      cum += rs.rtmass[d];
    }
    above += cum;
    const uint32_t digit = 255u - (uint32_t)sel;
    prefix |= digit << shift;
    pmask |= 255u << shift;
    if (pass == 3) {
      out.at_count = rs.rtcnt[sel];
      out.at_weight = rs.rtmass[sel];
    }
    __syncthreads();
  }
  out.tau = prefix;
  out.above = above;
  out.target = target;
  return out;
}

// The id of the nth (1-based) element, in ascending id order over the
// cluster, for which pred(local index) holds.  Same result in all CTAs.
template <int NT, class Pred>
SPEC_DEV int nth_in_cluster(int n, int lo, int nth, Pred pred, int rank, int CS, int& ph,
                            Sh<NT / 32>& sh) {
  // each warp counts one contiguous range of ids, 32 consecutive ids per step
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = ((n + NW - 1) / NW + 31) / 32 * 32;
  const int s0 = min(warp * seg, n), s1 = min(s0 + seg, n);
  int c = 0;  // warp-uniform
  for (int k0 = s0; k0 < s1; k0 += 32) {
    const int k = k0 + lane;
    c += __popc(__ballot_sync(kFull, k < s1 && pred(k)));
  }
  int tot;
  const int excl = __shfl_sync(kFull, block_excl_scan_i<NT>(lane == 0 ? c : 0, &tot, sh), 0);
  exchange(Post{{(unsigned long long)tot, 0ull, 0ull, 0ull}}, CS, ph, sh);
  int before = 0, owner = -1;
  for (int r = 0; r < CS; ++r) {
    const int tr = (int)sh.gath[r].w[0];
    if (owner < 0 && before + tr >= nth) owner = r;
    if (owner < 0) before += tr;
  }
  int found = INT_MAX;
  if (owner == rank) {
    const int local = nth - before;
    if (excl < local && local <= excl + c) {  // warp-uniform: this warp holds it
      int cnt = excl;
      for (int k0 = s0; k0 < s1; k0 += 32) {
        const int k = k0 + lane;
        unsigned b = __ballot_sync(kFull, k < s1 && pred(k));
        if (cnt + __popc(b) >= local) {
          for (int i = cnt + 1; i < local; ++i) b &= b - 1u;  // drop the lower set bits
          found = lo + k0 + __ffs(b) - 1;
          break;
        }
        cnt += __popc(b);
      }
    }
  }
  found = block_min_i<NT>(found, sh);
  exchange(Post{{(unsigned long long)(unsigned)found, 0ull, 0ull, 0ull}}, CS, ph, sh);
  return owner < 0 ? INT_MAX : (int)(unsigned)sh.gath[owner].w[0];
}

// tau / tie of the top-k then top-p cut by exact radix selection; E in buf.
template <int NT, class EK>
SPEC_DEV Cut cut_radix(const SP& p, const float* lrow, EK ek, int n, int lo,
                       const RadixScratch& rs, int rank, int CS, int& ph, Sh<NT / 32>& sh) {
  Cut c{2, 0.f, 0u, INT_MAX};
  if (p.top_k > 0 && p.top_k < p.V) {
    const Sel s = radix_select<NT>(
        lrow, n, false, 0.0, (unsigned long long)p.top_k, [](int, uint32_t) { return true; },
        [](int) { return 1ull; }, rs, CS);
    const int need = (int)(s.target - s.above);
    c.tau = s.tau;
    if ((uint32_t)need >= s.at_count) {
      c.tie = INT_MAX;
    } else {
      const uint32_t tau = s.tau;
      c.tie = nth_in_cluster<NT>(
          n, lo, need, [&](int k) { return okey(__ldg(lrow + k)) == tau; }, rank, CS, ph, sh);
    }
  }
  if (p.top_p > 0.f && p.top_p < 1.f) {
    const uint32_t tk = c.tau;
    const int tc = c.tie;
    auto keep_k = [&](int k, uint32_t key) { return is_kept(key, lo + k, tk, tc); };
    auto mass = [&](int k) {
      return (unsigned long long)__float2ull_rn(ek(k) * 1099511627776.0f);  // 2^40
    };
    const Sel s = radix_select<NT>(lrow, n, true, (double)p.top_p, 0ull, keep_k, mass, rs, CS);
    const unsigned long long e_tau = s.at_count ? s.at_weight / s.at_count : 0ull;
    unsigned long long need = 1;
    if (e_tau > 0 && s.target > s.above) need = (s.target - s.above + e_tau - 1) / e_tau;
    if (need < 1) need = 1;
    if (need > s.at_count) need = s.at_count;
    const uint32_t tau = s.tau;
    int tie;
    if (need == s.at_count) {
      tie = (tau == tk) ? tc : INT_MAX;
    } else {
      tie = nth_in_cluster<NT>(
          n, lo, (int)need,
          [&](int k) {
            const uint32_t key = okey(__ldg(lrow + k));
            return key == tau && is_kept(key, lo + k, tk, tc);
          },
          rank, CS, ph, sh);
    }
    c.tau = tau;
    c.tie = tie;
  }
  return c;
}

// the first child of node v after child c (storage order), -1 if none
SPEC_DEV int next_child(const int* par, int v, int c, int R) {
  for (int c2 = c + 1; c2 < R; ++c2)
    if (par[c2] == v) return c2;
  return -1;
}

// ---------------------------------------------------------------- the bin range of the cut
// Warp 0: the bin range [b_lo, b_hi] the top-k / top-p cut can fall in, from
// the octave totals (octf(o, count, m16 sum); lane = octave) and the bins of
// the octaves the crossings fall in (binf(b, count, m16 sum); lane = bin
// within the octave).  mode 1: found; 2: use the exact radix selection.
// kidx: the top-k cut's index among the members (-1: no top-k); members: the
// count in the range (-1: not known from the histogram).
template <int NT, class OctF, class BinF>
SPEC_DEV void find_range(bool topk, bool topp, int top_k, float top_p, unsigned long long zfx,
                         OctF octf, BinF binf, int* mode_o, int* b_lo_o, int* b_hi_o,
                         int* kidx_o) {
  const int lane = threadIdx.x & 31;
  unsigned long long oc_c = 0, oc_m = 0;
  octf(lane, oc_c, oc_m);
  oc_m = bin_fx(oc_m, 32 * lane);  // all bins of an octave share one exponent
  unsigned long long xc = oc_c, xm = oc_m;  // inclusive scans over octaves
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long tc = __shfl_up_sync(kFull, xc, o);
    const unsigned long long tmv = __shfl_up_sync(kFull, xm, o);
    if (lane >= o) { xc += tc; xm += tmv; }
  }
  const unsigned long long pc = xc - oc_c, pm = xm - oc_m;  // before each octave
  // cluster totals of the bins of octave o (lane j: bin 32 o + j)
  auto load_oct = [&](int o, unsigned long long& bc, unsigned long long& bmass) {
    unsigned long long mm = 0;
    bc = 0;
    binf(32 * o + lane, bc, mm);
    bmass = bin_fx(mm, 32 * o);
  };
  // inclusive scan over the lanes
  auto scan = [&](unsigned long long v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += t;
    }
    return v;
  };
  // first lane where po + running value reaches thr (31 if none)
  auto first_at = [&](unsigned long long po, unsigned long long incl,
                      unsigned long long thr) -> int {
    const unsigned h = __ballot_sync(kFull, po + incl >= thr);
    return h ? __ffs(h) - 1 : 31;
  };
  int mode = 1, b_lo = 0, b_hi = 0, kidx = -1, members = -1;
  if (topk) {
    const unsigned h = __ballot_sync(kFull, xc >= (unsigned long long)top_k);
    if (!h) {
      mode = 2;  // the k-th largest lies below 2^-32 of the maximum
    } else {
      const int ok = __ffs(h) - 1;
      unsigned long long bc, bmass;
      load_oct(ok, bc, bmass);
      const unsigned long long ic = scan(bc);
      const unsigned long long pck = __shfl_sync(kFull, pc, ok);
      const int jk = first_at(pck, ic, (unsigned long long)top_k);
      const int bk = 32 * ok + jk;
      b_lo = b_hi = bk;
      const int cnt_before_bk = (int)(pck + __shfl_sync(kFull, ic - bc, jk));
      kidx = top_k - cnt_before_bk - 1;
      members = (int)__shfl_sync(kFull, bc, jk);
      if (topp) {
        // the mass above bk, then the bin where top_p times it is reached
        const unsigned long long im = scan(bmass);
        const unsigned long long abk =
            __shfl_sync(kFull, pm, ok) + __shfl_sync(kFull, im - bmass, jk);
        const unsigned long long thr = mul_frac(abk, top_p);
        const unsigned h2 = __ballot_sync(kFull, xm >= thr);
        int ol = h2 ? __ffs(h2) - 1 : ok;
        if (ol > ok) ol = ok;
        unsigned long long lc = bc, lm = bmass, ilc = ic, ilm = im;
        if (ol != ok) {
          load_oct(ol, lc, lm);
          ilc = scan(lc);
          ilm = scan(lm);
        }
        int bl = 32 * ol + first_at(__shfl_sync(kFull, pm, ol), ilm, thr);
        if (bl > bk) bl = bk;
        b_lo = bl;
        // members in [b_lo, bk], and the count above b_lo
        const int jl = bl - 32 * ol;
        unsigned long long inrange;
        if (ol == ok) {
          inrange = (lane >= jl && lane <= jk) ? bc : 0;
        } else {
          inrange = (lane >= jl ? lc : 0) + (lane <= jk ? bc : 0) +
                    ((lane > ol && lane < ok) ? oc_c : 0);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) inrange += __shfl_xor_sync(kFull, inrange, o);
        members = (int)inrange;
        const int cnt_before_bl =
            (int)(__shfl_sync(kFull, pc, ol) + __shfl_sync(kFull, ilc - lc, jl));
        kidx = top_k - cnt_before_bl - 1;
      }
    }
  } else {
    const unsigned long long thr = mul_frac(zfx, top_p);
    const unsigned h = __ballot_sync(kFull, xm >= thr);
    if (!h) {
      mode = 2;
    } else {
      const int ol = __ffs(h) - 1;
      unsigned long long bc, bmass;
      load_oct(ol, bc, bmass);
      const int jl = first_at(__shfl_sync(kFull, pm, ol), scan(bmass), thr);
      b_lo = b_hi = 32 * ol + jl;
    }
  }
  if (mode == 1 && members > NT) mode = 2;  // the selection sorts at most NT members
  *mode_o = mode;
  *b_lo_o = b_lo;
  *b_hi_o = b_hi;
  *kidx_o = kidx;
}

// ---------------------------------------------------------------- the cut among the members
// Threads t < total hold member t (logit key, E bits), unsorted.  Sorts the
// members by key, descending (= logit desc, id asc): up to kRankSortMax
// members by rank (each member counts the larger keys; keys are distinct,
// the id is part of them), more by a bitonic network (shuffles inside a warp,
// shared memory across warps; xkey / xbits hold >= NT entries).  Then finds
// the cut on exact masses (units of 2^-44) running from a_lo, the mass above
// the members: the top-k member kidx (-1: no top-k), then (top-p) the first
// running mass >= top_p * Z_k.  Returns false if the cut does not lie among
// the members.
constexpr int kRankSortMax = 256;

template <int NT>
SPEC_DEV bool select_cut(unsigned long long key, uint32_t eb, int total, unsigned long long a_lo,
                         int kidx, bool topp, float top_p, unsigned long long zall_fx,
                         unsigned long long* xkey, uint32_t* xbits, Cut* cut, float* zkept,
                         Sh<NT / 32>& sh) {
  const int t = threadIdx.x;
  int P = 1;
  while (P < total) P <<= 1;
  if (total <= kRankSortMax) {
    if (t < total) {
      xkey[t] = key;
      xbits[t] = eb;
    }
    __syncthreads();
    int rank = 0;
    if (t < total) {
      // four independent counts: the shared-memory loads overlap
      int r4[4] = {0, 0, 0, 0};
      int j = 0;
      for (; j + 4 <= total; j += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) r4[u] += xkey[j + u] > key ? 1 : 0;
      }
      for (; j < total; ++j) r4[0] += xkey[j] > key ? 1 : 0;
      rank = (r4[0] + r4[1]) + (r4[2] + r4[3]);
    }
    __syncthreads();
    if (t < total) {
      xkey[rank] = key;
      xbits[rank] = eb;
    }
    __syncthreads();
    if (t < total) {
      key = xkey[t];
      eb = xbits[t];
    }
    P = 0;  // sorted: skip the network
  }
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      unsigned long long ok2;
      uint32_t ob;
      if (stride >= 32) {
        if (t < P) {
          xkey[t] = key;
          xbits[t] = eb;
        }
        __syncthreads();
        ok2 = (t < P) ? xkey[t ^ stride] : 0ull;
        ob = (t < P) ? xbits[t ^ stride] : 0u;
        __syncthreads();
      } else {
        ok2 = __shfl_xor_sync(kFull, key, stride);
        ob = __shfl_xor_sync(kFull, eb, stride);
      }
      const bool desc = (t & size) == 0;
      const bool lower = (t & stride) == 0;
      const bool take = lower ? (desc ? ok2 > key : ok2 < key) : (desc ? ok2 < key : ok2 > key);
      if (take) {
        key = ok2;
        eb = ob;
      }
    }
  }
  // thread t now holds the t-th largest member
  const bool live = t < total;
  const unsigned long long mt = live ? fx44(eb) : 0ull;
  const unsigned long long incl = a_lo + block_incl_scan_u64<NT>(mt, sh);  // mass through t
  const int last = (kidx >= 0) ? min(kidx, total - 1) : total - 1;
  if (t == 0) {
    sh.bi[5] = 0;
    if (kidx < 0) sh.zk = zall_fx;
  }
  __syncthreads();
  if (kidx >= 0 && t == last) sh.zk = incl;  // Z after top-k
  __syncthreads();
  const unsigned long long zk = sh.zk;
  int pick = -1;
  if (!topp) {
    if (t == last) pick = t;
  } else {
    const unsigned long long thr = mul_frac(zk, top_p);
    if (live && t <= last && incl - mt < thr && incl >= thr) pick = t;
  }
  if (pick >= 0) {  // unique: masses are positive
    sh.cut = Cut{1, __uint_as_float(eb), (uint32_t)(key >> 32), (int)(0xFFFFFFFFu - (uint32_t)key)};
    sh.zcut = incl;
    sh.bi[5] = 1;
  }
  __syncthreads();
  const bool ok = sh.bi[5] != 0;
  if (ok) {
    *cut = sh.cut;
    *zkept = (float)sh.zcut * (1.0f / 17592186044416.0f);  // 2^-44
  }
  __syncthreads();
  return ok;
}

// ---------------------------------------------------------------- row outcome
// Warp 0 of the row's (rank-0) CTA publishes the row's outcome; the warp that
// brings the sequence's counter to R assembles accepted_len, emitted, path
// and status from the R outcomes and resets the counter.
template <int NW>
SPEC_DEV void finish_row(const SP& p, int row, const Outcome& oc, Sh<NW>& sh) {
  const int lane = threadIdx.x & 31;
  const int R = p.R;
  const int b = row / R;
  int last = 0;
  if (lane == 0) {
    p.outcomes[row] = oc;
    __threadfence();
    last = atomicAdd(&p.seq_count[b], 1) == R - 1;
  }
  last = __shfl_sync(kFull, last, 0);
  if (!last) return;
  __threadfence();
  // warp 0 loads the sequence's outcomes (and its draft tokens) in parallel
  for (int r = lane; r < R; r += 32) {
    const int4 v = __ldcg(reinterpret_cast<const int4*>(&p.outcomes[(size_t)b * R + r]));
    sh.outs[r] = Outcome{v.x, v.y, v.z, v.w};
    sh.tok[r] = p.tree ? __ldg(&p.tokens[(size_t)b * R + r])
                       : (r < R - 1 ? __ldg(&p.tokens[(size_t)b * (R - 1) + r]) : -1);
  }
  __syncwarp();
  if (lane != 0) return;
  int32_t* emitted = p.emitted + (size_t)b * R;
  int nonfin = 0, status = 0, acc = 0, k = 0;
  for (int r = 0; r < R; ++r) nonfin |= sh.outs[r].flags;
  if (nonfin) {
    acc = -1;
    status = SPEC_SEQ_NONFINITE;
  } else if (!p.tree) {
    for (int r = 0; r < R; ++r) {
      const Outcome& o = sh.outs[r];
      status |= o.status;
      if (r < R - 1 && o.accept) {
        const int x = sh.tok[r];
        emitted[k++] = x;
        ++acc;
        if (x == p.eos) break;
        continue;
      }
      emitted[k++] = o.token;
      break;
    }
  } else {
    int32_t* path = p.path + (size_t)b * R;
    int v = 0;
    while (true) {
      const Outcome& o = sh.outs[v];
      status |= o.status;
      if (o.accept > v) {
        const int t = sh.tok[o.accept];
        emitted[k++] = t;
        path[acc++] = o.accept;
        v = o.accept;
        if (t == p.eos) break;
        continue;
      }
      emitted[k++] = o.token;
      break;
    }
  }
  for (int c = (nonfin ? 0 : k); c < R; ++c) emitted[c] = -1;
  if (p.tree)
    for (int c = (nonfin ? 0 : acc); c < R; ++c) p.path[(size_t)b * R + c] = -1;
  p.acc_len[b] = acc;
  if (p.status) p.status[b] = status;
  p.seq_count[b] = 0;
}

// ---------------------------------------------------------------- the kernel
// One cluster per target row.  Every row computes its own outcome:
//   chain row i < R-1: is draft i+1 accepted? if not, the correction drawn
//     from norm(max(0, p_i - q_i));  chain row R-1: the bonus drawn from p;
//   tree node v: the first accepted child (residual p' updated after each
//     rejected child) or, if none, the final token drawn from p'.
// The cluster that finishes a sequence's last row assembles the sequence.
template <int NT, bool FAST, bool TR>
__global__ void __launch_bounds__(NT, 512 / NT) sampler_kernel(const SP p) {
  constexpr int NW = NT / 32;
  constexpr int kWL = kListPerCTA / NW;
  extern __shared__ __align__(16) uint8_t dyn[];
  float* buf = reinterpret_cast<float*>(dyn);
  uint32_t* hcnt = reinterpret_cast<uint32_t*>(dyn + ((size_t)p.slice * 4 + 15) / 16 * 16);
  uint32_t* hm = hcnt + kHistPad;  // per-bin sums of m16 (this CTA)
  unsigned long long* mkey = reinterpret_cast<unsigned long long*>(hm + kHistPad);  // local members
  unsigned long long* gkey = mkey + kCandMax;  // gathered members
  uint32_t* mbits = reinterpret_cast<uint32_t*>(gkey + kCandMax);
  uint32_t* gbits = mbits + kCandMax;
  uint16_t* lists = reinterpret_cast<uint16_t*>(gbits + kCandMax);
  float* qb = reinterpret_cast<float*>(lists + kListPerCTA);  // q slice (full-vocabulary residuals)
  // the radix fallback reuses the member arrays (12 KB) as its scratch
  const RadixScratch rs{reinterpret_cast<uint32_t*>(mkey), mkey + 256, mkey + 768,
                        reinterpret_cast<uint32_t*>(mkey) + 2048};
  __shared__ Sh<NW> sh;

  const int CS = (int)cluster_nctarank();
  const int rank = (int)cluster_ctarank();
  const int row = blockIdx.x / CS;
  const int R = p.R;
  const int b = row / R;
  const int i = row % R;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lo = rank * p.slice;
  const int n = max(0, min(p.slice, p.V - lo));
  const float* lrow_full = p.logits + (size_t)row * p.V;
  const float* lrow = lrow_full + lo;
  // TR = false: untruncated, sampled chain rows (the truncation, tree and greedy
  // code is compiled out: each CTA runs its program once and fetches it cold)
  const bool tree = TR && p.tree != 0;
  const bool greedy = TR && p.greedy != 0;
  const bool topk = TR && p.top_k > 0 && p.top_k < p.V;
  const bool topp = TR && p.top_p > 0.f && p.top_p < 1.f;
  const bool trunc = TR && !greedy && (topk || topp);
  int ph = 0;

  // ---- 0. setup: barrier, histogram, tree shape, this row's probe token
  if (threadIdx.x == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
    sh.token_in = -1;
  }
  if (trunc)
    for (int k = threadIdx.x; k < kHist; k += NT) {
      hcnt[k] = 0u;
      hm[k] = 0u;
    }
  if (tree)
    for (int c = threadIdx.x; c < R; c += NT) {
      sh.par[c] = p.parent[(size_t)b * R + c];
      sh.tok[c] = p.tokens[(size_t)b * R + c];
    }
  __syncthreads();
  // the token whose E this row's first test needs (-1: no test)
  int probe = -1;
  if (!tree) {
    if (i < R - 1) probe = __ldg(&p.tokens[(size_t)b * (R - 1) + i]);
  } else {
    const int fc = next_child(sh.par, i, i, R);
    if (fc >= 0) probe = sh.tok[fc];
  }
  const float* qrow = nullptr;
  if (!greedy && p.q) {
    if (tree)
      qrow = p.q + ((size_t)b * R + i) * p.V;
    else if (i < R - 1)
      qrow = p.q + ((size_t)b * (R - 1) + i) * p.V;
  }
  // full-vocabulary residuals read q from shared memory (loaded with the logits)
  const bool q_sh = p.qsm && qrow != nullptr && n > 0;
  const bool chain_test = !tree && i < R - 1;
  float u_test = 0.f, u_last = 0.f, q_probe = 0.f;
  // the chain test's operands, loaded after the slice copies are issued: their
  // latency hides under the copies
  auto load_test_operands = [&]() {
    u_test = chain_test ? __ldg(&p.u[(size_t)b * R + i]) : 0.f;
    u_last = __ldg(&p.u[(size_t)b * R + (R - 1)]);
    q_probe = (chain_test && qrow != nullptr && probe >= 0 && probe < p.V) ? __ldg(&qrow[probe])
                                                                           : 0.f;
  };

  // ---- 1. the slice (and q's) into shared memory
  if (n > 0 && p.bulk) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&sh.bar, (uint32_t)n * (q_sh ? 8u : 4u));
      bulk_load(buf, lrow, (uint32_t)n * 4u, &sh.bar);
      if (q_sh) bulk_load(qb, qrow + lo, (uint32_t)n * 4u, &sh.bar);
    }
  }
  load_test_operands();
  if (n > 0) {
    if (p.bulk) {
      mbar_wait(&sh.bar, 0, p.err);
    } else {
      for (int k = threadIdx.x; k < n; k += NT) buf[k] = __ldg(lrow + k);
      __syncthreads();
    }
  }

  // ---- 2. maximum (NaN-propagating), greedy argmax
  float mx = -INFINITY, best = -INFINITY;
  int bid = INT_MAX;
  {
    const int n4 = n >> 2;
    const float4* b4 = reinterpret_cast<const float4*>(buf);
    for (int k4 = threadIdx.x; k4 < n4; k4 += NT) {
      const float4 v = b4[k4];
      mx = fmax_nan(fmax_nan(mx, v.x), fmax_nan(fmax_nan(v.y, v.z), v.w));
      if (greedy) {
        if (v.x > best) { best = v.x; bid = 4 * k4; }
        if (v.y > best) { best = v.y; bid = 4 * k4 + 1; }
        if (v.z > best) { best = v.z; bid = 4 * k4 + 2; }
        if (v.w > best) { best = v.w; bid = 4 * k4 + 3; }
      }
    }
    for (int k = 4 * n4 + threadIdx.x; k < n; k += NT) {
      const float v = buf[k];
      mx = fmax_nan(mx, v);
      if (greedy && v > best) { best = v; bid = k; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmax_nan(mx, __shfl_xor_sync(kFull, mx, o));
      const float ob = __shfl_xor_sync(kFull, best, o);
      const int oi = __shfl_xor_sync(kFull, bid, o);
      if (ob > best || (ob == best && oi < bid)) { best = ob; bid = oi; }
    }
    if (lane == 0) { sh.red_f[warp] = mx; sh.wsum[warp] = best; sh.red_i[warp] = bid; }
    __syncthreads();
    mx = sh.red_f[0]; best = sh.wsum[0]; bid = sh.red_i[0];
    for (int w = 1; w < NW; ++w) {
      mx = fmax_nan(mx, sh.red_f[w]);
      if (sh.wsum[w] > best || (sh.wsum[w] == best && sh.red_i[w] < bid)) {
        best = sh.wsum[w]; bid = sh.red_i[w];
      }
    }
    __syncthreads();
  }
  exchange(Post{{f2w(mx), f2w(best),
                 (unsigned long long)(unsigned)(bid == INT_MAX ? INT_MAX : lo + bid), 0ull}},
           CS, ph, sh);
  float m = -INFINITY;
  int argmax = INT_MAX;
  best = -INFINITY;
  for (int r = 0; r < CS; ++r) {
    m = fmax_nan(m, w2f(sh.gath[r].w[0]));
    const float ob = w2f(sh.gath[r].w[1]);
    const int oi = (int)(unsigned)sh.gath[r].w[2];
    if (ob > best || (ob == best && oi < argmax)) { best = ob; argmax = oi; }
  }
  const bool bad = isnan(m) || m == INFINITY || m == -INFINITY;
  Outcome oc{0, -1, 0, bad ? 1 : 0};
  bool drew = false;    // this row made a draw (same in every CTA of the cluster)
  int draw_token = -1;  // set by the draw's owner CTA only

  if (bad) {
    // no distribution: the sequence reports NONFINITE
  } else if (greedy) {
    if (!tree) {
      if (i < R - 1) oc.accept = (probe == argmax) ? 1 : 0;
    } else {
      oc.accept = -1;
      for (int c = i + 1; c < R; ++c)
        if (sh.par[c] == i && sh.tok[c] == argmax) { oc.accept = c; break; }
    }
    oc.token = argmax;
  } else {
    // ---- 3. E in place, Z (compensated per thread), histogram, probe value
    const float nm = -m, lfloor = m - 150.f * p.T;
    const float c_hi = p.c_hi, c_lo = p.c_lo, nmc = -m * p.c_hi;
    auto Eof = [&](float l) { return FAST ? fexp(l, c_hi, nmc) : texp(l, nm, lfloor, c_hi, c_lo); };
    float zs = 0.f, zc = 0.f;  // Kahan sum and compensation
    {
      const int n4 = n >> 2;
      float4* b4 = reinterpret_cast<float4*>(buf);
      for (int k4 = threadIdx.x; k4 < n4; k4 += NT) {
        const float4 v = b4[k4];
        float4 e;
        e.x = Eof(v.x);
        e.y = Eof(v.y);
        e.z = Eof(v.z);
        e.w = Eof(v.w);
        b4[k4] = e;
        const float ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float y = ev[j] - zc;
          const float t = zs + y;
          zc = (t - zs) - y;
          zs = t;
          if (trunc) {
            const uint32_t bits = __float_as_uint(ev[j]);
            const int bn = ebin(bits);
            if (topk) atomicAdd(&hcnt[bn], 1u);
            if (topp && bn < kBins) atomicAdd(&hm[bn], m16(bits));
          }
        }
      }
      for (int k = 4 * n4 + threadIdx.x; k < n; k += NT) {
        const float e = Eof(buf[k]);
        buf[k] = e;
        const float y = e - zc;
        const float t = zs + y;
        zc = (t - zs) - y;
        zs = t;
        if (trunc) {
          const uint32_t bits = __float_as_uint(e);
          const int bn = ebin(bits);
          if (topk) atomicAdd(&hcnt[bn], 1u);
          if (topp && bn < kBins) atomicAdd(&hm[bn], m16(bits));
        }
      }
    }
    const float zh = block_sum_f<NT>(zs, sh);  // includes barriers: buf and histogram complete
    const float zl = block_sum_f<NT>(-zc, sh);
    if (trunc && warp == 0) {  // per-octave totals of this CTA's bins
      uint32_t c = 0, mm = 0;
      for (int j = 0; j < 32; ++j) {
        c += hcnt[32 * lane + j];
        mm += hm[32 * lane + j];
      }
      sh.oct[lane] = c;
      sh.oct[32 + lane] = mm;
    }
    const bool pin = probe >= lo && probe < lo + n;
    exchange(Post{{f2w(zh), f2w(zl), f2w(pin ? buf[probe - lo] : 0.f), 0ull}}, CS, ph, sh);
    float e_probe = 0.f;
    if (probe >= 0 && probe < p.V) e_probe = w2f(sh.gath[probe / p.slice].w[2]);
    float zah = 0.f, zal = 0.f;  // Z of the whole row, float pair
    for (int r = 0; r < CS; ++r) df_acc(zah, zal, w2f(sh.gath[r].w[0]), w2f(sh.gath[r].w[1]));

    Cut cut{0, 0.f, 0u, INT_MAX};
    float zkept = zah + zal;
    int tmode = 0;
    if (trunc) {
      // ---- 4. the bin range the cut can fall in (warp 0): octave totals of
      // the cluster (lane = octave), then the bins of the octaves the
      // crossings fall in (lane = bin within the octave)
      if (warp == 0) {
        int mode, bl, bh, kx;
        find_range<NT>(
            topk, topp, p.top_k, p.top_p, fx44_pair(zah, zal),
            [&](int o, unsigned long long& c, unsigned long long& mm) {
              for (int r = 0; r < CS; ++r) {
                if (topk) c += dsmem_ld_u32(&sh.oct[o], r);
                if (topp) mm += dsmem_ld_u32(&sh.oct[32 + o], r);
              }
            },
            [&](int bb, unsigned long long& c, unsigned long long& mm) {
              for (int r = 0; r < CS; ++r) {
                if (topk) c += dsmem_ld_u32(&hcnt[bb], r);
                if (topp) mm += dsmem_ld_u32(&hm[bb], r);
              }
            },
            &mode, &bl, &bh, &kx);
        if (lane == 0) {
          sh.bi[0] = mode;
          sh.bi[1] = bl;
          sh.bi[2] = bh;
          sh.bi[3] = kx;
        }
      }
      __syncthreads();
      tmode = sh.bi[0];
      const int b_lo = sh.bi[1], b_hi = sh.bi[2], kidx = sh.bi[3];
      __syncthreads();

      if (tmode == 1) {
        // ---- 5. members of bins [b_lo, b_hi] and the exact mass above them
        if (threadIdx.x == 0) sh.bi[4] = 0;
        __syncthreads();
        unsigned long long above = 0;
        // E in bins <= b_hi  <=>  bits >= edge (bins count down from E = 1)
        const uint32_t edge = (uint32_t)(0x3F7FFFFF - ((b_hi + 1) << 18) + 1);
        auto visit = [&](int k, float e) {
          const uint32_t bits = __float_as_uint(e);
          if (bits < edge) return;
          const int bn = ebin(bits);
          if (bn < b_lo) {
            above += fx44(bits);
          } else if (bn <= b_hi) {
            const int slot = atomicAdd(&sh.bi[4], 1);
            if (slot < kCandMax) {
              mkey[slot] = ((unsigned long long)okey(__ldg(lrow + k)) << 32) |
                           (0xFFFFFFFFu - (uint32_t)(lo + k));
              mbits[slot] = bits;
            }
          }
        };
        {
          const int n4 = n >> 2;
          const float4* b4 = reinterpret_cast<const float4*>(buf);
          for (int k4 = threadIdx.x; k4 < n4; k4 += NT) {
            const float4 e = b4[k4];
            visit(4 * k4, e.x);
            visit(4 * k4 + 1, e.y);
            visit(4 * k4 + 2, e.z);
            visit(4 * k4 + 3, e.w);
          }
          for (int k = 4 * n4 + threadIdx.x; k < n; k += NT) visit(k, buf[k]);
        }
        above = block_sum_u64<NT>(above, sh);  // includes barriers: members complete
        exchange(Post{{(unsigned long long)sh.bi[4], above, 0ull, 0ull}}, CS, ph, sh);
        unsigned long long a_lo = 0;
        int total = 0;
        for (int r = 0; r < CS; ++r) {
          a_lo += sh.gath[r].w[1];
          total += (int)sh.gath[r].w[0];
        }
        if (total > NT || total < 1) {
          tmode = 2;  // too populous to sort here (top-p only: counted now)
        } else {
          // gather into registers: thread t holds member t
          const int t = threadIdx.x;
          unsigned long long key = 0ull;
          uint32_t eb = 0u;
          {
            int off = 0;
            for (int r = 0; r < CS; ++r) {
              const int cr = (int)sh.gath[r].w[0];
              if (t >= off && t < off + cr) {
                key = dsmem_ld_u64(&mkey[t - off], r);
                eb = dsmem_ld_u32(&mbits[t - off], r);
              }
              off += cr;
            }
          }
          if (!select_cut<NT>(key, eb, total, a_lo, kidx, topp, p.top_p,
                              fx44_pair(zah, zal), gkey, gbits,
                              &cut, &zkept, sh))
            tmode = 2;  // the rounded bin masses placed the cut one bin off
        }
      }
      if (tmode == 2) {
        // ---- 5'. exact radix selection over the logit keys
        cluster_sync();  // every CTA is done reading the others' member lists
        cut = cut_radix<NT>(p, lrow, [&](int k) { return buf[k]; }, n, lo, rs, rank, CS, ph, sh);
        // Z over the kept set (compensated per thread, fixed order)
        float s = 0.f, cmp = 0.f;
        for (int k = threadIdx.x; k < n; k += NT) {
          if (cut_keeps(cut, buf[k], lo + k, lrow_full)) {
            const float y = buf[k] - cmp;
            const float tt = s + y;
            cmp = (tt - s) - y;
            s = tt;
          }
        }
        const float hs = block_sum_f<NT>(s, sh);
        const float ls = block_sum_f<NT>(-cmp, sh);
        exchange(Post{{f2w(hs), f2w(ls), 0ull, 0ull}}, CS, ph, sh);
        float kh = 0.f, kl = 0.f;
        for (int r = 0; r < CS; ++r) df_acc(kh, kl, w2f(sh.gath[r].w[0]), w2f(sh.gath[r].w[1]));
        zkept = kh + kl;
      }
    }

    // ---- 6. (tree, p_out: on first use) zero the cut-off tail in place and
    // list each warp's kept positions
    const int rw = ((n + NW - 1) / NW + 3) / 4 * 4;
    Items<NW> it{false, lists, min(warp * rw, n), min((warp + 1) * rw, n), rw, n};
    bool kept_ready = !trunc, zeroed = !trunc;
    // zero: also clear buf outside the kept set (needed where buf is read by
    // position: the tree's probe values and p_out)
    auto ensure_kept = [&](bool zero) {
      if (kept_ready && (zeroed || !zero)) return;
      kept_ready = true;
      zeroed = zeroed || zero;
      int cntw = 0;
      uint16_t* myl = lists + warp * kWL;
      const int r1v = it.r0 + ((it.r1 - it.r0) & ~3);
      for (int s0 = it.r0; s0 < it.r1; s0 += 128) {
        const int k = s0 + 4 * lane;
        int c = 0;
        bool kp[4] = {false, false, false, false};
        if (k < r1v) {
          float4 e4 = *reinterpret_cast<const float4*>(buf + k);
          float ev[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            kp[u] = ev[u] > 0.f && cut_keeps(cut, ev[u], lo + k + u, lrow_full);
            if (!kp[u]) ev[u] = 0.f;
            c += kp[u] ? 1 : 0;
          }
          if (zero) *reinterpret_cast<float4*>(buf + k) = make_float4(ev[0], ev[1], ev[2], ev[3]);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (k + u < it.r1) {
              const float e = buf[k + u];
              kp[u] = e > 0.f && cut_keeps(cut, e, lo + k + u, lrow_full);
              if (!kp[u] && zero) buf[k + u] = 0.f;
              c += kp[u] ? 1 : 0;
            }
          }
        }
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int tt = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += tt;
        }
        int pos = cntw + incl - c;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (kp[u]) {
            if (pos < kWL) myl[pos] = (uint16_t)(k + u);
            ++pos;
          }
        cntw += __shfl_sync(kFull, incl, 31);
      }
      if (lane == 0) sh.list_n[warp] = cntw;
      it.listed = __syncthreads_and(cntw <= kWL ? 1 : 0) != 0;
    };
    const float invz = 1.0f / zkept;
    if (!FAST && p.p_out) {
      ensure_kept(true);
      float* dst = p.p_out + (size_t)row * p.V + lo;
      for (int k = threadIdx.x; k < n; k += NT) dst[k] = buf[k] * invz;
      // every thread has read buf before a residual draw rewrites it in place
      // (its warps own other elements than this loop's threads)
      __syncthreads();
    }

    const float u_final = u_last;
    const float* qlo = q_sh ? qb : (qrow ? qrow + lo : nullptr);
    if (!tree) {
      // ---- 7a. chain: the row's test, then its correction or bonus draw
      bool resid = false;
      if (i < R - 1) {
        const int x = probe;
        const bool xin = x >= 0 && x < p.V;
        const float qx = xin ? q_probe : 0.f;
        const float px = (xin && e_probe > 0.f && cut_keeps(cut, e_probe, x, lrow_full))
                             ? e_probe * invz : 0.f;
        if (qx == 0.f) oc.status |= SPEC_SEQ_QZERO;
        oc.accept = (u_test * qx < px) ? 1 : 0;
        resid = !oc.accept;
      }
      drew = i == R - 1 || resid;
      if (drew) {
        // truncated: the kept positions listed per warp (buf left as is);
        // otherwise (or when a list overflows) the whole warp range with the
        // cut applied inline
        ensure_kept(false);
        float t;
        if (it.listed)
          t = weight_pass<NT>(buf, it, resid ? 1 : 0, invz, qlo, q_sh, sh);
        else
          t = weight_full<NT>(buf, it.r0, it.r1, cut, lo, lrow_full, resid ? 1 : 0, invz, qlo,
                              q_sh, p.qbulk != 0, sh);
        exchange(Post{{f2w(t), 0ull, 0ull, 0ull}}, CS, ph, sh);
        int tokn = locate<NT>(buf, it, lo, u_final, rank, CS, sh);
        if (tokn == -2) {  // residual with zero mass (rounding only): draw from p
          oc.status |= SPEC_SEQ_RESID_ZERO;
          for (int k = it.r0 + lane; k < it.r1; k += 32)
            buf[k] = Eof(__ldg(lrow + k));
          __syncthreads();
          it.listed = false;
          const float t2 = weight_full<NT>(buf, it.r0, it.r1, cut, lo, lrow_full, 0, 1.f, qlo,
                                           q_sh, false, sh);
          exchange(Post{{f2w(t2), 0ull, 0ull, 0ull}}, CS, ph, sh);
          tokn = locate<NT>(buf, it, lo, u_final, rank, CS, sh);
        }
        draw_token = tokn;
      }
    } else {
      // ---- 7b. tree node: children in storage order against the running p'
      oc.accept = -1;
      float invw = invz;
      int nsteps = 0;
      float v_probe = (e_probe > 0.f && probe >= 0 && probe < p.V &&
                       cut_keeps(cut, e_probe, probe, lrow_full)) ? e_probe : 0.f;
      for (int c = next_child(sh.par, i, i, R); c >= 0; c = next_child(sh.par, i, c, R)) {
        const int t = sh.tok[c];
        const bool tin = t >= 0 && t < p.V;
        const float qt = tin ? __ldg(&qrow[t]) : 0.f;
        const float pt = tin ? v_probe * invw : 0.f;
        if (qt == 0.f) oc.status |= SPEC_SEQ_QZERO;
        if (__ldg(&p.u[(size_t)b * R + (c - 1)]) * qt < pt) {
          oc.accept = c;
          break;
        }
        // the next child's token: the exchange carries its p' value
        const int nc = next_child(sh.par, i, c, R);
        const int tn = nc >= 0 ? sh.tok[nc] : -1;
        const bool tnin = tn >= lo && tn < lo + n;
        // p' <- norm(max(0, p' - q_v))
        ensure_kept(true);
        if (threadIdx.x == 0) sh.invw_used[nsteps] = invw;
        const float wt = weight_pass<NT>(buf, it, 1, invw, qlo, q_sh, sh);
        exchange(Post{{f2w(wt), f2w(tnin ? buf[tn - lo] : 0.f), 0ull, 0ull}}, CS, ph, sh);
        float W = 0.f;
        for (int r = 0; r < CS; ++r) W += w2f(sh.gath[r].w[0]);
        const float vn = (tn >= 0 && tn < p.V) ? w2f(sh.gath[tn / p.slice].w[1]) : 0.f;
        if (W > 1e-37f) {
          invw = 1.0f / W;
          ++nsteps;
          v_probe = vn;
        } else {
          // zero mass (rounding only): keep p' -- rebuild it from the logits
          oc.status |= SPEC_SEQ_RESID_ZERO;
          const int cnt = it.count(sh);
          for (int j = lane; j < cnt; j += 32) {
            const int k = it.at(j);
            float e = Eof(__ldg(lrow + k));
            e = cut_keeps(cut, e, lo + k, lrow_full) ? e : 0.f;
            for (int s = 0; s < nsteps; ++s)
              e = residual_w(e, sh.invw_used[s],
                             e > 0.f ? (q_sh ? qlo[k] : __ldg(qlo + k)) : 0.f);
            buf[k] = e;
          }
          __syncthreads();
          exchange(Post{{0ull, f2w(tnin ? buf[tn - lo] : 0.f), 0ull, 0ull}}, CS, ph, sh);
          v_probe = (tn >= 0 && tn < p.V) ? w2f(sh.gath[tn / p.slice].w[1]) : 0.f;
        }
      }
      drew = oc.accept < 0;
      if (drew) {
        ensure_kept(true);
        const float t = weight_pass<NT>(buf, it, 0, 1.f, qlo, q_sh, sh);
        exchange(Post{{f2w(t), 0ull, 0ull, 0ull}}, CS, ph, sh);
        draw_token = locate<NT>(buf, it, lo, u_final, rank, CS, sh);
        if (draw_token == -2) oc.status |= SPEC_SEQ_RESID_ZERO;
      }
    }
  }

  // ---- 8. the draw's owner hands its token to rank 0; then rank 0 publishes
  if (draw_token >= 0 && threadIdx.x == 0) {
    if (rank == 0)
      sh.token_in = draw_token;
    else
      dsmem_st_s32(&sh.token_in, 0, draw_token);
  }
  cluster_sync();  // also: no CTA leaves while another may read its shared memory
  if (rank != 0 || threadIdx.x >= 32) return;
  if (drew) oc.token = sh.token_in;
  finish_row(p, row, oc, sh);
}

// ---------------------------------------------------------------- streaming kernel (many rows)
// One 1024-thread CTA per target row, used for truncated sampling when many
// rows run at once.  One evenly spaced sample per thread gives a reference
// maximum and a candidate floor that about kSBudget ids pass; then ONE sweep
// of the row from HBM (each warp its own contiguous id range) takes the
// maximum, Z relative to the reference (rescaled to the maximum after it) and
// appends every id at or above the floor, with its logit, to the warp's
// id-ordered candidate list in shared memory.  The histogram, the members of
// the crossing bins, the kept set and the draws all work on those lists.  A
// floor above the cut, or a list that overflows, falls back to further
// sweeps of the row.  No cluster exchanges: every SM works on its own rows.
// (The two-pass variant, PRE, takes the sweep's results from a pre-pass over
// all SMs instead.)
constexpr int kSNT = 1024;
constexpr int kSCap = 16384;    // list entries per row (kSCap / 32 per warp)
constexpr int kSBudget = 10240; // candidates a row's floor aims at (sampled estimate)
constexpr int kSListMaxV = 163840;  // rows up to this long are listed; longer ones are histogrammed whole

// Each warp of the row kernel owns one contiguous range of the row's ids
// (a multiple of 32 long); the two-pass variant's pre-pass sweeps each such
// range with one CTA of kSwW warps.
constexpr int kRangesPerRow = kSNT / 32;
constexpr int kSwW = 8;
constexpr int kSwNT = 32 * kSwW;
constexpr int kSWCap = kSCap / kRangesPerRow;  // list entries a row-kernel warp holds
constexpr int kSegCap = 128;  // list entries stored per pre-pass warp segment (kSwW per range)

__host__ __device__ inline int stream_range_width(int V) {
  return ((V + kRangesPerRow - 1) / kRangesPerRow + 31) / 32 * 32;
}
constexpr int kSamples = 1024;                 // samples per row for the floor
static_assert(kSamples == kSNT, "the floor samples are the row kernel's, one per thread");

// PRE: the pre-pass (sampler_sweep_kernel) has swept the row: the maximum, Z
// and the candidate lists are read from its results, not from the logits.
template <bool FAST, bool PRE>
__global__ void __launch_bounds__(kSNT, 1) sampler_stream_kernel(const SP p) {
  constexpr int NT = kSNT, NW = NT / 32, WCAP = kSCap / NW;
  extern __shared__ __align__(16) uint8_t dyn[];
  uint32_t* hcnt = reinterpret_cast<uint32_t*>(dyn);
  uint32_t* hm = hcnt + kHistPad;
  unsigned long long* xkey = reinterpret_cast<unsigned long long*>(hm + kHistPad);  // NT
  uint32_t* xbits = reinterpret_cast<uint32_t*>(xkey + NT);                          // NT
  int* lid = reinterpret_cast<int*>(xbits + NT);                                      // kSCap
  float* lval = reinterpret_cast<float*>(lid + kSCap);                                // kSCap
  const RadixScratch rs{reinterpret_cast<uint32_t*>(xkey), xkey + 256, xkey + 768,
                        reinterpret_cast<uint32_t*>(xkey) + 2048};
  __shared__ Sh<NW> sh;

  const int row = blockIdx.x;
  const int R = p.R, V = p.V;
  const int b = row / R;
  const int i = row % R;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* lrow = p.logits + (size_t)row * V;
  const bool topk = p.top_k > 0 && p.top_k < V;
  const bool topp = p.top_p > 0.f && p.top_p < 1.f;
  const bool trunc = topk || topp;
  const bool vec = p.bulk != 0;  // V % 4 == 0 and 16-byte aligned rows
  const int n4 = vec ? V / 4 : 0;
  const float4* l4 = reinterpret_cast<const float4*>(lrow);
  // the row is swept once (the lists keep what the cut needs): L2 need not keep it
  const uint64_t pol = PRE ? l2_keep_policy() : l2_first_policy();
  // every element of the row once: visit(k, l), four 16-byte loads in flight per thread
  auto sweep = [&](auto&& visit) {
    for (int base = threadIdx.x; base < n4; base += 4 * NT) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k4 = base + u * NT;
        v[u] = k4 < n4 ? ldg_keep4(l4 + k4, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k4 = base + u * NT;
        if (k4 < n4) {
          visit(4 * k4, v[u].x);
          visit(4 * k4 + 1, v[u].y);
          visit(4 * k4 + 2, v[u].z);
          visit(4 * k4 + 3, v[u].w);
        }
      }
    }
    for (int k = 4 * n4 + threadIdx.x; k < V; k += NT) visit(k, ldg_keep(lrow + k, pol));
  };
  int ph = 0;
  // the floor's sample (one per thread, evenly spaced) and the first 8 KB of
  // each warp's id range are requested before the setup: their latency hides
  // under it
  const float smp =
      PRE ? 0.f : ldg_keep(lrow + (int)(((long long)threadIdx.x * V) / NT), pol);
  if (!PRE) {
    const int rw0 = stream_range_width(V);
    const int a0 = min(warp * rw0, V), a1 = min((warp + 1) * rw0, V);
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (a0 + 1024 * q + 32 * lane < a1)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(lrow + a0 + 1024 * q + 32 * lane));
  }

  // ---- 0. setup
  if (threadIdx.x == 0) {
    sh.token_in = -1;
    sh.eprobe = 0.f;
    sh.bi[4] = 0;  // members found so far
  }
  if (trunc)
    for (int k = threadIdx.x; k < kHist; k += NT) {
      hcnt[k] = 0u;
      hm[k] = 0u;
    }
  if (p.tree)
    for (int c = threadIdx.x; c < R; c += NT) {
      sh.par[c] = p.parent[(size_t)b * R + c];
      sh.tok[c] = p.tokens[(size_t)b * R + c];
      sh.cpos[c] = -1;
    }
  __syncthreads();
  int probe = -1;
  if (!p.tree) {
    if (i < R - 1) probe = __ldg(&p.tokens[(size_t)b * (R - 1) + i]);
  } else {
    const int fc = next_child(sh.par, i, i, R);
    if (fc >= 0) probe = sh.tok[fc];
  }
  const float* qrow = nullptr;
  if (p.q) {
    if (p.tree)
      qrow = p.q + ((size_t)b * R + i) * V;
    else if (i < R - 1)
      qrow = p.q + ((size_t)b * (R - 1) + i) * V;
  }

  // each warp owns one contiguous id range of the row (a multiple of 32 long);
  // four logits of ids k..k+3 at a time (-inf past the range)
  const int rw = stream_range_width(V);
  const int r0 = min(warp * rw, V), r1 = min((warp + 1) * rw, V);
  auto load4 = [&](int k, float (&lv)[4]) {
    if (vec && k + 3 < r1) {
      const float4 v = ldg_keep4(reinterpret_cast<const float4*>(lrow + k), pol);
      lv[0] = v.x;
      lv[1] = v.y;
      lv[2] = v.z;
      lv[3] = v.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) lv[j] = k + j < r1 ? ldg_keep(lrow + k + j, pol) : -INFINITY;
    }
  };
  const unsigned lt = (1u << lane) - 1u;

  // ---- 1. the maximum (NaN-propagating) and Z.  PRE: every warp combines
  // the ranges' maxima (lane r holds range r's results).  Otherwise one sweep
  // of the row: one sample per thread, evenly spaced, gives a reference
  // maximum sref and the candidate floor Lf (a logit); the sweep then takes
  // the maximum, Z relative to sref (rescaled to the maximum after it) and a
  // bit per id at or above Lf
  float m;
  RangeStat st{0.f, 0.f, 0.f, 0};
  float Lf = INFINITY;              // candidate floor (+inf: no lists)
  float zh_sw = 0.f, zl_sw = 0.f;   // Z of the sweep (relative to m), float pair
  int cnt_sw = 0;                   // ids the sweep listed in this warp's range
  const float c_hi = p.c_hi, c_lo = p.c_lo, T150 = 150.f * p.T;
  if constexpr (PRE) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the pre-pass has completed
    st = p.stats[(size_t)row * kRangesPerRow + lane];
    m = st.m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(kFull, m, o));
    Lf = p.lfloor[2 * row];
  } else {
    // the samples' bin counters (the members' scratch, unused until the cut)
    uint32_t* scnt = reinterpret_cast<uint32_t*>(xkey);
    static_assert(NT == kBins, "one counter per thread, and one more");
    scnt[threadIdx.x] = 0u;
    if (threadIdx.x == 0) scnt[kBins] = 0u;
    float sm = smp;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm = fmax_nan(sm, __shfl_xor_sync(kFull, sm, o));
    if (lane == 0) sh.red_f[warp] = sm;
    __syncthreads();
    float sref = sh.red_f[0];
    for (int w = 1; w < NW; ++w) sref = fmax_nan(sref, sh.red_f[w]);
    const bool sref_ok = fabsf(sref) < INFINITY;  // uniform
    const float snmc = -sref * c_hi, snm = -sref, slfl = sref - T150;
    auto Eref = [&](float l) {
      return FAST ? fexp(l, c_hi, snmc) : texp(l, snm, slfl, c_hi, c_lo);
    };
    if (trunc && V <= kSListMaxV && sref_ok) {
      // the deepest bin of E relative to sref (32 per octave) whose sampled
      // count at or above it stays within the list budget, taken as a logit
      const float budget =
          topk ? fminf((float)kSBudget, 4.f * (float)p.top_k + 1024.f) : (float)kSBudget;
      const int ns = (int)(budget * (float)NT / (float)V);
      if (ns >= 1 && (!topk || p.top_k <= kSBudget / 2)) {
        atomicAdd(&scnt[ebin(__float_as_uint(Eref(smp)))], 1u);
        __syncthreads();
        if (warp == 0) {  // the largest b with count(sample bin <= b) <= ns
          // lane o: the count of octave o (bins 32 o .. 32 o + 31, 16-byte loads)
          const uint4* s4 = reinterpret_cast<const uint4*>(scnt + 32 * lane);
          uint32_t c = 0;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = s4[v];
            c += (x.x + x.y) + (x.z + x.w);
          }
          uint32_t incl = c;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t2 = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t2;
          }
          const unsigned h = __ballot_sync(kFull, incl > (uint32_t)ns);
          int bfs = kBins - 1;
          if (h) {
            // the crossing octave L: lane j takes bin 32 L + j, the running
            // count over the octave by a warp scan
            const int L = __ffs(h) - 1;
            const uint32_t base = __shfl_sync(kFull, incl - c, L);
            const uint32_t v = scnt[32 * L + lane];
            uint32_t run = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t t2 = __shfl_up_sync(kFull, run, o);
              if (lane >= o) run += t2;
            }
            const unsigned h2 = __ballot_sync(kFull, base + run > (uint32_t)ns);
            bfs = 32 * L + (__ffs(h2) - 1) - 1;  // h2 != 0: the octave's total crosses ns
          }
          if (lane == 0) sh.bi[6] = bfs;
        }
        __syncthreads();
        const int lo = sh.bi[6];
        if (lo >= 0) Lf = sref - (float)(lo + 1) * (p.T * kLn2 * (1.f / 32.f));
      }
    }
    const bool flagging = Lf < INFINITY;
    float mx = -INFINITY;
    uint64_t zs2 = f2_pack(0.f, 0.f), zc2 = f2_pack(0.f, 0.f);
    const uint64_t m1 = f2_pack(-1.f, -1.f);
    int* const wlid = lid + warp * WCAP;
    float* const wlval = lval + warp * WCAP;
    for (int s0 = r0; s0 < r1; s0 += 512) {  // warp-uniform
      // the chunk after the next one into L2 now (one 128-byte line per lane of
      // the first 16): the loads below then wait on L2 rather than on HBM
      if (lane < 16 && s0 + 1024 + 32 * lane < r1)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(lrow + s0 + 1024 + 32 * lane));
      float lv[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) load4(s0 + 128 * u + 4 * lane, lv[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = s0 + 128 * u + 4 * lane;
        float e[4];
        mx = fmax3_nan(mx, lv[u][0], lv[u][1]);
        mx = fmax3_nan(mx, lv[u][2], lv[u][3]);
        if (FAST) {  // the exponents' arguments two at a time (packed f32x2 FMA)
          const uint64_t c2 = f2_pack(c_hi, c_hi), n2 = f2_pack(snmc, snmc);
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(lv[u][0], lv[u][1]), c2, n2), x0, x1);
          f2_unpack(f2_fma(f2_pack(lv[u][2], lv[u][3]), c2, n2), x2, x3);
          e[0] = ex2_ftz(x0);
          e[1] = ex2_ftz(x1);
          e[2] = ex2_ftz(x2);
          e[3] = ex2_ftz(x3);  // 0 past the range
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) e[j] = Eref(lv[u][j]);
        }
        // Kahan summation of (e0 + e2, e1 + e3) in two packed streams
        const uint64_t y2 = f2_fma(zc2, m1, f2_add(f2_pack(e[0], e[1]), f2_pack(e[2], e[3])));
        const uint64_t t2 = f2_add(zs2, y2);
        zc2 = f2_fma(y2, m1, f2_fma(zs2, m1, t2));  // (t - s) - y
        zs2 = t2;
        if (flagging) {  // the ids at or above the floor, appended to the warp's list
          bool f[4];
          unsigned bal[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            f[j] = lv[u][j] >= Lf;  // false past the range (-inf)
            bal[j] = __ballot_sync(kFull, f[j]);
          }
          int pos = cnt_sw + __popc(bal[0] & lt) + __popc(bal[1] & lt) + __popc(bal[2] & lt) +
                    __popc(bal[3] & lt);  // ascending: lanes, then j
          if (cnt_sw + 128 <= WCAP) {  // warp-uniform: every entry of the group fits
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (f[j]) {
                wlid[pos] = k + j;
                wlval[pos] = lv[u][j];
                ++pos;
              }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (f[j]) {
                if (pos < WCAP) {
                  wlid[pos] = k + j;
                  wlval[pos] = lv[u][j];
                }
                ++pos;
              }
          }
          cnt_sw = __shfl_sync(kFull, pos, 31);  // the last lane's end: the warp's count
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax_nan(mx, __shfl_xor_sync(kFull, mx, o));
    __syncthreads();  // every thread has read sh.red_f above
    if (lane == 0) sh.red_f[warp] = mx;
    __syncthreads();
    m = sh.red_f[0];
    for (int w = 1; w < NW; ++w) m = fmax_nan(m, sh.red_f[w]);
    __syncthreads();  // every thread has m before the sums reuse sh.red_f
    float zs, zc;
    {
      float s0, s1, c0, c1;
      f2_unpack(zs2, s0, s1);
      f2_unpack(zc2, c0, c1);
      // the streams' sums added exactly (TwoSum: zs + err), the compensations
      // (excess over the true sums) added in
      zs = s0 + s1;
      const float bb = zs - s0;
      const float err = (s0 - (zs - bb)) + (s1 - bb);
      zc = (c0 + c1) - err;
    }
    const float Zh = block_sum_f<NT>(zs, sh), Zl = block_sum_f<NT>(-zc, sh);
    if (fabsf(m) < INFINITY) {  // uniform
      if (sref_ok && fabsf(Zh) < INFINITY) {
        // relative to m: times E(sref) relative to m, the product's error in the pair
        const float sc = FAST ? fexp(sref, c_hi, -m * c_hi) : texp(sref, -m, m - T150, c_hi, c_lo);
        zh_sw = Zh * sc;
        zl_sw = __fmaf_rn(Zh, sc, -zh_sw) + Zl * sc;
      } else {
        // E relative to sref overflowed (or no reference): Z again relative to m
        const float nm2 = -m, lfl2 = m - T150, nmc2 = -m * c_hi;
        float s2 = 0.f, c2 = 0.f;
        sweep([&](int, float l) {
          const float y = (FAST ? fexp(l, c_hi, nmc2) : texp(l, nm2, lfl2, c_hi, c_lo)) - c2;
          const float t = s2 + y;
          c2 = (t - s2) - y;
          s2 = t;
        });
        zh_sw = block_sum_f<NT>(s2, sh);
        zl_sw = block_sum_f<NT>(-c2, sh);
      }
    }
  }
  const bool bad = isnan(m) || m == INFINITY || m == -INFINITY;
  Outcome oc{0, -1, 0, bad ? 1 : 0};
  // the chain test's operands, loaded now: their latency hides under the next sweep
  const bool chain_test = !p.tree && i < R - 1;
  const float u_test = chain_test ? __ldg(&p.u[(size_t)b * R + i]) : 0.f;
  const float u_last = __ldg(&p.u[(size_t)b * R + (R - 1)]);
  const float q_probe =
      (chain_test && qrow != nullptr && probe >= 0 && probe < V) ? __ldg(&qrow[probe]) : 0.f;
  const float l_probe = (probe >= 0 && probe < V) ? __ldg(lrow + probe) : 0.f;

  if (!bad) {
    const float nm = -m, lfloor = m - 150.f * p.T;
    const float nmc = -m * c_hi;
    auto Eof = [&](float l) { return FAST ? fexp(l, c_hi, nmc) : texp(l, nm, lfloor, c_hi, c_lo); };
    auto hist = [&](uint32_t bits, int bn) {
      if (topk) atomicAdd(&hcnt[bn], 1u);
      if (topp && bn < kBins) atomicAdd(&hm[bn], m16(bits));
    };
    auto hist_e = [&](float e) {
      const uint32_t bits = __float_as_uint(e);
      hist(bits, ebin(bits));
    };

    // ---- 2. the listed bins: those whose every element lies at or above the
    // floor Lf, i.e. above the bin of E at Lf (taken 2^-12 high, which covers
    // the rounding of E); -1: no lists (every element histogrammed)
    int bf = -1;
    if (trunc && Lf < INFINITY) bf = ebin(__float_as_uint(Eof(Lf) * 1.000244140625f)) - 1;
    const bool listing = bf >= 0;

    // ---- 3. (PRE) Z: the ranges' Z combined
    if constexpr (PRE) {
      if (warp == 0) {
        // Z = sum over the ranges of Z_r E(m_r), in float pairs, fixed order
        const float sc = st.m == -INFINITY ? 0.f : Eof(st.m);
        float zh2 = st.zh * sc;
        float zl2 = __fmaf_rn(st.zh, sc, -zh2) + st.zl * sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float oh = __shfl_xor_sync(kFull, zh2, o);
          const float ol = __shfl_xor_sync(kFull, zl2, o);
          df_acc(zh2, zl2, oh, ol);
        }
        if (lane == 0) {
          sh.zpre[0] = zh2;
          sh.zpre[1] = zl2;
        }
      }
    }
    if (threadIdx.x == 0 && probe >= 0 && probe < V) sh.eprobe = Eof(l_probe);

    // ---- 4. the candidate lists: each warp lists the flagged ids of its
    // range in id order, then loads their logits; the histogram of the listed
    // elements of bins <= bf; without lists, or if a list overflowed, of every
    // element
    int cntw = 0;
    if (PRE) {
      // this warp's range list, copied from the pre-pass results: kSwW
      // segments in order (the entry j of the range lies in the last segment
      // whose offset is <= j)
      const int c = __shfl_sync(kFull, st.cnt, warp);
      cntw = listing ? c : 0;
      if (listing && c <= WCAP) {
        const size_t rg = (size_t)row * kRangesPerRow + warp;
        const int sc = lane < kSwW ? p.segcnt[rg * kSwW + lane] : 0;
        int incl = sc;
#pragma unroll
        for (int o = 1; o < kSwW; o <<= 1) {
          const int t2 = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t2;
        }
        int soff[kSwW];
#pragma unroll
        for (int k = 0; k < kSwW; ++k) soff[k] = __shfl_sync(kFull, incl - sc, k);
        const int32_t* gid = p.lid_g + rg * kSwW * kSegCap;
        const float* gval = p.lval_g + rg * kSwW * kSegCap;
        for (int j0 = 0; j0 < c; j0 += 256) {
          int idv[8];
          float lvv[8];  // eight entries in flight per lane
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + 32 * u + lane;
            int sg = 0, so = 0;  // the last segment whose offset is <= j (offsets ascend)
#pragma unroll
            for (int k = 1; k < kSwW; ++k)
              if (soff[k] <= j) {
                sg = k;
                so = soff[k];
              }
            const int at = sg * kSegCap + (j - so);
            idv[u] = j < c ? gid[at] : 0;
            lvv[u] = j < c ? gval[at] : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + 32 * u + lane;
            if (j < c) {
              lid[warp * WCAP + j] = idv[u];
              lval[warp * WCAP + j] = lvv[u];
              const uint32_t bits = __float_as_uint(Eof(lvv[u]));
              const int bn = ebin(bits);
              if (bn <= bf) hist(bits, bn);
            }
          }
        }
      }
    } else if (listing) {
      // the sweep listed the ids at or above the floor with their logits
      cntw = cnt_sw;
      if (cntw <= WCAP) {
        __syncwarp();
        const float* wv = lval + warp * WCAP;
        for (int j0 = 0; j0 < cntw; j0 += 128) {  // four entries per lane in flight
          float lv4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + 32 * u + lane;
            lv4[u] = j < cntw ? wv[j] : -INFINITY;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (j0 + 32 * u + lane < cntw) {
              const uint32_t bits = __float_as_uint(Eof(lv4[u]));
              const int bn = ebin(bits);
              if (bn <= bf) hist(bits, bn);  // a listed element of the partly listed bin: no
            }
          }
        }
      }
    }
    if (lane == 0) sh.list_n[warp] = cntw;
    const bool fit = __syncthreads_and(cntw <= WCAP ? 1 : 0) != 0;
    // lists hold every element that can be kept (ids, logits)
    bool cand_lists = listing && fit;
    if ((listing && !fit) || (trunc && !listing)) {
      for (int k = threadIdx.x; k < kHist; k += NT) {
        hcnt[k] = 0u;
        hm[k] = 0u;
      }
      __syncthreads();
      sweep([&](int, float l) { hist_e(Eof(l)); });
      bf = -1;
    }
    __syncthreads();  // the histogram (and, PRE, the Z pair) is complete
    const float zh = PRE ? sh.zpre[0] : zh_sw;
    const float zl = PRE ? sh.zpre[1] : zl_sw;
    const float e_probe = sh.eprobe;
    const unsigned long long zfx = fx44_pair(zh, zl);  // Z in units of 2^-44
    // a draft row that is likely to reject (p(x) <= E(x) / Z_kept is not
    // surely above u q(x)), or a tree node with children, reads q at its kept
    // ids for the residual: start those reads into L2 now, under the cut
    if (cand_lists && qrow != nullptr &&
        (p.tree ? probe >= 0 : (chain_test && !(u_test * q_probe * (zh + zl) < e_probe)))) {
      const int cnt = sh.list_n[warp];
      for (int j = lane; j < cnt; j += 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + lid[warp * WCAP + j]));
    }

    Cut cut{0, 0.f, 0u, INT_MAX};
    float zkept = zh + zl;
    if (trunc) {
      // ---- 5. the cut: bin range, members, selection (or the radix fallback)
      // every warp runs the search on the octave totals (a lone warp whose
      // siblings wait at a barrier runs its shuffles far slower)
      int f_mode = 2, f_lo = 0, f_hi = 0, f_k = -1;
      auto run_find = [&]() {
        {  // warp o: the totals of octave o
          uint32_t c = topk ? hcnt[32 * warp + lane] : 0u;
          unsigned long long mm = topp ? hm[32 * warp + lane] : 0u;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            c += __shfl_xor_sync(kFull, c, o);
            mm += __shfl_xor_sync(kFull, mm, o);
          }
          if (lane == 0) {
            sh.octc[warp] = c;
            sh.octm[warp] = mm;
          }
        }
        __syncthreads();
        find_range<NT>(
            topk, topp, p.top_k, p.top_p, zfx,
            [&](int o, unsigned long long& c, unsigned long long& mm) {
              c += sh.octc[o];
              mm += sh.octm[o];
            },
            [hcnt, hm, topk, topp](int bb, unsigned long long& c, unsigned long long& mm) {
              if (topk) c += hcnt[bb];
              if (topp) mm += hm[bb];
            },
            &f_mode, &f_lo, &f_hi, &f_k);
        __syncthreads();  // the totals may be rewritten by a second search
      };
      run_find();
      int tmode = f_mode;
      if (tmode == 2 && cand_lists) {
        // the cut lies below the listed bins: histogram the rest, search again
        sweep([&](int, float l) {
          const uint32_t bits = __float_as_uint(Eof(l));
          const int bn = ebin(bits);
          if (bn > bf) hist(bits, bn);
        });
        __syncthreads();
        run_find();
        tmode = f_mode;
        cand_lists = false;
      }
      int b_lo = f_lo, b_hi = f_hi, kidx = f_k;
      // a second attempt one bin wider on each side: the rounded bin masses
      // may place a cut that lies within their rounding of a bin edge one bin off
      for (int attempt = 0; tmode == 1 && attempt < 2; ++attempt) {
        if (attempt == 1) {
          if (b_lo > 0) {
            --b_lo;
            if (kidx >= 0) kidx += (int)hcnt[b_lo];  // the count above the range shrinks
          }
          if (b_hi < kBins - 1 && (!cand_lists || b_hi < bf)) ++b_hi;
          if (threadIdx.x == 0) sh.bi[4] = 0;
          __syncthreads();
        }
        // members of bins [b_lo, b_hi] and the exact mass above them; a logit
        // pre-filter (with margin) skips the E of elements below the range
        const uint32_t edge = (uint32_t)(0x3F7FFFFF - ((b_hi + 1) << 18) + 1);
        const float lpre = m + p.T * (__logf(__uint_as_float(edge)) - 1e-3f);
        unsigned long long above = 0;
        // an element that passed the pre-filter: above the range, a member, or below
        auto consider = [&](int k, float l) {
          const uint32_t bits = __float_as_uint(Eof(l));
          if (bits < edge) return;
          const int bn = ebin(bits);
          if (bn < b_lo) {
            above += fx44(bits);
          } else {
            const int slot = atomicAdd(&sh.bi[4], 1);
            if (slot < NT) {
              xkey[slot] = ((unsigned long long)okey(l) << 32) | (0xFFFFFFFFu - (uint32_t)k);
              xbits[slot] = bits;
            }
          }
        };
        if (!cand_lists) {
          // the pre-filter's survivors of each warp's range, compacted in id order
          // into the warp's list (id, logit); they include every element the cut
          // can keep
          int cw = 0;
          for (int s0 = r0; s0 < r1; s0 += 512) {
            float lv[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) load4(s0 + 128 * u + 4 * lane, lv[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k = s0 + 128 * u + 4 * lane;
              bool f[4];
              unsigned bal[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                f[j] = lv[u][j] >= lpre;
                bal[j] = __ballot_sync(kFull, f[j]);
              }
              int pos = cw + __popc(bal[0] & lt) + __popc(bal[1] & lt) + __popc(bal[2] & lt) +
                        __popc(bal[3] & lt);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (f[j]) {
                  if (pos < WCAP) {
                    lid[warp * WCAP + pos] = k + j;
                    lval[warp * WCAP + pos] = lv[u][j];
                  }
                  ++pos;
                }
              cw += __popc(bal[0]) + __popc(bal[1]) + __popc(bal[2]) + __popc(bal[3]);
            }
          }
          if (lane == 0) sh.list_n[warp] = cw;
          cand_lists = __syncthreads_and(cw <= WCAP ? 1 : 0) != 0;
        }
        if (cand_lists) {
          const int cnt = sh.list_n[warp];
          const int* wi = lid + warp * WCAP;
          const float* wv = lval + warp * WCAP;
          for (int j0 = 0; j0 < cnt; j0 += 128) {  // four entries per lane in flight
            int id4[4];
            float lv4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = j0 + 32 * u + lane;
              id4[u] = j < cnt ? wi[j] : 0;
              lv4[u] = j < cnt ? wv[j] : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (j0 + 32 * u + lane < cnt) consider(id4[u], lv4[u]);
          }
        } else {
          // the row, each warp its range, 32 consecutive ids per step, eight
          // steps' loads in flight
          for (int k0 = r0; k0 < r1; k0 += 256) {  // warp-uniform
            float lv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int k = k0 + 32 * u + lane;
              lv[u] = k < r1 ? ldg_keep(lrow + k, pol) : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int k = k0 + 32 * u + lane;
              if (k < r1 && lv[u] >= lpre) consider(k, lv[u]);
            }
          }
        }
        const unsigned long long a_lo = block_sum_u64<NT>(above, sh);  // barriers: members complete
        const int total = sh.bi[4];
        if (total > NT || total < 1) {
          tmode = 2;
        } else {
          const int t = threadIdx.x;
          const unsigned long long key = t < total ? xkey[t] : 0ull;
          const uint32_t eb = t < total ? xbits[t] : 0u;
          if (select_cut<NT>(key, eb, total, a_lo, kidx, topp, p.top_p,
                             zfx, xkey, xbits, &cut, &zkept, sh))
            break;
          if (attempt == 1) tmode = 2;
        }
      }
      if (tmode == 2) {
        cand_lists = false;
        cut = cut_radix<NT>(p, lrow, [&](int k) { return Eof(__ldg(lrow + k)); }, V, 0, rs, 0, 1,
                            ph, sh);
        float s = 0.f, cmp = 0.f;
        for (int k0 = threadIdx.x; k0 < V; k0 += 8 * NT) {
          float lv[8];  // eight logits in flight per thread
#pragma unroll
          for (int u = 0; u < 8; ++u) lv[u] = k0 + u * NT < V ? __ldg(lrow + k0 + u * NT) : 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int k = k0 + u * NT;
            if (k < V && is_kept(okey(lv[u]), k, cut.tau, cut.tie)) {
              const float y = Eof(lv[u]) - cmp;
              const float tt = s + y;
              cmp = (tt - s) - y;
              s = tt;
            }
          }
        }
        const float hs = block_sum_f<NT>(s, sh);
        const float ls = block_sum_f<NT>(-cmp, sh);
        zkept = hs + ls;
      }
      cut.mode = 2;  // from here on the kept test uses the logit keys
    }
    const float invz = 1.0f / zkept;
    auto kept_l = [&](float l, int id) { return !trunc || is_kept(okey(l), id, cut.tau, cut.tie); };

    // ---- 6. (on first use) list each warp's kept positions with their E
    bool listed = false, list_ready = false;
    auto ensure_list = [&]() {
      if (list_ready) return;
      list_ready = true;
      if (cand_lists) {
        // keep the candidates the cut keeps (in place, order preserved), logit -> E
        const int cnt = sh.list_n[warp];
        int kept = 0;
        for (int s0 = 0; s0 < cnt; s0 += 32) {
          const int j = s0 + lane;
          const int id = j < cnt ? lid[warp * WCAP + j] : 0;
          const float l = j < cnt ? lval[warp * WCAP + j] : 0.f;
          const bool kp = j < cnt && kept_l(l, id);
          const unsigned bal = __ballot_sync(kFull, kp);
          if (kp) {
            const int pos = kept + __popc(bal & ((1u << lane) - 1));
            lid[warp * WCAP + pos] = id;
            lval[warp * WCAP + pos] = Eof(l);
          }
          kept += __popc(bal);
        }
        __syncwarp();
        if (lane == 0) sh.list_n[warp] = kept;
        listed = true;
        __syncthreads();
      } else {
      int cntw = 0;
      for (int s0 = r0; s0 < r1; s0 += 512) {
        float lv[16];  // sixteen loads in flight per lane
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int k = s0 + 32 * u + lane;
          lv[u] = k < r1 ? ldg_keep(lrow + k, pol) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int k = s0 + 32 * u + lane;
          const bool kp = k < r1 && kept_l(lv[u], k);
          const unsigned bal = __ballot_sync(kFull, kp);
          const int pos = cntw + __popc(bal & ((1u << lane) - 1));
          if (kp && pos < WCAP) {
            lid[warp * WCAP + pos] = k;
            lval[warp * WCAP + pos] = Eof(lv[u]);
          }
          cntw += __popc(bal);
        }
      }
      if (lane == 0) sh.list_n[warp] = cntw;
      listed = __syncthreads_and(cntw <= WCAP ? 1 : 0) != 0;
      }
      // list positions of the node's children (binary search in the owning warp's list)
      if (listed && p.tree)
        for (int c = threadIdx.x; c < R; c += NT) {
          const int t = sh.tok[c];
          if (sh.par[c] != i || t < 0 || t >= V) continue;
          const int w = min(t / rw, NW - 1);
          int lo2 = 0, hi2 = sh.list_n[w];
          while (lo2 < hi2) {
            const int mid = (lo2 + hi2) >> 1;
            if (lid[w * WCAP + mid] < t) lo2 = mid + 1; else hi2 = mid;
          }
          if (lo2 < sh.list_n[w] && lid[w * WCAP + lo2] == t) sh.cpos[c] = w * WCAP + lo2;
        }
      __syncthreads();
    };
    if (p.p_out) {
      float* dst = p.p_out + (size_t)row * V;
      for (int k = threadIdx.x; k < V; k += NT) {
        const float l = __ldg(lrow + k);
        dst[k] = kept_l(l, k) ? Eof(l) * invz : 0.f;
      }
    }

    // weights of the listed items (mode 1: max(0, v * invw - q) stored back):
    // per-warp sums in sh.wsum, the CTA total returned (fixed order)
    auto list_weights = [&](int mode, float invw) -> float {
      // every warp is done with the previous weights (sh.wsum, and the list values
      // a tree node's child test read from any warp's list) before they change
      __syncthreads();
      const int cnt = min(sh.list_n[warp], WCAP);
      float acc = 0.f;
      for (int j0 = 0; j0 < cnt; j0 += 256) {  // eight q loads in flight per lane
        float vv[8], qq[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + 32 * u + lane;
          vv[u] = j < cnt ? lval[warp * WCAP + j] : 0.f;
        }
        if (mode == 1) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + 32 * u + lane;
            qq[u] = (j < cnt && vv[u] > 0.f) ? __ldg(qrow + lid[warp * WCAP + j]) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + 32 * u + lane;
            if (j < cnt) {
              vv[u] = residual_w(vv[u], invw, qq[u]);
              lval[warp * WCAP + j] = vv[u];
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += vv[u];  // ascending j, as one lane's stride
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      if (lane == 0) sh.wsum[warp] = acc;
      __syncthreads();
      float t = 0.f;
      for (int w = 0; w < NW; ++w) t += sh.wsum[w];
      return t;
    };
    // the first listed id whose running weight (ascending id) exceeds u * W
    auto list_locate = [&](float u, float W) -> int {
      const float target = u * W;
      int ow = -1, lw = -1;
      float wpre = 0.f, base_ow = 0.f, base_lw = 0.f;
      for (int w = 0; w < NW; ++w) {
        const float t = sh.wsum[w];
        if (t > 0.f) {
          if (ow < 0 && wpre + t > target) { ow = w; base_ow = wpre; }
          lw = w;
          base_lw = wpre;
        }
        wpre += t;
      }
      if (ow < 0) { ow = lw; base_ow = base_lw; }
      if (ow < 0) return -1;
      if (warp == ow) {
        const int cnt = min(sh.list_n[ow], WCAP);
        const int c = ((cnt + 31) / 32) | 1;
        const int j0 = min(lane * c, cnt), j1 = min(j0 + c, cnt);
        float ls = 0.f;
        for (int j = j0; j < j1; ++j) ls += lval[ow * WCAP + j];
        const float tw = target - base_ow;
        float incl = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned hit = __ballot_sync(kFull, ls > 0.f && incl > tw);
        const unsigned nz = __ballot_sync(kFull, ls > 0.f);
        const int L = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : -1);
        int found = -1;
        if (lane == L) {
          const float tl = tw - (incl - ls);
          float run = 0.f;
          int lastk = -1;
          for (int j = j0; j < j1; ++j) {
            const float v = lval[ow * WCAP + j];
            if (v > 0.f) {
              lastk = lid[ow * WCAP + j];
              run += v;
              if (run > tl) { found = lastk; break; }
            }
          }
          if (found < 0) found = lastk;
        }
        found = __shfl_sync(kFull, found, L < 0 ? 0 : L);
        if (lane == 0) sh.bi[7] = found;
      }
      __syncthreads();
      const int t = sh.bi[7];
      __syncthreads();
      return t;
    };
    // the same over the whole row with the weights recomputed (kept set too
    // large to list): w = kept ? (mode 1: max(0, E * invz - q); mode 0: E) : 0
    auto wfull = [&](int k, int mode) -> float {
      const float l = __ldg(lrow + k);
      if (!kept_l(l, k)) return 0.f;
      const float e = Eof(l);
      return mode == 1 ? residual_w(e, invz, __ldg(qrow + k)) : e;
    };
    auto full_draw = [&](int mode, float u) -> int {
      float acc = 0.f;
      for (int k = r0 + lane; k < r1; k += 32) acc += wfull(k, mode);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      if (lane == 0) sh.wsum[warp] = acc;
      __syncthreads();
      float W = 0.f;
      for (int w = 0; w < NW; ++w) W += sh.wsum[w];
      if (!(W > 0.f)) return -2;
      const float target = u * W;
      int ow = -1, lw = -1;
      float wpre = 0.f, base_ow = 0.f, base_lw = 0.f;
      for (int w = 0; w < NW; ++w) {
        const float t = sh.wsum[w];
        if (t > 0.f) {
          if (ow < 0 && wpre + t > target) { ow = w; base_ow = wpre; }
          lw = w;
          base_lw = wpre;
        }
        wpre += t;
      }
      if (ow < 0) { ow = lw; base_ow = base_lw; }
      if (warp == ow) {
        const int wr0 = min(ow * rw, V), wr1 = min((ow + 1) * rw, V);
        const int c = ((wr1 - wr0 + 31) / 32) | 1;
        const int j0 = min(wr0 + lane * c, wr1), j1 = min(j0 + c, wr1);
        float ls = 0.f;
        for (int k = j0; k < j1; ++k) ls += wfull(k, mode);
        const float tw = target - base_ow;
        float incl = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned hit = __ballot_sync(kFull, ls > 0.f && incl > tw);
        const unsigned nz = __ballot_sync(kFull, ls > 0.f);
        const int L = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : -1);
        int found = -1;
        if (lane == L) {
          const float tl = tw - (incl - ls);
          float run = 0.f;
          for (int k = j0; k < j1; ++k) {
            const float v = wfull(k, mode);
            if (v > 0.f) {
              found = k;
              run += v;
              if (run > tl) break;
            }
          }
        }
        found = __shfl_sync(kFull, found, L < 0 ? 0 : L);
        if (lane == 0) sh.bi[7] = found;
      }
      __syncthreads();
      const int t = sh.bi[7];
      __syncthreads();
      return t;
    };

    const float u_final = u_last;
    if (!p.tree) {
      // ---- 7a. chain: the row's test, then its correction or bonus draw
      bool resid = false;
      if (i < R - 1) {
        const int x = probe;
        const bool xin = x >= 0 && x < V;
        const float qx = xin ? q_probe : 0.f;
        const float px = (xin && e_probe > 0.f && kept_l(l_probe, x)) ? e_probe * invz : 0.f;
        if (qx == 0.f) oc.status |= SPEC_SEQ_QZERO;
        oc.accept = (u_test * qx < px) ? 1 : 0;
        resid = !oc.accept;
      }
      if (i == R - 1 || resid) {
        ensure_list();
        int tokn;
        if (listed) {
          const float W = list_weights(resid ? 1 : 0, invz);
          tokn = W > 0.f ? list_locate(u_final, W) : -2;
        } else {
          tokn = full_draw(resid ? 1 : 0, u_final);
        }
        if (tokn == -2) {  // residual with zero mass (rounding only): draw from p
          oc.status |= SPEC_SEQ_RESID_ZERO;
          tokn = full_draw(0, u_final);
        }
        oc.token = tokn;
      }
    } else {
      // ---- 7b. tree node: children in storage order against the running p'
      ensure_list();  // the host routes here only trees whose kept set fits the lists
      oc.accept = -1;
      float invw = invz;
      int nsteps = 0;
      for (int c = next_child(sh.par, i, i, R); c >= 0; c = next_child(sh.par, i, c, R)) {
        const int t = sh.tok[c];
        const bool tin = t >= 0 && t < V;
        const float qt = tin ? __ldg(&qrow[t]) : 0.f;
        const float pt = (tin && sh.cpos[c] >= 0) ? lval[sh.cpos[c]] * invw : 0.f;
        if (qt == 0.f) oc.status |= SPEC_SEQ_QZERO;
        if (__ldg(&p.u[(size_t)b * R + (c - 1)]) * qt < pt) {
          oc.accept = c;
          break;
        }
        if (threadIdx.x == 0) sh.invw_used[nsteps] = invw;
        const float W = list_weights(1, invw);  // p' <- norm(max(0, p' - q_v))
        if (W > 1e-37f) {
          invw = 1.0f / W;
          ++nsteps;
        } else {
          // zero mass (rounding only): keep p' -- rebuild it from the logits
          oc.status |= SPEC_SEQ_RESID_ZERO;
          const int cnt = min(sh.list_n[warp], WCAP);
          for (int j = lane; j < cnt; j += 32) {
            const int id = lid[warp * WCAP + j];
            float e = Eof(__ldg(lrow + id));
            for (int s2 = 0; s2 < nsteps; ++s2)
              e = residual_w(e, sh.invw_used[s2], e > 0.f ? __ldg(qrow + id) : 0.f);
            lval[warp * WCAP + j] = e;
          }
          __syncthreads();
        }
      }
      if (oc.accept < 0) {
        const float W = list_weights(0, 1.f);
        oc.token = W > 0.f ? list_locate(u_final, W) : -1;
        if (!(W > 0.f)) oc.status |= SPEC_SEQ_RESID_ZERO;
      }
    }
  }
  if (threadIdx.x >= 32) return;
  finish_row(p, row, oc, sh);
}

// ---------------------------------------------------------------- streaming pre-pass (many rows)
// Pass 1 of the two-pass streaming sampler, in two kernels.
//  * sampler_floor_kernel: each row's candidate floor, from 1024 evenly
//    spaced samples: the deepest bin (32 per octave of E relative to the
//    samples' maximum) whose sample count at or above it stays within the
//    list budget, taken as a logit.
//  * sampler_sweep_kernel: every row swept from HBM once, by one CTA per
//    warp range of the row kernel (32 per row: the sweep spreads evenly over
//    every SM, eight CTAs resident per SM).  The CTA copies its whole range
//    into shared memory at once (16-byte cp.async: about 150 KB in flight per
//    SM), then in one pass computes the range's maximum, Z relative to the
//    row samples' maximum (rescaled to the range's), and the ballots of the
//    ids at or above the floor, from which it writes their list (ascending,
//    with their logits).
// The row kernel (pass 2) starts from these results.  Both launches after
// the first are programmatic dependents: they start while the previous one
// finishes and wait for its results (griddepcontrol.wait) only where they
// need them.
constexpr int kSwMaxPieces = 64;  // 128-id pieces per range (ranges of up to 8192 ids)
constexpr int kSwCTAs = 5;        // pre-pass CTAs per SM (two range buffers each)


// The row's candidate floor as a logit (+inf: no lists).  Every thread
// returns the same value; contains barriers (call from uniform control flow).
template <bool FAST>
SPEC_DEV float row_floor(const SP& p, const float* lrow, uint64_t pol, uint32_t* scnt,
                         float* sred, int* sbf, float* smax_out) {
  const int V = p.V, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool topk = p.top_k > 0 && p.top_k < V;
  const bool topp = p.top_p > 0.f && p.top_p < 1.f;
  const float budget =
      topk ? fminf((float)kSBudget, 4.f * (float)p.top_k + 1024.f) : (float)kSBudget;
  const int ns = (int)(budget * (float)kSamples / (float)V);
  const bool want = (topk || topp) && V <= kSListMaxV && ns >= 1 &&
                    (!topk || p.top_k <= kSBudget / 2);
  constexpr int SPT = kSamples / kSwNT;  // samples per thread
  float smp[SPT];
  float sm = -INFINITY;
#pragma unroll
  for (int u = 0; u < SPT; ++u) {
    const long long j = threadIdx.x + kSwNT * u;
    smp[u] = ldg_keep(lrow + (int)((j * V) / kSamples), pol);
    sm = fmax_nan(sm, smp[u]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sm = fmax_nan(sm, __shfl_xor_sync(kFull, sm, o));
  if (lane == 0) sred[warp] = sm;
  for (int k = threadIdx.x; k < kHist; k += kSwNT) scnt[k] = 0u;
  __syncthreads();
  float smax = sred[0];
  for (int w = 1; w < kSwW; ++w) smax = fmax_nan(smax, sred[w]);
  *smax_out = smax;
  if (!want || !(fabsf(smax) < INFINITY)) return INFINITY;  // uniform
  const float nm = -smax, lfl = smax - 150.f * p.T, nmc = -smax * p.c_hi;
#pragma unroll
  for (int u = 0; u < SPT; ++u) {
    const float e = FAST ? fexp(smp[u], p.c_hi, nmc) : texp(smp[u], nm, lfl, p.c_hi, p.c_lo);
    atomicAdd(&scnt[ebin(__float_as_uint(e))], 1u);
  }
  __syncthreads();
  if (warp == 0) {
    // the deepest bin b whose samples in bins <= b number at most ns
    uint32_t c = 0;
    for (int b = 32 * lane; b < 32 * lane + 32; ++b) c += scnt[b];
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned h = __ballot_sync(kFull, incl > (uint32_t)ns);
    int bfs = kBins - 1;
    if (h) {
      const int L = __ffs(h) - 1;
      uint32_t run = __shfl_sync(kFull, incl - c, L);
      bfs = 32 * L + 31;
      for (int b = 32 * L; b < 32 * L + 32; ++b) {
        run += scnt[b];
        if (run > (uint32_t)ns) {
          bfs = b - 1;
          break;
        }
      }
    }
    if (lane == 0) *sbf = bfs;
  }
  __syncthreads();
  const int bfs = *sbf;
  if (bfs < 0) return INFINITY;
  // E >= 2^-(bfs + 1)/32 relative to smax  <=>  l >= smax - (bfs + 1) T ln2 / 32
  return smax - (float)(bfs + 1) * (p.T * kLn2 * (1.f / 32.f));
}

template <bool FAST>
__global__ void __launch_bounds__(kSwNT) sampler_floor_kernel(const SP p) {
  __shared__ uint32_t scnt[kHist];
  __shared__ float sred[kSwW];
  __shared__ int sbf;
  // the sweep may start now: it waits for this kernel before reading the floors
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int row = blockIdx.x;
  float smax;
  const float Lf = row_floor<FAST>(p, p.logits + (size_t)row * p.V, l2_first_policy(), scnt,
                                   sred, &sbf, &smax);
  if (threadIdx.x == 0) {
    p.lfloor[2 * row] = Lf;
    p.lfloor[2 * row + 1] = smax;
  }
}

// One warp range (item = row * 32 + range) whose logits are in buf: its
// maximum, Z and list.  Warp k takes a contiguous run of 128-id pieces (lane
// l reads ids 32 j + l of a piece, so ballot j is 32 consecutive ids in
// order) and appends the flagged ids of its run, ascending, to its own
// segment of the range's list (kSegCap entries; more marks the range as
// overflowing).  Every thread calls it; it ends with a barrier, after which
// buf and the shared arrays may be reused.
template <bool FAST>
SPEC_DEV void sweep_range(const SP& p, int item, float* buf, float* wmax, float* wzh, float* wzl,
                          int* wcnt, uint16_t* stage) {
  const int row = item / kRangesPerRow, w = item % kRangesPerRow;
  const int V = p.V, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rw = stream_range_width(V);
  const int r0 = min(w * rw, V), r1 = min((w + 1) * rw, V);
  const int n = r1 - r0, npc = (n + 127) / 128;  // ids, 128-id pieces
  for (int k = n + t; k < 128 * npc; k += kSwNT) buf[k] = -INFINITY;  // the pad
  const float Lf = p.lfloor[2 * row], sref = p.lfloor[2 * row + 1];
  const float c_hi = p.c_hi, c_lo = p.c_lo, T150 = 150.f * p.T;
  __syncthreads();
  // one pass: the maximum, Z relative to the samples' maximum sref (rescaled
  // to the range's maximum below), and the flagged ids
  const unsigned lt = (1u << lane) - 1u;
  const int ppw = (npc + kSwW - 1) / kSwW;
  const int q0 = min(warp * ppw, npc), q1 = min(q0 + ppw, npc);
  uint16_t* wst = stage + warp * kSegCap;  // this warp's staged offsets (within the range)
  float mx = -INFINITY, zs = 0.f, zc = 0.f;
  int run = 0;  // warp-uniform: ids appended to this warp's segment
  {
    const float nm = -sref, lfl = sref - T150, nmc = -sref * c_hi;
    for (int q = q0; q < q1; ++q) {
      float l[4], e[4];
      uint32_t bal[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        l[j] = buf[128 * q + 32 * j + lane];
        mx = fmax_nan(mx, l[j]);
        e[j] = FAST ? fexp(l[j], c_hi, nmc) : texp(l[j], nm, lfl, c_hi, c_lo);
        bal[j] = __ballot_sync(kFull, l[j] >= Lf);
      }
      const float y = ((e[0] + e[1]) + (e[2] + e[3])) - zc;  // Kahan
      const float tt = zs + y;
      zc = (tt - zs) - y;
      zs = tt;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pos = run + __popc(bal[j] & lt);
        if (((bal[j] >> lane) & 1u) && pos < kSegCap) wst[pos] = (uint16_t)(128 * q + 32 * j + lane);
        run += __popc(bal[j]);
      }
    }
  }
  __syncwarp();  // the warp's staged offsets are written
  {  // its segment, coalesced: ids and their logits
    int32_t* oid = p.lid_g + ((size_t)item * kSwW + warp) * kSegCap;
    float* oval = p.lval_g + ((size_t)item * kSwW + warp) * kSegCap;
    for (int e = lane; e < min(run, kSegCap); e += 32) {
      const int off = wst[e];
      oid[e] = r0 + off;
      oval[e] = buf[off];
    }
  }
  float zh = zs, zl = -zc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmax_nan(mx, __shfl_xor_sync(kFull, mx, o));
    zh += __shfl_xor_sync(kFull, zh, o);
    zl += __shfl_xor_sync(kFull, zl, o);
  }
  if (lane == 0) {
    wmax[warp] = mx;
    wzh[warp] = zh;
    wzl[warp] = zl;
    wcnt[warp] = run;
    p.segcnt[(size_t)item * kSwW + warp] = run;
  }
  __syncthreads();
  float M = wmax[0], Zh = wzh[0], Zl = wzl[0];
  int total = 0;
  bool over = false;
  for (int i = 0; i < kSwW; ++i) {
    if (i > 0) {
      M = fmax_nan(M, wmax[i]);
      Zh += wzh[i];
      Zl += wzl[i];
    }
    total += wcnt[i];
    over |= wcnt[i] > kSegCap;
  }
  RangeStat res{M, 0.f, 0.f, over ? kSWCap + 1 : total};
  if (fabsf(M) < INFINITY) {  // uniform; else Z is not needed
    if (fabsf(Zh) < INFINITY) {
      // Z relative to M: times E(sref) relative to M, the product's error kept in the pair
      const float sc = FAST ? fexp(sref, c_hi, -M * c_hi) : texp(sref, -M, M - T150, c_hi, c_lo);
      const float h = Zh * sc;
      res.zh = h;
      res.zl = __fmaf_rn(Zh, sc, -h) + Zl * sc;
    } else {
      // E relative to sref overflowed (a range far above the samples): Z again
      // relative to M, from the logits still in shared memory
      const float nm = -M, lfl = M - T150, nmc = -M * c_hi;
      float s2 = 0.f, c2 = 0.f;
      for (int k = t; k < 128 * npc; k += kSwNT) {
        const float e = FAST ? fexp(buf[k], c_hi, nmc) : texp(buf[k], nm, lfl, c_hi, c_lo);
        const float y = e - c2, tt = s2 + y;
        c2 = (tt - s2) - y;
        s2 = tt;
      }
      float h = s2, lo = -c2;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        h += __shfl_xor_sync(kFull, h, o);
        lo += __shfl_xor_sync(kFull, lo, o);
      }
      __syncthreads();  // every thread has read wzh / wzl above
      if (lane == 0) {
        wzh[warp] = h;
        wzl[warp] = lo;
      }
      __syncthreads();
      for (int i = 0; i < kSwW; ++i) {
        res.zh += wzh[i];
        res.zl += wzl[i];
      }
    }
  } else {
    res.cnt = 0;
  }
  if (t == 0) p.stats[item] = res;
  __syncthreads();
}

// Persistent: each CTA loops over items blockIdx.x, + gridDim.x, ...; the
// next item's logits are copied into the second buffer (16-byte cp.async,
// L2 -> shared) while the current one is processed.  Rows that are not
// 16-byte aligned (V % 4 != 0) are loaded with plain loads instead.
template <bool FAST>
__global__ void __launch_bounds__(kSwNT, kSwCTAs) sampler_sweep_kernel(const SP p) {
  extern __shared__ __align__(16) uint8_t dyn[];  // two buffers of `cap` floats
  __shared__ float wmax[kSwW], wzh[kSwW], wzl[kSwW];
  __shared__ int wcnt[kSwW];
  __shared__ uint16_t stage[kSwW * kSegCap];  // flagged offsets staged per warp
  const int V = p.V, t = threadIdx.x;
  const int rw = stream_range_width(V);
  const int cap = (rw + 127) / 128 * 128;
  const int items = p.B * p.R * kRangesPerRow;
  const uint64_t pol = l2_first_policy();
  float* bufs = reinterpret_cast<float*>(dyn);
  auto issue = [&](int item, float* buf) {
    const int row = item / kRangesPerRow, w = item % kRangesPerRow;
    const int r0 = min(w * rw, V), n = min((w + 1) * rw, V) - r0;
    const float* src = p.logits + (size_t)row * V + r0;
    if (p.bulk != 0) {  // V % 4 == 0: r0 and n are multiples of 4
      const uint32_t sbuf = smem_u32(buf);
      for (int q = t; q < n / 4; q += kSwNT)
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                         sbuf + 16 * q),
                     "l"(src + 4 * q), "l"(pol)
                     : "memory");
    } else {
      for (int k = t; k < n; k += kSwNT) buf[k] = ldg_keep(src + k, pol);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  int item = blockIdx.x;
  if (item < items) issue(item, bufs);
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the floors are written
  for (int k = 0; item < items; ++k, item += gridDim.x) {
    const int nxt = item + gridDim.x;
    if (nxt < items) {
      issue(nxt, bufs + ((k + 1) & 1) * cap);
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // this item's copies have landed
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    sweep_range<FAST>(p, item, bufs + (k & 1) * cap, wmax, wzh, wzl, wcnt, stage);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- host side
struct SampPlan {
  int CS, slice, NT;
  size_t smem;  // dynamic shared memory bytes
};

size_t dyn_smem(size_t slice_bytes, bool qsm) {
  const size_t sb = (slice_bytes + 15) / 16 * 16;
  return sb + 2 * (size_t)kHistPad * 4 + 2 * (size_t)kCandMax * 12 + (size_t)kListPerCTA * 2 +
         (qsm ? sb : 0);
}

int num_sms_cached() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = 152;
  }
  return n;
}

int cluster_size(int V) { return std::min(kMaxCS, std::max(1, (V + 16383) / 16384)); }

int slice_of(int V, int CS) { return ((V + CS - 1) / CS + 3) / 4 * 4; }

SampPlan plan_sampler(int B, int R, int V, bool qsm) {
  SampPlan pl;
  pl.CS = cluster_size(V);
  pl.slice = slice_of(V, pl.CS);
  // few rows: one 512-thread CTA per SM; many rows: two 256-thread CTAs per SM
  const long long ctas = (long long)B * R * pl.CS;
  pl.NT = ctas <= num_sms_cached() ? 512 : 256;
  pl.smem = dyn_smem((size_t)pl.slice * 4, qsm);
  return pl;
}

// Workspace: header, row outcomes, sequence counters; with `pre`, the
// streaming pre-pass results after them (see SP).
struct SampWs {
  size_t out, cnt, stats, lfloor, lid, lval, segcnt, end;
};

// Sequences per call.  The per-sequence counters sit at one place for every
// shape, right after the header: a completed call leaves them at zero, so a
// workspace serves later calls of any batch size or block length.
constexpr int kMaxSeqs = 65536;

SampWs samp_ws(int B, int R, bool pre) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)B * R;
  SampWs w;
  size_t off = sizeof(WsHeader);
  w.cnt = off;
  off += up((size_t)kMaxSeqs * sizeof(int32_t));
  w.out = off;
  off += up(rows * sizeof(Outcome));
  w.stats = w.lfloor = w.lid = w.lval = w.segcnt = 0;
  if (pre) {
    w.stats = off;
    off += up(rows * kRangesPerRow * sizeof(RangeStat));
    w.lfloor = off;
    off += up(rows * 2 * sizeof(float));
    const size_t seg = rows * kRangesPerRow * kSwW;
    w.lid = off;
    off += up(seg * kSegCap * sizeof(int32_t));
    w.lval = off;
    off += up(seg * kSegCap * sizeof(float));
    w.segcnt = off;
    off += up(seg * sizeof(int32_t));
  }
  w.end = off;
  return w;
}

// many rows: the streaming kernels (with truncated sampling) rather than clusters
bool many_rows(int B, int R, int V) {
  return (long long)B * R * cluster_size(V) > 2LL * num_sms_cached();
}

template <int NT, bool FAST, bool TR>
spec_status launch_nt(const SP& prm, const SampPlan& pl, int rows, cudaStream_t st) {
  // once per device, at the largest size, so graph captures need no setup
  static PerDeviceOnce<int> smem_once;
  const spec_status ra = ensure_smem_limit(smem_once, (const void*)sampler_kernel<NT, FAST, TR>,
                                           (int)dyn_smem(kMaxSliceBytes, true));
  if (ra != SPEC_OK) return ra;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.CS * rows), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, sampler_kernel<NT, FAST, TR>, prm) != cudaSuccess) return SPEC_ECUDA;
  return launch_status();
}

size_t stream_smem(int V) {
  (void)V;
  return 2 * (size_t)kHistPad * 4 + (size_t)kSNT * 12 + (size_t)kSCap * 8;
}

// the row kernel, after the pre-pass when PRE (a programmatic dependent: its
// CTAs start as the pre-pass's last ones finish and wait for its results)
template <bool FAST, bool PRE>
spec_status launch_stream(const SP& prm, int rows, cudaStream_t st) {
  static PerDeviceOnce<int> smem_once;  // once per device, at the largest size
  const spec_status ra = ensure_smem_limit(smem_once, (const void*)sampler_stream_kernel<FAST, PRE>,
                                           (int)stream_smem(kSListMaxV));
  if (ra != SPEC_OK) return ra;
  if (PRE) {
    constexpr int kSwSmemMax = 2 * kSwMaxPieces * 128 * (int)sizeof(float);
    const int sw_smem = 2 * ((stream_range_width(prm.V) + 127) / 128 * 128) * (int)sizeof(float);
    if (sw_smem > kSwSmemMax) return SPEC_EUNSUPPORTED;
    static PerDeviceOnce<int> sw_once;  // once per device, at the largest size
    const spec_status rb =
        ensure_smem_limit(sw_once, (const void*)sampler_sweep_kernel<FAST>, kSwSmemMax);
    if (rb != SPEC_OK) return rb;
    sampler_floor_kernel<FAST><<<(unsigned)rows, kSwNT, 0, st>>>(prm);
    spec_status rs = launch_status();
    if (rs != SPEC_OK) return rs;
    cudaLaunchConfig_t c1 = {};
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sampler_sweep_kernel<FAST>, kSwNT,
                                                      (size_t)sw_smem) != cudaSuccess ||
        per_sm < 1)
      return SPEC_ECUDA;
    const long long items = (long long)rows * kRangesPerRow;
    c1.gridDim = dim3((unsigned)std::min<long long>(items, (long long)per_sm * num_sms_cached()),
                      1, 1);
    c1.blockDim = dim3(kSwNT, 1, 1);
    c1.dynamicSmemBytes = (size_t)sw_smem;
    c1.stream = st;
    cudaLaunchAttribute a1[1];
    a1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a1[0].val.programmaticStreamSerializationAllowed = 1;
    c1.attrs = a1;
    c1.numAttrs = 1;
    if (cudaLaunchKernelEx(&c1, sampler_sweep_kernel<FAST>, prm) != cudaSuccess) return SPEC_ECUDA;
    rs = launch_status();
    if (rs != SPEC_OK) return rs;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows, 1, 1);
  cfg.blockDim = dim3(kSNT, 1, 1);
  cfg.dynamicSmemBytes = stream_smem(prm.V);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // a cluster of one (its radix fallback
  attr[0].val.clusterDim.x = 1;                        // uses the cluster exchange helpers)
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PRE ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, sampler_stream_kernel<FAST, PRE>, prm) != cudaSuccess)
    return SPEC_ECUDA;
  return launch_status();
}

spec_status launch_sampler(SP prm, int B, int R, int V, size_t ws_bytes, cudaStream_t st) {
  // full-vocabulary residuals (no truncation) stage q's slice in shared memory
  const bool trunc = (prm.top_k > 0 && prm.top_k < V) || (prm.top_p > 0.f && prm.top_p < 1.f);
  // many truncated rows: one streaming CTA per row (every SM busy, no
  // cluster exchanges); trees only when their kept set fits the lists
  {
    if (many_rows(B, R, V) && trunc && !prm.greedy &&
        (!prm.tree || (prm.top_k > 0 && prm.top_k <= kSCap / (kSNT / 32)))) {
      prm.slice = V;
      // two passes when the workspace holds the pre-pass results
      const SampWs w = samp_ws(B, R, true);
      if (ws_bytes >= w.end) {
        uint8_t* base = reinterpret_cast<uint8_t*>(prm.err);
        prm.stats = reinterpret_cast<RangeStat*>(base + w.stats);
        prm.lfloor = reinterpret_cast<float*>(base + w.lfloor);
        prm.lid_g = reinterpret_cast<int32_t*>(base + w.lid);
        prm.lval_g = reinterpret_cast<float*>(base + w.lval);
        prm.segcnt = reinterpret_cast<int32_t*>(base + w.segcnt);
        return prm.p_out ? launch_stream<false, true>(prm, B * R, st)
                         : launch_stream<true, true>(prm, B * R, st);
      }
      return prm.p_out ? launch_stream<false, false>(prm, B * R, st)
                       : launch_stream<true, false>(prm, B * R, st);
    }
  }
  prm.qsm = (!prm.greedy && prm.qbulk && !trunc) ? 1 : 0;
  const SampPlan pl = plan_sampler(B, R, V, prm.qsm != 0);
  if ((size_t)pl.slice * 4 > kMaxSliceBytes) return SPEC_EUNSUPPORTED;
  prm.slice = pl.slice;
  const bool tr = (trunc && !prm.greedy) || prm.tree || prm.greedy;  // else: the compact variant
  if (prm.p_out) {
    if (tr)
      return pl.NT == 512 ? launch_nt<512, false, true>(prm, pl, B * R, st)
                          : launch_nt<256, false, true>(prm, pl, B * R, st);
    return pl.NT == 512 ? launch_nt<512, false, false>(prm, pl, B * R, st)
                        : launch_nt<256, false, false>(prm, pl, B * R, st);
  }
  if (tr)
    return pl.NT == 512 ? launch_nt<512, true, true>(prm, pl, B * R, st)
                        : launch_nt<256, true, true>(prm, pl, B * R, st);
  return pl.NT == 512 ? launch_nt<512, true, false>(prm, pl, B * R, st)
                      : launch_nt<256, true, false>(prm, pl, B * R, st);
}

spec_status check_cfg(const spec_sampler* cfg) {
  if (!cfg) return SPEC_EINVAL;
  if (!cfg->greedy && !(cfg->temperature > 0.f)) return SPEC_EINVAL;
  if (cfg->top_k < 0 || !(cfg->top_p > 0.f) || cfg->top_p > 1.f) return SPEC_EINVAL;
  return SPEC_OK;
}

SP base_params(const float* logits, const float* q, const float* u, int B, int R, int V,
               const spec_sampler* cfg, void* ws) {
  SP prm{};
  prm.logits = logits;
  prm.q = q;
  prm.u = u;
  prm.B = B;
  prm.R = R;
  prm.V = V;
  prm.T = cfg->temperature > 0.f ? cfg->temperature : 1.f;
  const double c = 1.0 / ((double)prm.T * 0.6931471805599453);
  prm.c_hi = (float)c;
  prm.c_lo = (float)(c - (double)prm.c_hi);
  prm.top_k = cfg->top_k;
  prm.top_p = cfg->top_p;
  prm.greedy = cfg->greedy ? 1 : 0;
  prm.eos = cfg->eos_id;
  const SampWs sw = samp_ws(B, R, false);
  uint8_t* w = static_cast<uint8_t*>(ws);
  prm.err = reinterpret_cast<int32_t*>(w);
  prm.outcomes = reinterpret_cast<Outcome*>(w + sw.out);
  prm.seq_count = reinterpret_cast<int32_t*>(w + sw.cnt);
  prm.bulk = (V % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) ? 1 : 0;
  prm.qbulk = (q && V % 4 == 0 && (reinterpret_cast<uintptr_t>(q) & 15) == 0) ? 1 : 0;
  return prm;
}

bool slice_fits(int V) { return (size_t)slice_of(V, cluster_size(V)) * 4 <= kMaxSliceBytes; }

}  // namespace

extern "C" size_t spec_accept_sample_workspace_size(int B, int R, int V) {
  if (B < 0 || R < 1 || V < 1) return 0;
  return samp_ws(B, R, false).end;
}

extern "C" size_t spec_accept_sample_workspace_size_two_pass(int B, int R, int V) {
  if (B < 0 || R < 1 || V < 1) return 0;
  return samp_ws(B, R, many_rows(B, R, V)).end;
}

extern "C" spec_status spec_accept_sample(const float* target_logits, const float* draft_probs,
                                          const int32_t* draft_tokens, const float* uniforms,
                                          int B, int R, int V, const spec_sampler* cfg,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* accepted_len, int32_t* emitted, float* p_out,
                                          int32_t* status_per_seq, void* stream) {
  const spec_status cs = check_cfg(cfg);
  if (cs != SPEC_OK) return cs;
  if (B < 0 || R < 1 || V < 1) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !accepted_len || !emitted || !workspace) return SPEC_EINVAL;
  if (R > 1 && !draft_tokens) return SPEC_EINVAL;
  if (!cfg->greedy && (!uniforms || (R > 1 && !draft_probs))) return SPEC_EINVAL;
  if (R > kMaxN || B > kMaxSeqs || (long long)B * R * kMaxCS > INT_MAX) return SPEC_EUNSUPPORTED;
  if (!slice_fits(V)) return SPEC_EUNSUPPORTED;
  if (workspace_bytes < samp_ws(B, R, false).end) return SPEC_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return SPEC_EINVAL;
  SP prm = base_params(target_logits, draft_probs, uniforms, B, R, V, cfg, workspace);
  prm.tokens = draft_tokens;
  prm.tree = 0;
  prm.acc_len = accepted_len;
  prm.emitted = emitted;
  prm.p_out = cfg->greedy ? nullptr : p_out;
  prm.status = status_per_seq;
  return launch_sampler(prm, B, R, V, workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" spec_status spec_accept_sample_tree(const float* target_logits,
                                               const float* draft_probs,
                                               const int32_t* node_tokens, const int32_t* parent,
                                               const float* uniforms, int B, int N, int V,
                                               const spec_sampler* cfg, void* workspace,
                                               size_t workspace_bytes, int32_t* accepted_len,
                                               int32_t* path_nodes, int32_t* emitted, float* p_out,
                                               int32_t* status_per_seq, void* stream) {
  const spec_status cs = check_cfg(cfg);
  if (cs != SPEC_OK) return cs;
  if (B < 0 || N < 2 || V < 1) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !node_tokens || !parent || !accepted_len || !path_nodes || !emitted ||
      !workspace)
    return SPEC_EINVAL;
  if (!cfg->greedy && (!uniforms || !draft_probs)) return SPEC_EINVAL;
  if (N > kMaxN || B > kMaxSeqs || (long long)B * N * kMaxCS > INT_MAX) return SPEC_EUNSUPPORTED;
  if (!slice_fits(V)) return SPEC_EUNSUPPORTED;
  if (workspace_bytes < samp_ws(B, N, false).end) return SPEC_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return SPEC_EINVAL;
  SP prm = base_params(target_logits, draft_probs, uniforms, B, N, V, cfg, workspace);
  prm.tokens = node_tokens;
  prm.parent = parent;
  prm.tree = 1;
  prm.acc_len = accepted_len;
  prm.path = path_nodes;
  prm.emitted = emitted;
  prm.p_out = cfg->greedy ? nullptr : p_out;
  prm.status = status_per_seq;
  return launch_sampler(prm, B, N, V, workspace_bytes, static_cast<cudaStream_t>(stream));
}
