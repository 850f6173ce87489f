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
// one slice of the vocabulary once and every later pass -- max, normaliser,
// the top-k / top-p radix selection, the p output -- runs from shared
// memory, with cluster-wide reductions over DSMEM.  Rows are independent,
// so all B*R rows run at once.  The cluster that finishes a sequence's last
// row (an atomic counter per sequence) runs the left-to-right walk and then
// the correction / bonus draw: a cluster-wide prefix sum over the drawn row
// in ascending id order.  The draft-tree walk keeps the running residual p'
// dense in the same distributed shared memory.
//
// Numerics: exp((l - m)/T) is evaluated with the difference and quotient
// carried in two floats, so p matches a float64 evaluation to ~3e-7
// relative; normalisers use per-thread compensated sums and a float64 tree;
// top-p masses are accumulated in 2^-40 fixed point so the selection is
// deterministic.
#include <algorithm>
#include <climits>

#include "common.cuh"

namespace {

constexpr int kST = 512;
constexpr int kSW = kST / 32;
constexpr int kMaxCS = 8;
constexpr int kMaxN = 64;
constexpr unsigned kFull = 0xffffffffu;
constexpr size_t kMaxSliceBytes = 200 * 1024;

struct RowStat {
  float m;
  float Z;
  uint32_t tau;
  int32_t tie_cut;
  int32_t argmax;
  int32_t flags;
  int32_t pad[2];
};

struct SP {
  const float* logits;
  const float* q;
  const int32_t* tokens;
  const int32_t* parent;
  const float* u;
  int B, R, V, slice;
  float T, invT;
  int top_k;
  float top_p;
  int greedy, eos, tree, bulk;
  RowStat* stats;
  int32_t* seq_count;
  int32_t* err;
  int32_t* acc_len;
  int32_t* emitted;
  int32_t* path;
  float* p_out;
  int32_t* status;
};

struct alignas(16) Slot {
  unsigned long long a, b;
};

struct Shared {
  double red_d[kSW];
  float red_f[kSW];
  int red_i[kSW];
  uint32_t red_u[kSW];
  unsigned long long red_ull[kSW];
  Slot slots[4];
  unsigned long long hmass[2][256];
  uint32_t hcnt[2][256];
  unsigned long long tot_mass[256];
  uint32_t tot_cnt[256];
  int bi[8];
  float bf[8];
  uint32_t bu[8];
  unsigned long long bull[2];
  int par[kMaxN];
  int tok[kMaxN];
  uint64_t bar;
};

// order-preserving key: larger float -> larger key; -0 and +0 share a key
SPEC_DEV uint32_t okey(float x) {
  uint32_t u = __float_as_uint(x);
  if (x == 0.f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// exp((l - m) / T): the difference l - m (two-sum) and the quotient (FMA
// remainder) are carried in two floats; exp(hi + lo) = exp(hi) * (1 + lo).
SPEC_DEV float texp(float l, float m, float T, float invT) {
  if (l == -INFINITY) return 0.f;
  const float s = l - m;
  const float bv = s - l;
  const float av = s - bv;
  const float e = (l - av) + (-m - bv);
  const float qh = s * invT;
  const float r = fmaf(-qh, T, s);
  const float ql = (r + e) * invT;
  return expf(qh) * (1.0f + ql);
}

SPEC_DEV bool is_kept(uint32_t key, int id, uint32_t tau, int tie) {
  return key > tau || (key == tau && id <= tie);
}

// ---------------------------------------------------------------- block reductions
SPEC_DEV double block_sum_d(double v, Shared& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) sh.red_d[w] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int i = 0; i < kSW; ++i) t += sh.red_d[i];
  __syncthreads();
  return t;
}

// (max value, lowest id among maxima); non-finite flag OR-ed
SPEC_DEV void block_max_arg(float& v, int& id, Shared& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFull, v, o);
    const int oi = __shfl_xor_sync(kFull, id, o);
    if (ov > v || (ov == v && oi < id)) {
      v = ov;
      id = oi;
    }
  }
  if (lane == 0) {
    sh.red_f[w] = v;
    sh.red_i[w] = id;
  }
  __syncthreads();
  v = sh.red_f[0];
  id = sh.red_i[0];
  for (int i = 1; i < kSW; ++i) {
    const float ov = sh.red_f[i];
    const int oi = sh.red_i[i];
    if (ov > v || (ov == v && oi < id)) {
      v = ov;
      id = oi;
    }
  }
  __syncthreads();
}

SPEC_DEV int block_or(int v, Shared& sh) {
  v = __reduce_or_sync(kFull, (unsigned)v);
  if ((threadIdx.x & 31) == 0) sh.red_i[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = 0;
  for (int i = 0; i < kSW; ++i) t |= sh.red_i[i];
  __syncthreads();
  return t;
}

SPEC_DEV int block_min_i(int v, Shared& sh) {
  v = __reduce_min_sync(kFull, v);
  if ((threadIdx.x & 31) == 0) sh.red_i[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = INT_MAX;
  for (int i = 0; i < kSW; ++i) t = min(t, sh.red_i[i]);
  __syncthreads();
  return t;
}

// exclusive scan of one float per thread (fixed order); returns the
// exclusive prefix and writes the block total to *total.
SPEC_DEV float block_excl_scan_f(float v, float* total, Shared& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh.red_f[w] = incl;
  __syncthreads();
  float base = 0.f;
  for (int i = 0; i < w; ++i) base += sh.red_f[i];
  const float excl = base + (incl - v);
  __syncthreads();
  // total computed exactly the way the last element's running value is
  if (threadIdx.x == kST - 1) sh.red_f[0] = excl + v;
  __syncthreads();
  *total = sh.red_f[0];
  __syncthreads();
  return excl;
}

SPEC_DEV int block_excl_scan_i(int v, int* total, Shared& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh.red_i[w] = incl;
  __syncthreads();
  int base = 0;
  for (int i = 0; i < w; ++i) base += sh.red_i[i];
  __syncthreads();
  if (threadIdx.x == kST - 1) sh.red_i[0] = base + incl;
  __syncthreads();
  *total = sh.red_i[0];
  __syncthreads();
  return base + incl - v;
}

// ---------------------------------------------------------------- cluster exchange
// Every CTA posts one Slot; afterwards thread-local copies of all CS slots
// (rank order) are available to warp 0 lanes < CS.  Slots rotate over four
// buffers so that a slot is never rewritten before every reader has passed
// the next cluster barrier.
SPEC_DEV Slot cluster_post_get(Slot mine, int& ph, Shared& sh, uint32_t rank_to_read) {
  Slot* s = &sh.slots[ph & 3];
  if (threadIdx.x == 0) *s = mine;
  cluster_sync();
  Slot r;
  r.a = dsmem_ld_u64(&s->a, rank_to_read);
  r.b = dsmem_ld_u64(&s->b, rank_to_read);
  ++ph;
  return r;
}

SPEC_DEV double cluster_sum_d(double v, int CS, int& ph, Shared& sh) {
  Slot mine{(unsigned long long)__double_as_longlong(v), 0ull};
  double t = 0.0;
  // every thread reads every rank (CS <= 8 DSMEM loads), in rank order
  Slot* s = &sh.slots[ph & 3];
  if (threadIdx.x == 0) *s = mine;
  cluster_sync();
  for (int r = 0; r < CS; ++r) t += __longlong_as_double((long long)dsmem_ld_u64(&s->a, r));
  ++ph;
  return t;
}

SPEC_DEV unsigned long long cluster_sum_u64(unsigned long long v, int CS, int& ph, Shared& sh) {
  Slot* s = &sh.slots[ph & 3];
  if (threadIdx.x == 0) s->a = v;
  cluster_sync();
  unsigned long long t = 0;
  for (int r = 0; r < CS; ++r) t += dsmem_ld_u64(&s->a, r);
  ++ph;
  return t;
}

// value of CTA `src` (posted by every CTA; only src's value is used)
SPEC_DEV Slot cluster_from(Slot mine, int src, int& ph, Shared& sh) {
  return cluster_post_get(mine, ph, sh, (uint32_t)src);
}

// ---------------------------------------------------------------- helpers on the slice
struct Slice {
  float* buf;  // shared memory, n floats
  int lo, n;
};

// Load logits row into the slice buffer (TMA bulk copy when aligned).
SPEC_DEV void load_row(const SP& p, const float* row, Slice& sl, Shared& sh, uint32_t& bar_phase) {
  __syncthreads();  // every reader of the previous contents is done
  if (sl.n <= 0) {
    __syncthreads();
    return;
  }
  if (p.bulk) {
    if (threadIdx.x == 0) {
      fence_proxy_async();  // order earlier generic writes before the async copy
      mbar_arrive_expect_tx(&sh.bar, (uint32_t)sl.n * 4u);
      bulk_load(sl.buf, row + sl.lo, (uint32_t)sl.n * 4u, &sh.bar);
    }
    mbar_wait(&sh.bar, bar_phase, p.err);
    bar_phase ^= 1u;
  } else {
    for (int i = threadIdx.x; i < sl.n; i += kST) sl.buf[i] = row[sl.lo + i];
  }
  __syncthreads();
}

// The id (global) of the nth (1-based) element, in ascending id order over
// the cluster, for which pred(local index) holds.  Same result in all CTAs.
template <class Pred>
SPEC_DEV int nth_in_cluster(const Slice& sl, int nth, Pred pred, int rank, int CS, int& ph,
                            Shared& sh) {
  const int seg = (sl.n + kST - 1) / kST;
  const int s0 = min(threadIdx.x * seg, sl.n), s1 = min(s0 + seg, sl.n);
  int c = 0;
  for (int k = s0; k < s1; ++k) c += pred(k) ? 1 : 0;
  int tot;
  const int excl = block_excl_scan_i(c, &tot, sh);
  // rank prefix
  Slot* s = &sh.slots[ph & 3];
  if (threadIdx.x == 0) s->a = (unsigned long long)tot;
  cluster_sync();
  int before = 0, owner = -1;
  for (int r = 0; r < CS; ++r) {
    const int tr = (int)dsmem_ld_u64(&s->a, r);
    if (owner < 0 && before + tr >= nth) owner = r;
    if (owner < 0) before += tr;
  }
  ++ph;
  int found = INT_MAX;
  if (owner == rank) {
    const int local = nth - before;
    if (excl < local && local <= excl + c) {
      int cnt = excl;
      for (int k = s0; k < s1; ++k)
        if (pred(k) && ++cnt == local) {
          found = sl.lo + k;
          break;
        }
    }
  }
  found = block_min_i(found, sh);
  Slot mine{(unsigned long long)(unsigned)found, 0ull};
  const Slot o = cluster_from(mine, owner < 0 ? 0 : owner, ph, sh);
  return owner < 0 ? INT_MAX : (int)(unsigned)o.a;
}

// Radix selection, most significant digit first, of the position in
// (key desc, id asc) order where the running weight reaches `target`.
// Weight = 1 per element (by_mass = false) or its 2^-40 fixed-point mass.
// Elements considered: those with keep(k).  Returns tau (exact key), the
// weight strictly above tau, and the count/weight at tau.
struct Sel {
  uint32_t tau;
  unsigned long long above;
  unsigned long long at_weight;
  unsigned long long total;
  uint32_t at_count;
};

template <class Keep, class Weight>
SPEC_DEV Sel radix_select(const Slice& sl, bool target_is_fraction, double frac,
                          unsigned long long target_abs, Keep keep, Weight weight, int CS, int& ph,
                          Shared& sh) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, pmask = 0;
  unsigned long long above = 0, target = target_abs, total = 0;
  Sel out{};
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int h = pass & 1;
    for (int i = threadIdx.x; i < 256; i += kST) {
      sh.hmass[h][i] = 0ull;
      sh.hcnt[h][i] = 0u;
    }
    __syncthreads();
    const int iters = (sl.n + kST - 1) / kST;
    for (int it = 0; it < iters; ++it) {
      const int k = threadIdx.x + it * kST;
      bool act = false;
      uint32_t key = 0;
      unsigned long long wgt = 0;
      if (k < sl.n) {
        key = okey(sl.buf[k]);
        act = ((key & pmask) == prefix) && keep(k, key);
        if (act) wgt = weight(k);
      }
      const uint32_t digit = (key >> shift) & 255u;
      const unsigned peers = __match_any_sync(kFull, act ? digit : 256u + lane);
      // fixed-point weight <= 2^41: split so 32-lane sums fit in 32 bits
      const unsigned hi = __reduce_add_sync(peers, (unsigned)(wgt >> 20));
      const unsigned lo = __reduce_add_sync(peers, (unsigned)(wgt & 0xFFFFFull));
      if (act && lane == __ffs(peers) - 1) {
        atomicAdd(&sh.hcnt[h][digit], (unsigned)__popc(peers));
        atomicAdd(&sh.hmass[h][digit], ((unsigned long long)hi << 20) + lo);
      }
    }
    __syncthreads();
    cluster_sync();
    for (int d = threadIdx.x; d < 256; d += kST) {
      unsigned long long m = 0;
      uint32_t c = 0;
      for (int r = 0; r < CS; ++r) {
        m += dsmem_ld_u64(&sh.hmass[h][d], r);
        c += dsmem_ld_u32(&sh.hcnt[h][d], r);
      }
      sh.tot_mass[d] = m;
      sh.tot_cnt[d] = c;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane L holds digits 255-8L .. 248-8L (descending)
      unsigned long long ls = 0;
      for (int j = 0; j < 8; ++j) ls += sh.tot_mass[255 - 8 * lane - j];
      if (pass == 0) {
        unsigned long long t = ls;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
        total = t;
        if (target_is_fraction) {
          const double thr = ceil(frac * (double)t);
          target = thr < 1.0 ? 1ull : (unsigned long long)thr;
          if (target > t) target = t;
        }
      }
      unsigned long long incl = ls;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned long long need = target - above;
      const unsigned hit = __ballot_sync(kFull, incl >= need);
      const int L = hit ? __ffs(hit) - 1 : 31;
      if (lane == L) {
        unsigned long long cum = incl - ls;
        int dsel = 248 - 8 * L;
        for (int j = 0; j < 8; ++j) {
          const int d = 255 - 8 * L - j;
          if (cum + sh.tot_mass[d] >= need) {
            dsel = d;
            break;
          }
          cum += sh.tot_mass[d];
        }
        sh.bu[0] = (uint32_t)dsel;
        sh.bull[0] = cum;  // weight in digits above dsel (within the prefix)
      }
      if (lane == 0) sh.bull[1] = total;
    }
    __syncthreads();
    const uint32_t dsel = sh.bu[0];
    above += sh.bull[0];
    total = sh.bull[1];
    if (pass == 0 && target_is_fraction) {
      const double thr = ceil(frac * (double)total);
      target = thr < 1.0 ? 1ull : (unsigned long long)thr;
      if (target > total) target = total;
    }
    prefix |= dsel << shift;
    pmask |= 255u << shift;
    if (pass == 3) {
      out.at_count = sh.tot_cnt[dsel];
      out.at_weight = sh.tot_mass[dsel];
    }
    __syncthreads();
  }
  out.tau = prefix;
  out.above = above;
  out.total = total;
  // stash the target for the caller (needed for the tie count)
  sh.bull[0] = target;
  __syncthreads();
  return out;
}

// Draw: the first id whose running sum (ascending id order over the
// cluster) of the slice values exceeds u * total.  Returns -2 if the total
// is zero.  Same result in all CTAs.
SPEC_DEV int draw_from_slice(const Slice& sl, float u, int rank, int CS, int& ph, Shared& sh) {
  const int seg = (sl.n + kST - 1) / kST;
  const int s0 = min(threadIdx.x * seg, sl.n), s1 = min(s0 + seg, sl.n);
  float run = 0.f;
  for (int k = s0; k < s1; ++k) run += sl.buf[k];
  float tot;
  const float excl = block_excl_scan_f(run, &tot, sh);
  Slot* s = &sh.slots[ph & 3];
  if (threadIdx.x == 0) s->a = (unsigned long long)__float_as_uint(tot);
  cluster_sync();
  float prefix = 0.f, my_prefix = 0.f;
  float tots[kMaxCS];
  for (int r = 0; r < CS; ++r) {
    tots[r] = __uint_as_float((uint32_t)dsmem_ld_u64(&s->a, r));
  }
  ++ph;
  float pre[kMaxCS + 1];
  pre[0] = 0.f;
  for (int r = 0; r < CS; ++r) pre[r + 1] = pre[r] + tots[r];
  const float W = pre[CS];
  if (!(W > 0.f)) return -2;
  const float target = u * W;
  int owner = -1;
  for (int r = 0; r < CS; ++r)
    if (owner < 0 && tots[r] > 0.f && pre[r] + tots[r] > target) owner = r;
  if (owner < 0)
    for (int r = CS - 1; r >= 0; --r)
      if (owner < 0 && tots[r] > 0.f) owner = r;
  prefix = pre[owner];
  (void)my_prefix;
  int found = INT_MAX;
  if (owner == rank) {
    if (prefix + (excl + run) > target || threadIdx.x == kST - 1) {
      float acc = 0.f;
      for (int k = s0; k < s1; ++k) {
        acc += sl.buf[k];
        if (prefix + (excl + acc) > target) {
          found = k;
          break;
        }
      }
    }
  }
  found = block_min_i(found, sh);
  if (owner == rank && found == INT_MAX) {
    // rounding left nothing above target: take the last nonzero entry
    int last = -1;
    for (int k = s0; k < s1; ++k)
      if (sl.buf[k] > 0.f) last = k;
    const int neg = block_min_i(-last, sh);  // -(largest index)
    found = (neg <= 0) ? -neg : INT_MAX;
  }
  Slot mine{(unsigned long long)(unsigned)(found == INT_MAX ? 0 : sl.lo + found), 0ull};
  const Slot o = cluster_from(mine, owner, ph, sh);
  return (int)(unsigned)o.a;
}

SPEC_DEV RowStat load_stat(const RowStat* s) {
  RowStat r;
  const int4* src = reinterpret_cast<const int4*>(s);
  const int4 a = __ldcg(src), b2 = __ldcg(src + 1);
  memcpy(&r, &a, 16);
  memcpy(reinterpret_cast<char*>(&r) + 16, &b2, 16);
  return r;
}

// p_row(x) from the row's statistics and one logit
SPEC_DEV float p_of(const SP& p, const RowStat& st, float l, int id) {
  if (!is_kept(okey(l), id, st.tau, st.tie_cut)) return 0.f;
  return texp(l, st.m, p.T, p.invT) / st.Z;
}

// Fill the slice with p of row `row` (logits already loaded in the slice).
SPEC_DEV void slice_to_p(const SP& p, const RowStat& st, Slice& sl) {
  for (int k = threadIdx.x; k < sl.n; k += kST) sl.buf[k] = p_of(p, st, sl.buf[k], sl.lo + k);
  __syncthreads();
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kST, 1) sampler_kernel(const SP p) {
  extern __shared__ __align__(16) float sbuf[];
  __shared__ Shared sh;
  const int rank = (int)cluster_ctarank();
  const int CS = (int)cluster_nctarank();
  const int row = blockIdx.y;
  const int b = row / p.R;
  const int i = row % p.R;
  Slice sl{sbuf, rank * p.slice, 0};
  sl.n = max(0, min(p.slice, p.V - sl.lo));
  int ph = 0;
  uint32_t bar_phase = 0;
  if (threadIdx.x == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- 1. the row into shared memory
  load_row(p, p.logits + (size_t)row * p.V, sl, sh, bar_phase);

  // ---- 2. max, lowest-id argmax, non-finite check
  float mv = -INFINITY;
  int mi = INT_MAX;
  int bad = 0;
  for (int k = threadIdx.x; k < sl.n; k += kST) {
    const float x = sl.buf[k];
    if (isnan(x) || x == INFINITY) bad = 1;
    if (x > mv || (x == mv && sl.lo + k < mi)) {
      mv = x;
      mi = sl.lo + k;
    }
  }
  bad = block_or(bad, sh);
  block_max_arg(mv, mi, sh);
  {
    Slot* s = &sh.slots[ph & 3];
    if (threadIdx.x == 0) {
      s->a = ((unsigned long long)__float_as_uint(mv) << 32) | (unsigned)mi;
      s->b = (unsigned long long)bad;
    }
    cluster_sync();
    for (int r = 0; r < CS; ++r) {
      const unsigned long long a = dsmem_ld_u64(&s->a, r);
      const float ov = __uint_as_float((uint32_t)(a >> 32));
      const int oi = (int)(uint32_t)a;
      bad |= (int)dsmem_ld_u64(&s->b, r);
      if (ov > mv || (ov == mv && oi < mi)) {
        mv = ov;
        mi = oi;
      }
    }
    ++ph;
  }
  if (mv == -INFINITY) bad = 1;  // every token banned: no distribution
  const float m = mv;
  RowStat st{};
  st.m = m;
  st.argmax = mi;
  st.flags = bad;
  st.tau = 0u;
  st.tie_cut = INT_MAX;
  st.Z = 1.f;

  if (!p.greedy && !bad) {
    // ---- 3. truncation (top-k by count, then top-p by mass)
    if (p.top_k > 0 && p.top_k < p.V) {
      const Sel s = radix_select(
          sl, false, 0.0, (unsigned long long)p.top_k, [](int, uint32_t) { return true; },
          [](int) { return 1ull; }, CS, ph, sh);
      const unsigned long long target = sh.bull[0];
      const int need = (int)(target - s.above);  // ties at tau to keep (>= 1)
      st.tau = s.tau;
      if ((uint32_t)need >= s.at_count) {
        st.tie_cut = INT_MAX;
      } else {
        const uint32_t tau = s.tau;
        st.tie_cut = nth_in_cluster(
            sl, need, [&](int k) { return okey(sl.buf[k]) == tau; }, rank, CS, ph, sh);
      }
    }
    if (p.top_p > 0.f && p.top_p < 1.f) {
      const uint32_t tk = st.tau;
      const int tc = st.tie_cut;
      const float T = p.T, invT = p.invT;
      auto keep_k = [&](int k, uint32_t key) { return is_kept(key, sl.lo + k, tk, tc); };
      auto mass = [&](int k) {
        const float e = texp(sl.buf[k], m, T, invT);
        return (unsigned long long)__float2ull_rn(e * 1099511627776.0f);  // 2^40
      };
      const Sel s = radix_select(sl, true, (double)p.top_p, 0ull, keep_k, mass, CS, ph, sh);
      const unsigned long long target = sh.bull[0];
      const unsigned long long e_tau = s.at_count ? s.at_weight / s.at_count : 0ull;
      unsigned long long need = 1;
      if (e_tau > 0 && target > s.above) need = (target - s.above + e_tau - 1) / e_tau;
      if (need < 1) need = 1;
      if (need > s.at_count) need = s.at_count;
      const uint32_t tau = s.tau;
      int tie;
      if (need == s.at_count) {
        tie = (tau == tk) ? tc : INT_MAX;
      } else {
        tie = nth_in_cluster(
            sl, (int)need,
            [&](int k) {
              const uint32_t key = okey(sl.buf[k]);
              return key == tau && is_kept(key, sl.lo + k, tk, tc);
            },
            rank, CS, ph, sh);
      }
      st.tau = tau;
      st.tie_cut = tie;
    }
    // ---- 4. normaliser over the kept set (compensated per thread, fp64 tree)
    float sum = 0.f, cmp = 0.f;
    for (int k = threadIdx.x; k < sl.n; k += kST) {
      const float x = sl.buf[k];
      if (!is_kept(okey(x), sl.lo + k, st.tau, st.tie_cut)) continue;
      const float y = texp(x, m, p.T, p.invT) - cmp;
      const float t = sum + y;
      cmp = (t - sum) - y;
      sum = t;
    }
    double z = block_sum_d((double)sum - (double)cmp, sh);
    z = cluster_sum_d(z, CS, ph, sh);
    st.Z = (float)z;
    if (p.p_out) {
      float* dst = p.p_out + (size_t)row * p.V + sl.lo;
      for (int k = threadIdx.x; k < sl.n; k += kST) dst[k] = p_of(p, st, sl.buf[k], sl.lo + k);
    }
  }

  // ---- 5. publish the row statistics; the last row of a sequence continues
  if (rank == 0 && threadIdx.x == 0) {
    p.stats[row] = st;
    __threadfence();
    const int old = atomicAdd(&p.seq_count[b], 1);
    sh.bi[0] = (old == p.R - 1) ? 1 : 0;
  }
  cluster_sync();
  const int last = (int)dsmem_ld_u32(&sh.bi[0], 0);
  cluster_sync();
  if (!last) return;
  __threadfence();

  const int R = p.R;
  int32_t* emitted = p.emitted + (size_t)b * R;
  int status = 0;
  int k_emit = 0;

  // ---- 6a. greedy walks (thread 0 of rank 0 writes the outputs)
  if (p.greedy) {
    if (rank == 0 && threadIdx.x == 0) {
      int nonfin = 0;
      for (int r = 0; r < R; ++r) nonfin |= load_stat(&p.stats[(size_t)b * R + r]).flags;
      int acc = 0;
      if (nonfin) {
        status |= SPEC_SEQ_NONFINITE;
        acc = -1;
      } else if (!p.tree) {
        for (int r = 0; r < R; ++r) {
          const int a = load_stat(&p.stats[(size_t)b * R + r]).argmax;
          if (r == R - 1) {
            emitted[k_emit++] = a;
            break;
          }
          const int x = p.tokens[(size_t)b * (R - 1) + r];
          if (x == a) {
            emitted[k_emit++] = x;
            ++acc;
            if (x == p.eos) break;
          } else {
            emitted[k_emit++] = a;
            break;
          }
        }
      } else {
        int v = 0;
        while (true) {
          const int a = load_stat(&p.stats[(size_t)b * R + v]).argmax;
          int nxt = -1;
          for (int c = v + 1; c < R; ++c)
            if (p.parent[(size_t)b * R + c] == v && p.tokens[(size_t)b * R + c] == a) {
              nxt = c;
              break;
            }
          emitted[k_emit++] = a;
          if (nxt >= 0) p.path[(size_t)b * R + acc++] = nxt;
          if (nxt < 0 || a == p.eos) break;
          v = nxt;
        }
        for (int c = acc; c < R; ++c) p.path[(size_t)b * R + c] = -1;
      }
      for (int c = (nonfin ? 0 : k_emit); c < R; ++c) emitted[c] = -1;
      if (nonfin && p.tree)
        for (int c = 0; c < R; ++c) p.path[(size_t)b * R + c] = -1;
      p.acc_len[b] = acc;
      if (p.status) p.status[b] = status;
      p.seq_count[b] = 0;
    }
    return;
  }

  // ---- 6b. sampling: read statistics of every row of this sequence
  int nonfin = 0;
  for (int r = 0; r < R; ++r) nonfin |= load_stat(&p.stats[(size_t)b * R + r]).flags;
  if (nonfin) {
    if (rank == 0 && threadIdx.x == 0) {
      for (int c = 0; c < R; ++c) emitted[c] = -1;
      if (p.tree)
        for (int c = 0; c < R; ++c) p.path[(size_t)b * R + c] = -1;
      p.acc_len[b] = -1;
      if (p.status) p.status[b] = SPEC_SEQ_NONFINITE;
      p.seq_count[b] = 0;
    }
    return;
  }

  const float u_final = p.u[(size_t)b * R + (R - 1)];
  if (!p.tree) {
    // chain walk: thread 0 of every CTA computes the same decisions
    int acc = 0, draw_row = -1, resid = 0, stop = 0;
    for (int r = 0; r < R - 1; ++r) {
      const int x = p.tokens[(size_t)b * (R - 1) + r];
      float px = 0.f, qx = 0.f;
      if (x >= 0 && x < p.V) {
        const RowStat srow = load_stat(&p.stats[(size_t)b * R + r]);
        px = p_of(p, srow, __ldcg(&p.logits[((size_t)b * R + r) * p.V + x]), x);
        qx = __ldcg(&p.q[((size_t)b * (R - 1) + r) * p.V + x]);
      }
      if (qx == 0.f) status |= SPEC_SEQ_QZERO;
      if (p.u[(size_t)b * R + r] * qx < px) {
        ++acc;
        if (x == p.eos) {
          stop = 1;
          break;
        }
      } else {
        draw_row = r;
        resid = 1;
        break;
      }
    }
    if (!stop && draw_row < 0) draw_row = R - 1;
    int tok = -1;
    if (!stop) {
      const RowStat sr = load_stat(&p.stats[(size_t)b * R + draw_row]);
      load_row(p, p.logits + ((size_t)b * R + draw_row) * p.V, sl, sh, bar_phase);
      const float* qrow = p.q + ((size_t)b * (R - 1) + (resid ? draw_row : 0)) * p.V + sl.lo;
      for (int k = threadIdx.x; k < sl.n; k += kST) {
        const float pv = p_of(p, sr, sl.buf[k], sl.lo + k);
        sl.buf[k] = resid ? fmaxf(pv - __ldcg(&qrow[k]), 0.f) : pv;
      }
      __syncthreads();
      tok = draw_from_slice(sl, u_final, rank, CS, ph, sh);
      if (tok == -2) {
        // residual with zero mass (rounding only): draw from p instead
        status |= SPEC_SEQ_RESID_ZERO;
        load_row(p, p.logits + ((size_t)b * R + draw_row) * p.V, sl, sh, bar_phase);
        slice_to_p(p, sr, sl);
        tok = draw_from_slice(sl, u_final, rank, CS, ph, sh);
      }
    }
    if (rank == 0 && threadIdx.x == 0) {
      for (int r = 0; r < acc; ++r) emitted[r] = p.tokens[(size_t)b * (R - 1) + r];
      int kk = acc;
      if (!stop) emitted[kk++] = tok;
      for (int c = kk; c < R; ++c) emitted[c] = -1;
      p.acc_len[b] = acc;
      if (p.status) p.status[b] = status;
      p.seq_count[b] = 0;
    }
    cluster_sync();  // keep every CTA's shared memory alive until all reads finish
    return;
  }

  // ---- 6c. tree walk with a dense running residual p' in the slices
  const int N = R;
  for (int c = threadIdx.x; c < N; c += kST) {
    sh.par[c] = p.parent[(size_t)b * N + c];
    sh.tok[c] = p.tokens[(size_t)b * N + c];
  }
  __syncthreads();
  int v = 0, acc = 0, done = 0;
  int32_t* path = p.path + (size_t)b * N;
  {
    const RowStat s0 = load_stat(&p.stats[(size_t)b * N]);
    load_row(p, p.logits + (size_t)b * N * p.V, sl, sh, bar_phase);
    slice_to_p(p, s0, sl);
  }
  while (!done) {
    int moved = 0;
    for (int c = v + 1; c < N && !moved; ++c) {
      if (sh.par[c] != v) continue;
      const int t = sh.tok[c];
      cluster_sync();  // p' complete everywhere
      float pt = 0.f;
      if (t >= 0 && t < p.V) {
        const int owner = t / p.slice;
        pt = dsmem_ld_f32(&sl.buf[t - owner * p.slice], (uint32_t)owner);
      }
      cluster_sync();  // nobody rewrites p' before every CTA has read it
      const float qx = (t >= 0 && t < p.V) ? __ldcg(&p.q[((size_t)b * N + v) * p.V + t]) : 0.f;
      if (qx == 0.f) status |= SPEC_SEQ_QZERO;
      if (p.u[(size_t)b * N + (c - 1)] * qx < pt) {
        if (rank == 0 && threadIdx.x == 0) {
          emitted[acc] = t;
          path[acc] = c;
        }
        ++acc;
        v = c;
        moved = 1;
        if (t == p.eos) {
          done = 1;
        } else {
          const RowStat sv = load_stat(&p.stats[(size_t)b * N + v]);
          load_row(p, p.logits + ((size_t)b * N + v) * p.V, sl, sh, bar_phase);
          slice_to_p(p, sv, sl);
        }
      } else {
        // p' <- norm(max(0, p' - q_v))
        const float* qrow = p.q + ((size_t)b * N + v) * p.V + sl.lo;
        float sum = 0.f, cmp = 0.f;
        for (int k = threadIdx.x; k < sl.n; k += kST) {
          const float y = fmaxf(sl.buf[k] - __ldcg(&qrow[k]), 0.f) - cmp;
          const float tt = sum + y;
          cmp = (tt - sum) - y;
          sum = tt;
        }
        double W = block_sum_d((double)sum - (double)cmp, sh);
        W = cluster_sum_d(W, CS, ph, sh);
        if (W > 0.0) {
          const float Wf = (float)W;
          for (int k = threadIdx.x; k < sl.n; k += kST)
            sl.buf[k] = fmaxf(sl.buf[k] - __ldcg(&qrow[k]), 0.f) / Wf;
        } else {
          status |= SPEC_SEQ_RESID_ZERO;
        }
        __syncthreads();
      }
    }
    if (!moved && !done) {
      const int tok = draw_from_slice(sl, u_final, rank, CS, ph, sh);
      if (rank == 0 && threadIdx.x == 0) emitted[acc] = tok;
      done = 1;
      if (rank == 0 && threadIdx.x == 0) {
        for (int c = acc + 1; c < N; ++c) emitted[c] = -1;
      }
    } else if (done && rank == 0 && threadIdx.x == 0) {
      for (int c = acc; c < N; ++c) emitted[c] = -1;
    }
  }
  if (rank == 0 && threadIdx.x == 0) {
    for (int c = acc; c < N; ++c) path[c] = -1;
    p.acc_len[b] = acc;
    if (p.status) p.status[b] = status;
    p.seq_count[b] = 0;
  }
  cluster_sync();
}

// ---------------------------------------------------------------- host side
struct SampPlan {
  int CS, slice;
  size_t smem;
};

SampPlan plan_sampler(int V) {
  SampPlan pl;
  pl.CS = std::min(kMaxCS, std::max(1, (V + 16383) / 16384));
  pl.slice = ((V + pl.CS - 1) / pl.CS + 3) / 4 * 4;
  pl.smem = (size_t)pl.slice * 4;
  return pl;
}

size_t samp_ws(int B, int R, size_t* off_stats, size_t* off_cnt) {
  size_t off = sizeof(WsHeader);
  *off_stats = off;
  off += ((size_t)B * R * sizeof(RowStat) + 255) / 256 * 256;
  *off_cnt = off;
  off += ((size_t)B * sizeof(int32_t) + 255) / 256 * 256;
  return off;
}

spec_status launch_sampler(SP prm, int B, int R, int V, cudaStream_t st) {
  const SampPlan pl = plan_sampler(V);
  prm.slice = pl.slice;
  if (pl.smem > kMaxSliceBytes) return SPEC_EUNSUPPORTED;
  static bool attr_set = false;  // once, at the largest size, so graph captures need no setup
  if (!attr_set) {
    if (cudaFuncSetAttribute(sampler_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kMaxSliceBytes) != cudaSuccess)
      return SPEC_ECUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.CS, B * R, 1);
  cfg.blockDim = dim3(kST, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, sampler_kernel, prm) != cudaSuccess) return SPEC_ECUDA;
  return launch_status();
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
  prm.invT = 1.0f / prm.T;
  prm.top_k = cfg->top_k;
  prm.top_p = cfg->top_p;
  prm.greedy = cfg->greedy ? 1 : 0;
  prm.eos = cfg->eos_id;
  size_t off_stats, off_cnt;
  samp_ws(B, R, &off_stats, &off_cnt);
  uint8_t* w = static_cast<uint8_t*>(ws);
  prm.err = reinterpret_cast<int32_t*>(w);
  prm.stats = reinterpret_cast<RowStat*>(w + off_stats);
  prm.seq_count = reinterpret_cast<int32_t*>(w + off_cnt);
  prm.bulk = (V % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) ? 1 : 0;
  return prm;
}

}  // namespace

extern "C" size_t spec_accept_sample_workspace_size(int B, int R, int V) {
  (void)V;
  if (B < 0 || R < 1) return 0;
  size_t a, c;
  return samp_ws(B, R, &a, &c);
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
  if (R > kMaxN || B * R > 65535) return SPEC_EUNSUPPORTED;
  if (plan_sampler(V).smem > kMaxSliceBytes) return SPEC_EUNSUPPORTED;
  size_t a, c;
  if (workspace_bytes < samp_ws(B, R, &a, &c)) return SPEC_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return SPEC_EINVAL;
  SP prm = base_params(target_logits, draft_probs, uniforms, B, R, V, cfg, workspace);
  prm.tokens = draft_tokens;
  prm.tree = 0;
  prm.acc_len = accepted_len;
  prm.emitted = emitted;
  prm.p_out = cfg->greedy ? nullptr : p_out;
  prm.status = status_per_seq;
  return launch_sampler(prm, B, R, V, static_cast<cudaStream_t>(stream));
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
  if (N > kMaxN || B * N > 65535) return SPEC_EUNSUPPORTED;
  if (plan_sampler(V).smem > kMaxSliceBytes) return SPEC_EUNSUPPORTED;
  size_t a, c;
  if (workspace_bytes < samp_ws(B, N, &a, &c)) return SPEC_EINVAL;
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
  return launch_sampler(prm, B, N, V, static_cast<cudaStream_t>(stream));
}
