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
// one slice of the vocabulary once; max, exp values, normaliser, the
// top-k / top-p cut and the draws all run from shared memory, with
// cluster-wide reductions gathered by one warp over DSMEM.  Every row
// computes its own outcome independently (its draft test, and its
// correction draw if it rejects; the last row's bonus draw; for a tree node
// the first accepted child under the running residual, or its final draw),
// so all B*R rows run at once and nothing waits on a serial walk.  The
// cluster that finishes a sequence's last row assembles the outcomes.
//
// Numerics: exp((l - m)/T) is evaluated with the difference and quotient
// carried in two floats (p matches a float64 evaluation to ~3e-7 relative);
// sums are per-thread compensated and combined as float pairs in a fixed
// order, so results are deterministic.  top-k / top-p: a 1/16-nat histogram
// (below the row maximum) locates the crossing bin, its members are sorted
// exactly by (logit desc, id asc); an exact radix selection is the fallback
// for crossing bins too populous to sort.
#include <algorithm>
#include <climits>

#include "common.cuh"

namespace {

constexpr int kST = 512;
constexpr int kSW = kST / 32;
constexpr int kMaxCS = 8;
constexpr int kMaxN = 64;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kCandMax = 1024;                 // sortable members of one crossing bin
constexpr size_t kMaxSliceBytes = 84 * 1024;   // per CTA: logits + exp slices, each this size

// Outcome of one target row, written by its cluster.
struct Outcome {
  int32_t accept;  // chain: 1 if the row's draft is accepted; tree: accepted child or -1
  int32_t token;   // correction / bonus / final token of this row (-1 if none)
  int32_t status;  // SPEC_SEQ_* bits raised by this row
  int32_t flags;   // 1 if the row's logits are not finite
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
  int greedy, eos, tree, bulk, qbulk;
  Outcome* outcomes;
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

struct DF {  // hi + lo, |lo| <= ulp(hi)/2
  float hi, lo;
};

struct Shared {
  float red_f[kSW];
  int red_i[kSW];
  DF red_df[kSW];
  Slot slots[4];
  Slot gath[kMaxCS];
  uint32_t hcnt[256];
  float hmass[256];
  uint32_t tcnt[256];
  float tmass[256];
  uint32_t rcnt[2][256];
  unsigned long long rmass[2][256];
  unsigned long long rtmass[256];
  uint32_t rtcnt[256];
  int bi[8];
  DF bdf[2];
  int par[kMaxN];
  int tok[kMaxN];
  Outcome outs[kMaxN];
  uint64_t bar;
};

// ---------------------------------------------------------------- scalar helpers
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

SPEC_DEV DF df_norm(float a, float b) {  // fast two-sum, |a| >= |b| or a == 0
  const float s = a + b;
  return DF{s, b - (s - a)};
}

SPEC_DEV DF df_add(DF a, DF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb) + a.lo + b.lo;
  return df_norm(s, e);
}

struct Kahan {
  float s = 0.f, c = 0.f;
  SPEC_DEV void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  SPEC_DEV DF df() const { return df_norm(s, -c); }
};

SPEC_DEV double df_d(DF a) { return (double)a.hi + (double)a.lo; }

// ---------------------------------------------------------------- block reductions
SPEC_DEV DF block_sum_df(DF v, Shared& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = df_add(v, DF{__shfl_xor_sync(kFull, v.hi, o), __shfl_xor_sync(kFull, v.lo, o)});
  if (lane == 0) sh.red_df[w] = v;
  __syncthreads();
  if (w == 0) {
    DF x = lane < kSW ? sh.red_df[lane] : DF{0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      x = df_add(x, DF{__shfl_xor_sync(kFull, x.hi, o), __shfl_xor_sync(kFull, x.lo, o)});
    if (lane == 0) sh.bdf[0] = x;
  }
  __syncthreads();
  const DF t = sh.bdf[0];
  __syncthreads();
  return t;
}

// (max value, lowest id among maxima)
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

// exclusive scan of one float per thread (fixed order); *total = block total
// computed the way the last thread's running value is.
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
// Every CTA posts one Slot; warp 0 fetches all CS slots (lane r <- rank r)
// into sh.gath, which every thread then reads locally.  Posting slots rotate
// over four buffers so a slot is never rewritten before every reader is past
// the next cluster barrier.
SPEC_DEV void cluster_allgather(Slot mine, int CS, int& ph, Shared& sh) {
  Slot* s = &sh.slots[ph & 3];
  if (threadIdx.x == 0) *s = mine;
  cluster_sync();
  if ((int)threadIdx.x < CS) {
    Slot r;
    r.a = dsmem_ld_u64(&s->a, threadIdx.x);
    r.b = dsmem_ld_u64(&s->b, threadIdx.x);
    sh.gath[threadIdx.x] = r;
  }
  __syncthreads();
  ++ph;
}

SPEC_DEV Slot cluster_from(Slot mine, int src, int CS, int& ph, Shared& sh) {
  cluster_allgather(mine, CS, ph, sh);
  return sh.gath[src];
}

SPEC_DEV Slot slot_df(DF v) {
  return Slot{(unsigned long long)__float_as_uint(v.hi), (unsigned long long)__float_as_uint(v.lo)};
}

SPEC_DEV DF cluster_sum_df(DF v, int CS, int& ph, Shared& sh) {
  cluster_allgather(slot_df(v), CS, ph, sh);
  DF t{0.f, 0.f};
  for (int r = 0; r < CS; ++r)
    t = df_add(t, DF{__uint_as_float((uint32_t)sh.gath[r].a),
                     __uint_as_float((uint32_t)sh.gath[r].b)});
  return t;
}

// ---------------------------------------------------------------- the slice
struct Slice {
  float* buf;  // shared memory, n floats
  int lo, n;
};

// Load a row slice into shared memory (TMA bulk copy when aligned).
SPEC_DEV void load_row(const SP& p, const float* row, Slice& sl, Shared& sh, uint32_t& bar_phase) {
  __syncthreads();  // every reader of the previous contents is done
  if (sl.n <= 0) return;
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

// coarse bin of a logit: 1/16 nat below the row maximum, 255 = beyond 16 nats
SPEC_DEV int coarse_bin(float l, float m, float scale16) {
  const float d = (m - l) * scale16;  // monotone non-increasing in l
  return d < 255.f ? (int)d : 255;
}

// Deterministic cluster sum of E over the elements with pred(k).
template <class Pred>
SPEC_DEV DF cluster_masked_sum(const Slice& sl, const float* E, Pred pred, int CS, int& ph,
                               Shared& sh) {
  Kahan acc;
  for (int k = threadIdx.x; k < sl.n; k += kST)
    if (pred(k)) acc.add(E[k]);
  return cluster_sum_df(block_sum_df(acc.df(), sh), CS, ph, sh);
}

// First index d in [0, n) (n <= 256) where the running sum of val[0..d]
// reaches target; -1 if none.  Warp 0 scans 8 bins per lane; the result is
// broadcast to the block.
template <class T>
SPEC_DEV int first_reaching(const T* val, int n, double target, Shared& sh) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    double ls = 0.0;
    for (int j = 0; j < 8; ++j)
      if (8 * lane + j < n) ls += (double)val[8 * lane + j];
    double incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(kFull, incl >= target);
    int res = -1;
    if (hit) {
      const int L = __ffs(hit) - 1;
      if (lane == L) {
        double cum = incl - ls;
        for (int j = 0; j < 8; ++j) {
          const int d = 8 * L + j;
          if (d >= n) break;
          cum += (double)val[d];
          if (cum >= target) {
            res = d;
            break;
          }
        }
      }
      res = __shfl_sync(kFull, res, L);
    }
    if (lane == 0) sh.bi[2] = res;
  }
  __syncthreads();
  const int r = sh.bi[2];
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------- crossing-bin sort
SPEC_DEV uint64_t cand_of(float l, int id) {
  return ((uint64_t)okey(l) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)id);
}
SPEC_DEV uint32_t cand_key(uint64_t c) { return (uint32_t)(c >> 32); }
SPEC_DEV int cand_id(uint64_t c) { return (int)(0xFFFFFFFFu - (uint32_t)c); }

struct Scratch {
  uint64_t *cand, *gk, *sk;
  float *candE, *ge, *se;
};

struct Sorted {
  uint64_t* key;  // CTA 0: members sorted by (logit desc, id asc)
  float* E;       // their exp values, same order
  int n;
};

// Gather the elements with pred(k) (with their exp values) from every CTA
// into CTA 0 and rank-sort them there.  The caller guarantees the cluster
// count is <= kCandMax.  Same n in every CTA; keys valid in CTA 0 only.
template <class Pred>
SPEC_DEV Sorted gather_sort(const Slice& sl, const float* E, const Scratch& sc, Pred pred, int rank,
                            int CS, int& ph, Shared& sh) {
  if (threadIdx.x == 0) sh.bi[1] = 0;
  __syncthreads();
  for (int k = threadIdx.x; k < sl.n; k += kST) {
    if (pred(k)) {
      const int slot = atomicAdd(&sh.bi[1], 1);
      if (slot < kCandMax) {
        sc.cand[slot] = cand_of(sl.buf[k], sl.lo + k);
        sc.candE[slot] = E[k];
      }
    }
  }
  __syncthreads();
  const int mine = min(sh.bi[1], kCandMax);
  cluster_allgather(Slot{(unsigned long long)mine, 0ull}, CS, ph, sh);
  int cnt[kMaxCS];
  int total = 0;
  for (int r = 0; r < CS; ++r) {
    cnt[r] = (int)sh.gath[r].a;
    total += cnt[r];
  }
  total = min(total, kCandMax);
  if (rank == 0) {
    int off = 0;
    for (int r = 0; r < CS; ++r) {
      for (int j = threadIdx.x; j < cnt[r] && off + j < kCandMax; j += kST) {
        sc.gk[off + j] = dsmem_ld_u64(&sc.cand[j], r);
        sc.ge[off + j] = dsmem_ld_f32(&sc.candE[j], r);
      }
      off += cnt[r];
    }
    __syncthreads();
    // rank sort: keys are distinct (ids are), rank = number of larger keys
    for (int i = threadIdx.x; i < total; i += kST) {
      const uint64_t c = sc.gk[i];
      int rk = 0;
      for (int j = 0; j < total; ++j) rk += sc.gk[j] > c ? 1 : 0;
      sc.sk[rk] = c;
      sc.se[rk] = sc.ge[i];
    }
    __syncthreads();
  }
  cluster_sync();  // other CTAs' candidate lists stay intact until CTA 0 has copied them
  return Sorted{sc.sk, sc.se, total};
}

// In CTA 0: the first sorted index j whose base + sum(E[0..j]) reaches thr
// (float-pair sums, fixed order), with that running sum; (-1, 0) if none.
SPEC_DEV void sorted_crossing(const Sorted& so, DF base, double thr, int* idx, DF* at, Shared& sh) {
  const int per = (so.n + kST - 1) / kST;
  const int s0 = min((int)threadIdx.x * per, so.n), s1 = min(s0 + per, so.n);
  DF run{0.f, 0.f};
  for (int j = s0; j < s1; ++j) run = df_add(run, DF{so.E[j], 0.f});
  // inclusive scan over the lanes, then over the warps, in a fixed order
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  DF incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF t = DF{__shfl_up_sync(kFull, incl.hi, o), __shfl_up_sync(kFull, incl.lo, o)};
    if (lane >= o) incl = df_add(t, incl);
  }
  const DF lanes_before = DF{__shfl_up_sync(kFull, incl.hi, 1), __shfl_up_sync(kFull, incl.lo, 1)};
  if (lane == 31) sh.red_df[w] = incl;
  __syncthreads();
  DF excl = base;
  for (int i = 0; i < w; ++i) excl = df_add(excl, sh.red_df[i]);
  if (lane > 0) excl = df_add(excl, lanes_before);
  __syncthreads();
  int found = INT_MAX;
  DF val{0.f, 0.f};
  if (df_d(df_add(excl, run)) >= thr) {
    DF acc = excl;
    for (int j = s0; j < s1; ++j) {
      acc = df_add(acc, DF{so.E[j], 0.f});
      if (df_d(acc) >= thr) {
        found = j;
        val = acc;
        break;
      }
    }
  }
  const int f = block_min_i(found, sh);
  if (found == f && f != INT_MAX) sh.bdf[1] = val;
  __syncthreads();
  *idx = (f == INT_MAX) ? -1 : f;
  *at = (f == INT_MAX) ? DF{0.f, 0.f} : sh.bdf[1];
  __syncthreads();
}

// In CTA 0: float-pair sum (fixed order) of the first n sorted exp values.
SPEC_DEV DF sorted_head_sum(const Sorted& so, int n, Shared& sh) {
  const int per = (n + kST - 1) / kST;
  const int s0 = min((int)threadIdx.x * per, n), s1 = min(s0 + per, n);
  DF run{0.f, 0.f};
  for (int j = s0; j < s1; ++j) run = df_add(run, DF{so.E[j], 0.f});
  return block_sum_df(run, sh);
}

struct Trunc {
  uint32_t tau;
  int tie;
  DF Z;
  bool ok;
};

// Top-k then top-p by coarse bins + an exact sort of the crossing bin.
// ok = false when a crossing bin is too populous (the caller falls back to
// the exact radix selection).
SPEC_DEV Trunc truncate_fast(const SP& p, const Slice& sl, const float* E, const Scratch& sc,
                             float m, DF Zall, int rank, int CS, int& ph, Shared& sh) {
  Trunc tr{0u, INT_MAX, Zall, true};
  const float s16 = p.invT * 16.f;
  for (int d = threadIdx.x; d < 256; d += kST) {
    sh.hcnt[d] = 0u;
    sh.hmass[d] = 0.f;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < sl.n; k += kST) {
    const int bn = coarse_bin(sl.buf[k], m, s16);
    if (bn < 255) {
      atomicAdd(&sh.hcnt[bn], 1u);
      atomicAdd(&sh.hmass[bn], E[k]);
    }
  }
  __syncthreads();
  cluster_sync();
  // cluster totals: thread d sums bin d over the ranks
  for (int d = threadIdx.x; d < 256; d += kST) {
    uint32_t c = 0;
    float mm = 0.f;
    for (int r = 0; r < CS; ++r) {
      c += dsmem_ld_u32(&sh.hcnt[d], r);
      mm += dsmem_ld_f32(&sh.hmass[d], r);
    }
    sh.tcnt[d] = c;
    sh.tmass[d] = mm;
  }
  __syncthreads();
  int bk = 254;  // last bin (partly) kept by top-k
  if (p.top_k > 0 && p.top_k < p.V) {
    const int bsel = first_reaching(sh.tcnt, 255, (double)p.top_k, sh);
    if (bsel < 0 || sh.tcnt[bsel] > (uint32_t)kCandMax) {
      tr.ok = false;
      return tr;
    }
    uint32_t above_cnt = 0;
    for (int d = 0; d < bsel; ++d) above_cnt += sh.tcnt[d];
    const int need = p.top_k - (int)above_cnt;
    const DF above = cluster_masked_sum(
        sl, E, [&](int k) { return coarse_bin(sl.buf[k], m, s16) < bsel; }, CS, ph, sh);
    const Sorted so = gather_sort(
        sl, E, sc, [&](int k) { return coarse_bin(sl.buf[k], m, s16) == bsel; }, rank, CS, ph, sh);
    const int nn = min(need, so.n);
    Slot mine{0ull, 0ull};
    if (rank == 0) {
      const DF part = sorted_head_sum(so, nn, sh);
      if (threadIdx.x == 0) mine = Slot{so.key[nn - 1], slot_df(part).a | (slot_df(part).b << 32)};
    }
    const Slot o = cluster_from(mine, 0, CS, ph, sh);
    const DF part = DF{__uint_as_float((uint32_t)o.b), __uint_as_float((uint32_t)(o.b >> 32))};
    tr.tau = cand_key(o.a);
    tr.tie = cand_id(o.a);
    tr.Z = df_add(above, part);
    bk = bsel;
  }
  if (p.top_p > 0.f && p.top_p < 1.f) {
    const double thr = (double)p.top_p * df_d(tr.Z);
    const uint32_t tk = tr.tau;
    const int tc = tr.tie;
    int bp = first_reaching(sh.tmass, bk + 1, thr, sh);
    if (bp < 0) bp = bk;
    for (int attempt = 0; attempt < 6; ++attempt) {
      if (bp < 0 || bp > bk || sh.tcnt[bp] > (uint32_t)kCandMax) break;
      const int bsel = bp;
      const DF above = cluster_masked_sum(
          sl, E,
          [&](int k) {
            const float l = sl.buf[k];
            return coarse_bin(l, m, s16) < bsel && is_kept(okey(l), sl.lo + k, tk, tc);
          },
          CS, ph, sh);
      if (df_d(above) >= thr) {  // the crossing lies in an earlier bin
        --bp;
        continue;
      }
      const Sorted so = gather_sort(
          sl, E, sc,
          [&](int k) {
            const float l = sl.buf[k];
            return coarse_bin(l, m, s16) == bsel && is_kept(okey(l), sl.lo + k, tk, tc);
          },
          rank, CS, ph, sh);
      Slot mine{~0ull, 0ull};
      if (rank == 0) {
        int idx;
        DF at;
        sorted_crossing(so, above, thr, &idx, &at, sh);
        if (threadIdx.x == 0 && idx >= 0)
          mine = Slot{so.key[idx], slot_df(at).a | (slot_df(at).b << 32)};
      }
      const Slot o = cluster_from(mine, 0, CS, ph, sh);
      if (o.a == ~0ull) {  // not in this bin: move on to the next one
        ++bp;
        continue;
      }
      tr.tau = cand_key(o.a);
      tr.tie = cand_id(o.a);
      tr.Z = DF{__uint_as_float((uint32_t)o.b), __uint_as_float((uint32_t)(o.b >> 32))};
      return tr;
    }
    tr.ok = false;
  }
  return tr;
}

// ---------------------------------------------------------------- exact radix fallback
// Radix selection, most significant digit first, of the position in
// (key desc, id asc) order where the running weight reaches the target.
// Weight = 1 per element (top-k) or its 2^-40 fixed-point mass (top-p).
struct Sel {
  uint32_t tau;
  unsigned long long above, at_weight, target;
  uint32_t at_count;
};

template <class Keep, class Weight>
SPEC_DEV Sel radix_select(const Slice& sl, bool target_is_fraction, double frac,
                          unsigned long long target_abs, Keep keep, Weight weight, int CS, int& ph,
                          Shared& sh) {
  uint32_t prefix = 0, pmask = 0;
  unsigned long long above = 0, target = target_abs;
  Sel out{};
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int h = pass & 1;
    for (int i = threadIdx.x; i < 256; i += kST) {
      sh.rmass[h][i] = 0ull;
      sh.rcnt[h][i] = 0u;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < sl.n; k += kST) {
      const uint32_t key = okey(sl.buf[k]);
      if ((key & pmask) == prefix && keep(k, key)) {
        const uint32_t digit = (key >> shift) & 255u;
        atomicAdd(&sh.rcnt[h][digit], 1u);
        atomicAdd(&sh.rmass[h][digit], weight(k));
      }
    }
    __syncthreads();
    cluster_sync();
    for (int d = threadIdx.x; d < 256; d += kST) {
      unsigned long long mm = 0;
      uint32_t c = 0;
      for (int r = 0; r < CS; ++r) {
        mm += dsmem_ld_u64(&sh.rmass[h][d], r);
        c += dsmem_ld_u32(&sh.rcnt[h][d], r);
      }
      sh.rtmass[255 - d] = mm;  // descending digit order
      sh.rtcnt[255 - d] = c;
    }
    __syncthreads();
    if (pass == 0 && target_is_fraction) {
      unsigned long long tot = 0;
      for (int d = 0; d < 256; ++d) tot += sh.rtmass[d];
      const double thr = ceil(frac * (double)tot);
      target = thr < 1.0 ? 1ull : (unsigned long long)thr;
      if (target > tot) target = tot;
    }
    // first descending digit whose running weight reaches target - above
    const unsigned long long need = target - above;
    unsigned long long cum = 0;
    int sel = 255;
    for (int d = 0; d < 256; ++d) {  // every thread, identical result
      if (cum + sh.rtmass[d] >= need) {
        sel = d;
        break;
      }
      cum += sh.rtmass[d];
    }
    above += cum;
    const uint32_t digit = 255u - (uint32_t)sel;
    prefix |= digit << shift;
    pmask |= 255u << shift;
    if (pass == 3) {
      out.at_count = sh.rtcnt[sel];
      out.at_weight = sh.rtmass[sel];
    }
    __syncthreads();
  }
  out.tau = prefix;
  out.above = above;
  out.target = target;
  return out;
}

// The id (global) of the nth (1-based) element, in ascending id order over
// the cluster, for which pred(local index) holds.  Same result in all CTAs.
template <class Pred>
SPEC_DEV int nth_in_cluster(const Slice& sl, int nth, Pred pred, int rank, int CS, int& ph,
                            Shared& sh) {
  const int seg = (sl.n + kST - 1) / kST;
  const int s0 = min((int)threadIdx.x * seg, sl.n), s1 = min(s0 + seg, sl.n);
  int c = 0;
  for (int k = s0; k < s1; ++k) c += pred(k) ? 1 : 0;
  int tot;
  const int excl = block_excl_scan_i(c, &tot, sh);
  cluster_allgather(Slot{(unsigned long long)tot, 0ull}, CS, ph, sh);
  int before = 0, owner = -1;
  for (int r = 0; r < CS; ++r) {
    const int tr = (int)sh.gath[r].a;
    if (owner < 0 && before + tr >= nth) owner = r;
    if (owner < 0) before += tr;
  }
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
  const Slot o = cluster_from(Slot{(unsigned long long)(unsigned)found, 0ull},
                              owner < 0 ? 0 : owner, CS, ph, sh);
  return owner < 0 ? INT_MAX : (int)(unsigned)o.a;
}

SPEC_DEV Trunc truncate_radix(const SP& p, const Slice& sl, float m, int rank, int CS, int& ph,
                              Shared& sh) {
  Trunc tr{0u, INT_MAX, DF{0.f, 0.f}, true};
  cluster_sync();  // other CTAs may still read this CTA's coarse histogram
  if (p.top_k > 0 && p.top_k < p.V) {
    const Sel s = radix_select(
        sl, false, 0.0, (unsigned long long)p.top_k, [](int, uint32_t) { return true; },
        [](int) { return 1ull; }, CS, ph, sh);
    const int need = (int)(s.target - s.above);
    tr.tau = s.tau;
    if ((uint32_t)need >= s.at_count) {
      tr.tie = INT_MAX;
    } else {
      const uint32_t tau = s.tau;
      tr.tie = nth_in_cluster(
          sl, need, [&](int k) { return okey(sl.buf[k]) == tau; }, rank, CS, ph, sh);
    }
  }
  if (p.top_p > 0.f && p.top_p < 1.f) {
    const uint32_t tk = tr.tau;
    const int tc = tr.tie;
    const float T = p.T, invT = p.invT;
    auto keep_k = [&](int k, uint32_t key) { return is_kept(key, sl.lo + k, tk, tc); };
    auto mass = [&](int k) {
      const float e = texp(sl.buf[k], m, T, invT);
      return (unsigned long long)__float2ull_rn(e * 1099511627776.0f);  // 2^40
    };
    const Sel s = radix_select(sl, true, (double)p.top_p, 0ull, keep_k, mass, CS, ph, sh);
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
      tie = nth_in_cluster(
          sl, (int)need,
          [&](int k) {
            const uint32_t key = okey(sl.buf[k]);
            return key == tau && is_kept(key, sl.lo + k, tk, tc);
          },
          rank, CS, ph, sh);
    }
    tr.tau = tau;
    tr.tie = tie;
  }
  return tr;
}

// ---------------------------------------------------------------- the draw
// The first id whose running sum (ascending id order over the cluster) of
// the slice values exceeds u * total; -2 if the total is zero.  Same result
// in all CTAs.
SPEC_DEV int draw_from_slice(const Slice& sl, float u, int rank, int CS, int& ph, Shared& sh) {
  const int seg = (sl.n + kST - 1) / kST;
  const int s0 = min((int)threadIdx.x * seg, sl.n), s1 = min(s0 + seg, sl.n);
  float run = 0.f;
  for (int k = s0; k < s1; ++k) run += sl.buf[k];
  float tot;
  const float excl = block_excl_scan_f(run, &tot, sh);
  cluster_allgather(Slot{(unsigned long long)__float_as_uint(tot), 0ull}, CS, ph, sh);
  float pre[kMaxCS + 1], tots[kMaxCS];
  pre[0] = 0.f;
  for (int r = 0; r < CS; ++r) {
    tots[r] = __uint_as_float((uint32_t)sh.gath[r].a);
    pre[r + 1] = pre[r] + tots[r];
  }
  const float W = pre[CS];
  if (!(W > 0.f)) return -2;
  const float target = u * W;
  int owner = -1;
  for (int r = 0; r < CS; ++r)
    if (owner < 0 && tots[r] > 0.f && pre[r] + tots[r] > target) owner = r;
  if (owner < 0)
    for (int r = CS - 1; r >= 0; --r)
      if (owner < 0 && tots[r] > 0.f) owner = r;
  const float prefix = pre[owner];
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
    found = block_min_i(found, sh);
    if (found == INT_MAX) {
      // rounding left nothing above target: take the last nonzero entry
      int last = -1;
      for (int k = s0; k < s1; ++k)
        if (sl.buf[k] > 0.f) last = k;
      const int neg = block_min_i(-last, sh);  // -(largest index)
      found = (neg <= 0) ? -neg : INT_MAX;
    }
  }
  const Slot o = cluster_from(
      Slot{(unsigned long long)(unsigned)(found == INT_MAX ? 0 : sl.lo + found), 0ull}, owner, CS,
      ph, sh);
  return (int)(unsigned)o.a;
}

// ---------------------------------------------------------------- the kernel
// One cluster per target row.  Every row computes its own outcome:
//   chain row i < R-1: is draft i+1 accepted? if not, the correction drawn
//     from norm(max(0, p_i - q_i));  chain row R-1: the bonus drawn from p;
//   tree node v: the first accepted child (residual p' updated after each
//     rejected child) or, if none, the final token drawn from p'.
// The cluster that finishes a sequence's last row assembles the sequence.
__global__ void __launch_bounds__(kST, 1) sampler_kernel(const SP p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  float* Lb = reinterpret_cast<float*>(dyn);
  float* Eb = Lb + p.slice;
  Scratch sc;
  sc.cand = reinterpret_cast<uint64_t*>(Eb + p.slice);
  sc.gk = sc.cand + kCandMax;
  sc.sk = sc.gk + kCandMax;
  sc.candE = reinterpret_cast<float*>(sc.sk + kCandMax);
  sc.ge = sc.candE + kCandMax;
  sc.se = sc.ge + kCandMax;
  __shared__ Shared sh;
  const int rank = (int)cluster_ctarank();
  const int CS = (int)cluster_nctarank();
  const int row = blockIdx.y;
  const int R = p.R;
  const int b = row / R;
  const int i = row % R;
  Slice sl{Lb, rank * p.slice, 0};
  sl.n = max(0, min(p.slice, p.V - sl.lo));
  Slice sw{Eb, sl.lo, sl.n};
  int ph = 0;
  uint32_t bar_phase = 0;

  // the q row this row may need for its residual: warm it into L2 now
  const float* qrow = nullptr;
  if (!p.greedy && p.q) {
    if (p.tree)
      qrow = p.q + ((size_t)b * R + i) * p.V;
    else if (i < R - 1)
      qrow = p.q + ((size_t)b * (R - 1) + i) * p.V;
  }
  if (threadIdx.x == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
    if (qrow && p.qbulk && sl.n > 0) prefetch_l2(qrow + sl.lo, (uint32_t)sl.n * 4u);
  }
  if (p.tree)
    for (int c = threadIdx.x; c < R; c += kST) {
      sh.par[c] = p.parent[(size_t)b * R + c];
      sh.tok[c] = p.tokens[(size_t)b * R + c];
    }
  // scalars of this row's test, loaded early
  float u_test = 0.f, u_final = 0.f;
  int x_draft = -1;
  if (!p.greedy) {
    u_final = __ldg(&p.u[(size_t)b * R + (R - 1)]);
    if (!p.tree && i < R - 1) {
      u_test = __ldg(&p.u[(size_t)b * R + i]);
      x_draft = __ldg(&p.tokens[(size_t)b * (R - 1) + i]);
    }
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
  cluster_allgather(Slot{((unsigned long long)__float_as_uint(mv) << 32) | (unsigned)mi,
                         (unsigned long long)bad},
                    CS, ph, sh);
  for (int r = 0; r < CS; ++r) {
    const unsigned long long a = sh.gath[r].a;
    const float ov = __uint_as_float((uint32_t)(a >> 32));
    const int oi = (int)(uint32_t)a;
    bad |= (int)sh.gath[r].b;
    if (ov > mv || (ov == mv && oi < mi)) {
      mv = ov;
      mi = oi;
    }
  }
  if (mv == -INFINITY) bad = 1;  // every token banned: no distribution
  const float m = mv;
  Outcome oc{0, -1, 0, bad};

  if (p.greedy) {
    // ---- greedy: the argmax decides everything
    if (!bad) {
      if (!p.tree) {
        if (i < R - 1) oc.accept = (__ldg(&p.tokens[(size_t)b * (R - 1) + i]) == mi) ? 1 : 0;
        oc.token = mi;
      } else {
        oc.accept = -1;
        for (int c = i + 1; c < R; ++c)
          if (sh.par[c] == i && sh.tok[c] == mi) {
            oc.accept = c;
            break;
          }
        oc.token = mi;
      }
    }
  } else if (!bad) {
    // ---- 3. exp values, normaliser, truncation
    Kahan acc;
    for (int k = threadIdx.x; k < sl.n; k += kST) {
      const float e = texp(sl.buf[k], m, p.T, p.invT);
      Eb[k] = e;
      acc.add(e);
    }
    const DF zall = cluster_sum_df(block_sum_df(acc.df(), sh), CS, ph, sh);
    Trunc tr{0u, INT_MAX, zall, true};
    if ((p.top_k > 0 && p.top_k < p.V) || (p.top_p > 0.f && p.top_p < 1.f)) {
      tr = truncate_fast(p, sl, Eb, sc, m, zall, rank, CS, ph, sh);
      if (!tr.ok) {
        tr = truncate_radix(p, sl, m, rank, CS, ph, sh);
        const uint32_t tau = tr.tau;
        const int tie = tr.tie;
        tr.Z = cluster_masked_sum(
            sl, Eb, [&](int k) { return is_kept(okey(sl.buf[k]), sl.lo + k, tau, tie); }, CS,
            ph, sh);
      }
    }
    const float invZ = 1.0f / (float)df_d(tr.Z);
    const bool truncated = tr.tau != 0u || tr.tie != INT_MAX;
    // p in place of the exp values (0 outside the kept set)
    if (truncated) {
      for (int k = threadIdx.x; k < sl.n; k += kST)
        Eb[k] = is_kept(okey(sl.buf[k]), sl.lo + k, tr.tau, tr.tie) ? Eb[k] * invZ : 0.f;
    } else {
      for (int k = threadIdx.x; k < sl.n; k += kST) Eb[k] *= invZ;
    }
    __syncthreads();
    if (p.p_out) {
      float* dst = p.p_out + (size_t)row * p.V + sl.lo;
      for (int k = threadIdx.x; k < sl.n; k += kST) dst[k] = Eb[k];
    }

    if (!p.tree) {
      // ---- 4a. chain: this row's test, then its correction or bonus draw
      bool draw = true;
      bool resid = false;
      if (i < R - 1) {
        const int x = x_draft;
        const bool xin = x >= 0 && x < p.V;
        const float qx = xin ? __ldg(&qrow[x]) : 0.f;
        cluster_sync();  // p complete in every CTA
        const float px =
            xin ? dsmem_ld_f32(&Eb[x - (x / p.slice) * p.slice], (uint32_t)(x / p.slice)) : 0.f;
        if (qx == 0.f) oc.status |= SPEC_SEQ_QZERO;
        oc.accept = (u_test * qx < px) ? 1 : 0;
        cluster_sync();  // nobody rewrites p before every CTA has read p(x)
        draw = !oc.accept;
        resid = true;
      }
      if (draw) {
        if (resid) {
          for (int k = threadIdx.x; k < sl.n; k += kST)
            Eb[k] = fmaxf(Eb[k] - __ldg(&qrow[sl.lo + k]), 0.f);
          __syncthreads();
        }
        int tok = draw_from_slice(sw, u_final, rank, CS, ph, sh);
        if (tok == -2) {  // residual with zero mass (rounding only): draw from p
          oc.status |= SPEC_SEQ_RESID_ZERO;
          for (int k = threadIdx.x; k < sl.n; k += kST)
            Eb[k] = is_kept(okey(sl.buf[k]), sl.lo + k, tr.tau, tr.tie)
                        ? texp(sl.buf[k], m, p.T, p.invT) * invZ
                        : 0.f;
          __syncthreads();
          tok = draw_from_slice(sw, u_final, rank, CS, ph, sh);
        }
        oc.token = tok;
      }
    } else {
      // ---- 4b. tree node: children in storage order against the running p'
      oc.accept = -1;
      for (int c = i + 1; c < R; ++c) {
        if (sh.par[c] != i) continue;
        const int t = sh.tok[c];
        const bool tin = t >= 0 && t < p.V;
        const float qx = tin ? __ldg(&qrow[t]) : 0.f;
        cluster_sync();  // p' complete everywhere
        const float pt =
            tin ? dsmem_ld_f32(&Eb[t - (t / p.slice) * p.slice], (uint32_t)(t / p.slice)) : 0.f;
        cluster_sync();  // nobody rewrites p' before every CTA has read it
        if (qx == 0.f) oc.status |= SPEC_SEQ_QZERO;
        if (__ldg(&p.u[(size_t)b * R + (c - 1)]) * qx < pt) {
          oc.accept = c;
          break;
        }
        // p' <- norm(max(0, p' - q_v))
        Kahan w;
        for (int k = threadIdx.x; k < sl.n; k += kST)
          w.add(fmaxf(Eb[k] - __ldg(&qrow[sl.lo + k]), 0.f));
        const DF W = cluster_sum_df(block_sum_df(w.df(), sh), CS, ph, sh);
        const float Wf = (float)df_d(W);
        if (Wf > 0.f) {
          const float invW = 1.0f / Wf;
          for (int k = threadIdx.x; k < sl.n; k += kST)
            Eb[k] = fmaxf(Eb[k] - __ldg(&qrow[sl.lo + k]), 0.f) * invW;
        } else {
          oc.status |= SPEC_SEQ_RESID_ZERO;
        }
        __syncthreads();
      }
      if (oc.accept < 0) oc.token = draw_from_slice(sw, u_final, rank, CS, ph, sh);
    }
  }

  // ---- 5. publish the outcome; the last row of the sequence assembles it
  cluster_sync();  // every CTA is done with the others' shared memory
  if (rank != 0 || threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
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

// ---------------------------------------------------------------- host side
struct SampPlan {
  int CS, slice;
  size_t smem;  // bytes of one slice buffer
};

SampPlan plan_sampler(int V) {
  SampPlan pl;
  pl.CS = std::min(kMaxCS, std::max(1, (V + 16383) / 16384));
  pl.slice = ((V + pl.CS - 1) / pl.CS + 3) / 4 * 4;
  pl.smem = (size_t)pl.slice * 4;
  return pl;
}

size_t dyn_smem(size_t slice_bytes) {
  return 2 * slice_bytes + 3 * (size_t)kCandMax * (sizeof(uint64_t) + sizeof(float));
}

size_t samp_ws(int B, int R, size_t* off_out, size_t* off_cnt) {
  size_t off = sizeof(WsHeader);
  *off_out = off;
  off += ((size_t)B * R * sizeof(Outcome) + 255) / 256 * 256;
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
                             (int)dyn_smem(kMaxSliceBytes)) != cudaSuccess)
      return SPEC_ECUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.CS, B * R, 1);
  cfg.blockDim = dim3(kST, 1, 1);
  cfg.dynamicSmemBytes = dyn_smem(pl.smem);
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
  size_t off_out, off_cnt;
  samp_ws(B, R, &off_out, &off_cnt);
  uint8_t* w = static_cast<uint8_t*>(ws);
  prm.err = reinterpret_cast<int32_t*>(w);
  prm.outcomes = reinterpret_cast<Outcome*>(w + off_out);
  prm.seq_count = reinterpret_cast<int32_t*>(w + off_cnt);
  prm.bulk = (V % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) ? 1 : 0;
  prm.qbulk = (q && V % 4 == 0 && (reinterpret_cast<uintptr_t>(q) & 15) == 0) ? 1 : 0;
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
