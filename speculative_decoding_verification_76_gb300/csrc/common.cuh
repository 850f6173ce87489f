// Shared device helpers for libspecverify (sm_103a).  Inline PTX wrappers for
// mbarrier, bulk copies, thread-block clusters / distributed shared memory and
// the warp-level MMA; the host-side per-device setup helper.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spec_verify.h"
#include "dev_once.h"

#define SPEC_DEV __device__ __forceinline__

// Workspace header: every workspace starts with this block (256 bytes).
struct WsHeader {
  int32_t error;      // first error word written by a bounded wait
  int32_t pad[63];
};
static_assert(sizeof(WsHeader) == 256, "header");

// Wall-clock bound of every spin on an mbarrier: far beyond any legitimate
// wait (microseconds), short enough that a broken phase cannot hang the GPU.
#define SPEC_WAIT_NS 2000000000ull

SPEC_DEV void set_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- mbarrier
SPEC_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SPEC_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

SPEC_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

SPEC_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

SPEC_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

SPEC_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

SPEC_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

SPEC_DEV uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait that may suspend the thread for up to `ns` nanoseconds while the
// phase is incomplete (returns as soon as it completes).
SPEC_DEV bool mbar_try_wait_ns(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (and records an error) if the phase does not
// complete within limit_ns (SPEC_WAIT_NS unless a test lowers it).  The fast
// path touches no global memory: it polls with suspended waits; only a wait
// that has already lasted long checks the clock and whether another wait of
// this launch has given up.
SPEC_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                        uint64_t limit_ns = SPEC_WAIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  for (int it = 0; it < 64; ++it)
    if (mbar_try_wait_ns(bar, parity, 1000)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    // once any wait of this launch has given up, later waits give up at once
    if (err && *reinterpret_cast<volatile int32_t*>(err) != 0) return false;
    for (int it = 0; it < 256; ++it)
      if (mbar_try_wait_ns(bar, parity, 1000)) return true;
    if (global_ns() - t0 > limit_ns) break;
  }
  set_error(err, SPEC_ERR_MBAR_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
SPEC_DEV void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- clusters
SPEC_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

SPEC_DEV uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier with release/acquire semantics (all threads of all CTAs).
SPEC_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                   : "memory");
}

// Address of the same shared-memory variable in CTA `rank` of this cluster.
SPEC_DEV uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}



SPEC_DEV uint32_t dsmem_ld_u32(const void* local, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(dsmem_addr(local, rank)) : "memory");
  return v;
}

SPEC_DEV unsigned long long dsmem_ld_u64(const void* local, uint32_t rank) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(dsmem_addr(local, rank)) : "memory");
  return v;
}

SPEC_DEV void dsmem_st_s32(void* local, uint32_t rank, int32_t v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(dsmem_addr(local, rank)), "r"(v) : "memory");
}

// ---------------------------------------------------------------- warp MMA (bf16)
SPEC_DEV void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

SPEC_DEV void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D (fp32)
SPEC_DEV void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

SPEC_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed pairs of fp32 (sm_100+ f32x2 arithmetic: one instruction, two lanes
// of the pair, each rounded as the scalar operation would be).
SPEC_DEV uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
SPEC_DEV void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
SPEC_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
SPEC_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
SPEC_DEV uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
SPEC_DEV float fmax3(float a, float b, float c) {  // three-input maximum (sm_100+)
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x on the special-function unit (PTX ex2.approx; ~2 ulp).
SPEC_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

SPEC_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

SPEC_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Status helpers shared by the host entry points.
#define SPEC_CUDA_TRY(expr)                          \
  do {                                               \
    cudaError_t e_ = (expr);                         \
    if (e_ != cudaSuccess) return SPEC_ECUDA;        \
  } while (0)

static inline spec_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// Raise `func`'s dynamic shared-memory limit to `bytes` on the current device,
// once per device and thread-safely (`once` is the launch site's record).
// Device ordinals beyond the record's range set the attribute on every call.
static inline spec_status ensure_smem_limit(PerDeviceOnce<int>& once, const void* func, int bytes) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ECUDA;
  auto set = [&](int*) {
    return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
                   cudaSuccess
               ? 0
               : 1;
  };
  const int rc = once.run(dev, set);
  if (rc == -1) return set(nullptr) == 0 ? SPEC_OK : SPEC_ECUDA;
  return rc == 0 ? SPEC_OK : SPEC_ECUDA;
}
