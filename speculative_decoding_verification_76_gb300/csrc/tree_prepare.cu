// spec_tree_prepare: ancestor bitmask, depth and position id of every node
// of a flattened draft tree.  "Speculative Decoding" (atlas), section
// "Chains, trees and visibility": a node sees the accepted prefix, its
// ancestors and itself; position ids follow depth, not storage order.
//
// One warp per sequence.  Because parent[i] < i (storage order is a
// topological order), mask[i] = mask[parent[i]] | (1 << i) and
// depth[i] = depth[parent[i]] + 1 can be filled in increasing i; the warp
// does it as log2(R) rounds of pointer jumping so no lane waits on a chain.
#include "common.cuh"

namespace {

__global__ void tree_prepare_kernel(const int32_t* __restrict__ parent,
                                    const int32_t* __restrict__ ctx_len, int B, int R,
                                    uint64_t* __restrict__ anc_mask, int32_t* __restrict__ pos_ids,
                                    int32_t* __restrict__ status) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= B) return;
  const int b = warp;
  // two nodes per lane: i = lane and lane + 32
  int par[2], jump[2], depth[2];
  uint64_t mask[2];
  bool bad = false;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    int p = -1;
    if (i < R) {
      p = parent ? parent[(size_t)b * R + i] : i - 1;
      if (i == 0 ? p != -1 : (p < 0 || p >= i)) bad = true;
    }
    par[k] = (i < R && !bad) ? p : -1;
    jump[k] = par[k];
    depth[k] = (i < R && par[k] >= 0) ? 1 : 0;
    mask[k] = (i < R) ? (1ull << i) : 0ull;
  }
  bad = __any_sync(0xffffffffu, bad);
  // pointer jumping: after round r, jump = 2^r-th ancestor, mask covers the
  // 2^r nearest ancestors, depth counts them.
  for (int round = 0; round < 6; ++round) {
    int j[2];
    uint64_t m[2];
    int d[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int a = jump[k];
      // read node a's state (owned by lane a & 31, slot a >> 5)
      const int src_lane = a < 0 ? 0 : (a & 31);
      const int slot = a < 0 ? 0 : (a >> 5);
      const int ja0 = __shfl_sync(0xffffffffu, jump[0], src_lane);
      const int ja1 = __shfl_sync(0xffffffffu, jump[1], src_lane);
      const uint64_t ma0 = __shfl_sync(0xffffffffu, mask[0], src_lane);
      const uint64_t ma1 = __shfl_sync(0xffffffffu, mask[1], src_lane);
      const int da0 = __shfl_sync(0xffffffffu, depth[0], src_lane);
      const int da1 = __shfl_sync(0xffffffffu, depth[1], src_lane);
      if (a >= 0) {
        j[k] = slot ? ja1 : ja0;
        m[k] = mask[k] | (slot ? ma1 : ma0);
        d[k] = depth[k] + (slot ? da1 : da0);
      } else {
        j[k] = -1;
        m[k] = mask[k];
        d[k] = depth[k];
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      jump[k] = j[k];
      mask[k] = m[k];
      depth[k] = d[k];
    }
  }
  const int ctx = ctx_len[b];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < R) {
      anc_mask[(size_t)b * R + i] = bad ? 0ull : mask[k];
      if (pos_ids) pos_ids[(size_t)b * R + i] = bad ? 0 : ctx + depth[k];
    }
  }
  if (status && lane == 0) status[b] = bad ? SPEC_SEQ_BAD_TREE : 0;
}

}  // namespace

extern "C" const char* spec_status_str(spec_status s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_EINVAL: return "SPEC_EINVAL: invalid argument";
    case SPEC_EUNSUPPORTED: return "SPEC_EUNSUPPORTED: outside the supported envelope";
    case SPEC_ECUDA: return "SPEC_ECUDA: CUDA call failed";
    case SPEC_ETIMEOUT: return "SPEC_ETIMEOUT: bounded device wait ran out";
  }
  return "unknown spec_status";
}

extern "C" spec_status spec_tree_prepare(const int32_t* parent, const int32_t* ctx_len, int B,
                                         int R, uint64_t* anc_mask, int32_t* pos_ids,
                                         int32_t* status_per_seq, void* stream) {
  if (B < 0 || R < 1 || R > 64 || !ctx_len || !anc_mask) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  const int threads = 128;
  const int blocks = (B * 32 + threads - 1) / threads;
  tree_prepare_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(parent, ctx_len, B, R, anc_mask,
                                                                    pos_ids, status_per_seq);
  return launch_status();
}

extern "C" spec_status spec_workspace_error(const void* workspace, int32_t* host_err,
                                            void* stream) {
  if (!workspace || !host_err) return SPEC_EINVAL;
  SPEC_CUDA_TRY(cudaMemcpyAsync(host_err, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                (cudaStream_t)stream));
  SPEC_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  return SPEC_OK;
}
