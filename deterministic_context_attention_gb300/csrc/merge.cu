// merge.cu -- canonical merge of a partial-state table (HBM-bound).
//
// The table holds states (o_b, lse_b, b) produced by any number of logical CP
// ranks, in any arrival order.  The merge first sorts them by
// global_block_index -- a counting sort of slab ids into an index
// [sequence][block] -- and then folds every (row, head) left to right in
// ascending block order with the canonical fold, writing out (FP32 and/or
// BF16, downcast only here) and lse ("WS2 Attention PR5 Drift Benchmark",
// Transformer Engine Reuse: build states, sort by global_block_index, apply
// the correction arithmetic; Report Contract: merge order global_block_index,
// downcast at final write).  No atomics touch a result; a duplicate or
// missing block is reported through the device error word.
#include <cuda_runtime.h>

#include "numerics.cuh"
#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {

// Rows needing block b of sequence s: rows i with kv_len - q_len + i >= b*B.
__device__ __forceinline__ int first_row_of_block(int b, int B, int q_len, int kv_len) {
  return max(0, b * B - (kv_len - q_len));
}

// One CTA: index[s][b] = slab id, then check every slab owns its slot.
__global__ void __launch_bounds__(1024) rlk_merge_index_kernel(const __grid_constant__ MergeParams p) {
  const int n_idx = p.num_seqs * p.max_blocks;
  for (int i = threadIdx.x; i < n_idx; i += blockDim.x) p.index[i] = -1;
  __syncthreads();
  for (int64_t sid = threadIdx.x; sid < p.n_slabs; sid += blockDim.x) {
    const Slab sl = p.slabs[sid];
    bool ok = sl.seq >= 0 && sl.seq < p.num_seqs && sl.block >= 0 && sl.block < p.max_blocks;
    if (ok) {
      const int q_len = p.cu_q[sl.seq + 1] - p.cu_q[sl.seq];
      const int kv_len = p.cu_k[sl.seq + 1] - p.cu_k[sl.seq];
      ok = sl.block * p.block < kv_len &&
           sl.row_begin == first_row_of_block(sl.block, p.block, q_len, kv_len) &&
           sl.row_count == q_len - sl.row_begin && sl.offset >= 0;
    }
    if (ok) p.index[sl.seq * p.max_blocks + sl.block] = static_cast<int32_t>(sid);
    else report_error(p.err, kErrBadSlab, 0x501);
  }
  __syncthreads();
  for (int64_t sid = threadIdx.x; sid < p.n_slabs; sid += blockDim.x) {
    const Slab sl = p.slabs[sid];
    if (sl.seq >= 0 && sl.seq < p.num_seqs && sl.block >= 0 && sl.block < p.max_blocks &&
        p.index[sl.seq * p.max_blocks + sl.block] != static_cast<int32_t>(sid))
      report_error(p.err, kErrDuplicateBlock, 0x502);
  }
}

// One warp per (query row, head); lane l holds elements 4l..4l+3.
__global__ void __launch_bounds__(256) rlk_merge_fold_kernel(const __grid_constant__ MergeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t total = p.total_rows * p.hq;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
       w += warps) {
    const int64_t tok = w / p.hq;
    const int h = static_cast<int>(w - tok * p.hq);
    int s = 0;
    {  // sequence of packed row tok
      int lo = 0, hi = p.num_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cu_q[mid] <= tok) lo = mid; else hi = mid - 1;
      }
      s = lo;
    }
    const int q_len = p.cu_q[s + 1] - p.cu_q[s];
    const int kv_len = p.cu_k[s + 1] - p.cu_k[s];
    const int i = static_cast<int>(tok - p.cu_q[s]);
    const int pos = kv_len - q_len + i;
    const int nb = pos / p.block + 1;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    bool bad = false;
    // Blocks are visited in groups of 32: lane j resolves block b0 + j (slab,
    // pair, lse) and the group's state rows are then streamed in order.
    for (int b0 = 0; b0 < nb; b0 += 32) {
      int64_t my_pair = -1;
      float my_lse = -INFINITY;
      const int b = b0 + lane;
      if (b < nb) {
        const int sid = p.index[s * p.max_blocks + b];
        if (sid >= 0) {
          const Slab sl = p.slabs[sid];
          const int r = i - sl.row_begin;
          if (r >= 0 && r < sl.row_count) {
            my_pair = sl.offset + static_cast<int64_t>(h) * sl.row_count + r;
            my_lse = p.state_lse[my_pair];
          }
        }
      }
      if (__any_sync(0xffffffffu, b < nb && my_pair < 0)) bad = true;
      const int n_here = min(32, nb - b0);
      int64_t pair = __shfl_sync(0xffffffffu, my_pair, 0);
      float4 cur = make_float4(0.f, 0.f, 0.f, 0.f);
      if (pair >= 0) cur = *reinterpret_cast<const float4*>(p.state_o + pair * kHeadDim + 4 * lane);
      for (int j = 0; j < n_here; ++j) {
        const float lb = __shfl_sync(0xffffffffu, my_lse, j);
        float4 nxt = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j + 1 < n_here) {
          const int64_t np = __shfl_sync(0xffffffffu, my_pair, j + 1);
          if (np >= 0) nxt = *reinterpret_cast<const float4*>(p.state_o + np * kHeadDim + 4 * lane);
        }
        if (lb != -INFINITY) {
          if (L == -INFINITY) {
            O = cur;
            L = lb;
          } else {
            float Lp, alpha, beta;
            fold_coeffs(L, lb, Lp, alpha, beta);
            O.x = fold_elem(O.x, cur.x, alpha, beta);
            O.y = fold_elem(O.y, cur.y, alpha, beta);
            O.z = fold_elem(O.z, cur.z, alpha, beta);
            O.w = fold_elem(O.w, cur.w, alpha, beta);
            L = Lp;
          }
        }
        cur = nxt;
      }
    }
    if (bad) {
      if (lane == 0) report_error(p.err, kErrMissingBlock, 0x503);
      O = make_float4(NAN, NAN, NAN, NAN);
      L = NAN;
    }
    const int64_t row = tok * p.hq + h;
    if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + row * kHeadDim + 4 * lane) = O;
    if (p.out_bf16)
      *reinterpret_cast<uint2*>(p.out_bf16 + row * kHeadDim + 4 * lane) =
          make_uint2(pack_bf16x2(O.x, O.y), pack_bf16x2(O.z, O.w));
    if (p.lse && lane == 0) p.lse[row] = L;
  }
}

cudaError_t launch_merge(const MergeParams& p, int num_sms, cudaStream_t stream) {
  rlk_merge_index_kernel<<<1, 1024, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = p.total_rows * p.hq;
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // 8 CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  rlk_merge_fold_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace rlk

// ---------------------------------------------------------------- no-alloc variant
// Scratch for callers that cannot allocate device memory: the merge's
// (sequence, block) -> slab index lives in this file-scope array instead of a
// caller-supplied workspace.  Every GPU that loads the library holds it until
// the process exits.
namespace rlk {

static __device__ __align__(256) int32_t g_merge_index_scratch[kNoAllocIndexEntries];

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  (In host code the array's name is
// only a host-side stand-in; the kernels must receive this address.)
cudaError_t merge_noalloc_scratch(int32_t** ptr, int64_t* entries) {
  static int32_t* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!addr[dev]) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_merge_index_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<int32_t*>(a);
  }
  *ptr = addr[dev];
  *entries = kNoAllocIndexEntries;
  return cudaSuccess;
}

}  // namespace rlk
