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

// A slab of this launch's sequence range the merge may read: its sequence,
// block and row range agree with the problem, and its hq * row_count state
// rows lie inside the table.  (ls: the slab's sequence relative to the range.)
__device__ __forceinline__ bool slab_ok(const MergeParams& p, const Slab& sl, int ls) {
  if (ls < 0 || ls >= p.num_seqs || sl.block < 0 || sl.block >= p.max_blocks) return false;
  const int q_len = p.cu_q[ls + 1] - p.cu_q[ls];
  const int kv_len = p.cu_k[ls + 1] - p.cu_k[ls];
  return sl.block * p.block < kv_len && sl.row_begin == first_row_of_block(sl.block, p.block, q_len, kv_len) &&
         sl.row_count == q_len - sl.row_begin && sl.offset >= 0 &&
         sl.offset <= p.n_pairs - static_cast<int64_t>(p.hq) * sl.row_count;
}

// One CTA: index[s][b] = slab id for the slabs of this launch's sequence
// range, then check every valid slab owns its slot (a slab that fails
// slab_ok is reported and never indexed, so its block counts as missing
// unless another slab supplies it).  Slabs of other ranges of the call are
// left to those ranges' launches; a sequence id outside the call is bad.
__global__ void __launch_bounds__(1024) rlk_merge_index_kernel(const __grid_constant__ MergeParams p) {
  const int n_idx = p.num_seqs * p.max_blocks;
  for (int i = threadIdx.x; i < n_idx; i += blockDim.x) p.index[i] = -1;
  __syncthreads();
  for (int64_t sid = threadIdx.x; sid < p.n_slabs; sid += blockDim.x) {
    const Slab sl = p.slabs[sid];
    const int ls = sl.seq - p.seq_base;
    if (sl.seq < 0 || sl.seq >= p.total_seqs) report_error(p.err, kErrBadSlab, 0x501);
    else if (ls < 0 || ls >= p.num_seqs) continue;
    else if (slab_ok(p, sl, ls)) p.index[ls * p.max_blocks + sl.block] = static_cast<int32_t>(sid);
    else report_error(p.err, kErrBadSlab, 0x501);
  }
  __syncthreads();
  for (int64_t sid = threadIdx.x; sid < p.n_slabs; sid += blockDim.x) {
    const Slab sl = p.slabs[sid];
    const int ls = sl.seq - p.seq_base;
    if (slab_ok(p, sl, ls) && p.index[ls * p.max_blocks + sl.block] != static_cast<int32_t>(sid))
      report_error(p.err, kErrDuplicateBlock, 0x502);
  }
}

// Four threads per (query row, head) pair, eight heads of one row per warp:
// thread q of a pair holds elements 16m + 4q .. 16m + 4q + 3 (m = 0..7), so
// a pair's four threads move 64 contiguous bytes per instruction, and each
// thread follows its pair's fold coefficients itself (the coefficient chain
// is serial per pair; a quarter of a row per thread keeps it cheap).  The
// warp's pairs share the row's blocks: lane j resolves the slab of block
// b0 + j for all of them.  State rows stream through a per-thread ring of
// asynchronous copies into shared memory (kMergeStages deep), so two blocks
// per pair are in flight while one folds; a thread reads only its own slots.
constexpr int kMergeHeadsPerWarp = 8;
constexpr int kMergeThreads = 256;
constexpr int kMergeStages = 3;
constexpr int kMergeSmem = kMergeStages * (8 * kMergeThreads * 16 + kMergeThreads * 4);

__global__ void __launch_bounds__(kMergeThreads, 2) rlk_merge_fold_kernel(const __grid_constant__ MergeParams p) {
  extern __shared__ __align__(16) uint8_t msm[];
  float4* ring = reinterpret_cast<float4*>(msm);  // [stage][m][thread]
  float* lring = reinterpret_cast<float*>(msm + kMergeStages * 8 * kMergeThreads * 16);  // [stage][thread]
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int sub = lane >> 2;  // pair within the warp
  const int qq = lane & 3;    // element quarter
  const int chunks = (p.hq + kMergeHeadsPerWarp - 1) / kMergeHeadsPerWarp;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t total = p.total_rows * chunks;
  // issue the copies of one state row quarter (and its lse) into ring slot st;
  // a missing state gets lse = -inf and no data (the fold skips it)
  auto issue = [&](int64_t pr, int st) {
    if (pr >= 0) {
      const float4* src = reinterpret_cast<const float4*>(p.state_o + pr * kHeadDim) + qq;
#pragma unroll
      for (int m = 0; m < 8; ++m) cp_async16(&ring[(st * 8 + m) * kMergeThreads + tid], src + 4 * m);
      cp_async4(&lring[st * kMergeThreads + tid], p.state_lse + pr);
    } else {
      lring[st * kMergeThreads + tid] = -INFINITY;
    }
  };
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (tid >> 5); w < total; w += warps) {
    const int64_t tok = w / chunks;
    const int h = static_cast<int>(w - tok * chunks) * kMergeHeadsPerWarp + sub;
    const bool hv = h < p.hq;  // lanes past the last head take part in the warp's shuffles only
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
    float4 O[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) O[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    bool bad = false;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      // lane j: the slab of block b0 + j (same for every head of the row)
      int64_t my_off = 0;
      int my_rb = 0, my_rc = 0;
      bool my_ok = false;
      const int b = b0 + lane;
      if (b < nb) {
        const int sid = p.index[s * p.max_blocks + b];
        if (sid >= 0) {
          const Slab sl = p.slabs[sid];
          const int r = i - sl.row_begin;
          if (r >= 0 && r < sl.row_count) {
            my_off = sl.offset;
            my_rb = sl.row_begin;
            my_rc = sl.row_count;
            my_ok = true;
          }
        }
      }
      if (__any_sync(0xffffffffu, b < nb && !my_ok)) bad = true;
      const int n_here = min(32, nb - b0);
      // state pair of this thread's head for block b0 + j (-1: none)
      auto pair_of = [&](int j) -> int64_t {
        const int64_t off = __shfl_sync(0xffffffffu, my_off, j);
        const int rb = __shfl_sync(0xffffffffu, my_rb, j);
        const int rc = __shfl_sync(0xffffffffu, my_rc, j);
        const bool ok = __shfl_sync(0xffffffffu, my_ok, j);
        return (ok && hv) ? off + static_cast<int64_t>(h) * rc + (i - rb) : -1;
      };
      // prologue: blocks 0 and 1 of the group in flight
#pragma unroll
      for (int j = 0; j < kMergeStages - 1; ++j) {
        if (j < n_here) issue(pair_of(j), j);
        cp_async_commit();
      }
      for (int j = 0; j < n_here; ++j) {
        const int jn = j + kMergeStages - 1;
        if (jn < n_here) issue(pair_of(jn), jn % kMergeStages);
        cp_async_commit();
        cp_async_wait<kMergeStages - 1>();  // this thread's copies of block j have landed
        const int st = j % kMergeStages;
        const float lc = lring[st * kMergeThreads + tid];
        if (lc != -INFINITY) {
          if (L == -INFINITY) {
#pragma unroll
            for (int m = 0; m < 8; ++m) O[m] = ring[(st * 8 + m) * kMergeThreads + tid];
            L = lc;
          } else {
            float Lp, alpha, beta;
            fold_coeffs(L, lc, Lp, alpha, beta);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const float4 c = ring[(st * 8 + m) * kMergeThreads + tid];
              O[m].x = fold_elem(O[m].x, c.x, alpha, beta);
              O[m].y = fold_elem(O[m].y, c.y, alpha, beta);
              O[m].z = fold_elem(O[m].z, c.z, alpha, beta);
              O[m].w = fold_elem(O[m].w, c.w, alpha, beta);
            }
            L = Lp;
          }
        }
      }
      cp_async_wait<0>();  // no copy outlives the group (the ring is reused)
    }
    if (!hv) continue;
    if (bad) {
      if (lane == 0) report_error(p.err, kErrMissingBlock, 0x503);
#pragma unroll
      for (int m = 0; m < 8; ++m) O[m] = make_float4(NAN, NAN, NAN, NAN);
      L = NAN;
    }
    const int64_t row = tok * p.hq + h;
    if (p.out_f32) {
      float4* dst = reinterpret_cast<float4*>(p.out_f32 + row * kHeadDim) + qq;
#pragma unroll
      for (int m = 0; m < 8; ++m) dst[4 * m] = O[m];
    }
    if (p.out_bf16) {
      uint2* dst = reinterpret_cast<uint2*>(p.out_bf16 + row * kHeadDim) + qq;
#pragma unroll
      for (int m = 0; m < 8; ++m) dst[4 * m] = make_uint2(pack_bf16x2(O[m].x, O[m].y), pack_bf16x2(O[m].z, O[m].w));
    }
    if (p.lse && qq == 0) p.lse[row] = L;
  }
}

cudaError_t configure_merge_kernels() {
  return cudaFuncSetAttribute(rlk_merge_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSmem);
}

cudaError_t launch_merge(const MergeParams& p, int num_sms, cudaStream_t stream) {
  rlk_merge_index_kernel<<<1, 1024, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = p.total_rows * ((p.hq + kMergeHeadsPerWarp - 1) / kMergeHeadsPerWarp);
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 2;  // 2 CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  rlk_merge_fold_kernel<<<static_cast<int>(blocks), kMergeThreads, kMergeSmem, stream>>>(p);
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

// Device address of the scratch array on the current device.  (In host code
// the array's name is only a host-side stand-in; the kernels must receive
// this address.)  The library looks it up once per device, with that device
// current, in its per-device set-up.
cudaError_t merge_noalloc_scratch(int32_t** ptr, int64_t* entries) {
  void* a = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&a, g_merge_index_scratch);
  if (e != cudaSuccess) return e;
  *ptr = static_cast<int32_t*>(a);
  *entries = kNoAllocIndexEntries;
  return cudaSuccess;
}

}  // namespace rlk
