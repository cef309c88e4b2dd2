// rope.cu -- rotary position embedding of packed BF16 rows [T, H, 128].
//
// The pages compose RoPE before attention, the attention reading post-RoPE
// Q/K, and require decode replay to keep cache, position and RoPE identical
// to prefill ("WS2 Attention PR5 Drift Benchmark", Scope; "[WS2][Attention]
// H100 validation and reproduction guide", PR stack: decode KV-cache replay
// and cache/position/RoPE identity).  Canonical form (the same in every
// kernel that rotates, so a row's bits depend only on its values and
// position): rotate-half pairs (i, i + 64); c, s from the FP32 table the host
// builds (cos / sin of p * theta^(-2i/128) in double, one rounding each);
//   y_i      = bf16_rn(fma(x_i, c, -(x_{i+64} * s)))
//   y_{i+64} = bf16_rn(fma(x_{i+64}, c, x_i * s))
// with the products rounded to FP32 on their own.
//
// The pass is HBM-bound: 256 B read and 256 B written per (token, head) row;
// the table (512 B per position) stays in L2.  A thread takes 8 pairs of one
// row -- 16 B from each half, so a warp reads four rows' halves as whole
// 128-byte lines -- and the grid strides over rows.
#include <cuda_runtime.h>

#include <algorithm>

#include "numerics.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kRopeThreads = 256;

// Rotate the 8 pairs held in a (first half) and b (second half).
__device__ __forceinline__ void rope8(uint4& a, uint4& b, const float4& c0, const float4& c1, const float4& s0,
                                      const float4& s1) {
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  rope_words8(a, b, c, s);
}

__global__ void __launch_bounds__(kRopeThreads) rlk_rope_kernel(const __grid_constant__ RopeParams p) {
  __shared__ int32_t s_cu[kMaxSeqs + 1];
  __shared__ int32_t s_pos0[kMaxSeqs];
  for (int i = threadIdx.x; i <= p.num_seqs; i += blockDim.x) s_cu[i] = p.cu[i];
  for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) s_pos0[i] = p.pos0[i];
  __syncthreads();
  const int64_t units1 = p.rows * 8, units = units1 + p.rows2 * 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units; u += stride) {
    // units of the first tensor, then of the second
    const bool second = u >= units1;
    const int64_t uu = second ? u - units1 : u;
    const int heads = second ? p.heads2 : p.heads;
    const int64_t row = uu >> 3;
    const int j = static_cast<int>(uu & 7);
    const int tok = static_cast<int>(row / heads);
    // the sequence holding tok: the last s with cu[s] <= tok (empty
    // sequences share their start with the next one)
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_cu[mid] <= tok) lo = mid;
      else hi = mid - 1;
    }
    const int pos = s_pos0[lo] + (tok - s_cu[lo]);
    const uint4* xr = reinterpret_cast<const uint4*>((second ? p.x2 : p.x) + row * kHeadDim);
    uint4 a = xr[j], b = xr[8 + j];
    const float4* t = reinterpret_cast<const float4*>(p.table + static_cast<int64_t>(pos) * kHeadDim);
    const float4 c0 = __ldg(t + 2 * j), c1 = __ldg(t + 2 * j + 1);
    const float4 s0 = __ldg(t + 16 + 2 * j), s1 = __ldg(t + 16 + 2 * j + 1);
    rope8(a, b, c0, c1, s0, s1);
    const int64_t ys = (second || p.y_stride == 0) ? kHeadDim : p.y_stride;
    uint4* yr = reinterpret_cast<uint4*>((second ? p.y2 : p.y) + row * ys);
    yr[j] = a;
    yr[8 + j] = b;
  }
}

}  // namespace

cudaError_t launch_rope(const RopeParams& p, int num_sms, cudaStream_t stream) {
  const int64_t units = (p.rows + p.rows2) * 8;
  if (units == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((units + kRopeThreads - 1) / kRopeThreads, static_cast<int64_t>(num_sms) * 16);
  rlk_rope_kernel<<<static_cast<int>(blocks), kRopeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace rlk
