// bwd.cu -- deterministic backward of causal GQA attention for sm_103a.
//
// Three kernels, one stream, no atomics on any result:
//   preprocess  Delta_i = sum_d dout_id * out_id (fixed order), written with
//               lse transposed to [Hq][T] for coalesced per-block reads;
//   dK/dV       one CTA per (sequence, KV head g, KV block j).  For query
//               blocks i = j .. last in ascending order, and within each for
//               the query heads of group g in ascending order, it recomputes
//               S^T = K_j Q_i^T and dP^T = V_j dO_i^T on the tensor core, forms
//               P^T = exp(S^T - lse) and dS^T = P^T (dP^T - Delta), and
//               accumulates dV += P^T dO and dK += dS^T Q in TMEM (FP32), with
//               P^T and dS^T each split into BF16 hi + lo parts;
//   dQ          one CTA per (sequence, query head, query block i): for KV
//               blocks j = 0 .. i ascending, S = Q_i K_j^T, dP = dO_i V_j^T,
//               dS as above, dQ += dS K_j in TMEM.
// The reduction order of every dK/dV/dQ element is therefore fixed by the
// block decomposition alone, so the result is bitwise identical across
// logical CP ranks and repeated runs ("[WS2][Attention] H100 validation and
// reproduction guide", Acceptance: dQ/dK/dV max abs 0.0 at 2/4/8 ranks;
// "WS2 Attention PR5 Drift Benchmark", Scope: optional backward dq, dk, dv).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <memory>
#include <type_traits>
#include <vector>

#include "../../include/rlk_attn.h"
#include "numerics.cuh"
#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {


constexpr float kLog2e = 1.44269504088896340736f;

struct alignas(16) BwdItem {
  int32_t seq;
  int32_t head;   // dK/dV: KV head g; dQ: query head h
  int32_t block;  // dK/dV: KV block j; dQ: first row of the query tile
  int32_t rows;   // dQ: rows of the tile written; dK/dV: unused
};

constexpr int kMaxBwdTiles = 1800;

// The item list holds tiles; item i is head i mod item_heads of tile
// i / item_heads (the heads of a tile are adjacent in the longest-first
// order), so a launch takes kMaxBwdTiles * heads items.
struct BwdParams {
  ErrWord* err;
  int32_t hq, hkv, group, num_items;
  int32_t item_heads, pad0;
  int64_t t_pad;        // row stride of the transposed lse / Delta
  float scale, scale_log2;
  const float* lse_t;   // [hq][t_pad]
  const float* delta_t; // [hq][t_pad]
  float* dq;
  float* dk;
  float* dv;
  int32_t cu[kMaxSeqs + 1];
  BwdItem items[kMaxBwdTiles];
};

__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int item) {
  const int t = item / p.item_heads;
  BwdItem it = p.items[t];
  it.head = item - t * p.item_heads;
  return it;
}

// ------------------------------------------------------------------ preprocess
struct PrepParams {
  int32_t hq;
  int64_t rows, t_pad;
  const float* out;
  const uint16_t* dout;
  const float* lse;
  float* lse_t;
  float* delta_t;
};

// One warp per (row, head): lane l takes elements 4l..4l+3 (fma in order),
// then a fixed xor butterfly.
__global__ void __launch_bounds__(256) rlk_bwd_prep_kernel(const __grid_constant__ PrepParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * 8;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); w < p.rows * p.hq; w += warps) {
    const int64_t row = w / p.hq;
    const int h = static_cast<int>(w - row * p.hq);
    const float4 o = *reinterpret_cast<const float4*>(p.out + w * kHeadDim + 4 * lane);
    const uint2 d = *reinterpret_cast<const uint2*>(p.dout + w * kHeadDim + 4 * lane);
    float acc = __fmul_rn(bf16_lo_as_f32(d.x), o.x);
    acc = __fmaf_rn(bf16_hi_as_f32(d.x), o.y, acc);
    acc = __fmaf_rn(bf16_lo_as_f32(d.y), o.z, acc);
    acc = __fmaf_rn(bf16_hi_as_f32(d.y), o.w, acc);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    if (lane == 0) {
      p.delta_t[static_cast<int64_t>(h) * p.t_pad + row] = acc;
      p.lse_t[static_cast<int64_t>(h) * p.t_pad + row] = p.lse[w];
    }
  }
}

// ------------------------------------------------------------------ shared layout
template <int KIND>
struct BwdLayoutT {
  static constexpr int kTile = 128 * kHeadDim * 2;  // one 128 x 128 BF16 tile (two 64-column halves)
  static constexpr int kHalf = 128 * 128;
  static constexpr int kResOff = 0;                 // resident pair (K_j,V_j) or (Q_i,dO_i)
  static constexpr int kStreamOff = 2 * kTile;
  // dK/dV: two stages of the streamed pair (Q_i, dO_i).  dQ: K_j in a ring of
  // three slots (read by S and by the accumulation) and V_j in a ring of two
  // (read by dP only): step t + 1's K loads into the slot of step t - 2,
  // released by that step's accumulation, while steps t - 1 and t may still
  // read theirs, so the load waits for no accumulation of the last two steps.
  static constexpr int kStages = 2, kKSlots = 3, kVSlots = 2;
  static constexpr int kVOff = kStreamOff + kKSlots * kTile;  // dQ
  static constexpr int kStreamBytes = KIND == 0 ? kStages * 2 * kTile : (kKSlots + kVSlots) * kTile;
  // per-warp copies of a step's column statistics (dK/dV): [buf 2][warp 8][lse2, Delta][64] floats
  static constexpr int kVecOff = kStreamOff + kStreamBytes;
  static constexpr int kVecBytes = KIND == 0 ? 2 * 8 * 2 * 64 * 4 : 0;
  static constexpr int kBarOff = kVecOff + kVecBytes;
  // barriers; S/dP and P/dS barriers come in pairs, one per 64-column half of a step
  // (dQ's P/dS pair is double-buffered by step parity: kPFull + 2 (s & 1) + c)
  static constexpr int kResFull = 0, kResEmpty = 1, kStFull = 2, kStEmpty = 5, kVEmpty = 8, kSFull = 10, kPFull = 12,
                       kAccFull = 16, kAccEmpty = 17, kSDPRead = 18, kNumBars = 19;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kTotal = kMiscOff + 16;
  static constexpr int kAlloc = kTotal + 1024;
};
using BwdLayout = BwdLayoutT<0>;
static_assert(BwdLayoutT<1>::kAlloc <= 227 * 1024, "dQ shared memory");

__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int k) {  // K-major operand, K-step k (16 elements)
  return sdesc_sw128(tile + (k >> 2) * BwdLayout::kHalf + (k & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int k) {  // MN-major operand, K-step k (16 rows)
  return sdesc_sw128(tile + k * 16 * 128, BwdLayout::kHalf, 1024);
}

// Per-element backward arithmetic of both kernels (one rounding per step):
//   p  = 2^fma(s, scale_log2, -lse log2 e)     (0 where masked)
//   ds = p * (dp - Delta)
// KIND 0: dK/dV (rows = keys of block j, columns = query rows);
// KIND 1: dQ    (rows = query rows,       columns = keys of block j).
template <int KIND>
__global__ void __launch_bounds__(384, 1)
    rlk_bwd_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_do) {
  using L = BwdLayoutT<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  float* vecs = reinterpret_cast<float*>(smem + L::kVecOff);  // [buf][warp][lse2, delta][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bars[L::kResFull], 1);
    mbar_init(&bars[L::kResEmpty], 1);
    for (int s = 0; s < L::kKSlots; ++s) {  // dK/dV uses the first kStages of them
      mbar_init(&bars[L::kStFull + s], 1);
      mbar_init(&bars[L::kStEmpty + s], 1);
    }
    for (int s = 0; s < L::kVSlots; ++s) mbar_init(&bars[L::kVEmpty + s], 1);
    for (int h = 0; h < 2; ++h) mbar_init(&bars[L::kSFull + h], 1);
    for (int h = 0; h < 4; ++h) mbar_init(&bars[L::kPFull + h], 256);  // the eight elementwise warps
    mbar_init(&bars[L::kAccFull], 1);
    mbar_init(&bars[L::kAccEmpty], 256);
    mbar_init(&bars[L::kSDPRead], 256);  // dQ: the eight elementwise warps have read dP
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s = tmem, tm_dp = tmem + 128, tm_acc0 = tmem + 256, tm_acc1 = tmem + 384;
  // dQ: S (then dS over it) and dP rotate through three 128-column areas
  // (the fourth holds the accumulator): step s puts S in area s mod 3 and
  // dP in area (s + 1) mod 3
  auto dq_area = [&](uint32_t i) { return tmem + (i == 2 ? 384u : 128u * i); };
  const uint32_t res_addr = smem_u32(smem + L::kResOff);
  uint8_t* st_base = smem + L::kStreamOff;

  // steps of an item: dK/dV: (query block i from j to the last) x (heads of the
  // group); dQ: KV blocks 0 .. last of the tile.
  auto item_steps = [&](const BwdItem& it, int& len, int& nsteps) {
    len = p.cu[it.seq + 1] - p.cu[it.seq];
    if (KIND == 0) {
      const int nq = (len + 127) / 128;
      nsteps = (nq - it.block) * p.group;
    } else {
      nsteps = (it.block + it.rows - 1) / 128 + 1;
    }
  };

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    uint32_t res_it = 0, st_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int g_ = static_cast<int>(gridDim.x), c_ = static_cast<int>(blockIdx.x);
      const int item = round * g_ + ((round & 1) ? g_ - 1 - c_ : c_);  // snake order over the longest-first list
      if (item >= p.num_items) continue;
      const BwdItem it = bwd_item(p, item);
      int len, nsteps;
      item_steps(it, len, nsteps);
      const int tok0 = p.cu[it.seq];
      bool ok = mbar_wait(&bars[L::kResEmpty], (res_it & 1) ^ 1, abort, p.err, 0x601);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[L::kResFull], 2 * L::kTile);
        uint8_t* a = smem + L::kResOff;
        if (KIND == 0) {
          const int r = tok0 + it.block * 128;
          tma_load_3d(a, &tm_k, &bars[L::kResFull], 0, it.head, r);
          tma_load_3d(a + L::kHalf, &tm_k, &bars[L::kResFull], 64, it.head, r);
          tma_load_3d(a + L::kTile, &tm_v, &bars[L::kResFull], 0, it.head, r);
          tma_load_3d(a + L::kTile + L::kHalf, &tm_v, &bars[L::kResFull], 64, it.head, r);
        } else {
          const int r = tok0 + it.block;
          tma_load_3d(a, &tm_q, &bars[L::kResFull], 0, it.head, r);
          tma_load_3d(a + L::kHalf, &tm_q, &bars[L::kResFull], 64, it.head, r);
          tma_load_3d(a + L::kTile, &tm_do, &bars[L::kResFull], 0, it.head, r);
          tma_load_3d(a + L::kTile + L::kHalf, &tm_do, &bars[L::kResFull], 64, it.head, r);
        }
      }
      ++res_it;
      for (int t = 0; t < nsteps; ++t) {
        if (KIND == 1) {
          // K_j into slot t mod 3 (free once the accumulation of the step
          // three back is done), V_j into slot t mod 2 (free once the dP of
          // the step two back is done); both land on the K slot's barrier
          const uint32_t ks = st_it % L::kKSlots, vs = st_it % L::kVSlots;
          ok = mbar_wait(&bars[L::kStEmpty + ks], ((st_it / L::kKSlots) & 1) ^ 1, abort, p.err, 0x602);
          ok = ok && mbar_wait(&bars[L::kVEmpty + vs], ((st_it / L::kVSlots) & 1) ^ 1, abort, p.err, 0x607);
          if (!__all_sync(0xffffffffu, ok)) break;
          if (lane == 0) {
            uint8_t* dk = st_base + ks * L::kTile;
            uint8_t* dvs = smem + L::kVOff + vs * L::kTile;
            const int g = it.head / p.group;
            const int r = tok0 + t * 128;
            mbar_arrive_expect_tx(&bars[L::kStFull + ks], 2 * L::kTile);
            tma_load_3d(dk, &tm_k, &bars[L::kStFull + ks], 0, g, r);
            tma_load_3d(dk + L::kHalf, &tm_k, &bars[L::kStFull + ks], 64, g, r);
            tma_load_3d(dvs, &tm_v, &bars[L::kStFull + ks], 0, g, r);
            tma_load_3d(dvs + L::kHalf, &tm_v, &bars[L::kStFull + ks], 64, g, r);
          }
          ++st_it;
          continue;
        }
        const uint32_t stage = st_it % L::kStages;
        ok = mbar_wait(&bars[L::kStEmpty + stage], ((st_it / L::kStages) & 1) ^ 1, abort, p.err, 0x602);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane == 0) {
          uint8_t* d = st_base + stage * 2 * L::kTile;
          mbar_arrive_expect_tx(&bars[L::kStFull + stage], 2 * L::kTile);
          if (KIND == 0) {
            const int i = it.block + t / p.group;
            const int h = it.head * p.group + t % p.group;
            const int r = tok0 + i * 128;
            tma_load_3d(d, &tm_q, &bars[L::kStFull + stage], 0, h, r);
            tma_load_3d(d + L::kHalf, &tm_q, &bars[L::kStFull + stage], 64, h, r);
            tma_load_3d(d + L::kTile, &tm_do, &bars[L::kStFull + stage], 0, h, r);
            tma_load_3d(d + L::kTile + L::kHalf, &tm_do, &bars[L::kStFull + stage], 64, h, r);
          } else {
            const int g = it.head / p.group;
            const int r = tok0 + t * 128;
            tma_load_3d(d, &tm_k, &bars[L::kStFull + stage], 0, g, r);
            tma_load_3d(d + L::kHalf, &tm_k, &bars[L::kStFull + stage], 64, g, r);
            tma_load_3d(d + L::kTile, &tm_v, &bars[L::kStFull + stage], 0, g, r);
            tma_load_3d(d + L::kTile + L::kHalf, &tm_v, &bars[L::kStFull + stage], 64, g, r);
          }
        }
        ++st_it;
      }
      if (*abort) break;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // dK/dV: each step's S/dP is issued as two N = 64 halves (columns 0-63,
    // 64-127 of TMEM and of the step's query rows), so the elementwise step
    // of one half runs while the tensor core works on the other:
    //   S/dP_0(t) S/dP_1(t) | acc_0(t) S/dP_0(t+1) | acc_1(t) S/dP_1(t+1) | ...
    // where acc_c takes K-steps 4c..4c+3 (hi, then lo) of dV and dK.  The
    // tensor core runs them in issue order, so S/dP_c(t+1) overwrites the
    // half only after acc_c(t) has read it.  dQ issues S/dP whole (below).
    constexpr uint32_t kIdK = idesc_bf16(128, 64, false, false);   // both operands K-major, N = 64
    constexpr uint32_t kIdMN = idesc_bf16(128, 128, false, true);  // A in TMEM, B MN-major
    uint32_t res_it = 0, st_it = 0, s_it = 0, acc_it = 0;
    // the whole warp walks the K-steps (warp-uniform descriptors) and the
    // elected lane issues each MMA: a lone lane in a divergent branch issues
    // them slower than the tensor core runs them
    const uint32_t leader = elect_one_sync();
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int g_ = static_cast<int>(gridDim.x), c_ = static_cast<int>(blockIdx.x);
      const int item = round * g_ + ((round & 1) ? g_ - 1 - c_ : c_);  // snake order over the longest-first list
      if (item >= p.num_items) continue;
      const BwdItem it = bwd_item(p, item);
      int len, nsteps;
      item_steps(it, len, nsteps);
      bool ok = mbar_wait(&bars[L::kResFull], res_it & 1, abort, p.err, 0x611);
      if (!__all_sync(0xffffffffu, ok)) break;
      ++res_it;
      // S^T|S and dP^T|dP of half c of step t (stream stage of step t)
      auto issue_sdp = [&](uint32_t st_addr, int c) {
        const uint32_t boff = static_cast<uint32_t>(c) * 64 * 128;  // rows 64c.. of the streamed tiles
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (leader) umma_ss(tm_s + 64 * c, kdesc(res_addr, k), kdesc(st_addr + boff, k), kIdK, k > 0);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (leader)
            umma_ss(tm_dp + 64 * c, kdesc(res_addr + L::kTile, k), kdesc(st_addr + L::kTile + boff, k), kIdK, k > 0);
        if (leader) umma_commit(&bars[L::kSFull + c]);
        __syncwarp();
      };
      // dK/dV: K-steps 4c..4c+3 of the accumulators (first: the item's first product)
      auto issue_acc = [&](uint32_t st_addr, int c, bool first) {
        const int k0 = 4 * c;
        if (KIND == 0) {
          // dV += P^T dO ; dK += dS^T Q   (B operands MN-major: N = D, K = query rows)
#pragma unroll
          for (int k = k0; k < k0 + 4; ++k)
            if (leader)
              umma_ts(tm_acc0, tm_s + 16 * k, mndesc(st_addr + L::kTile, k), kIdMN, (first && k == k0) ? 0u : 1u);
#pragma unroll
          for (int k = k0; k < k0 + 4; ++k)
            if (leader) umma_ts(tm_acc0, tm_s + 16 * k + 8, mndesc(st_addr + L::kTile, k), kIdMN, 1u);
#pragma unroll
          for (int k = k0; k < k0 + 4; ++k)
            if (leader) umma_ts(tm_acc1, tm_dp + 16 * k, mndesc(st_addr, k), kIdMN, (first && k == k0) ? 0u : 1u);
#pragma unroll
          for (int k = k0; k < k0 + 4; ++k)
            if (leader) umma_ts(tm_acc1, tm_dp + 16 * k + 8, mndesc(st_addr, k), kIdMN, 1u);
        }
        __syncwarp();
      };
      auto stage_addr = [&](uint32_t si) { return smem_u32(st_base + (si % L::kStages) * 2 * L::kTile); };
      bool fail = false;
      if constexpr (KIND == 1) {
        // dQ: one N = 128 S/dP per step.  Its single accumulator makes S/dP
        // the larger part of its tensor work, so N = 64 halves' lower MMA
        // rate would cost more than their overlap gains (measured 1.6 %
        // slower for the whole backward).  With the accumulator in 128 of
        // the 512 TMEM columns, S/dS and dP rotate through the other three
        // areas; step t + 1's S/dP overwrites only step t's dP and step
        // t - 1's dS, so it is issued as soon as the elementwise warps have
        // read step t's dP (their first act), ahead of step t's accumulation:
        //   S/dP(t+1) acc_0(t) acc_1(t) | S/dP(t+2) acc_0(t+1) acc_1(t+1) | ...
        // The elementwise warps can then run one step ahead of the waits on
        // their P/dS barriers, which are therefore kept per step parity.
        constexpr uint32_t kIdK128 = idesc_bf16(128, 128, false, false);
        auto k_slot = [&](uint32_t si) { return smem_u32(st_base + (si % L::kKSlots) * L::kTile); };
        auto v_slot = [&](uint32_t si) { return smem_u32(smem + L::kVOff + (si % L::kVSlots) * L::kTile); };
        auto issue_sdp128 = [&](uint32_t si, bool last, uint32_t s) {
          const uint32_t ts = dq_area(s % 3), tdp = dq_area((s + 1) % 3);
          const uint32_t ka = k_slot(si), va = v_slot(si);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (leader) umma_ss(ts, kdesc(res_addr, k), kdesc(ka, k), kIdK128, k > 0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (leader) umma_ss(tdp, kdesc(res_addr + L::kTile, k), kdesc(va, k), kIdK128, k > 0);
          if (leader) {
            umma_commit(&bars[L::kSFull]);
            umma_commit(&bars[L::kSFull + 1]);
            umma_commit(&bars[L::kVEmpty + si % L::kVSlots]);  // V_j is read by dP only
            if (last) umma_commit(&bars[L::kResEmpty]);  // the item's last S/dP: the resident pair is free
          }
          __syncwarp();
        };
        // dQ += dS K_j over K-steps 4c..4c+3, with dS in area tds and K_j at ka
        auto issue_acc_dq = [&](uint32_t ka, int c, bool first, uint32_t tds) {
          const int k0 = 4 * c;
#pragma unroll
          for (int k = k0; k < k0 + 4; ++k)
            if (leader) umma_ts(tm_acc0, tds + 16 * k, mndesc(ka, k), kIdMN, (first && k == k0) ? 0u : 1u);
#pragma unroll
          for (int k = k0; k < k0 + 4; ++k)
            if (leader) umma_ts(tm_acc0, tds + 16 * k + 8, mndesc(ka, k), kIdMN, 1u);
          __syncwarp();
        };
        {
          bool w = mbar_wait(&bars[L::kStFull + st_it % L::kKSlots], (st_it / L::kKSlots) & 1, abort, p.err, 0x613);
          if (!__all_sync(0xffffffffu, w)) break;
          tc_fence_after();
          issue_sdp128(st_it, nsteps == 1, s_it);
        }
        ok = mbar_wait(&bars[L::kAccEmpty], (acc_it & 1) ^ 1, abort, p.err, 0x612);
        if (!__all_sync(0xffffffffu, ok)) break;
        for (int t = 0; t < nsteps; ++t) {
          const uint32_t cur = st_it, nxt = st_it + 1;
          const bool more = t + 1 < nsteps;
          const uint32_t tds = dq_area(s_it % 3);
          const uint32_t pf = L::kPFull + 2 * (s_it & 1), pph = (s_it >> 1) & 1;
          // this step's dP has been read: the next step's S/dP goes into its
          // area and into that of the previous step's dS (read by
          // accumulations issued before it), ahead of this step's accumulation
          bool w = mbar_wait(&bars[L::kSDPRead], s_it & 1, abort, p.err, 0x616);
          if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
          if (more) {
            w = mbar_wait(&bars[L::kStFull + nxt % L::kKSlots], (nxt / L::kKSlots) & 1, abort, p.err, 0x615);
            if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
            tc_fence_after();
            issue_sdp128(nxt, t + 2 == nsteps, s_it + 1);
          }
          w = mbar_wait(&bars[pf], pph, abort, p.err, 0x614);
          if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
          tc_fence_after();
          issue_acc_dq(k_slot(cur), 0, t == 0, tds);
          w = mbar_wait(&bars[pf + 1], pph, abort, p.err, 0x614);
          if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
          tc_fence_after();
          issue_acc_dq(k_slot(cur), 1, false, tds);
          if (leader) {
            umma_commit(&bars[L::kStEmpty + cur % L::kKSlots]);  // K_j no longer read
            if (!more) umma_commit(&bars[L::kAccFull]);
          }
          __syncwarp();
          ++s_it;
          ++st_it;
        }
        if (fail) break;
        ++acc_it;
        continue;
      }
      {
        bool w = mbar_wait(&bars[L::kStFull + st_it % L::kStages], (st_it / L::kStages) & 1, abort, p.err, 0x613);
        if (!__all_sync(0xffffffffu, w)) break;
        tc_fence_after();
        issue_sdp(stage_addr(st_it), 0);
        issue_sdp(stage_addr(st_it), 1);
        if (nsteps == 1) {
          if (leader) umma_commit(&bars[L::kResEmpty]);  // the item's last S/dP: the resident pair is free
          __syncwarp();
        }
      }
      // the accumulators are free once the previous item's epilogue read them
      ok = mbar_wait(&bars[L::kAccEmpty], (acc_it & 1) ^ 1, abort, p.err, 0x612);
      if (!__all_sync(0xffffffffu, ok)) break;
      for (int t = 0; t < nsteps; ++t) {
        const uint32_t cur = st_it, nxt = st_it + 1;
        const bool more = t + 1 < nsteps;
        for (int c = 0; c < 2; ++c) {
          bool w = mbar_wait(&bars[L::kPFull + c], s_it & 1, abort, p.err, 0x614);
          if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
          tc_fence_after();
          issue_acc(stage_addr(cur), c, t == 0 && c == 0);
          if (c == 1 && leader) {
            umma_commit(&bars[L::kStEmpty + cur % L::kStages]);  // step t's stage is no longer read
            if (!more) umma_commit(&bars[L::kAccFull]);
          }
          __syncwarp();
          if (more) {
            if (c == 0) {
              w = mbar_wait(&bars[L::kStFull + nxt % L::kStages], (nxt / L::kStages) & 1, abort, p.err, 0x615);
              if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
              tc_fence_after();
            }
            issue_sdp(stage_addr(nxt), c);
            if (c == 1 && t + 2 == nsteps) {
              if (leader) umma_commit(&bars[L::kResEmpty]);  // the item's last S/dP: the resident pair is free
              __syncwarp();
            }
          }
        }
        if (fail) break;
        ++s_it;
        ++st_it;
      }
      if (fail) break;
      ++acc_it;
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ P / dS (+ epilogue)
    // The tensor core hands over the two column halves of a step one after
    // the other, and all eight warps work on each half in turn: warp w takes
    // TMEM lane quadrant w mod 4 and the 32 columns 64 c + 32 (w / 4) .. of
    // half c.  (Two warps per SMSP on every half: a single warp per SMSP is
    // latency-bound on the arithmetic.)  The epilogue splits the same way:
    // warps 0-3 write dV (dQ: columns 0-63), warps 4-7 dK (dQ: 64-127).
    const int wq = warp & 3, wh = warp >> 2;
    const int r = wq * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    uint32_t s_it = 0, acc_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int g_ = static_cast<int>(gridDim.x), c_ = static_cast<int>(blockIdx.x);
      const int item = round * g_ + ((round & 1) ? g_ - 1 - c_ : c_);  // snake order over the longest-first list
      if (item >= p.num_items) continue;
      const BwdItem it = bwd_item(p, item);
      int len, nsteps;
      item_steps(it, len, nsteps);
      const int tok0 = p.cu[it.seq];
      // dQ: this thread's row statistics are fixed for the item
      float row_lse2 = 0.f, row_delta = 0.f;
      int row_pos = 0;
      bool row_ok = false;
      if (KIND == 1) {
        row_pos = it.block + r;
        row_ok = r < it.rows && row_pos < len;
        if (row_ok) {
          const int64_t idx = static_cast<int64_t>(it.head) * p.t_pad + tok0 + row_pos;
          row_lse2 = __fmul_rn(p.lse_t[idx], kLog2e);
          row_delta = p.delta_t[idx];
        }
      }
      const int key_pos = (KIND == 0) ? it.block * 128 + r : 0;
      // dK/dV: the column statistics (lse, Delta of the step's query rows) of
      // this warp's columns in both halves, loaded one step ahead
      float nl[2] = {0.f, 0.f}, nd[2] = {0.f, 0.f};
      auto load_stats = [&](int t) {
        const int i = it.block + t / p.group;
        const int h = it.head * p.group + t % p.group;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int qp = i * 128 + 64 * c + 32 * wh + lane;
          const int64_t idx = static_cast<int64_t>(h) * p.t_pad + tok0 + qp;
          nl[c] = qp < len ? p.lse_t[idx] : 0.f;
          nd[c] = qp < len ? p.delta_t[idx] : 0.f;
        }
      };
      if (KIND == 0) load_stats(0);
      bool fail = false;
      for (int t = 0; t < nsteps; ++t) {
        float* vb = vecs + ((s_it & 1) * 8 + warp) * 128;  // [half][lse2 32, Delta 32] of this warp's columns
        int col0;  // position of column 0 of this step
        if (KIND == 0) {
          col0 = (it.block + t / p.group) * 128;
#pragma unroll
          for (int c = 0; c < 2; ++c) {  // each warp stages its own copy (warp-local sync only)
            vb[64 * c + lane] = __fmul_rn(nl[c], kLog2e);
            vb[64 * c + 32 + lane] = nd[c];
          }
          __syncwarp();
          if (t + 1 < nsteps) load_stats(t + 1);
        } else {
          col0 = t * 128;
        }
        const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
        const uint32_t ts_e = (KIND == 0) ? tm_s : dq_area(s_it % 3);
        const uint32_t tdp_e = (KIND == 0) ? tm_dp : dq_area((s_it + 1) % 3);
        const uint32_t tds_e = (KIND == 0) ? tm_dp : ts_e;  // dQ writes dS over S
        // dQ: both halves of S/dP complete together; dP of both is read
        // first, so the MMA warp can issue the next step's S/dP over it
        // while this step's P and dS are formed
        uint32_t dq_dp0[32], dq_dp1[32];
        if constexpr (KIND == 1) {
          bool w = mbar_wait(&bars[L::kSFull], s_it & 1, abort, p.err, 0x621);
          w = w && mbar_wait(&bars[L::kSFull + 1], s_it & 1, abort, p.err, 0x621);
          if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
          tc_fence_after();
          tmem_ld32(tdp_e + lane_off + 32 * wh, dq_dp0);
          tmem_ld32(tdp_e + lane_off + 64 + 32 * wh, dq_dp1);
          tmem_ld_wait(dq_dp0);
          tmem_ld_wait(dq_dp1);
          tc_fence_before();
          mbar_arrive(&bars[L::kSDPRead]);
        }
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          if (KIND == 0) {
            bool w = mbar_wait(&bars[L::kSFull + c], s_it & 1, abort, p.err, 0x621);
            if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
            tc_fence_after();
          }
          const int colc = 64 * c + 32 * wh;  // first column of this warp's 32
          // every element of this warp's columns is visible: no per-element mask
          bool full;
          if (KIND == 0)
            full = __all_sync(0xffffffffu, key_pos < len && col0 + colc + 31 < len && col0 + colc >= key_pos);
          else
            full = __all_sync(0xffffffffu, row_ok && col0 + colc + 31 <= row_pos);
          uint32_t sr[32], dr[32];
          tmem_ld32(ts_e + lane_off + colc, sr);
          if (KIND == 0) tmem_ld32(tdp_e + lane_off + colc, dr);
          tmem_ld_wait(sr);
          if (KIND == 0) {
            tmem_ld_wait(dr);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) dr[e] = c ? dq_dp1[e] : dq_dp0[e];
          }
          const float* vc = vb + 64 * c;
          uint32_t pw[32], dw[32];
          // the masked form only on tiles that need it: a warp-uniform branch
          // inside the unrolled loop would cut it into one short block per
          // pair and expose the exp -> split latency chain of every pair
          auto arith = [&](auto masked) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float4 l4 = make_float4(row_lse2, row_lse2, row_lse2, row_lse2);
              float4 d4 = make_float4(row_delta, row_delta, row_delta, row_delta);
              if (KIND == 0) {
                l4 = *reinterpret_cast<const float4*>(vc + e);
                d4 = *reinterpret_cast<const float4*>(vc + 32 + e);
              }
              const float la[4] = {l4.x, l4.y, l4.z, l4.w};
              const float da[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
              for (int u = 0; u < 4; u += 2) {
                // p = 2^(s scale_log2 - lse log2 e), ds = p (dp - Delta); a
                // masked element has p = 0, hence ds = 0
                const float2 x = ffma2(make_float2(__uint_as_float(sr[e + u]), __uint_as_float(sr[e + u + 1])), sl2,
                                       make_float2(-la[u], -la[u + 1]));
                float2 pp = make_float2(ex2_hw(x.x), ex2_hw(x.y));
                if constexpr (decltype(masked)::value) {
                  const int cA = colc + e + u, cB = cA + 1;
                  bool okA, okB;
                  if (KIND == 0) {
                    okA = key_pos < len && col0 + cA < len && col0 + cA >= key_pos;
                    okB = key_pos < len && col0 + cB < len && col0 + cB >= key_pos;
                  } else {
                    okA = row_ok && col0 + cA <= row_pos;
                    okB = row_ok && col0 + cB <= row_pos;
                  }
                  pp.x = okA ? pp.x : 0.0f;
                  pp.y = okB ? pp.y : 0.0f;
                }
                const float2 ds = fmul2(pp, fsub2(make_float2(__uint_as_float(dr[e + u]), __uint_as_float(dr[e + u + 1])),
                                                  make_float2(da[u], da[u + 1])));
                // a 16-column group of TMEM holds one K-step: its 8 hi words, then its 8 lo words
                const int slot = ((e + u) >> 4) * 16 + (((e + u) & 15) >> 1);
                uint32_t hi, lo;
                if (KIND == 0) {  // dQ reads only dS
                  split_pair2(pp, hi, lo);
                  pw[slot] = hi;
                  pw[slot + 8] = lo;
                }
                split_pair2(ds, hi, lo);
                dw[slot] = hi;
                dw[slot + 8] = lo;
              }
            }
          };
          if (full)
            arith(std::false_type{});
          else
            arith(std::true_type{});
          if (KIND == 0) tmem_st32(tm_s + lane_off + colc, pw);
          tmem_st32(tds_e + lane_off + colc, dw);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars[L::kPFull + (KIND == 1 ? 2 * (s_it & 1) : 0) + c]);
        }
        if (fail) break;
        ++s_it;
      }
      if (fail) break;
      // ---------------------------------------------------------- epilogue
      bool w = mbar_wait(&bars[L::kAccFull], acc_it & 1, abort, p.err, 0x631);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      {
        float* dst_base;
        bool ok;
        float mul;
        uint32_t src;
        if (KIND == 0) {
          // warps 0-3: dV (the raw sum), warps 4-7: dK (times the softmax scale)
          const int kp = it.block * 128 + r;
          ok = kp < len;
          const int64_t row = static_cast<int64_t>(tok0 + kp) * p.hkv + it.head;
          dst_base = (wh == 0 ? p.dv : p.dk) + row * kHeadDim;
          mul = (wh == 0) ? 1.0f : p.scale;
          src = (wh == 0 ? tm_acc0 : tm_acc1) + lane_off;
        } else {
          // dQ (times the softmax scale): warps 0-3 columns 0-63, warps 4-7 64-127
          const int qp = it.block + r;
          ok = r < it.rows && qp < len;
          const int64_t row = static_cast<int64_t>(tok0 + qp) * p.hq + it.head;
          dst_base = p.dq + row * kHeadDim + 64 * wh;
          mul = p.scale;
          src = tm_acc0 + lane_off + 64 * wh;
        }
        const int nchunks = (KIND == 0) ? 4 : 2;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t x[32];
          tmem_ld32(src + 32 * c, x);
          tmem_ld_wait(x);
          if (ok) {
            float4* dst = reinterpret_cast<float4*>(dst_base + 32 * c);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float v0 = __uint_as_float(x[e]), v1 = __uint_as_float(x[e + 1]);
              float v2 = __uint_as_float(x[e + 2]), v3 = __uint_as_float(x[e + 3]);
              if (mul != 1.0f) {
                v0 = __fmul_rn(v0, mul);
                v1 = __fmul_rn(v1, mul);
                v2 = __fmul_rn(v2, mul);
                v3 = __fmul_rn(v3, mul);
              }
              dst[e / 4] = make_float4(v0, v1, v2, v3);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[L::kAccEmpty]);
      ++acc_it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    if (*abort) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_map_bwd(CUtensorMap* m, const void* base, uint64_t heads, uint64_t rows) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  cuuint64_t dims[3] = {128, heads, rows};
  cuuint64_t strides[2] = {256, 256 * heads};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::vector<int> cp_chunks_owner(int n, int cp, int layout, int rank, std::vector<std::pair<int, int>>* ranges) {
  std::vector<int> owner;
  const int chunks = layout == 0 ? cp : 2 * cp;
  for (int c = 0; c < chunks; ++c) {
    const int b = static_cast<int>(static_cast<int64_t>(c) * n / chunks);
    const int e = static_cast<int>(static_cast<int64_t>(c + 1) * n / chunks);
    const int r = layout == 0 ? c : (c < cp ? c : 2 * cp - 1 - c);
    if (ranges && r == rank && e > b) ranges->push_back({b, e});
    owner.push_back(r);
  }
  return owner;
}

int owner_of(int pos, int n, int cp, int layout) {
  const int chunks = layout == 0 ? cp : 2 * cp;
  for (int c = 0; c < chunks; ++c) {
    const int b = static_cast<int>(static_cast<int64_t>(c) * n / chunks);
    const int e = static_cast<int>(static_cast<int64_t>(c + 1) * n / chunks);
    if (pos >= b && pos < e) return layout == 0 ? c : (c < cp ? c : 2 * cp - 1 - c);
  }
  return -1;
}

template <int KIND>
cudaError_t launch_bwd(BwdParams* bp, const std::vector<BwdItem>& tiles, int heads, const CUtensorMap& mq,
                       const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo, int num_sms,
                       cudaStream_t stream) {
  auto kern = rlk_bwd_kernel<KIND>;
  cudaError_t e = cudaSuccess;
  bp->item_heads = heads;
  for (size_t i0 = 0; i0 < tiles.size(); i0 += kMaxBwdTiles) {
    const size_t n = std::min(tiles.size() - i0, static_cast<size_t>(kMaxBwdTiles));
    std::copy(tiles.begin() + i0, tiles.begin() + i0 + n, bp->items);
    bp->num_items = static_cast<int32_t>(n) * heads;
    const int grid = std::min(bp->num_items, num_sms);
    kern<<<grid, 384, BwdLayoutT<KIND>::kAlloc, stream>>>(*bp, mq, mk, mv, mdo);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

static_assert(sizeof(BwdParams) + 4 * sizeof(CUtensorMap) + 256 <= 32764, "backward parameters");

cudaError_t configure_bwd_kernels() {
  cudaError_t e = cudaFuncSetAttribute(rlk_bwd_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BwdLayoutT<0>::kAlloc);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(rlk_bwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdLayoutT<1>::kAlloc);
}

size_t backward_workspace_bytes(const rlk_attn_params* prm, const int32_t* cu) {
  const size_t t_pad = static_cast<size_t>(cu[prm->num_seqs]) + 128;
  return (2 * t_pad * prm->num_q_heads * sizeof(float) + 255) / 256 * 256;
}

rlk_status run_backward(const rlk_attn_params* prm, const void* q, const void* k, const void* v,
                        const float* out_f32, const void* dout, const float* lse, const int32_t* cu,
                        int32_t cp_rank, float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                        ErrWord* err, int num_sms, cudaStream_t stream) {
  (void)workspace_bytes;
  const int T = cu[prm->num_seqs];
  if (T == 0) return RLK_OK;
  if (prm->kv_block_size != 128) return RLK_ERR_UNSUPPORTED;
  const int64_t t_pad = static_cast<int64_t>(T) + 128;
  float* lse_t = static_cast<float*>(workspace);
  float* delta_t = lse_t + t_pad * prm->num_q_heads;

  // preprocess
  PrepParams pp;
  pp.hq = prm->num_q_heads;
  pp.rows = T;
  pp.t_pad = t_pad;
  pp.out = out_f32;
  pp.dout = static_cast<const uint16_t*>(dout);
  pp.lse = lse;
  pp.lse_t = lse_t;
  pp.delta_t = delta_t;
  {
    int64_t blocks = (static_cast<int64_t>(T) * prm->num_q_heads + 7) / 8;
    blocks = std::min<int64_t>(blocks, static_cast<int64_t>(num_sms) * 8);
    rlk_bwd_prep_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return RLK_ERR_CUDA;
  }

  CUtensorMap mq, mk, mv, mdo;
  if (!make_map_bwd(&mq, q, prm->num_q_heads, T) || !make_map_bwd(&mk, k, prm->num_kv_heads, T) ||
      !make_map_bwd(&mv, v, prm->num_kv_heads, T) || !make_map_bwd(&mdo, dout, prm->num_q_heads, T))
    return RLK_ERR_CUDA;

  auto bp = std::make_unique<BwdParams>();
  std::memset(bp.get(), 0, sizeof(BwdParams));
  bp->err = err;
  bp->hq = prm->num_q_heads;
  bp->hkv = prm->num_kv_heads;
  bp->group = prm->num_q_heads / prm->num_kv_heads;
  bp->t_pad = t_pad;
  bp->scale = prm->softmax_scale;
  bp->scale_log2 = static_cast<float>(static_cast<double>(prm->softmax_scale) * 1.4426950408889634073599);
  bp->lse_t = lse_t;
  bp->delta_t = delta_t;
  bp->dq = dq;
  bp->dk = dk;
  bp->dv = dv;
  for (int s = 0; s <= prm->num_seqs; ++s) bp->cu[s] = cu[s];

  // dK/dV tiles: (seq, KV block), most query blocks first, each taken by
  // every KV head; dQ tiles: (seq, query tile), most KV blocks first, each
  // taken by every query head
  std::vector<std::pair<int, BwdItem>> kv;
  std::vector<std::pair<int, BwdItem>> qi;
  for (int s = 0; s < prm->num_seqs; ++s) {
    const int len = cu[s + 1] - cu[s];
    const int nb = (len + 127) / 128;
    for (int j = 0; j < nb; ++j) {
      if (cp_rank >= 0 && owner_of(j * 128, len, prm->cp_size, prm->cp_layout) != cp_rank) continue;
      kv.push_back({nb - j, BwdItem{s, 0, j, 128}});
    }
    std::vector<std::pair<int, int>> ranges;
    if (cp_rank < 0) ranges.push_back({0, len});
    else cp_chunks_owner(len, prm->cp_size, prm->cp_layout, cp_rank, &ranges);
    for (auto& rg : ranges)
      for (int r0 = rg.first; r0 < rg.second; r0 += 128) {
        const int rows = std::min(128, rg.second - r0);
        const int cost = (r0 + rows - 1) / 128 + 1;
        qi.push_back({cost, BwdItem{s, 0, r0, rows}});
      }
  }
  auto by_cost = [](const std::pair<int, BwdItem>& a, const std::pair<int, BwdItem>& b) { return a.first > b.first; };
  std::stable_sort(kv.begin(), kv.end(), by_cost);
  std::stable_sort(qi.begin(), qi.end(), by_cost);
  std::vector<BwdItem> tiles;
  for (auto& x : kv) tiles.push_back(x.second);
  if (!tiles.empty() &&
      launch_bwd<0>(bp.get(), tiles, prm->num_kv_heads, mq, mk, mv, mdo, num_sms, stream) != cudaSuccess)
    return RLK_ERR_CUDA;
  tiles.clear();
  for (auto& x : qi) tiles.push_back(x.second);
  if (!tiles.empty() &&
      launch_bwd<1>(bp.get(), tiles, prm->num_q_heads, mq, mk, mv, mdo, num_sms, stream) != cudaSuccess)
    return RLK_ERR_CUDA;
  return RLK_OK;
}

}  // namespace rlk
