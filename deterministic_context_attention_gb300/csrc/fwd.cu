// fwd.cu -- forward engine for sm_103a: fused causal prefill, partial-state
// production, and paged-KV decode.
//
// One persistent CTA per SM walks a static, longest-first list of work items.
// An item is 128 query rows of one query head (prefill / states) or the query
// heads of one KV head of one decode sequence.  For each global KV block b of
// the item, in ascending order, the CTA computes the block state of every row
//   state_b = (o_b, lse_b, b)
// ("WS2 Attention PR5 Drift Benchmark", Transformer Engine Reuse) with full
// block arithmetic: S = Q K_b^T on the tensor core (tcgen05, FP32 in TMEM),
// block softmax statistics in FP32, PV = P_hi V_b + P_lo V_b with P split into
// two BF16 parts, o_b = PV / l_b.  The fused and decode modes fold the states
// on chip in ascending global_block_index order with the canonical fold; the
// states mode writes every state to the caller's state table instead.  Because
// all three modes run this one pipeline and the functions of numerics.cuh,
// a state has the same bits whichever mode, tile position or logical CP rank
// produced it ("[WS2][Attention] H100 validation and reproduction guide",
// Status and Acceptance: fixed merge order, full-KV arithmetic retained, max
// abs 0.0 across ranks).
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  correction / epilogue: thread r owns TMEM lane r (row r)
//   warps 4-7  softmax: thread r owns TMEM lane r, writes P_hi/P_lo to TMEM
//              over its scores (per 16-key MMA step: 8 columns hi, 8 lo)
//   warp  8    TMA producer (Q tile, K/V blocks or pages)
//   warp  9    TMEM allocator and MMA issuer (also zeroes V rows past the
//              valid length of a partial block)
//   warps 10-11 idle (the block is sized in whole warpgroups, the unit in
//              which registers are granted)
// TMEM (512 columns): S/P double buffer [0,256), PV [256,384), O [384,512).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>

#include "numerics.cuh"
#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {

template <int B>
struct FwdLayout {
  static constexpr int kStages = (B == 128) ? 2 : 4;
  static constexpr int kQBytes = kTileRows * kHeadDim * 2;  // 32 KB, two 64-column halves
  static constexpr int kQHalf = kTileRows * 128;            // bytes of one half
  static constexpr int kKVHalf = B * 128;                   // bytes of one 64-column half
  static constexpr int kKVBytes = 2 * kKVHalf;              // K (or V) of one block
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQBytes;                    // stage s: K then V
  static constexpr int kBarOff = kKVOff + kStages * 2 * kKVBytes;
  // barrier indices
  static constexpr int kQFull = 0, kQEmpty = 1, kKVFull = 2, kKVEmpty = 2 + kStages,
                       kSFull = 2 + 2 * kStages, kPFull = kSFull + 2, kPVFull = kPFull + 2,
                       kPVEmpty = kPVFull + 1, kStatsFull = kPVEmpty + 1,
                       kNumBars = kStatsFull + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base (u32), abort (i32)
  static constexpr int kStatsOff = (kMiscOff + 16 + 15) / 16 * 16;
  static constexpr int kTotal = kStatsOff + 4 * kTileRows * 8;
  static constexpr int kAlloc = kTotal + 1024;
};

struct ItemInfo {
  int seq, head, row_begin, row_count, nb, blk0, q_len, kv_len, q_tok0, k_tok0;
  int slab_rb, slab_rc;
  int64_t slab_off;
};

template <int MODE>
__device__ __forceinline__ ItemInfo item_info(const FwdParams& p, int item) {
  ItemInfo it;
  if (MODE == kModeDecode) {
    const FwdTile& t = p.tiles[item];
    it.seq = t.seq;
    it.head = t.row_begin;  // KV head g; rows are query heads g*group .. g*group+group-1
    it.row_begin = 0;
    it.row_count = p.group;
    it.kv_len = p.cu_k[t.seq];
    it.q_len = 1;
    it.q_tok0 = t.seq;
    it.k_tok0 = 0;
    it.blk0 = 0;
    it.nb = (it.kv_len + p.block - 1) / p.block;
    it.slab_rb = it.slab_rc = 0;
    it.slab_off = 0;
  } else {
    const int tile = item / p.hq;
    const FwdTile& t = p.tiles[tile];
    it.seq = t.seq;
    it.head = item - tile * p.hq;
    it.row_begin = t.row_begin;
    it.row_count = t.row_count;
    it.q_tok0 = p.cu_q[t.seq];
    it.k_tok0 = p.cu_k[t.seq];
    it.q_len = p.cu_q[t.seq + 1] - it.q_tok0;
    it.kv_len = p.cu_k[t.seq + 1] - it.k_tok0;
    if (MODE == kModeStates) {
      it.blk0 = t.block;
      it.nb = 1;
    } else {
      const int pmax = it.kv_len - it.q_len + t.row_begin + t.row_count - 1;
      it.blk0 = 0;
      it.nb = pmax / p.block + 1;
    }
    it.slab_off = t.slab_offset;
    it.slab_rb = t.slab_row_begin;
    it.slab_rc = t.slab_row_count;
  }
  return it;
}

// Keys of block b visible to a row at key position pos (prefix of the block).
__device__ __forceinline__ int visible_keys(int pos, int kv_len, int b, int B) {
  const int last = min(pos, kv_len - 1);
  return max(0, min(B, last - b * B + 1));
}

template <int B, int MODE>
__global__ void __launch_bounds__(384, 1)
    rlk_fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = FwdLayout<B>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  float2* stats = reinterpret_cast<float2*>(smem + L::kStatsOff);  // [4][128]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bars[L::kQFull], 1);
    mbar_init(&bars[L::kQEmpty], 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars[L::kKVFull + s], 1);
      mbar_init(&bars[L::kKVEmpty + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[L::kSFull + s], 1);
      mbar_init(&bars[L::kPFull + s], 128);
    }
    mbar_init(&bars[L::kPVFull], 1);
    mbar_init(&bars[L::kPVEmpty], 128);
    for (int s = 0; s < 4; ++s) mbar_init(&bars[L::kStatsFull + s], 128);
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
  const uint32_t tm_s = tmem;          // S/P buffers: + 128 * buf
  const uint32_t tm_pv = tmem + 256;
  const uint32_t tm_o = tmem + 384;

  const uint32_t q_addr = smem_u32(smem + L::kQOff);
  uint8_t* kv_base = smem + L::kKVOff;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    uint32_t kv_it = 0, q_it = 0;
    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
      const ItemInfo it = item_info<MODE>(p, item);
      bool ok = mbar_wait(&bars[L::kQEmpty], (q_it & 1) ^ 1, abort, p.err, 0x101);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        if (MODE == kModeDecode) {
          mbar_arrive_expect_tx(&bars[L::kQFull], p.group * kHeadDim * 2);
          tma_load_3d(smem + L::kQOff, &tm_q, &bars[L::kQFull], 0, it.head * p.group, it.seq);
          tma_load_3d(smem + L::kQOff + L::kQHalf, &tm_q, &bars[L::kQFull], 64, it.head * p.group, it.seq);
        } else {
          mbar_arrive_expect_tx(&bars[L::kQFull], L::kQBytes);
          const int row0 = it.q_tok0 + it.row_begin;
          tma_load_3d(smem + L::kQOff, &tm_q, &bars[L::kQFull], 0, it.head, row0);
          tma_load_3d(smem + L::kQOff + L::kQHalf, &tm_q, &bars[L::kQFull], 64, it.head, row0);
        }
      }
      ++q_it;
      const int g = (MODE == kModeDecode) ? it.head : it.head / p.group;
      for (int j = 0; j < it.nb; ++j) {
        const int b = it.blk0 + j;
        const uint32_t stage = kv_it % S;
        ok = mbar_wait(&bars[L::kKVEmpty + stage], ((kv_it / S) & 1) ^ 1, abort, p.err, 0x102);
        if (!__all_sync(0xffffffffu, ok)) break;
        uint8_t* kd = kv_base + stage * 2 * L::kKVBytes;
        uint8_t* vd = kd + L::kKVBytes;
        if (MODE != kModeDecode) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars[L::kKVFull + stage], 2 * L::kKVBytes);
            const int r = it.k_tok0 + b * B;
            tma_load_3d(kd, &tm_k, &bars[L::kKVFull + stage], 0, g, r);
            tma_load_3d(kd + L::kKVHalf, &tm_k, &bars[L::kKVFull + stage], 64, g, r);
            tma_load_3d(vd, &tm_v, &bars[L::kKVFull + stage], 0, g, r);
            tma_load_3d(vd + L::kKVHalf, &tm_v, &bars[L::kKVFull + stage], 64, g, r);
          }
        } else {
          const int ps = p.page_size;
          const int n_tok = min(B, it.kv_len - b * B);
          const int n_pg = (n_tok + ps - 1) / ps;
          if (lane == 0) mbar_arrive_expect_tx(&bars[L::kKVFull + stage], n_pg * ps * 512);
          __syncwarp();
          if (lane < n_pg) {
            int32_t pe = p.page_table[static_cast<int64_t>(it.seq) * p.max_pages + b * (B / ps) + lane];
            if (pe < 0 || pe >= p.n_pages) {
              report_error(p.err, kErrBadPage, 0x103);
              pe = p.n_pages;  // out of range: the copy reads the zero fill
            }
            const int r = pe * ps;
            const int off = lane * ps * 128;
            tma_load_3d(kd + off, &tm_k, &bars[L::kKVFull + stage], 0, g, r);
            tma_load_3d(kd + L::kKVHalf + off, &tm_k, &bars[L::kKVFull + stage], 64, g, r);
            tma_load_3d(vd + off, &tm_v, &bars[L::kKVFull + stage], 0, g, r);
            tma_load_3d(vd + L::kKVHalf + off, &tm_v, &bars[L::kKVFull + stage], 64, g, r);
          }
        }
        ++kv_it;
      }
      if (*abort) break;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdescS = idesc_bf16(128, B, false, false);
    constexpr uint32_t kIdescPV = idesc_bf16(128, kHeadDim, false, true);
    uint32_t kv_it = 0, s_it = 0, pv_it = 0, q_it = 0;
    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
      const ItemInfo it = item_info<MODE>(p, item);
      bool ok = mbar_wait(&bars[L::kQFull], q_it & 1, abort, p.err, 0x201);
      if (!__all_sync(0xffffffffu, ok)) break;
      ++q_it;
      const uint32_t kvb = kv_it, sb0 = s_it;
      auto issue_s = [&](int j) -> bool {
        const uint32_t kvi = kvb + j;
        const uint32_t stage = kvi % S;
        bool w = mbar_wait(&bars[L::kKVFull + stage], (kvi / S) & 1, abort, p.err, 0x202);
        if (!__all_sync(0xffffffffu, w)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_addr = smem_u32(kv_base + stage * 2 * L::kKVBytes);
          const uint32_t d = tm_s + ((sb0 + j) & 1) * 128;
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t half = k >> 2, sub = (k & 3) * 32;
            const uint64_t ad = sdesc_sw128(q_addr + half * L::kQHalf + sub, 16, 1024);
            const uint64_t bd = sdesc_sw128(k_addr + half * L::kKVHalf + sub, 16, 1024);
            umma_ss(d, ad, bd, kIdescS, k > 0 ? 1u : 0u);
          }
          umma_commit(&bars[L::kSFull + ((sb0 + j) & 1)]);
        }
        __syncwarp();
        return true;
      };
      if (!issue_s(0)) break;
      bool fail = false;
      for (int j = 0; j < it.nb; ++j) {
        if (j + 1 < it.nb) {
          if (!issue_s(j + 1)) { fail = true; break; }
        } else {
          if (lane == 0) umma_commit(&bars[L::kQEmpty]);  // Q no longer read
          __syncwarp();
        }
        const uint32_t sidx = sb0 + j;
        const uint32_t buf = sidx & 1;
        bool w = mbar_wait(&bars[L::kPFull + buf], (sidx >> 1) & 1, abort, p.err, 0x203);
        w = w && mbar_wait(&bars[L::kPVEmpty], (pv_it & 1) ^ 1, abort, p.err, 0x204);
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        const uint32_t stage = (kvb + j) % S;
        uint8_t* vd = kv_base + stage * 2 * L::kKVBytes + L::kKVBytes;
        // V rows past the valid keys of a partial block may hold stale or
        // non-finite data; P is exactly 0 there, so zero them (0 * NaN = NaN).
        const int b = it.blk0 + j;
        const int valid = min(B, it.kv_len - b * B);
        if (valid < B) {
          const int nrow = B - valid;
          for (int i = lane; i < nrow * 16; i += 32) {
            const int row = valid + (i >> 4);
            const int part = i & 15;  // 16 B pieces: 8 per half-row, 2 halves
            uint4* dst = reinterpret_cast<uint4*>(vd + (part >> 3) * L::kKVHalf + row * 128 + (part & 7) * 16);
            *dst = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t v_addr = smem_u32(vd);
          const uint32_t a0 = tm_s + buf * 128;
#pragma unroll
          for (int k = 0; k < B / 16; ++k) {
            const uint64_t bd = sdesc_sw128(v_addr + k * 16 * 128, L::kKVHalf, 1024);
            umma_ts(tm_pv, a0 + 16 * k, bd, kIdescPV, k > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int k = 0; k < B / 16; ++k) {
            const uint64_t bd = sdesc_sw128(v_addr + k * 16 * 128, L::kKVHalf, 1024);
            umma_ts(tm_pv, a0 + 16 * k + 8, bd, kIdescPV, 1u);
          }
          umma_commit(&bars[L::kPVFull]);
          umma_commit(&bars[L::kKVEmpty + stage]);
        }
        __syncwarp();
        ++pv_it;
      }
      if (fail) break;
      kv_it += it.nb;
      s_it += it.nb;
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax
    const int r = tid - 128;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t s_it = 0, st_it = 0;
    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
      const ItemInfo it = item_info<MODE>(p, item);
      const bool valid = r < it.row_count;
      const int pos = (MODE == kModeDecode) ? it.kv_len - 1 : it.kv_len - it.q_len + it.row_begin + r;
      bool fail = false;
      for (int j = 0; j < it.nb; ++j) {
        const int b = it.blk0 + j;
        const uint32_t buf = s_it & 1;
        bool w = mbar_wait(&bars[L::kSFull + buf], (s_it >> 1) & 1, abort, p.err, 0x301);
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        tc_fence_after();
        const uint32_t ta = tm_s + lane_off + buf * 128;
        const int nvis = valid ? visible_keys(pos, it.kv_len, b, B) : 0;
        // pass 1: row max over the visible keys
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < B / 32; ++c) {
          uint32_t raw[32];
          tmem_ld32(ta + 32 * c, raw);
          tmem_ld_wait(raw);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            m = fmaxf(m, scaled_score(__uint_as_float(raw[e]), 32 * c + e, nvis, p.scale_log2));
        }
        // pass 2: probabilities, canonical partial sums, P = P_hi + P_lo.  The
        // words of keys 16k..16k+15 go to columns 16k..16k+15 (8 hi, then 8 lo),
        // the columns their scores came from.
        float part[32];
        const bool has = nvis > 0;
#pragma unroll
        for (int c = 0; c < B / 32; ++c) {
          uint32_t raw[32];
          tmem_ld32(ta + 32 * c, raw);
          tmem_ld_wait(raw);
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int key = 32 * c + e;
            float p0 = prob(scaled_score(__uint_as_float(raw[e]), key, nvis, p.scale_log2), m);
            float p1 = prob(scaled_score(__uint_as_float(raw[e + 1]), key + 1, nvis, p.scale_log2), m);
            if (!has) { p0 = 0.0f; p1 = 0.0f; }
            partial_add(part, key, p0);
            partial_add(part, key + 1, p1);
            uint32_t hi, lo;
            split_pair(p0, p1, hi, lo);
            const int slot = (e >> 4) * 16 + ((e & 15) >> 1);  // K-step (e/16), word within it
            w[slot] = hi;
            w[slot + 8] = lo;
          }
          tmem_st32(ta + 32 * c, w);
        }
        float lse_b = -INFINITY, rcp = 0.0f;
        if (has) block_stats(m, partial_tree(part), lse_b, rcp);
        tmem_st_wait();
        tc_fence_before();
        stats[(st_it & 3) * kTileRows + r] = make_float2(lse_b, rcp);
        mbar_arrive(&bars[L::kPFull + buf]);
        mbar_arrive(&bars[L::kStatsFull + (st_it & 3)]);
        ++s_it;
        ++st_it;
      }
      if (fail) break;
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ correction / epilogue
    const int r = tid;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t pv_it = 0, st_it = 0;
    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
      const ItemInfo it = item_info<MODE>(p, item);
      const bool valid = r < it.row_count;
      float Lrun = -INFINITY;
      bool fail = false;
      for (int j = 0; j < it.nb; ++j) {
        bool w = mbar_wait(&bars[L::kPVFull], pv_it & 1, abort, p.err, 0x401);
        w = w && mbar_wait(&bars[L::kStatsFull + (st_it & 3)], (st_it >> 2) & 1, abort, p.err, 0x402);
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        tc_fence_after();
        const float2 st = stats[(st_it & 3) * kTileRows + r];
        const float lse_b = st.x, rcp = st.y;
        const bool has = valid && (lse_b != -INFINITY);
        if (MODE == kModeStates) {
          const int64_t pair = it.slab_off + static_cast<int64_t>(it.head) * it.slab_rc +
                               (it.row_begin + r - it.slab_rb);
          float4* dst = reinterpret_cast<float4*>(p.state_o + pair * kHeadDim);
#pragma unroll
          for (int c = 0; c < kHeadDim / 32; ++c) {
            uint32_t x[32];
            tmem_ld32(tm_pv + lane_off + 32 * c, x);
            tmem_ld_wait(x);
            if (has) {
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                dst[(32 * c + e) / 4] = make_float4(state_elem(__uint_as_float(x[e]), rcp),
                                                    state_elem(__uint_as_float(x[e + 1]), rcp),
                                                    state_elem(__uint_as_float(x[e + 2]), rcp),
                                                    state_elem(__uint_as_float(x[e + 3]), rcp));
            }
          }
          if (has) p.state_lse[pair] = lse_b;
        } else {
          float Lp = 0.f, alpha = 0.f, beta = 0.f;
          if (j > 0 && has) fold_coeffs(Lrun, lse_b, Lp, alpha, beta);
#pragma unroll
          for (int c = 0; c < kHeadDim / 32; ++c) {
            uint32_t x[32], y[32];
            tmem_ld32(tm_pv + lane_off + 32 * c, x);
            tmem_ld_wait(x);
            if (j > 0) {
              tmem_ld32(tm_o + lane_off + 32 * c, y);
              tmem_ld_wait(y);
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float o = state_elem(__uint_as_float(x[e]), rcp);
              if (j == 0) {
                y[e] = __float_as_uint(o);
              } else if (has) {
                y[e] = __float_as_uint(fold_elem(__uint_as_float(y[e]), o, alpha, beta));
              }
            }
            tmem_st32(tm_o + lane_off + 32 * c, y);
          }
          tmem_st_wait();
          if (has) Lrun = (j == 0) ? lse_b : Lp;
        }
        tc_fence_before();
        mbar_arrive(&bars[L::kPVEmpty]);
        ++pv_it;
        ++st_it;
      }
      if (fail) break;
      if (MODE != kModeStates) {
        // epilogue: O and L are final; write FP32 / BF16 rows and lse
        int64_t row_idx;
        if (MODE == kModeDecode) row_idx = static_cast<int64_t>(it.seq) * p.hq + it.head * p.group + r;
        else row_idx = static_cast<int64_t>(it.q_tok0 + it.row_begin + r) * p.hq + it.head;
#pragma unroll
        for (int c = 0; c < kHeadDim / 32; ++c) {
          uint32_t y[32];
          tmem_ld32(tm_o + lane_off + 32 * c, y);
          tmem_ld_wait(y);
          if (valid) {
            if (p.out_f32) {
              float4* dst = reinterpret_cast<float4*>(p.out_f32 + row_idx * kHeadDim + 32 * c);
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                dst[e / 4] = make_float4(__uint_as_float(y[e]), __uint_as_float(y[e + 1]),
                                         __uint_as_float(y[e + 2]), __uint_as_float(y[e + 3]));
            }
            if (p.out_bf16) {
              uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + row_idx * kHeadDim + 32 * c);
#pragma unroll
              for (int e = 0; e < 32; e += 8)
                dst[e / 8] = make_uint4(pack_bf16x2(__uint_as_float(y[e]), __uint_as_float(y[e + 1])),
                                        pack_bf16x2(__uint_as_float(y[e + 2]), __uint_as_float(y[e + 3])),
                                        pack_bf16x2(__uint_as_float(y[e + 4]), __uint_as_float(y[e + 5])),
                                        pack_bf16x2(__uint_as_float(y[e + 6]), __uint_as_float(y[e + 7])));
            }
          }
        }
        if (valid && p.lse) p.lse[row_idx] = Lrun;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    if (*abort) {
      // let copies already in flight land before the CTA's memory is released
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- launchers
template <int B, int MODE>
static cudaError_t launch_fwd_t(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t stream) {
  using L = FwdLayout<B>;
  auto kern = rlk_fwd_kernel<B, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, 384, L::kAlloc, stream>>>(p, tq, tk, tv);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, kern) == cudaSuccess)
      fprintf(stderr, "rlk_fwd_kernel<%d,%d>: %d registers, max %d threads/block, %zu B dynamic smem\n", B, MODE,
              a.numRegs, a.maxThreadsPerBlock, static_cast<size_t>(L::kAlloc));
  }
  return e;
}

cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t stream) {
  if (p.block == 128) {
    switch (p.mode) {
      case kModeFused: return launch_fwd_t<128, kModeFused>(p, tq, tk, tv, grid, stream);
      case kModeStates: return launch_fwd_t<128, kModeStates>(p, tq, tk, tv, grid, stream);
      case kModeDecode: return launch_fwd_t<128, kModeDecode>(p, tq, tk, tv, grid, stream);
    }
  } else if (p.block == 64) {
    switch (p.mode) {
      case kModeFused: return launch_fwd_t<64, kModeFused>(p, tq, tk, tv, grid, stream);
      case kModeStates: return launch_fwd_t<64, kModeStates>(p, tq, tk, tv, grid, stream);
      case kModeDecode: return launch_fwd_t<64, kModeDecode>(p, tq, tk, tv, grid, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace rlk
