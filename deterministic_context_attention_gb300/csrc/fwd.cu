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
// Warp roles (512 threads, four warpgroups):
//   warps 0-3  correction / epilogue: thread r owns TMEM lane r (row r) and
//              keeps the running O of its row in registers
//   warps 4-7  softmax, keys [0, B/2) of every block; warps 12-15 softmax,
//              keys [B/2, B): thread r of either group owns TMEM lane r and
//              reads its half of the row's S once into registers (the half's
//              maximum comes with the load); the two warps of a TMEM lane
//              quadrant exchange the half maxima and half sums through shared
//              memory, then write P_hi/P_lo over their half of S (per 16-key
//              MMA step: 8 columns hi, then 8 lo)
//   warp  8    TMA producer (Q tile; K and V blocks or pages, separate rings)
//   warp  9    TMEM allocator and MMA issuer (also zeroes V rows past the
//              valid length of a partial block)
//   warps 10-11 idle (registers are granted per warpgroup: warps 8-11 run
//              with 48, warps 0-3 with 208, the softmax groups with 128)
// TMEM (512 columns): S/P double buffer [0,256), PV double buffer [256,512).
// Per block the tensor core runs S_{b+1} then PV_b, so the softmax of block
// b+1 overlaps PV_b and the correction of block b overlaps both.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>

#include "numerics.cuh"
#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {

// Four warpgroups (512 threads, 128 registers per thread at launch),
// re-split per warpgroup: correction 208, the two softmax groups 128 each,
// producer / MMA 48.
constexpr int kThreads = 512;
constexpr int kRegsLaunch = 128;
constexpr int kRegsCorrection = 208;
constexpr int kRegsSoftmax = 128;
constexpr int kRegsProducer = 48;
static_assert(kRegsCorrection + 2 * kRegsSoftmax + kRegsProducer <= 4 * kRegsLaunch, "register split");

template <int B>
struct FwdLayout {
  static constexpr int kSK = (B == 128) ? 3 : 4;         // K ring
  static constexpr int kSV = (B == 128) ? 2 : 4;         // V ring
  static constexpr int kStatsRing = 8;
  static constexpr int kQBytes = kTileRows * kHeadDim * 2;  // 32 KB, two 64-column halves
  static constexpr int kQHalf = kTileRows * 128;            // bytes of one half
  static constexpr int kKVHalf = B * 128;                   // bytes of one 64-column half
  static constexpr int kKVBytes = 2 * kKVHalf;              // K (or V) of one block
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kSK * kKVBytes;
  static constexpr int kBarOff = kVOff + kSV * kKVBytes;
  static constexpr int kQFull = 0, kQEmpty = 1, kKFull = 2, kKEmpty = kKFull + kSK, kVFull = kKEmpty + kSK,
                       kVEmpty = kVFull + kSV, kSFull = kVEmpty + kSV, kPFull = kSFull + 2, kPVFull = kPFull + 2,
                       kPVEmpty = kPVFull + 2, kStatsFull = kPVEmpty + 2, kXch = kStatsFull + kStatsRing,
                       kQRot = kXch + 4, kNumBars = kQRot + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base (u32), abort (i32)
  static constexpr int kStatsOff = (kMiscOff + 16 + 15) / 16 * 16;
  // softmax exchange: the half maxima and half sums of every row, [2][128] each
  static constexpr int kXchOff = kStatsOff + kStatsRing * kTileRows * 8;
  static constexpr int kPageWin = 512;  // decode: page ids cached per window
  static constexpr int kPageOff = kXchOff + 2 * 2 * kTileRows * 4;
  // epilogue staging: per correction warp 32 rows x 128 B (one column chunk)
  static constexpr int kEpiOff = kPageOff + 2 * kPageWin * 4;
  static constexpr int kEpiBytes = 4 * 32 * 128;
  static constexpr int kTotal = kEpiOff + kEpiBytes;
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= 232448, "forward shared memory");
  static_assert(kEpiOff % 16 == 0, "staging alignment");
};

struct ItemInfo {
  int seq, head, row_begin, row_count, nb, blk0, q_len, kv_len, q_tok0, k_tok0;
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
      it.nb = t.slab_row_count;  // a run of consecutive blocks of the rank
    } else {
      const int pmax = it.kv_len - it.q_len + t.row_begin + t.row_count - 1;
      it.blk0 = 0;
      it.nb = pmax / p.block + 1;
    }
    it.slab_off = t.slab_offset;
  }
  return it;
}

// Item of this CTA in round k of the static schedule: CTAs take one item per
// round from the longest-first list, in ascending CTA order on even rounds
// and descending on odd ones, which evens out the per-CTA work.  A CTA's item
// index grows with the round, so its loop ends at the first round without one.
__device__ __forceinline__ int snake_item(int round) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return round * g + ((round & 1) ? g - 1 - c : c);
}

// Keys of block b visible to a row at key position pos (prefix of the block).
__device__ __forceinline__ int visible_keys(int pos, int kv_len, int b, int B) {
  const int last = min(pos, kv_len - 1);
  return max(0, min(B, last - b * B + 1));
}

// Decode places query head i of a KV head's group in tile row (TMEM lane)
// 32 * (i % 4) + i / 4, so a small group is spread over the four lane
// quadrants and each warp of a group works on one of its rows (a warp reaches
// only its own 32 lanes).  Prefill and states rows map one to one.
template <int MODE>
__device__ __forceinline__ int row_of_lane(int r) {
  return MODE == kModeDecode ? 4 * (r & 31) + (r >> 5) : r;
}
__device__ __forceinline__ int decode_lane_of_row(int i) { return 32 * (i & 3) + (i >> 2); }

__device__ __forceinline__ void setmaxnreg_inc208() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
}
__device__ __forceinline__ void setmaxnreg_dec48() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 48;" ::: "memory");
}

// Softmax of one row's half block (the H = B/2 keys [h H, (h+1) H) of global
// block b), from a single read of the half's S.  The H/32 column chunks are
// loaded together (each load also returns its chunk's maximum) into s; with
// masking, keys at or past hv (the visible keys of this half) are set to
// -inf first, so their probability is exactly 0.  The half's maximum is
// returned; after the maxima of both halves are exchanged, half_probs forms
// the probabilities in place and their canonical half sum.
template <int NC>
__device__ __forceinline__ float half_load(uint32_t ta, bool full, int hv, uint32_t (&s)[NC][32]) {
  float mx[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) tmem_ld32_max(ta + 32 * c, s[c], mx[c]);
  tmem_ld_wait_only();
#pragma unroll
  for (int c = 0; c < NC; ++c) tmem_tie(s[c], mx[c]);
  float m = -INFINITY;
  if (full) {
#pragma unroll
    for (int c = 0; c < NC; ++c) m = fmaxf(m, mx[c]);
  } else {
    const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        s[c][e] = 32 * c + e < hv ? s[c][e] : ninf;
        s[c][e + 1] = 32 * c + e + 1 < hv ? s[c][e + 1] : ninf;
        m = fmax3(m, __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]));
      }
    }
  }
  return m;
}

// p = 2^fma(S, scale_log2, -mc) for the half's keys, chunk by chunk: the
// words become (hi, lo) = split(p_2i, p_2i+1) in key-pair order and each
// 16-key MMA step is stored over its S columns; returns the canonical half
// sum: partial j (j < 16) adds the half's keys j, j + 16, j + 32, ... in
// ascending order, and the 16 partials combine by the 8-4-2-1 tree.
template <int NC>
__device__ __forceinline__ float half_probs(uint32_t ta, uint32_t (&s)[NC][32], float scale_log2, float mc) {
  const float2 sc = make_float2(scale_log2, scale_log2);
  const float2 nm = make_float2(-mc, -mc);
  float part[16];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float2 x = ffma2(make_float2(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), sc, nm);
      const float2 pr = make_float2(ex2_hw(x.x), ex2_hw(x.y));
      const int j = e & 15;
      if (c == 0 && e < 16) {
        part[j] = pr.x;
        part[j + 1] = pr.y;
      } else {
        const float2 acc = fadd2(make_float2(part[j], part[j + 1]), pr);
        part[j] = acc.x;
        part[j + 1] = acc.y;
      }
      uint32_t hi, lo;
      split_pair2(pr, hi, lo);
      s[c][e] = hi;
      s[c][e + 1] = lo;
      // each 16-key MMA step's words go out as soon as they exist
      if ((e & 15) == 14) tmem_st16_hilo(ta + 32 * c + (e & 16), &s[c][e & 16]);
    }
  }
  return partial_tree(part);
}

// RoPE of one quarter of a query row in the shared-memory tile (128-byte
// swizzle, two 64-column halves of kQHalf bytes): pairs 32h .. 32h + 31 of
// row r, i.e. 16-byte chunks 4h .. 4h + 3 of the first half and the chunks at
// the same swizzled offsets of the second half.  trow: the row's position in
// the table, advanced to cos[32h] (sin follows 64 floats later).  One chunk
// at a time (the table lines were prefetched into L1), so few registers are
// live.
__device__ __forceinline__ void rope_row_quarter(const float* trow, uint8_t* q_tile, int r, int h) {
  const float4* t4 = reinterpret_cast<const float4*>(trow);
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    const float4 x0 = __ldg(t4 + 2 * cc), x1 = __ldg(t4 + 2 * cc + 1);
    const float4 y0 = __ldg(t4 + 16 + 2 * cc), y1 = __ldg(t4 + 16 + 2 * cc + 1);
    const float c[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const float sn[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
    const int pj = (4 * h + cc) ^ (r & 7);
    uint4* pa = reinterpret_cast<uint4*>(q_tile + r * 128 + pj * 16);
    uint4* pb = reinterpret_cast<uint4*>(q_tile + FwdLayout<128>::kQHalf + r * 128 + pj * 16);
    uint4 a = *pa, b = *pb;
    rope_words8(a, b, c, sn);
    *pa = a;
    *pb = b;
  }
}
// Bring a quarter row of the table (128 B of cos, 128 B of sin) towards the
// SM ahead of its use.
__device__ __forceinline__ void rope_prefetch(const float* trow) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(trow));
  asm volatile("prefetch.global.L1 [%0];" ::"l"(trow + 64));
}

// ROPE (fused mode only): the query tile is rotated in shared memory by the
// softmax warps before the first S of each item (the table in p.rope_table).
template <int B, int MODE, bool ROPE>
__global__ void __launch_bounds__(512, 1)
    rlk_fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = FwdLayout<B>;
  constexpr int SK = L::kSK, SV = L::kSV, SR = L::kStatsRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  float2* stats = reinterpret_cast<float2*>(smem + L::kStatsOff);  // [ring][128]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bars[L::kQFull], 1);
    mbar_init(&bars[L::kQEmpty], 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(&bars[L::kKFull + s], 1);
      mbar_init(&bars[L::kKEmpty + s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&bars[L::kVFull + s], 1);
      mbar_init(&bars[L::kVEmpty + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[L::kSFull + s], 1);
      mbar_init(&bars[L::kPFull + s], 256);
      mbar_init(&bars[L::kPVFull + s], 1);
      mbar_init(&bars[L::kPVEmpty + s], 128);
    }
    for (int s = 0; s < SR; ++s) mbar_init(&bars[L::kStatsFull + s], 128);
    for (int s = 0; s < 4; ++s) mbar_init(&bars[L::kXch + s], 64);
    mbar_init(&bars[L::kQRot], 256);
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
  const uint32_t tm_pv = tmem + 256;   // PV buffers: + 128 * buf

  const uint32_t q_addr = smem_u32(smem + L::kQOff);
  uint8_t* k_base = smem + L::kKOff;
  uint8_t* v_base = smem + L::kVOff;

  if (warp >= 8 && warp < 12) {
    setmaxnreg_dec48();
    if (warp == 8) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      uint32_t k_it = 0, v_it = 0, q_it = 0;
      // decode: the page ids of the current sequence, cached in two 512-entry
      // windows (V trails K by one block, so both may be live at a boundary)
      int32_t* page_cache = reinterpret_cast<int32_t*>(smem + L::kPageOff);
      int cached_win0 = -1, cached_win1 = -1;
      // load K (IS_V false) or V of block b into its ring slot; false on abort
      auto load_kv = [&](const ItemInfo& it, int g, int b, bool is_v) -> bool {
        const uint32_t idx = is_v ? v_it : k_it;
        const int S = is_v ? SV : SK;
        const uint32_t stage = idx % S;
        uint64_t* empty = &bars[(is_v ? L::kVEmpty : L::kKEmpty) + stage];
        uint64_t* full = &bars[(is_v ? L::kVFull : L::kKFull) + stage];
        bool ok = mbar_wait(empty, ((idx / S) & 1) ^ 1, abort, p.err, is_v ? 0x103 : 0x102);
        if (!__all_sync(0xffffffffu, ok)) return false;
        uint8_t* dst = (is_v ? v_base : k_base) + stage * L::kKVBytes;
        const CUtensorMap* map = is_v ? &tm_v : &tm_k;
        if (MODE != kModeDecode) {
          if (lane == 0) {
            mbar_arrive_expect_tx(full, L::kKVBytes);
            const int r = it.k_tok0 + b * B;
            tma_load_3d(dst, map, full, 0, g, r);
            tma_load_3d(dst + L::kKVHalf, map, full, 64, g, r);
          }
        } else {
          const int ps = p.page_size;
          const int n_tok = min(B, it.kv_len - b * B);
          const int n_pg = (n_tok + ps - 1) / ps;
          const int pg0 = b * (B / ps);           // first page of the block (B/ps divides the window)
          const int win = pg0 / L::kPageWin, wbuf = win & 1;
          int32_t* wc = page_cache + wbuf * L::kPageWin;
          if ((wbuf ? cached_win1 : cached_win0) != win) {
            const int seq_pages = (it.kv_len + ps - 1) / ps;
            const int32_t* row = p.page_table + static_cast<int64_t>(it.seq) * p.max_pages;
            // four loads of the lane in flight at a time (one after another
            // they serialise on the memory latency)
#pragma unroll
            for (int t0 = 0; t0 < L::kPageWin / 32; t0 += 4) {
              int32_t pg[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int gp = win * L::kPageWin + lane + 32 * (t0 + t);
                pg[t] = gp < seq_pages ? __ldg(row + gp) : -1;
              }
#pragma unroll
              for (int t = 0; t < 4; ++t) wc[lane + 32 * (t0 + t)] = pg[t];
            }
            __syncwarp();
            if (wbuf) cached_win1 = win; else cached_win0 = win;
          }
          if (lane == 0) mbar_arrive_expect_tx(full, n_pg * ps * 256);
          __syncwarp();
          if (lane < n_pg) {
            int32_t pe = wc[(pg0 + lane) % L::kPageWin];
            if (pe < 0 || pe >= p.n_pages) {
              report_error(p.err, kErrBadPage, 0x104);
              pe = p.n_pages;  // out of range: the copy reads the zero fill
            }
            const int r = pe * ps;
            const int off = lane * ps * 128;
            tma_load_3d(dst + off, map, full, 0, g, r);
            tma_load_3d(dst + L::kKVHalf + off, map, full, 64, g, r);
          }
        }
        if (is_v) ++v_it; else ++k_it;
        return true;
      };
      for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
        const int item = snake_item(round);
        if (item >= p.num_items) continue;
        const ItemInfo it = item_info<MODE>(p, item);
        bool ok = mbar_wait(&bars[L::kQEmpty], (q_it & 1) ^ 1, abort, p.err, 0x101);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane == 0) {
          if (MODE == kModeDecode) {
            // one TMA row per query head, into the row of its lane quadrant
            mbar_arrive_expect_tx(&bars[L::kQFull], p.group * kHeadDim * 2);
            for (int i = 0; i < p.group; ++i) {
              uint8_t* dst = smem + L::kQOff + decode_lane_of_row(i) * 128;
              tma_load_3d(dst, &tm_q, &bars[L::kQFull], 0, it.head * p.group + i, it.seq);
              tma_load_3d(dst + L::kQHalf, &tm_q, &bars[L::kQFull], 64, it.head * p.group + i, it.seq);
            }
          } else {
            mbar_arrive_expect_tx(&bars[L::kQFull], L::kQBytes);
            const int row0 = it.q_tok0 + it.row_begin;
            tma_load_3d(smem + L::kQOff, &tm_q, &bars[L::kQFull], 0, it.head, row0);
            tma_load_3d(smem + L::kQOff + L::kQHalf, &tm_q, &bars[L::kQFull], 64, it.head, row0);
          }
        }
        ++q_it;
        const int g = (MODE == kModeDecode) ? it.head : it.head / p.group;
        cached_win0 = cached_win1 = -1;  // a new sequence's page ids
        // consumption order: K_0, K_1, V_0, K_2, V_1, ...
        bool fail = false;
        for (int j = 0; j <= it.nb && !fail; ++j) {
          if (j < it.nb && !load_kv(it, g, it.blk0 + j, false)) fail = true;
          if (!fail && j >= 1 && !load_kv(it, g, it.blk0 + j - 1, true)) fail = true;
        }
        if (fail || *abort) break;
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescS = idesc_bf16(128, B, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(128, kHeadDim, false, true);
      const Desc qd0 = make_desc(q_addr, 16, 1024);
      const uint32_t leader = elect_one_sync();
      uint32_t k_it = 0, v_it = 0, s_it = 0, pv_it = 0, q_it = 0;
      // the next item's descriptor (two levels of dependent global loads,
      // ~700 cycles) is read while the current item runs, not between the
      // last PV and the next item's first S
      ItemInfo nxt;
      if (snake_item(0) < p.num_items) nxt = item_info<MODE>(p, snake_item(0));
      for (int round = 0; snake_item(round) < p.num_items; ++round) {
        const ItemInfo it = nxt;
        // with RoPE in the prefill the softmax warps hand over the rotated tile
        bool ok = mbar_wait(&bars[ROPE ? L::kQRot : L::kQFull], q_it & 1, abort, p.err, 0x201);
        if (!__all_sync(0xffffffffu, ok)) break;
        ++q_it;
        const uint32_t kb = k_it, vb = v_it, sb = s_it, pb = pv_it;
        auto issue_s = [&](int j) -> bool {
          const uint32_t ki = kb + j;
          const uint32_t stage = ki % SK;
          bool w = mbar_wait(&bars[L::kKFull + stage], (ki / SK) & 1, abort, p.err, 0x202);
          if (!__all_sync(0xffffffffu, w)) return false;
          tc_fence_after();
          // the whole warp walks the K-steps (warp-uniform descriptors); the
          // elected lane issues
          const Desc kd0 = make_desc(smem_u32(k_base + stage * L::kKVBytes), 16, 1024);
          const uint32_t d = tm_s + ((sb + j) & 1) * 128;
          // S = Q K^T: K-steps 0-3 in the first 64-column half, 4-7 in the second
          if (leader) mma_ss<0>(d, qd0, 0, kd0, 0, kIdescS);
#pragma unroll
          for (int k = 1; k < kHeadDim / 16; ++k)
            if (leader)
              mma_ss<1>(d, qd0, (k >> 2) * (L::kQHalf >> 4) + (k & 3) * 2, kd0, (k >> 2) * (L::kKVHalf >> 4) + (k & 3) * 2,
                        kIdescS);
          if (leader) {
            umma_commit(&bars[L::kSFull + ((sb + j) & 1)]);
            umma_commit(&bars[L::kKEmpty + stage]);
          }
          __syncwarp();
          return true;
        };
        if (!issue_s(0)) break;
        if (snake_item(round + 1) < p.num_items) nxt = item_info<MODE>(p, snake_item(round + 1));
        bool fail = false;
        for (int j = 0; j < it.nb; ++j) {
          if (j + 1 < it.nb) {
            if (!issue_s(j + 1)) { fail = true; break; }
          } else {
            if (leader) umma_commit(&bars[L::kQEmpty]);  // Q no longer read
            __syncwarp();
          }
          const uint32_t sidx = sb + j, buf = sidx & 1;
          const uint32_t vi = vb + j, vstage = vi % SV;
          const uint32_t pvi = pb + j, pvbuf = pvi & 1;
          // V_j and the PV buffer are normally ready: their checks come before
          // the wait for P_j, so only that wait's wake-up follows the softmax
          bool w = mbar_wait(&bars[L::kVFull + vstage], (vi / SV) & 1, abort, p.err, 0x204);
          w = w && mbar_wait(&bars[L::kPVEmpty + pvbuf], ((pvi >> 1) & 1) ^ 1, abort, p.err, 0x205);
          w = w && mbar_wait(&bars[L::kPFull + buf], (sidx >> 1) & 1, abort, p.err, 0x203);
          if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
          uint8_t* vd = v_base + vstage * L::kKVBytes;
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
          {
            const Desc vdd = make_desc(smem_u32(vd), L::kKVHalf, 1024);
            const uint32_t a0 = tm_s + buf * 128;
            const uint32_t d = tm_pv + pvbuf * 128;
            // PV = P_hi V + P_lo V; K-step k reads V rows 16k..16k+15 (2048 B)
            if (leader) mma_ts<0>(d, a0, vdd, 0, kIdescPV);
#pragma unroll
            for (int k = 1; k < B / 16; ++k)
              if (leader) mma_ts<1>(d, a0 + 16 * k, vdd, k * 128, kIdescPV);
#pragma unroll
            for (int k = 0; k < B / 16; ++k)
              if (leader) mma_ts<1>(d, a0 + 16 * k + 8, vdd, k * 128, kIdescPV);
            if (leader) {
              umma_commit(&bars[L::kPVFull + pvbuf]);
              umma_commit(&bars[L::kVEmpty + vstage]);
            }
          }
          __syncwarp();
        }
        if (fail) break;
        k_it += it.nb;
        v_it += it.nb;
        s_it += it.nb;
        pv_it += it.nb;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // group h (warps 4-7: h = 0, warps 12-15: h = 1) takes keys
    // [h B/2, (h+1) B/2) of every global block; row r is TMEM lane r in both
    constexpr int HB = B / 2, NC = HB / 32;
    const int h = warp >= 12 ? 1 : 0;
    const int r = tid - (h ? 384 : 128);
    const int quad = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    uint64_t* xbar = &bars[L::kXch + quad];  // the quadrant's two warps meet here
    uint32_t x_par = 0, q_par = 0;
    float* xmax = reinterpret_cast<float*>(smem + L::kXchOff);  // [2][128]
    float* xsum = xmax + 2 * kTileRows;                          // [2][128]
    uint32_t s_it = 0, st_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int item = snake_item(round);
      if (item >= p.num_items) continue;
      const ItemInfo it = item_info<MODE>(p, item);
      const bool valid = row_of_lane<MODE>(r) < it.row_count;
      // a warp none of whose rows is written (decode: all but the first)
      // only takes part in the barriers
      const bool warp_rows = __any_sync(0xffffffffu, valid);
      const int pos = (MODE == kModeDecode) ? it.kv_len - 1 : it.kv_len - it.q_len + it.row_begin + r;
      bool fail = false;
      if (ROPE) {
        // RoPE of the item's query tile, in place in shared memory, while the
        // tensor core finishes the previous item: thread (h, r) rotates row
        // r's pairs 32h .. 32h + 31 -- 16-byte chunks 4h .. 4h + 3 of the
        // first half, whose partners (element i + 64) sit at the same
        // swizzled offset of the second half.  The table rows are fetched
        // before the tile lands.
        if (valid) rope_prefetch(p.rope_table + static_cast<int64_t>(pos) * kHeadDim + 32 * h);
        bool w = mbar_wait(&bars[L::kQFull], q_par, abort, p.err, 0x304);
        q_par ^= 1;
        if (!__all_sync(0xffffffffu, w)) break;
        if (valid) rope_row_quarter(p.rope_table + static_cast<int64_t>(pos) * kHeadDim + 32 * h, smem + L::kQOff, r, h);
        fence_proxy_async_smem();  // the tensor core reads the tile through the async proxy
        mbar_arrive(&bars[L::kQRot]);
      }
      for (int j = 0; j < it.nb; ++j) {
        const int b = it.blk0 + j;
        const uint32_t buf = s_it & 1;
        bool w = mbar_wait(&bars[L::kSFull + buf], (s_it >> 1) & 1, abort, p.err, 0x301);
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        tc_fence_after();
        const uint32_t ta = tm_s + lane_off + buf * 128 + h * HB;
        const int nvis = valid ? visible_keys(pos, it.kv_len, b, B) : 0;
        const bool has = nvis > 0;
        const int hv = min(max(nvis - h * HB, 0), HB);  // visible keys of this half
        // every row of the warp that is written sees all keys of the half: no
        // masking (a row that is not written may hold anything: MMA rows are
        // independent and its state is never stored)
        const bool full = __all_sync(0xffffffffu, !valid || hv == HB);
        uint32_t sv[NC][32];
        float lse_b = -INFINITY, rcp = 0.0f, mc = 0.0f;
        if (warp_rows) xmax[h * kTileRows + r] = half_load<NC>(ta, full, hv, sv);
        mbar_arrive(xbar);
        w = mbar_wait(xbar, x_par, abort, p.err, 0x302);
        x_par ^= 1;
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        if (warp_rows) {
          const float m = fmaxf(xmax[r], xmax[kTileRows + r]);  // exact
          mc = has ? __fmul_rn(m, p.scale_log2) : 0.0f;
          xsum[h * kTileRows + r] = half_probs<NC>(ta, sv, p.scale_log2, mc);
        }
        // P is in TMEM: the PV product may start while the half sums are
        // exchanged and the block statistics formed (only the correction
        // warps read those)
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[L::kPFull + buf]);
        mbar_arrive(xbar);
        w = mbar_wait(xbar, x_par, abort, p.err, 0x303);
        x_par ^= 1;
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        if (h == 0 && warp_rows && has) block_stats(mc, __fadd_rn(xsum[r], xsum[kTileRows + r]), lse_b, rcp);
        if (h == 0) {
          stats[(st_it % SR) * kTileRows + r] = make_float2(lse_b, rcp);
          mbar_arrive(&bars[L::kStatsFull + (st_it % SR)]);
        }
        ++s_it;
        ++st_it;
      }
      if (fail) break;
    }
  } else {
    // ------------------------------------------------------------ correction / epilogue
    setmaxnreg_inc208();
    const int r = tid;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t pv_it = 0, st_it = 0;
    float O[kHeadDim];
#pragma unroll
    for (int e = 0; e < kHeadDim; ++e) O[e] = 0.0f;
    // in the fused mode the next item's descriptor is read ahead: the
    // epilogue already puts these warps behind the PV products at an item
    // start.  The states mode reads it in place: its epilogue stores the
    // states block by block, and there the read-ahead measured ~6 % slower.
    ItemInfo nxt;
    if (MODE == kModeFused && snake_item(0) < p.num_items) nxt = item_info<MODE>(p, snake_item(0));
    for (int round = 0; snake_item(round) < p.num_items; ++round) {
      ItemInfo it;
      if (MODE == kModeFused) {
        it = nxt;
        if (snake_item(round + 1) < p.num_items) nxt = item_info<MODE>(p, snake_item(round + 1));
      } else {
        it = item_info<MODE>(p, snake_item(round));
      }
      const bool valid = row_of_lane<MODE>(r) < it.row_count;
      const bool warp_rows = __any_sync(0xffffffffu, valid);
      float Lrun = -INFINITY;
      int64_t slab_off = it.slab_off;  // states: the slab of block blk0 + j
      bool fail = false;
      for (int j = 0; j < it.nb; ++j) {
        const uint32_t buf = pv_it & 1;
        bool w = mbar_wait(&bars[L::kPVFull + buf], (pv_it >> 1) & 1, abort, p.err, 0x401);
        w = w && mbar_wait(&bars[L::kStatsFull + (st_it % SR)], (st_it / SR) & 1, abort, p.err, 0x402);
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        tc_fence_after();
        const uint32_t ta = tm_pv + lane_off + buf * 128;
        const float2 st = stats[(st_it % SR) * kTileRows + r];
        const float lse_b = st.x, rcp = st.y;
        const bool has = valid && (lse_b != -INFINITY);
        uint32_t x0[32], x1[32];
        if (!warp_rows) {
          tc_fence_before();
          mbar_arrive(&bars[L::kPVEmpty + buf]);
        } else if (MODE == kModeStates) {
          tmem_ld32(ta, x0);
          tmem_ld32(ta + 32, x1);
          // the warp's 32 rows are consecutive pairs of the slab: their
          // state rows are one contiguous 16 KB span
          const int slab_rb = max(0, (it.blk0 + j) * B - (it.kv_len - it.q_len));
          const int slab_rc = it.q_len - slab_rb;
          const int64_t pair = slab_off + static_cast<int64_t>(it.head) * slab_rc + (it.row_begin + r - slab_rb);
          slab_off += static_cast<int64_t>(slab_rc) * p.hq;
          const int64_t pair0 = pair - lane;
          const uint32_t has_mask = __ballot_sync(0xffffffffu, has);
          // each 32-column chunk goes through shared memory (chunk j of a
          // row in slot j ^ (row & 7)) and leaves as whole 128-byte lines,
          // four rows per store instruction
          float4* stg = reinterpret_cast<float4*>(smem + L::kEpiOff + (warp & 3) * (32 * 128));
          auto put_chunk = [&](const uint32_t (&xa)[32], int c) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              stg[lane * 8 + (j ^ (lane & 7))] =
                  make_float4(state_elem(__uint_as_float(xa[4 * j]), rcp), state_elem(__uint_as_float(xa[4 * j + 1]), rcp),
                              state_elem(__uint_as_float(xa[4 * j + 2]), rcp), state_elem(__uint_as_float(xa[4 * j + 3]), rcp));
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int rr = 4 * k + (lane >> 3), jj = lane & 7;
              const float4 v = stg[rr * 8 + (jj ^ (rr & 7))];
              if ((has_mask >> rr) & 1u)
                reinterpret_cast<float4*>(p.state_o + (pair0 + rr) * kHeadDim + 32 * c)[jj] = v;
            }
            __syncwarp();
          };
          tmem_ld_wait(x0);
          tmem_ld_wait(x1);
          if (has_mask) {
            put_chunk(x0, 0);
            put_chunk(x1, 1);
          }
          tmem_ld32(ta + 64, x0);
          tmem_ld32(ta + 96, x1);
          tmem_ld_wait(x0);
          tmem_ld_wait(x1);
          tc_fence_before();
          mbar_arrive(&bars[L::kPVEmpty + buf]);  // PV read: the buffer is free
          if (has_mask) {
            put_chunk(x0, 2);
            put_chunk(x1, 3);
          }
          if (has) p.state_lse[pair] = lse_b;
        } else {
          tmem_ld32(ta, x0);
          float Lp = 0.f, alpha = 0.f, beta = 0.f;
          if (j > 0 && has) fold_coeffs(Lrun, lse_b, Lp, alpha, beta);  // overlaps the PV load
          const float2 rc2 = make_float2(rcp, rcp), al2 = make_float2(alpha, alpha), be2 = make_float2(beta, beta);
          // o_b = PV * (1/l); O = fma(o_b, beta, O * alpha)  (packed, two lanes at a time)
          auto fold32 = [&](const uint32_t (&xa)[32], int o0) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 oa = fmul2(make_float2(__uint_as_float(xa[e]), __uint_as_float(xa[e + 1])), rc2);
              if (j == 0) {
                O[o0 + e] = oa.x;
                O[o0 + e + 1] = oa.y;
              } else if (has) {
                const float2 ra = ffma2(oa, be2, fmul2(make_float2(O[o0 + e], O[o0 + e + 1]), al2));
                O[o0 + e] = ra.x;
                O[o0 + e + 1] = ra.y;
              }
            }
          };
          tmem_ld_wait(x0);
          tmem_ld32(ta + 32, x1);
          fold32(x0, 0);
          tmem_ld_wait(x1);
          tmem_ld32(ta + 64, x0);
          fold32(x1, 32);
          tmem_ld_wait(x0);
          tmem_ld32(ta + 96, x1);
          fold32(x0, 64);
          tmem_ld_wait(x1);
          tc_fence_before();
          mbar_arrive(&bars[L::kPVEmpty + buf]);  // PV read: the buffer is free
          fold32(x1, 96);
          if (has) Lrun = (j == 0) ? lse_b : Lp;
        }
        ++pv_it;
        ++st_it;
      }
      if (fail) break;
      if (MODE == kModeFused) {
        // epilogue: O and L are final.  Each warp stages its 32 rows through
        // shared memory one 128-byte column chunk at a time (chunk j of a
        // row in slot j ^ (row & 7), so neither side conflicts on banks) and
        // writes four whole rows' chunks per store instruction.
        float4* stg = reinterpret_cast<float4*>(smem + L::kEpiOff + (warp & 3) * (32 * 128));
        const int r0 = (warp & 3) * 32;
        const int64_t row_base = static_cast<int64_t>(it.q_tok0 + it.row_begin) * p.hq + it.head;
        auto write_chunks = [&](auto&& store) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lane >> 3), jj = lane & 7;
            const int tr = r0 + rr;
            const float4 v = stg[rr * 8 + (jj ^ (rr & 7))];
            if (tr < it.row_count) store(row_base + static_cast<int64_t>(tr) * p.hq, jj, v);
          }
        };
        if (p.out_f32) {
#pragma unroll
          for (int c = 0; c < kHeadDim / 32; ++c) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              stg[lane * 8 + (j ^ (lane & 7))] =
                  make_float4(O[32 * c + 4 * j], O[32 * c + 4 * j + 1], O[32 * c + 4 * j + 2], O[32 * c + 4 * j + 3]);
            __syncwarp();
            write_chunks([&](int64_t row_idx, int jj, const float4& v) {
              reinterpret_cast<float4*>(p.out_f32 + row_idx * kHeadDim + 32 * c)[jj] = v;
            });
            __syncwarp();
          }
        }
        if (p.out_bf16) {
#pragma unroll
          for (int c = 0; c < kHeadDim / 64; ++c) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int e = 64 * c + 8 * j;
              const uint4 w = make_uint4(pack_bf16x2(O[e], O[e + 1]), pack_bf16x2(O[e + 2], O[e + 3]),
                                         pack_bf16x2(O[e + 4], O[e + 5]), pack_bf16x2(O[e + 6], O[e + 7]));
              stg[lane * 8 + (j ^ (lane & 7))] = *reinterpret_cast<const float4*>(&w);
            }
            __syncwarp();
            write_chunks([&](int64_t row_idx, int jj, const float4& v) {
              reinterpret_cast<float4*>(p.out_bf16 + row_idx * kHeadDim + 64 * c)[jj] = v;
            });
            __syncwarp();
          }
        }
        if (p.lse && valid) p.lse[row_base + static_cast<int64_t>(r) * p.hq] = Lrun;
      } else if (MODE == kModeDecode && valid) {
        // epilogue (decode): the group's rows are spread over the lane
        // quadrants; few rows, written directly
        const int64_t row_idx = static_cast<int64_t>(it.seq) * p.hq + it.head * p.group + row_of_lane<MODE>(r);
        if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(p.out_f32 + row_idx * kHeadDim);
#pragma unroll
          for (int e = 0; e < kHeadDim; e += 4) dst[e / 4] = make_float4(O[e], O[e + 1], O[e + 2], O[e + 3]);
        }
        if (p.out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + row_idx * kHeadDim);
#pragma unroll
          for (int e = 0; e < kHeadDim; e += 8)
            dst[e / 8] = make_uint4(pack_bf16x2(O[e], O[e + 1]), pack_bf16x2(O[e + 2], O[e + 3]),
                                    pack_bf16x2(O[e + 4], O[e + 5]), pack_bf16x2(O[e + 6], O[e + 7]));
        }
        if (p.lse) p.lse[row_idx] = Lrun;
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
template <int B, int MODE, bool ROPE>
static cudaError_t configure_fwd_t() {
  using L = FwdLayout<B>;
  auto kern = rlk_fwd_kernel<B, MODE, ROPE>;
  // The warpgroup register split (208 / 128 / 128 / 48) needs the launch to
  // grant 128 registers per thread; with fewer, setmaxnreg.inc would wait
  // forever.
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, kern);
  if (e != cudaSuccess) return e;
  if (a.numRegs < kRegsLaunch) {
    fprintf(stderr, "rlk_fwd_kernel<%d,%d,%d>: %d registers at launch, the warpgroup split needs %d\n", B, MODE,
            ROPE ? 1 : 0, a.numRegs, kRegsLaunch);
    return cudaErrorInvalidConfiguration;
  }
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
}

cudaError_t configure_fwd_kernels() {
  cudaError_t e;
  if ((e = configure_fwd_t<128, kModeFused, false>()) != cudaSuccess) return e;
  if ((e = configure_fwd_t<128, kModeFused, true>()) != cudaSuccess) return e;
  if ((e = configure_fwd_t<128, kModeStates, false>()) != cudaSuccess) return e;
  if ((e = configure_fwd_t<128, kModeDecode, false>()) != cudaSuccess) return e;
  if ((e = configure_fwd_t<64, kModeFused, false>()) != cudaSuccess) return e;
  if ((e = configure_fwd_t<64, kModeFused, true>()) != cudaSuccess) return e;
  if ((e = configure_fwd_t<64, kModeStates, false>()) != cudaSuccess) return e;
  return configure_fwd_t<64, kModeDecode, false>();
}

template <int B, int MODE, bool ROPE>
static cudaError_t launch_fwd_t(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t stream) {
  rlk_fwd_kernel<B, MODE, ROPE><<<grid, kThreads, FwdLayout<B>::kAlloc, stream>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t stream) {
  const bool rope = p.rope_table != nullptr;
  if (p.block == 128) {
    switch (p.mode) {
      case kModeFused:
        return rope ? launch_fwd_t<128, kModeFused, true>(p, tq, tk, tv, grid, stream)
                    : launch_fwd_t<128, kModeFused, false>(p, tq, tk, tv, grid, stream);
      case kModeStates: return launch_fwd_t<128, kModeStates, false>(p, tq, tk, tv, grid, stream);
      case kModeDecode: return launch_fwd_t<128, kModeDecode, false>(p, tq, tk, tv, grid, stream);
    }
  } else if (p.block == 64) {
    switch (p.mode) {
      case kModeFused:
        return rope ? launch_fwd_t<64, kModeFused, true>(p, tq, tk, tv, grid, stream)
                    : launch_fwd_t<64, kModeFused, false>(p, tq, tk, tv, grid, stream);
      case kModeStates: return launch_fwd_t<64, kModeStates, false>(p, tq, tk, tv, grid, stream);
      case kModeDecode: return launch_fwd_t<64, kModeDecode, false>(p, tq, tk, tv, grid, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace rlk
