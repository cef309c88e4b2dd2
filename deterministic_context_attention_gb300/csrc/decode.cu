// decode.cu -- paged-KV decode for sm_103a in transposed form.
//
// A decode step has one query token per sequence, so the query rows of one
// (sequence, KV head) item are only the group's query heads (4 for 32 / 8).
// The forward engine's 128-row tile would leave 124 of its 128 MMA rows
// idle; this kernel instead puts the KV block's 128 keys on the MMA's M side:
//   S^T = K_b Q^T        (M = 128 keys, N = 16 query columns, K = 128 dims)
//   O^T = V_b^T P^T      (M = 128 dims, N = 16 query columns, K = 128 keys)
// with the group padded to N = 16 by zero rows.  The block state of every
// query head is the same as the prefill's ("WS2 Attention PR5 Drift
// Benchmark", Transformer Engine Reuse: state_b = (o_b, lse_b, b)) and every
// floating-point step is the one numerics.cuh defines, in the same order:
// the block maximum (exact), p = 2^fma(S, scale_log2, -m scale_log2), the
// canonical row sum (per 64-key half, key c to partial c mod 16 in
// ascending key order and the fixed 8-4-2-1 tree; then half 0 + half 1), P = P_hi + P_lo, PV accumulated over the hi
// K-steps then the lo K-steps, o_b = PV / l and the canonical fold in
// ascending global_block_index order.  The tensor core gives the same bits
// for a product and for its transposed formulation, so a decode row equals
// the prefill's last row of the same sequence bit for bit.
//
// Warp roles (512 threads):
//   warps 0-3   correction / epilogue: thread d owns TMEM lane d (head
//               dimension d) and keeps the running O of every query head
//   warps 4-7   softmax of the even blocks, warps 8-11 of the odd blocks:
//               thread t owns TMEM lane t (key t of the block)
//   warp  12    TMA producer of the group's query rows and the K pages
//   warp  13    TMA producer of the V pages
//   warp  14    TMEM allocator and issuer of the S^T products
//   warp  15    issuer of the O^T (PV) products (two issuers: these small
//               MMAs are issue-bound, 7 % on a few long sequences)
// Split decode with the fold on chip adds CTAs past the work items, on SMs
// the producers leave free, whose warps fold one (sequence, KV head, query
// head) each as the producers write the block states.
// TMEM (128 columns): S^T ring [0,64), O^T ring [64,128), 16 columns a slot.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>

#include "numerics.cuh"
#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kDThreads = 512;
constexpr int kDN = 16;  // MMA N: the group's query heads, padded with zero rows

struct DecLayout {
  static constexpr int B = 128;
  static constexpr int kSK = 3, kSV = 2;  // K and V rings
  static constexpr int kPS = 2;           // P^T operand slots
  static constexpr int kSS = 4, kOS = 4;  // TMEM rings of S^T and O^T
  static constexpr int kSR = 8;           // statistics ring
  static constexpr int kKVHalf = B * 128;                 // one 64-dim half of a K or V block
  static constexpr int kKVBytes = 2 * kKVHalf;
  static constexpr int kTHalf = kDN * 128;                // one 64-column half of a 16-row operand
  static constexpr int kTBytes = 2 * kTHalf;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTBytes;
  static constexpr int kVOff = kKOff + kSK * kKVBytes;
  static constexpr int kPOff = kVOff + kSV * kKVBytes;    // [slot][hi, lo] tiles
  // per softmax group: block maxima float [2][4][kDecodeMaxGroup] and
  // partial sums float [2][4][kDecodeMaxGroup][32], double-buffered by block
  static constexpr int kRedBytes = 2 * 4 * kDecodeMaxGroup * 4;
  static constexpr int kPartBytes = 2 * 4 * kDecodeMaxGroup * 32 * 4;
  static constexpr int kRedOff = kPOff + kPS * 2 * kTBytes;
  static constexpr int kPartOff = kRedOff + 2 * kRedBytes;
  static constexpr int kStatsOff = kPartOff + 2 * kPartBytes;  // float2 [kSR][kDecodeMaxGroup]
  static constexpr int kBarOff = kStatsOff + kSR * kDecodeMaxGroup * 8;
  static constexpr int kQFull = 0, kQEmpty = 1, kKFull = 2, kKEmpty = kKFull + kSK, kVFull = kKEmpty + kSK,
                       kVEmpty = kVFull + kSV, kSFull = kVEmpty + kSV, kSEmpty = kSFull + kSS,
                       kPFull = kSEmpty + kSS, kPEmpty = kPFull + kPS, kOFull = kPEmpty + kPS,
                       kOEmpty = kOFull + kOS, kStatsFull = kOEmpty + kOS, kSyncMax = kStatsFull + kSR,
                       kSyncPart = kSyncMax + 4, kQRope = kSyncPart + 4,  // sync: [group][parity]
                       kFillDone = kQRope + 1,  // split decode: the table fill (correction + softmax warps)
                       kNumBars = kFillDone + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base (u32), abort (i32)
  static constexpr int kPageWin = 512;                     // page ids cached per window (one per producer)
  static constexpr int kPageOff = (kMiscOff + 16 + 15) / 16 * 16;
  static constexpr int kTotal = kPageOff + 2 * kPageWin * 4;
  static constexpr int kAlloc = kTotal + 1024;
};
static_assert(DecLayout::kAlloc <= 232448, "decode shared memory");
static_assert(DecLayout::kPageWin == 1 << 9, "the producers index the page window with shifts by 9");
static_assert(DecLayout::kKOff % 1024 == 0 && DecLayout::kVOff % 1024 == 0 && DecLayout::kPOff % 1024 == 0,
              "128-byte-swizzled tiles start on 1024-byte boundaries");

// Byte offset of element (row, col) of a 16-row operand tile of 128 BF16
// columns, stored K-major as two 64-column halves in the 128-byte swizzle
// (the layout a TMA load with 128-byte swizzle produces).
__device__ __forceinline__ uint32_t tile16_off(int row, int col) {
  const int half = col >> 6, c = col & 63;
  const uint32_t chunk = static_cast<uint32_t>(c >> 3) ^ static_cast<uint32_t>(row & 7);
  return static_cast<uint32_t>(half * DecLayout::kTHalf + row * 128) + chunk * 16 + static_cast<uint32_t>(c & 7) * 2;
}

__device__ __forceinline__ int dec_snake_item(int round) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return round * g + ((round & 1) ? g - 1 - c : c);
}

__device__ __forceinline__ float bf16_bits_as_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// One item: the query heads of KV head g of sequence seq against the global
// blocks b0, b0 + stride, ... (nb of them).  Plain decode: all of the
// sequence's blocks (stride 1), folded on chip.  Split decode (state_o set):
// a fixed range of them (stride 1), or with the fold on chip the blocks
// b = r (mod split_stride) of item r; their block states are written to the
// state table at pair (cu_q[seq] + b) * hq + head, for the merge kernel or
// the fold CTAs to fold.
struct DecItem {
  int seq, g, kv_len, b0, nb, stride;
};
__device__ __forceinline__ DecItem dec_item(const FwdParams& p, int item) {
  const FwdTile& t = p.tiles[item];
  DecItem d;
  d.seq = t.seq;
  d.g = t.row_begin;
  d.kv_len = p.cu_k[t.seq];
  d.stride = 1;
  if (p.state_o) {
    d.b0 = t.block;
    d.nb = t.slab_row_count;
    if (p.split_stride > 0) {
      d.stride = p.split_stride;
    }
  } else {
    d.b0 = 0;
    d.nb = (d.kv_len + DecLayout::B - 1) / DecLayout::B;
  }
  return d;
}

// Split decode with the fold on chip: thread t of the 384 correction and
// softmax threads writes its share of the item's state-table slots with
// kUnwritten (o_b as 16-byte pieces, then lse_b) before any of the item's
// states can land.
constexpr int kFillThreads = 384;
__device__ __forceinline__ void fill_item_slots(const FwdParams& p, const DecItem& di, int G, int t) {
  const int64_t blk0 = p.cu_q[di.seq] + di.b0;
  const int per = G * (kHeadDim / 4);  // 16-byte pieces of one block's states
  const float u = __uint_as_float(kUnwritten);
  const float4 u4 = make_float4(u, u, u, u);
  for (int i = t; i < di.nb * per; i += kFillThreads) {
    const int j = i / per;
    reinterpret_cast<float4*>(p.state_o + ((blk0 + static_cast<int64_t>(j) * di.stride) * p.hq + di.g * G) *
                                              kHeadDim)[i - j * per] = u4;
  }
  for (int i = t; i < di.nb * G; i += kFillThreads) {
    const int j = i / G;
    p.state_lse[(blk0 + static_cast<int64_t>(j) * di.stride) * p.hq + di.g * G + (i - j * G)] = u;
  }
}

// Row maximum of the 32 lanes of a warp (exact; every lane receives it).
__device__ __forceinline__ float warp_max(float v) {
  float m;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}

// Split decode with the fold on chip, the fold side: one warp folds query
// head q of the pair (seq, g) over the pair's block states in ascending block
// order as the producer CTAs write them -- the fold the correction role
// applies in the single pass, operation for operation, so the result is the
// same bit for bit.  Lane l folds head dimensions 4 l .. 4 l + 3 and every
// lane runs the head's lse chain (the same inputs, so no lane waits on
// another).
//
// C blocks at a time, the next chunk's reads in flight while the current one
// folds.  The table holds the all-ones NaN until a state lands (arithmetic
// never produces that pattern, and a 32-bit store lands whole, so a value
// that differs from it is the final one).  Reads are weak first (they overlap
// one another); values still unwritten, or stale, are read again with strong
// (device-scope relaxed) loads, which the memory model guarantees to see
// other SMs' stores eventually (a thread's strong loads complete one after
// another).  When the producers fill the table themselves (fill_flag set),
// the chain first waits until every item of the pair has published its
// flag: before that, an item's slots may still hold an earlier call's
// states.  Returns false on a timeout (reported) or an abort.
__device__ __noinline__ bool fold_chain_on_chip(const FwdParams& p, int seq, int g, int q, int lane,
                                                volatile int* abort) {
  constexpr int C = 8;
  const int G = p.group;
  const int nbp = (p.cu_k[seq] + DecLayout::B - 1) / DecLayout::B;
  const int64_t base = p.cu_q[seq];
  // lane i: the lse of block c0 + i; every lane: dimensions 4 lane .. of the
  // chunk's blocks (past the chunk: its last block, a valid value)
  auto lse_src = [&](int c0, int nc) { return p.state_lse + (base + c0 + min(lane, nc - 1)) * p.hq + g * G + q; };
  auto o_src = [&](int c0, int nc, int i) {
    return p.state_o + ((base + c0 + min(i, nc - 1)) * p.hq + g * G + q) * kHeadDim + 4 * lane;
  };
  auto issue = [&](int c0, float& lsl, float4 (&v)[C]) {
    const int nc = min(C, nbp - c0);
    lsl = ld_l2_weak(lse_src(c0, nc));
#pragma unroll
    for (int i = 0; i < C; ++i) v[i] = ld_l2_weak4(o_src(c0, nc, i));
  };
  auto unwritten4 = [](const float4& a) {
    return __float_as_uint(a.x) == kUnwritten || __float_as_uint(a.y) == kUnwritten ||
           __float_as_uint(a.z) == kUnwritten || __float_as_uint(a.w) == kUnwritten;
  };
  // until every value of the chunk has landed: strong re-reads of what is missing
  auto settle = [&](int c0, float& lsl, float4 (&v)[C]) -> bool {
    const int nc = min(C, nbp - c0);
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      uint32_t miss = static_cast<uint32_t>(__float_as_uint(lsl) == kUnwritten);
#pragma unroll
      for (int i = 0; i < C; ++i) miss |= static_cast<uint32_t>(unwritten4(v[i]));
      if (__all_sync(0xffffffffu, miss == 0)) return true;
      const bool late = __shfl_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitTimeoutNs, 0);
      if (late || *abort) {
        if (late && lane == 0) {
          *abort = 1;
          report_error(p.err, kErrDeviceTimeout, 0x901);
        }
        return false;
      }
      if (__float_as_uint(lsl) == kUnwritten) lsl = ld_l2_poll(lse_src(c0, nc));
#pragma unroll
      for (int i = 0; i < C; ++i)
        if (unwritten4(v[i])) v[i] = ld_l2_poll4(o_src(c0, nc, i));
    }
  };
  if (p.fill_flag) {
    // lane r (and r + 32): item r's flag; the warp barrier then orders every
    // lane's table reads after the acquiring loads
    const int nr = min(p.split_stride, nbp);
    const uint64_t* flag = p.fill_flag + (static_cast<int64_t>(seq) * p.hkv + g) * kMaxSplitK;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      bool filled = true;
      for (int r = lane; r < nr; r += 32) filled = ld_acquire_u64(flag + r) == p.fill_nonce && filled;
      if (__all_sync(0xffffffffu, filled)) break;
      const bool late = __shfl_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitTimeoutNs, 0);
      if (late || *abort) {
        if (late && lane == 0) {
          *abort = 1;
          report_error(p.err, kErrDeviceTimeout, 0x903);
        }
        return false;
      }
    }
    __syncwarp();
  }
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  float Lrun = -INFINITY;
  float lsl, lsn = 0.f;
  float4 v[C], vn[C];
  issue(0, lsl, v);
  for (int c0 = 0; c0 < nbp; c0 += C) {
    const int nc = min(C, nbp - c0);
    if (!settle(c0, lsl, v)) return false;
    if (c0 + C < nbp) issue(c0 + C, lsn, vn);  // lands while this chunk folds
#pragma unroll
    for (int i = 0; i < C; ++i) {
      if (i < nc) {
        const float lb = __shfl_sync(0xffffffffu, lsl, i);
        if (c0 + i == 0) {
          O = v[i];
          Lrun = lb;
        } else {
          float Lp, al, be;
          fold_coeffs(Lrun, lb, Lp, al, be);
          O.x = __fmaf_rn(v[i].x, be, __fmul_rn(O.x, al));
          O.y = __fmaf_rn(v[i].y, be, __fmul_rn(O.y, al));
          O.z = __fmaf_rn(v[i].z, be, __fmul_rn(O.z, al));
          O.w = __fmaf_rn(v[i].w, be, __fmul_rn(O.w, al));
          Lrun = Lp;
        }
      }
    }
    lsl = lsn;
#pragma unroll
    for (int i = 0; i < C; ++i) v[i] = vn[i];
  }
  const int64_t row = static_cast<int64_t>(seq) * p.hq + g * G + q;
  if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + row * kHeadDim + 4 * lane) = O;
  if (p.out_bf16) {
    const uint32_t w0 = pack_bf16x2(O.x, O.y), w1 = pack_bf16x2(O.z, O.w);
    *reinterpret_cast<uint2*>(p.out_bf16 + row * kHeadDim + 4 * lane) = make_uint2(w0, w1);
  }
  if (lane == 0 && p.lse) p.lse[row] = Lrun;
  return true;
}

// MG: the group's query heads rounded up to 1, 2, 4 or 8 (heads at or past
// the group size are skipped at run time).
// FOLD: the instance the split decode with the fold on chip launches (its
// CTAs past the items fold); the others never carry the fold code.
template <int MG, bool FOLD>
__global__ void __launch_bounds__(kDThreads, 1)
    rlk_decode_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = DecLayout;
  constexpr int B = L::B, SK = L::kSK, SV = L::kSV, PS = L::kPS, SS = L::kSS, OS = L::kOS, SR = L::kSR;
  static_assert(MG <= kDecodeMaxGroup && PS == 2, "decode layout");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  float2* stats = reinterpret_cast<float2*>(smem + L::kStatsOff);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.group;

  // operand rows at or past G are never written: they must read as zero
  for (int i = tid; i < L::kTBytes / 16; i += kDThreads)
    reinterpret_cast<uint4*>(smem + L::kQOff)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < PS * 2 * L::kTBytes / 16; i += kDThreads)
    reinterpret_cast<uint4*>(smem + L::kPOff)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
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
    for (int s = 0; s < SS; ++s) {
      mbar_init(&bars[L::kSFull + s], 1);
      mbar_init(&bars[L::kSEmpty + s], 128);
    }
    for (int s = 0; s < PS; ++s) {
      mbar_init(&bars[L::kPFull + s], 128);
      mbar_init(&bars[L::kPEmpty + s], 1);
    }
    for (int s = 0; s < OS; ++s) {
      mbar_init(&bars[L::kOFull + s], 1);
      mbar_init(&bars[L::kOEmpty + s], 128);
    }
    for (int s = 0; s < SR; ++s) mbar_init(&bars[L::kStatsFull + s], 128);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars[L::kSyncMax + s], 128);
      mbar_init(&bars[L::kSyncPart + s], 128);
    }
    mbar_init(&bars[L::kQRope], 128);
    mbar_init(&bars[L::kFillDone], kFillThreads);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 14) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s = tmem;       // S^T slots: + 16 * slot
  const uint32_t tm_o = tmem + 64;  // O^T slots: + 16 * slot
  uint8_t* q_tile = smem + L::kQOff;
  uint8_t* k_base = smem + L::kKOff;
  uint8_t* v_base = smem + L::kVOff;
  uint8_t* p_base = smem + L::kPOff;

  if (FOLD && static_cast<int>(blockIdx.x) >= p.num_items) {
    // ------------------------------------------------------------ fold CTA
    // split decode with the fold on chip: the CTAs past the items, on SMs
    // the producers leave free, fold one (sequence, KV head, query head)
    // chain a warp, in (sequence, KV head, query head) order
    const int chain = (static_cast<int>(blockIdx.x) - p.num_items) * (kDThreads / 32) + warp;
    const int per_seq = p.hkv * G;
    if (p.split_stride > 0 && chain < p.fold_seqs * per_seq) {
      const int seq = chain / per_seq, g = (chain % per_seq) / G, q = chain % G;
      fold_chain_on_chip(p, seq, g, q, lane, abort);
    }
  } else if (warp == 12 || warp == 13) {
    // ------------------------------------------------------------ producers
    // warp 12 loads the query rows and K, warp 13 V, so neither ring waits
    // on the other's free slots
    const bool is_v = warp == 13;
    const CUtensorMap* map = is_v ? &tm_v : &tm_k;
    if (lane == 0) {
      if (!is_v) tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(map);
    }
    const int S = is_v ? SV : SK;
    uint64_t* full_b = &bars[is_v ? L::kVFull : L::kKFull];
    uint64_t* empty_b = &bars[is_v ? L::kVEmpty : L::kKEmpty];
    uint8_t* ring = is_v ? v_base : k_base;
    // the page ids of the current sequence, one window cached per producer
    int32_t* wc = reinterpret_cast<int32_t*>(smem + L::kPageOff) + (is_v ? L::kPageWin : 0);
    uint32_t it_n = 0, q_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int item = dec_snake_item(round);
      if (item >= p.num_items) continue;
      const DecItem di = dec_item(p, item);
      const int seq = di.seq, g = di.g, kv_len = di.kv_len, nb = di.nb;
      if (!is_v) {
        bool ok = mbar_wait(&bars[L::kQEmpty], (q_it & 1) ^ 1, abort, p.err, 0x501);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane == 0) {
          // the group's query rows 0..G-1 of the 16-row operand tile
          mbar_arrive_expect_tx(&bars[L::kQFull], G * kHeadDim * 2);
          for (int i = 0; i < G; ++i) {
            tma_load_3d(q_tile + i * 128, &tm_q, &bars[L::kQFull], 0, g * G + i, seq);
            tma_load_3d(q_tile + L::kTHalf + i * 128, &tm_q, &bars[L::kQFull], 64, g * G + i, seq);
          }
        }
        ++q_it;
      }
      const int ps = p.page_size;
      const int seq_pages = (kv_len + ps - 1) / ps;
      const int32_t* prow = p.page_table + static_cast<int64_t>(seq) * p.max_pages;
      int cached = -1;  // a new sequence's page ids
      const int lg = 31 - __clz(B / ps);  // log2 of the pages per block
      bool fail = false;
      for (int j = 0; j < nb; ++j) {
        const int b = di.b0 + j * di.stride;  // global block
        const uint32_t stage = it_n % S;
        bool ok = mbar_wait(empty_b + stage, ((it_n / S) & 1) ^ 1, abort, p.err, is_v ? 0x503 : 0x502);
        if (!__all_sync(0xffffffffu, ok)) { fail = true; break; }
        uint8_t* dst = ring + stage * L::kKVBytes;
        const int n_tok = min(B, kv_len - b * B);
        const int n_pg = (n_tok + ps - 1) / ps;
        // the window holds the pages of 2^(9 - lg) consecutive blocks of the
        // item (a block's 2^lg pages: page_size is a power of two dividing B)
        const int win = j >> (9 - lg);
        if (cached != win) {
          // the lane's 16 loads all in flight before the first store (one
          // after another they took ~10 us, the whole start of a long item)
          int32_t pg[L::kPageWin / 32];
#pragma unroll
          for (int t = 0; t < L::kPageWin / 32; ++t) {
            const int i = lane + 32 * t;
            const int jj = (win << (9 - lg)) + (i >> lg);  // block of the item
            const int gp = ((di.b0 + jj * di.stride) << lg) + (i & ((1 << lg) - 1));
            pg[t] = (jj < nb && gp < seq_pages) ? __ldg(prow + gp) : -1;
          }
#pragma unroll
          for (int t = 0; t < L::kPageWin / 32; ++t) wc[lane + 32 * t] = pg[t];
          __syncwarp();
          cached = win;
        }
        if (lane == 0) mbar_arrive_expect_tx(full_b + stage, n_pg * ps * 256);
        __syncwarp();
        if (lane < n_pg) {
          int32_t pe = wc[((j & ((1 << (9 - lg)) - 1)) << lg) + lane];
          if (pe < 0 || pe >= p.n_pages) {
            report_error(p.err, kErrBadPage, 0x504);
            pe = p.n_pages;  // out of range: the copy reads the zero fill
          }
          const int r = pe * ps;
          const int off = lane * ps * 128;
          tma_load_3d(dst + off, map, full_b + stage, 0, g, r);
          tma_load_3d(dst + L::kKVHalf + off, map, full_b + stage, 64, g, r);
        }
        ++it_n;
      }
      if (fail || *abort) break;
    }
  } else if (warp == 14) {
    // ------------------------------------------------------------ S issuer
    constexpr uint32_t kIdS = idesc_bf16(128, kDN, false, false);  // A = K (K-major), B = Q (K-major)
    const Desc qd = make_desc(smem_u32(q_tile), 16, 1024);
    const uint32_t leader = elect_one_sync();
    uint32_t k_it = 0, s_it = 0, q_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int item = dec_snake_item(round);
      if (item >= p.num_items) continue;
      const DecItem di = dec_item(p, item);
      const int kv_len = di.kv_len, nb = di.nb;
      // with RoPE the correction warps hand over the rotated rows
      bool ok = mbar_wait(&bars[p.rope_table ? L::kQRope : L::kQFull], q_it & 1, abort, p.err, 0x601);
      if (!__all_sync(0xffffffffu, ok)) break;
      ++q_it;
      const uint32_t kb = k_it, sb = s_it;
      // S^T_j = K_j Q^T into S^T slot (sb + j) mod SS
      auto issue_s = [&](int j) -> bool {
        const uint32_t ki = kb + j, stage = ki % SK;
        const uint32_t si = sb + j, slot = si % SS;
        bool w = mbar_wait(&bars[L::kKFull + stage], (ki / SK) & 1, abort, p.err, 0x602);
        w = w && mbar_wait(&bars[L::kSEmpty + slot], ((si / SS) & 1) ^ 1, abort, p.err, 0x603);
        if (!__all_sync(0xffffffffu, w)) return false;
        tc_fence_after();
        {
          // the whole warp walks the K-steps (warp-uniform descriptors) and
          // the elected lane issues: a lone lane in a divergent branch issues
          // these small MMAs far slower than the tensor core runs them
          const Desc kd = make_desc(smem_u32(k_base + stage * L::kKVBytes), 16, 1024);
          const uint32_t d = tm_s + slot * 16;
          // K-steps over head dimensions: 0-3 in the first 64-dim half, 4-7 in the second
          if (leader) mma_ss<0>(d, kd, 0, qd, 0, kIdS);
#pragma unroll
          for (int s = 1; s < kHeadDim / 16; ++s)
            if (leader)
              mma_ss<1>(d, kd, (s >> 2) * (L::kKVHalf >> 4) + (s & 3) * 2, qd,
                        (s >> 2) * (L::kTHalf >> 4) + (s & 3) * 2, kIdS);
          if (leader) {
            umma_commit(&bars[L::kSFull + slot]);
            umma_commit(&bars[L::kKEmpty + stage]);
            if (j + 1 == nb) umma_commit(&bars[L::kQEmpty]);  // Q no longer read
          }
        }
        __syncwarp();
        return true;
      };
      // S runs as far ahead as the S^T ring allows; warp 15 issues the PV products
      bool fail = false;
      for (int j = 0; j < nb && !fail; ++j)
        if (!issue_s(j)) fail = true;
      if (fail) break;
      k_it += nb;
      s_it += nb;
    }
  } else if (warp == 15) {
    // ------------------------------------------------------------ PV issuer
    constexpr uint32_t kIdO = idesc_bf16(128, kDN, true, false);   // A = V^T (dims contiguous), B = P^T
    const uint32_t leader = elect_one_sync();
    uint32_t v_it = 0, o_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int item = dec_snake_item(round);
      if (item >= p.num_items) continue;
      const DecItem di = dec_item(p, item);
      const int kv_len = di.kv_len, nb = di.nb;
      const uint32_t vb = v_it, ob = o_it;
      bool fail = false;
      for (int j = 0; j < nb; ++j) {
        const uint32_t vi = vb + j, vstage = vi % SV;
        const uint32_t oi = ob + j, oslot = oi % OS, pslot = oi % PS;
        bool w = mbar_wait(&bars[L::kPFull + pslot], (oi / PS) & 1, abort, p.err, 0x604);
        w = w && mbar_wait(&bars[L::kVFull + vstage], (vi / SV) & 1, abort, p.err, 0x605);
        w = w && mbar_wait(&bars[L::kOEmpty + oslot], ((oi / OS) & 1) ^ 1, abort, p.err, 0x606);
        if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
        uint8_t* vd = v_base + vstage * L::kKVBytes;
        // V rows past the context may hold stale or non-finite data; P is
        // exactly 0 there, so zero them (0 * NaN = NaN)
        const int valid = min(B, kv_len - (di.b0 + j * di.stride) * B);
        if (valid < B) {
          const int nrow = B - valid;
          for (int i = lane; i < nrow * 16; i += 32) {
            const int row = valid + (i >> 4);
            const int piece = i & 15;  // 16 B pieces: 8 per half-row, 2 halves
            *reinterpret_cast<uint4*>(vd + (piece >> 3) * L::kKVHalf + row * 128 + (piece & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        {
          // O^T = V^T P_hi^T + V^T P_lo^T: K-step s covers keys 16s..16s+15
          // (V rows: 2048 B a step; P^T columns: 32 B a step within a half)
          const Desc vdd = make_desc(smem_u32(vd), L::kKVHalf, 1024);
          const Desc ph = make_desc(smem_u32(p_base + pslot * 2 * L::kTBytes), 16, 1024);
          const Desc pl = make_desc(smem_u32(p_base + pslot * 2 * L::kTBytes + L::kTBytes), 16, 1024);
          const uint32_t d = tm_o + oslot * 16;
          if (leader) mma_ss<0>(d, vdd, 0, ph, 0, kIdO);
#pragma unroll
          for (int s = 1; s < B / 16; ++s)
            if (leader) mma_ss<1>(d, vdd, s * 128, ph, (s >> 2) * (L::kTHalf >> 4) + (s & 3) * 2, kIdO);
#pragma unroll
          for (int s = 0; s < B / 16; ++s)
            if (leader) mma_ss<1>(d, vdd, s * 128, pl, (s >> 2) * (L::kTHalf >> 4) + (s & 3) * 2, kIdO);
          if (leader) {
            umma_commit(&bars[L::kOFull + oslot]);
            umma_commit(&bars[L::kVEmpty + vstage]);
            umma_commit(&bars[L::kPEmpty + pslot]);
          }
        }
        __syncwarp();
      }
      if (fail) break;
      v_it += nb;
      o_it += nb;
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // two groups of four warps take alternate blocks (group = block parity,
    // which is also the block's P^T slot)
    const int grp = warp >= 8 ? 1 : 0;
    const int t = tid - (grp ? 256 : 128);  // key lane
    const int w = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + L::kRedOff + grp * L::kRedBytes);
    float* part = reinterpret_cast<float*>(smem + L::kPartOff + grp * L::kPartBytes);
    const float sl = p.scale_log2;
    uint32_t s_it = 0, sy_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int item = dec_snake_item(round);
      if (item >= p.num_items) continue;
      const DecItem di = dec_item(p, item);
      const int kv_len = di.kv_len, nb = di.nb;
      if (FOLD && p.state_o && p.fill_flag) {
        // their share of the item's table fill (threads 128-383; the
        // correction warps take 0-127), released to the correction warps,
        // which wait for both shares before their first state store (one
        // item per CTA here, so a phase of the fill barrier is one item)
        fill_item_slots(p, di, G, tid);
        mbar_arrive(&bars[L::kFillDone]);
      }
      bool fail = false;
      for (int j = 0; j < nb; ++j, ++s_it) {
        if (static_cast<int>(s_it & 1) != grp) continue;  // the other group's block
        const uint32_t slot = s_it % SS;
        bool ok = mbar_wait(&bars[L::kSFull + slot], (s_it / SS) & 1, abort, p.err, 0x701);
        if (!__all_sync(0xffffffffu, ok)) { fail = true; break; }
        tc_fence_after();
        uint32_t raw[16];
        tmem_ld16(tm_s + lane_off + slot * 16, raw);
        tmem_ld_wait(raw);
        tc_fence_before();
        mbar_arrive(&bars[L::kSEmpty + slot]);
        const bool vis = (di.b0 + j * di.stride) * B + t < kv_len;
        const int rb = static_cast<int>(sy_it & 1);
        const uint32_t sy_par = (sy_it >> 1) & 1;
        // block maximum of every query head over the visible keys (exact)
#pragma unroll
        for (int q = 0; q < MG; ++q) {
          const float m = warp_max((q < G && vis) ? __uint_as_float(raw[q]) : -INFINITY);
          if (lane == 0) red[(rb * 4 + w) * MG + q] = m;
        }
        mbar_arrive(&bars[L::kSyncMax + grp * 2 + rb]);
        ok = mbar_wait(&bars[L::kSyncMax + grp * 2 + rb], sy_par, abort, p.err, 0x702);
        if (!__all_sync(0xffffffffu, ok)) { fail = true; break; }
        float mc[MG], pr[MG];
#pragma unroll
        for (int q = 0; q < MG; ++q) {
          const float* r4 = red + rb * 4 * MG + q;
          const float m = fmaxf(fmaxf(fmaxf(r4[0], r4[MG]), r4[2 * MG]), r4[3 * MG]);
          mc[q] = __fmul_rn(m, sl);
          pr[q] = (q < G && vis) ? prob(__uint_as_float(raw[q]), sl, -mc[q]) : 0.0f;
        }
        // P^T = P_hi^T + P_lo^T into the operand tiles of P slot grp
        ok = mbar_wait(&bars[L::kPEmpty + grp], ((s_it / PS) & 1) ^ 1, abort, p.err, 0x703);
        if (!__all_sync(0xffffffffu, ok)) { fail = true; break; }
        uint8_t* ph = p_base + grp * 2 * L::kTBytes;
#pragma unroll
        for (int q = 0; q < MG; ++q) {
          if (q < G) {
            const uint16_t hi = f32_to_bf16_rn(pr[q]);
            const uint16_t lo = f32_to_bf16_rn(__fsub_rn(pr[q], bf16_bits_as_f32(hi)));
            const uint32_t o = tile16_off(q, t);
            *reinterpret_cast<uint16_t*>(ph + o) = hi;
            *reinterpret_cast<uint16_t*>(ph + L::kTBytes + o) = lo;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[L::kPFull + grp]);
        // canonical row sums: per 64-key half of the block (warps 2h and
        // 2h + 1), key c goes to partial c mod 16, the partial adding keys j,
        // j + 16 (first warp's lanes j, j + 16), j + 32, j + 48 (second
        // warp's) in ascending order; the 8-4-2-1 tree of each half runs as a
        // butterfly over 16 lanes, and the block sum is half 0 + half 1 (lane
        // 0 holds it)
#pragma unroll
        for (int q = 0; q < MG; ++q) part[((rb * 4 + w) * MG + q) * 32 + lane] = pr[q];
        mbar_arrive(&bars[L::kSyncPart + grp * 2 + rb]);
        ok = mbar_wait(&bars[L::kSyncPart + grp * 2 + rb], sy_par, abort, p.err, 0x704);
        if (!__all_sync(0xffffffffu, ok)) { fail = true; break; }
        const uint32_t sslot = s_it % SR;
#pragma unroll
        for (int q = 0; q < MG; ++q) {
          if (q >= G || (q & 3) != w) continue;  // warp w sums query heads w, w + 4
          const float* pq = part + (rb * 4 * MG + q) * 32 + lane;
          const float* pw = pq - lane + (lane & 15);  // key (lane mod 16) of each warp's 32
          float a = __fadd_rn(__fadd_rn(__fadd_rn(pw[0], pw[16]), pw[MG * 32]), pw[MG * 32 + 16]);
          float a1 = __fadd_rn(__fadd_rn(__fadd_rn(pw[2 * MG * 32], pw[2 * MG * 32 + 16]), pw[3 * MG * 32]),
                               pw[3 * MG * 32 + 16]);
#pragma unroll
          for (int off = 8; off >= 1; off >>= 1) {
            a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, off));
            a1 = __fadd_rn(a1, __shfl_xor_sync(0xffffffffu, a1, off));
          }
          a = __fadd_rn(a, a1);
          if (lane == 0) {
            float lse_b, rcp;
            block_stats(mc[q], a, lse_b, rcp);
            stats[sslot * kDecodeMaxGroup + q] = make_float2(lse_b, rcp);
          }
        }
        mbar_arrive(&bars[L::kStatsFull + sslot]);
        ++sy_it;
      }
      if (fail) break;
    }
  } else {
    // ------------------------------------------------------------ correction / epilogue
    const int d = tid;  // head dimension lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t o_it = 0, rq_it = 0, fill_it = 0;
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.num_items; ++round) {
      const int item = dec_snake_item(round);
      if (item >= p.num_items) continue;
      const DecItem di = dec_item(p, item);
      const int seq = di.seq, g = di.g, nb = di.nb;
      const bool split = p.state_o != nullptr;
      if (p.rope_table) {
        // RoPE of the query rows at position kv_len - 1, in place: thread t
        // takes pairs 4u .. 4u+3 (u = t mod 16) of row t / 16; the pair's
        // second element sits at the same offset of the second half
        bool ok = mbar_wait(&bars[L::kQFull], rq_it & 1, abort, p.err, 0x803);
        if (!__all_sync(0xffffffffu, ok)) break;
        ++rq_it;
        const int i = tid >> 4, u = tid & 15;
        if (i < G) {
          const float* trow = p.rope_table + static_cast<int64_t>(di.kv_len - 1) * kHeadDim;
          const float4 c = __ldg(reinterpret_cast<const float4*>(trow) + u);
          const float4 s = __ldg(reinterpret_cast<const float4*>(trow + 64) + u);
          uint2* pa = reinterpret_cast<uint2*>(q_tile + tile16_off(i, 4 * u));
          uint2* pb = reinterpret_cast<uint2*>(q_tile + tile16_off(i, 64 + 4 * u));
          const uint2 a = *pa, b = *pb;
          const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
          const uint32_t wa[2] = {a.x, a.y}, wb[2] = {b.x, b.y};
          uint32_t ra[2], rb[2];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            float ya[2], yb[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * w + h;
              const float x0 = bf16_bits_as_f32(static_cast<uint16_t>(h ? (wa[w] >> 16) : wa[w]));
              const float x1 = bf16_bits_as_f32(static_cast<uint16_t>(h ? (wb[w] >> 16) : wb[w]));
              ya[h] = __fmaf_rn(x0, cc[e], -__fmul_rn(x1, ss[e]));
              yb[h] = __fmaf_rn(x1, cc[e], __fmul_rn(x0, ss[e]));
            }
            ra[w] = pack_bf16x2(ya[0], ya[1]);
            rb[w] = pack_bf16x2(yb[0], yb[1]);
          }
          *pa = make_uint2(ra[0], ra[1]);
          *pb = make_uint2(rb[0], rb[1]);
        }
        fence_proxy_async_smem();  // the tensor core reads the rows through the async proxy
        mbar_arrive(&bars[L::kQRope]);
      }
      if (FOLD && split && p.fill_flag) {
        // the item's slots of the state table hold kUnwritten before any of
        // its states can land (the fold takes any other value as landed);
        // the softmax warps fill a share (threads 128-383) at their item start;
        // the flag, set once the first block's state is written (the fill's
        // stores have long drained by then), tells the fold warps.  After the
        // query rotation, which the first S waits for.
        fill_item_slots(p, di, G, tid);
        // another warp's thread writes a slot's state: the barrier (release
        // on arrival, acquire on completion) orders every fill store before
        // every state store
        mbar_arrive(&bars[L::kFillDone]);
        const bool ok = mbar_wait(&bars[L::kFillDone], fill_it & 1, abort, p.err, 0x804);
        ++fill_it;
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      float O[MG];
#pragma unroll
      for (int q = 0; q < MG; ++q) O[q] = 0.0f;
      float Lrun = -INFINITY;  // lane q: running lse of query head q
      bool fail = false;
      for (int j = 0; j < nb; ++j) {
        const uint32_t sslot = o_it % SR, oslot = o_it % OS;
        bool ok = mbar_wait(&bars[L::kStatsFull + sslot], (o_it / SR) & 1, abort, p.err, 0x801);
        ok = ok && mbar_wait(&bars[L::kOFull + oslot], (o_it / OS) & 1, abort, p.err, 0x802);
        if (!__all_sync(0xffffffffu, ok)) { fail = true; break; }
        tc_fence_after();
        uint32_t raw[16];
        tmem_ld16(tm_o + lane_off + oslot * 16, raw);
        // fold coefficients of query head `lane` (overlap the TMEM load)
        float lb = -INFINITY, rc = 0.0f, al = 0.0f, be = 0.0f, Lp = 0.0f;
        if (lane < G) {
          const float2 st = stats[sslot * kDecodeMaxGroup + lane];
          lb = st.x;
          rc = st.y;
          if (j > 0 && !split) fold_coeffs(Lrun, lb, Lp, al, be);
        }
        tmem_ld_wait(raw);
        tc_fence_before();
        mbar_arrive(&bars[L::kOEmpty + oslot]);
        // o_b = PV * (1/l); O = fma(o_b, beta, O * alpha), or (split) the
        // block state written out
        const int64_t blk = p.cu_q[seq] + di.b0 + j * di.stride;  // state-table block
        const int64_t pair_b = blk * p.hq + g * G;
#pragma unroll
        for (int q = 0; q < MG; ++q) {
          const float rq = __shfl_sync(0xffffffffu, rc, q);
          const float aq = __shfl_sync(0xffffffffu, al, q);
          const float bq = __shfl_sync(0xffffffffu, be, q);
          if (q < G) {
            const float oa = __fmul_rn(__uint_as_float(raw[q]), rq);
            if (split) p.state_o[(pair_b + q) * kHeadDim + d] = oa;
            else O[q] = (j == 0) ? oa : __fmaf_rn(oa, bq, __fmul_rn(O[q], aq));
          }
        }
        if (split) {
          if (warp == 0 && lane < G) p.state_lse[pair_b + lane] = lb;
          if (FOLD && p.fill_flag && j == 0) {
            // the fill barrier and the releasing store order the four warps'
            // fill stores before the flag
            if (tid == 0)
              st_release_u64(p.fill_flag + (static_cast<int64_t>(seq) * p.hkv + g) * kMaxSplitK + di.b0,
                             p.fill_nonce);
          }
        } else if (lane < G) {
          Lrun = (j == 0) ? lb : Lp;
        }
        ++o_it;
      }
      if (fail) break;
      if (split) continue;
      // epilogue: O and L are final
#pragma unroll
      for (int q = 0; q < MG; ++q) {
        if (q < G) {
          const int64_t row = static_cast<int64_t>(seq) * p.hq + g * G + q;
          if (p.out_f32) p.out_f32[row * kHeadDim + d] = O[q];
          if (p.out_bf16) p.out_bf16[row * kHeadDim + d] = f32_to_bf16_rn(O[q]);
        }
      }
      if (warp == 0 && lane < G && p.lse) p.lse[static_cast<int64_t>(seq) * p.hq + g * G + lane] = Lrun;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 14) {
    if (*abort) {
      // let copies already in flight land before the CTA's memory is released
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int MG>
cudaError_t launch_decode_t(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, cudaStream_t stream) {
  rlk_decode_kernel<MG, false><<<grid, kDThreads, DecLayout::kAlloc, stream>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

// The split decode with the fold on chip: its fold warps wait for states
// that other CTAs of the launch publish, so every CTA must be resident at
// once -- a cooperative launch guarantees it (or fails).
template <int MG>
cudaError_t launch_decode_coop_t(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, int grid, cudaStream_t stream) {
  void* args[] = {const_cast<FwdParams*>(&p), const_cast<CUtensorMap*>(&tq), const_cast<CUtensorMap*>(&tk),
                  const_cast<CUtensorMap*>(&tv)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&rlk_decode_kernel<MG, true>), dim3(grid),
                                     dim3(kDThreads), args, DecLayout::kAlloc, stream);
}

// Split decode, second step: the canonical fold of one (sequence, query head)
// pair's block states in ascending global block order -- the operations the
// single-pass kernel applies on chip, so the result is the same bit for bit.
// One 128-thread CTA per pair, thread t owning head dimension t.  The fold is a
// chain over the blocks, so what bounds it is how many state bytes are in
// flight: chunks of kDmChunk block states (512 B of o plus the lse each) are
// staged through a kDmStages-deep ring of asynchronous copies, whole chunks
// landing while an earlier one folds.  Every thread recomputes the same fold
// coefficients from the staged lse values.
constexpr int kDmChunk = 32;
constexpr int kDmStages = 4;
constexpr int kDmThreads = kHeadDim;
constexpr int kDmStageBytes = kDmChunk * kHeadDim * 4 + kDmChunk * 4;
constexpr int kDmSmem = kDmStages * kDmStageBytes;
static_assert(kDmThreads == 128 && (kDmChunk * kHeadDim / 4) % kDmThreads == 0, "decode fold staging layout");

// The fold's own parameters: the decode's item list stays out of this launch.
struct DecFoldParams {
  const float* state_o;
  const float* state_lse;
  float* out_f32;
  uint16_t* out_bf16;
  float* lse;
  int32_t num_seqs, hq;
  int32_t block_base[kMaxSeqs + 1];  // first state-table block of each sequence
  int32_t ctx[kMaxSeqs + 1];         // context length of each sequence
};

__global__ void __launch_bounds__(kDmThreads) rlk_decode_merge_kernel(const __grid_constant__ DecFoldParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const int t = threadIdx.x;
  const int64_t total = static_cast<int64_t>(p.num_seqs) * p.hq;
  for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
    const int seq = static_cast<int>(w / p.hq);
    const int h = static_cast<int>(w - static_cast<int64_t>(seq) * p.hq);
    const int nb = (p.ctx[seq] + DecLayout::B - 1) / DecLayout::B;
    const int nchunks = (nb + kDmChunk - 1) / kDmChunk;
    const int64_t pair0 = static_cast<int64_t>(p.block_base[seq]) * p.hq + h;
    // chunk c -> stage c % kDmStages; a warp copies one block's 512 B of o
    auto issue = [&](int c) {
      if (c < nchunks) {
        uint8_t* st = dsm + (c % kDmStages) * kDmStageBytes;
        float* so = reinterpret_cast<float*>(st);
        float* sl = reinterpret_cast<float*>(st + kDmChunk * kHeadDim * 4);
#pragma unroll
        for (int k = 0; k < kDmChunk * kHeadDim / 4 / kDmThreads; ++k) {
          const int i = t + k * kDmThreads;
          const int j = i >> 5, seg = i & 31;
          const int b = c * kDmChunk + j;
          if (b < nb) {
            const int64_t pr = pair0 + static_cast<int64_t>(b) * p.hq;
            cp_async16(so + j * kHeadDim + seg * 4, p.state_o + pr * kHeadDim + seg * 4);
          }
        }
        if (t < kDmChunk && c * kDmChunk + t < nb) {
          const int64_t pr = pair0 + static_cast<int64_t>(c * kDmChunk + t) * p.hq;
          cp_async4(sl + t, p.state_lse + pr);
        }
      }
      cp_async_commit();  // empty groups keep the count uniform
    };
#pragma unroll
    for (int c = 0; c < kDmStages - 1; ++c) issue(c);
    float O = 0.f, L = -INFINITY;
    for (int c = 0; c < nchunks; ++c) {
      issue(c + kDmStages - 1);
      cp_async_wait<kDmStages - 1>();
      __syncthreads();
      const uint8_t* st = dsm + (c % kDmStages) * kDmStageBytes;
      const float* so = reinterpret_cast<const float*>(st);
      const float* sl = reinterpret_cast<const float*>(st + kDmChunk * kHeadDim * 4);
      const int jn = min(kDmChunk, nb - c * kDmChunk);
      const int j0 = c == 0 ? 1 : 0;
      if (c == 0) {
        O = so[t];
        L = sl[0];
      }
      auto fold1 = [&](int j) {
        float Lp, alpha, beta;
        fold_coeffs(L, sl[j], Lp, alpha, beta);
        O = fold_elem(O, so[j * kHeadDim + t], alpha, beta);
        L = Lp;
      };
      if (jn == kDmChunk) {
        // whole chunk: unrolled, so the loads and the O update sit beside
        // the serial lse chain instead of on it
#pragma unroll
        for (int j = 0; j < kDmChunk; ++j)
          if (j >= j0) fold1(j);
      } else {
        for (int j = j0; j < jn; ++j) fold1(j);
      }
      __syncthreads();  // the stage is refilled by the next iteration's issue
    }
    cp_async_wait<0>();
    const int64_t row = static_cast<int64_t>(seq) * p.hq + h;
    if (p.out_f32) p.out_f32[row * kHeadDim + t] = O;
    if (p.out_bf16) p.out_bf16[row * kHeadDim + t] = f32_to_bf16_rn(O);
    if (p.lse && t == 0) p.lse[row] = L;
  }
}

}  // namespace

bool decode_transposed_supported(const FwdParams& p) {
  return p.block == DecLayout::B && p.group >= 1 && p.group <= kDecodeMaxGroup && p.page_size >= 8 &&
         DecLayout::kPageWin % (DecLayout::B / p.page_size) == 0;
}

template <int MG>
cudaError_t configure_decode_mg() {
  cudaError_t e = cudaFuncSetAttribute(rlk_decode_kernel<MG, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DecLayout::kAlloc);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(rlk_decode_kernel<MG, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DecLayout::kAlloc);
}

cudaError_t configure_decode_kernels() {
  cudaError_t e;
  if ((e = configure_decode_mg<1>())) return e;
  if ((e = configure_decode_mg<2>())) return e;
  if ((e = configure_decode_mg<4>())) return e;
  if ((e = configure_decode_mg<8>())) return e;
  return cudaFuncSetAttribute(rlk_decode_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDmSmem);
}

cudaError_t launch_decode_merge(const FwdParams& p, int num_sms, cudaStream_t stream) {
  DecFoldParams f;
  f.state_o = p.state_o;
  f.state_lse = p.state_lse;
  f.out_f32 = p.out_f32;
  f.out_bf16 = p.out_bf16;
  f.lse = p.lse;
  f.num_seqs = p.num_tiles;  // the caller passes the sequence count here
  f.hq = p.hq;
  for (int s = 0; s <= kMaxSeqs; ++s) {
    f.block_base[s] = p.cu_q[s];
    f.ctx[s] = p.cu_k[s];
  }
  const int64_t pairs = static_cast<int64_t>(f.num_seqs) * f.hq;
  const int64_t blocks = std::min<int64_t>(std::max<int64_t>(pairs, 1), static_cast<int64_t>(num_sms) * 3);
  rlk_decode_merge_kernel<<<static_cast<int>(blocks), kDmThreads, kDmSmem, stream>>>(f);
  return cudaGetLastError();
}

cudaError_t launch_decode_cooperative(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, int grid, cudaStream_t stream) {
  if (p.group <= 1) return launch_decode_coop_t<1>(p, tq, tk, tv, grid, stream);
  if (p.group <= 2) return launch_decode_coop_t<2>(p, tq, tk, tv, grid, stream);
  if (p.group <= 4) return launch_decode_coop_t<4>(p, tq, tk, tv, grid, stream);
  return launch_decode_coop_t<8>(p, tq, tk, tv, grid, stream);
}

cudaError_t launch_decode(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          int grid, cudaStream_t stream) {
  if (p.group <= 1) return launch_decode_t<1>(p, tq, tk, tv, grid, stream);
  if (p.group <= 2) return launch_decode_t<2>(p, tq, tk, tv, grid, stream);
  if (p.group <= 4) return launch_decode_t<4>(p, tq, tk, tv, grid, stream);
  return launch_decode_t<8>(p, tq, tk, tv, grid, stream);
}

}  // namespace rlk
