// rlk_internal.h -- launch parameter blocks and limits shared by the host
// side of the C ABI and the kernels.  Not part of the public interface.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace rlk {

constexpr int kHeadDim = 128;           // D, the only head size the kernels take
constexpr int kMaxSeqs = 128;           // sequences per launch (their tables ride in kernel params)
constexpr int kMaxSeqsPerCall = 1 << 20;  // sequences per call: larger batches run as 128-sequence ranges
constexpr int kMaxTilesPerLaunch = 880; // work tiles per launch (kernel param space)
constexpr int kTileRows = 128;          // MMA M: query rows per tile
constexpr int kDecodeMaxGroup = 8;     // query heads per KV head the transposed decode kernel takes
constexpr int64_t kNoAllocIndexEntries = 65536;  // no-alloc merge scratch: (sequence, block) index entries
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // bounded mbarrier waits: 1 s
constexpr uint32_t kUnwritten = 0xFFFFFFFFu;  // state-table fill of the on-chip fold (a NaN arithmetic never makes)
constexpr int kMaxSplitK = 64;  // split decode: items per (sequence, KV head)

// device error word bits
constexpr unsigned kErrDeviceTimeout = 1u;
constexpr unsigned kErrBadPage = 2u;
constexpr unsigned kErrDuplicateBlock = 4u;
constexpr unsigned kErrMissingBlock = 8u;
constexpr unsigned kErrBadSlab = 16u;

struct ErrWord {
  unsigned int bits;
  unsigned int site;
};

enum FwdMode : int { kModeFused = 0, kModeStates = 1, kModeDecode = 2 };

// One unit of forward work: up to 128 query rows of one sequence (all query
// heads are looped inside the grid), or, for decode, one (sequence, KV head)
// whose query heads form the rows.
struct alignas(16) FwdTile {
  int32_t seq;
  int32_t row_begin;       // first query row, relative to the sequence's first query row
  int32_t row_count;       // rows of the tile that are written (<= 128)
  int32_t block;           // states mode, split decode: the first global block; otherwise -1
  int64_t slab_offset;     // states mode: first (row, head) pair of that block's slab
  int32_t slab_row_begin;  // unused (0)
  int32_t slab_row_count;  // states mode, split decode: consecutive blocks from `block`
};
// States mode: the slabs of consecutive blocks follow each other in the
// state table, and block b's slab covers rows max(0, b*B - (kv_len - q_len))
// .. q_len - 1 with (row, head) pair offset + head * rows + (row - first row),
// so an item derives every block's slab from the first one.

struct FwdParams {
  ErrWord* err;
  int32_t mode;
  int32_t hq, hkv, group;  // query heads, KV heads, hq / hkv
  int32_t block;           // KV block size (64 or 128)
  float scale_log2;        // softmax_scale * log2(e), rounded once on the host
  int32_t num_tiles;
  int32_t num_items;
  // fused / decode outputs
  float* out_f32;
  uint16_t* out_bf16;
  float* lse;
  // states outputs
  float* state_o;
  float* state_lse;
  // decode
  const int32_t* page_table;
  int32_t max_pages, page_size, n_pages;
  // split decode with the fold on chip: item r of a (sequence, KV head) takes
  // the blocks b = r, r + split_stride, ... (0: contiguous ranges, or the
  // whole sequence); the CTAs past the items fold the states of fold_seqs
  // sequences as the producers write them into the table.  Each item first
  // fills its own slots with kUnwritten and then stores fill_nonce (a value
  // new to every call) to fill_flag[(seq * hkv + g) * kMaxSplitK + r]; the
  // fold reads an item's slots once its flag holds the nonce
  int32_t split_stride, fold_seqs;
  uint64_t* fill_flag;
  uint64_t fill_nonce;
  // transposed decode: RoPE table [positions][cos 64, sin 64] (FP32); when
  // set, the query rows are rotated at position kv_len - 1 after they land
  const float* rope_table;
  // sequences: fused/states use cu_q / cu_k (packed offsets); decode uses
  // cu_k[s] as the context length of sequence s.
  int32_t cu_q[kMaxSeqs + 1];
  int32_t cu_k[kMaxSeqs + 1];
  FwdTile tiles[kMaxTilesPerLaunch];
};

// Merge (canonical fold of a partial-state table).
struct Slab {  // mirrors rlk_attn_slab
  int32_t seq, block, row_begin, row_count;
  int64_t offset;
  int32_t producer, reserved;
};

struct MergeParams {
  ErrWord* err;
  int32_t num_seqs, hq, block, max_blocks;
  int32_t seq_base;        // the slabs' sequence ids are seq_base + local index
  int32_t total_seqs;      // sequences of the whole call (slab ids outside are bad)
  int64_t total_rows;      // query rows over all sequences
  int64_t n_slabs;
  const Slab* slabs;       // device, arrival order
  const float* state_o;
  const float* state_lse;
  int64_t n_pairs;         // (row, head) pairs the state table holds
  int32_t* index;          // [num_seqs * max_blocks] slab id per (seq, block)
  float* out_f32;
  uint16_t* out_bf16;
  float* lse;
  int32_t cu_q[kMaxSeqs + 1];
  int32_t cu_k[kMaxSeqs + 1];
};

// RoPE pass over packed BF16 rows [T, heads, 128] (and optionally a second
// tensor [T, heads2, 128] of the same tokens); row i of sequence s sits at
// position pos0[s] + i.
struct RopeParams {
  const uint16_t* x;
  uint16_t* y;          // may equal x
  const uint16_t* x2;   // optional second tensor of the same tokens (K beside Q), or null
  uint16_t* y2;
  const float* table;   // [positions][cos 64, sin 64]
  int64_t rows;         // T * heads
  int64_t rows2;        // T * heads2
  int32_t heads, heads2, num_seqs;
  int32_t y_stride;     // elements from one (token, head) row of y to the next (0: 128)
  int32_t cu[kMaxSeqs + 1];
  int32_t pos0[kMaxSeqs];
};

// Per-device set-up, run once per device (with it current) before the first
// launch there: the kernels' dynamic shared memory limits and launch checks.
// Function attributes are per device, so every device a process uses needs
// its own call.
cudaError_t configure_fwd_kernels();
cudaError_t configure_decode_kernels();
cudaError_t configure_merge_kernels();
cudaError_t configure_bwd_kernels();
// Device address of the no-alloc merge's file-scope scratch on the current
// device, and its size in int32 entries.
cudaError_t merge_noalloc_scratch(int32_t** ptr, int64_t* entries);

}  // namespace rlk
