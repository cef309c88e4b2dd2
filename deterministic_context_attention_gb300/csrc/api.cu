// api.cu -- host side of the C ABI (include/rlk_attn.h): argument checks,
// the global block plan and logical CP partition, TMA tensor maps, the static
// longest-first work schedule, and kernel launches.  Nothing here allocates
// device memory or synchronises, except rlk_attn_check_device_error.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <random>
#include <string>
#include <type_traits>
#include <vector>

#include "../../include/rlk_attn.h"
#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {
cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, int num_sms, cudaStream_t stream);
bool decode_transposed_supported(const FwdParams& p);
cudaError_t launch_decode_merge(const FwdParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_rope(const RopeParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_decode(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          int grid, cudaStream_t stream);
cudaError_t launch_decode_cooperative(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, int grid, cudaStream_t stream);
rlk_status run_backward(const rlk_attn_params* prm, const void* q, const void* k, const void* v,
                        const float* out_f32, const void* dout, const float* lse,
                        const int32_t* cu, int32_t cp_rank, float* dq, float* dk, float* dv,
                        void* workspace, size_t workspace_bytes, ErrWord* err, int num_sms,
                        cudaStream_t stream);
size_t backward_workspace_bytes(const rlk_attn_params* prm, const int32_t* cu);
}  // namespace rlk

static_assert(sizeof(rlk::FwdParams) + 3 * sizeof(CUtensorMap) + 256 <= 32764,
              "forward kernel parameters exceed the 32 KB launch limit");
static_assert(sizeof(rlk::MergeParams) <= 4096, "merge parameters");
static_assert(sizeof(rlk_attn_slab) == sizeof(rlk::Slab), "slab layout");

// The device error word.  Host code reaches it through its device address,
// looked up once per device.
static __device__ rlk::ErrWord g_rlk_err;

namespace {

thread_local std::string g_last_error;

// Set while an entry point validates the sequence ranges of a batch larger
// than one launch's tables (over_ranges): each range's call then checks its
// arguments on the host and returns before it touches the device.
thread_local bool g_dry_run = false;

rlk_status fail(rlk_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

rlk_status ok() {
  g_last_error.clear();
  return RLK_OK;
}

// What the library keeps per device, set up once with that device current
// (under g_dev_mutex, so concurrent first calls from several host threads are
// safe): the SM count, the device addresses of the error word and of the
// no-alloc merge scratch, and the kernels' function attributes (which are
// per device).
struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  rlk::ErrWord* err = nullptr;
  int32_t* merge_scratch = nullptr;
  int64_t merge_scratch_entries = 0;
};
std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

rlk_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return fail(RLK_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(RLK_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_rlk_err);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
    d.err = static_cast<rlk::ErrWord*>(addr);
    e = rlk::merge_noalloc_scratch(&d.merge_scratch, &d.merge_scratch_entries);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "cudaGetSymbolAddress(merge scratch): %s", cudaGetErrorString(e));
    if ((e = rlk::configure_fwd_kernels()) != cudaSuccess || (e = rlk::configure_decode_kernels()) != cudaSuccess ||
        (e = rlk::configure_merge_kernels()) != cudaSuccess || (e = rlk::configure_bwd_kernels()) != cudaSuccess)
      return fail(RLK_ERR_CUDA, "kernel set-up on device %d: %s", dev, cudaGetErrorString(e));
    d.ready = true;
  }
  *out = &d;
  return RLK_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// BF16 tensor [d2][d1][128] as a 3-D map (innermost first), 128-byte swizzle,
// box {64, box1, box2}.
// Rows of 128 BF16 elements, head_bytes apart (256: packed [T, H, 128]).
rlk_status make_map(CUtensorMap* m, const void* base, uint64_t d1, uint64_t d2, uint32_t box1, uint32_t box2,
                    uint64_t head_bytes = 256) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(RLK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {128, d1, d2};
  cuuint64_t strides[2] = {head_bytes, head_bytes * d1};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RLK_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return RLK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rlk_status check_params(const rlk_attn_params* p) {
  if (!p) return fail(RLK_ERR_INVALID_ARGUMENT, "params is NULL");
  if (p->head_dim != rlk::kHeadDim) return fail(RLK_ERR_UNSUPPORTED, "head_dim %d: only 128 is supported", p->head_dim);
  if (p->num_q_heads < 1 || p->num_kv_heads < 1 || p->num_q_heads % p->num_kv_heads)
    return fail(RLK_ERR_INVALID_ARGUMENT, "heads %d / %d: Hkv must divide Hq", p->num_q_heads, p->num_kv_heads);
  if (p->num_q_heads / p->num_kv_heads > 128)
    return fail(RLK_ERR_UNSUPPORTED, "more than 128 query heads per KV head");
  if (p->causal != 1) return fail(RLK_ERR_UNSUPPORTED, "only causal attention is supported");
  if (p->kv_block_size != 64 && p->kv_block_size != 128)
    return fail(RLK_ERR_UNSUPPORTED, "kv_block_size %d: must be 64 or 128", p->kv_block_size);
  if (p->cp_size < 1 || p->cp_size > 8) return fail(RLK_ERR_INVALID_ARGUMENT, "cp_size %d not in 1..8", p->cp_size);
  if (p->cp_layout != 0 && p->cp_layout != 1) return fail(RLK_ERR_INVALID_ARGUMENT, "cp_layout %d", p->cp_layout);
  if (p->num_seqs < 1 || p->num_seqs > rlk::kMaxSeqsPerCall)
    return fail(RLK_ERR_UNSUPPORTED, "num_seqs %d not in 1..%d", p->num_seqs, rlk::kMaxSeqsPerCall);
  if (!(p->softmax_scale > 0.0f) || !std::isfinite(p->softmax_scale))
    return fail(RLK_ERR_INVALID_ARGUMENT, "softmax_scale must be finite and > 0");
  return RLK_OK;
}

rlk_status check_cu(const rlk_attn_params* p, const int32_t* cu_q, const int32_t* cu_k) {
  if (!cu_q || !cu_k) return fail(RLK_ERR_INVALID_ARGUMENT, "cu_seqlens is NULL");
  if (cu_q[0] != 0 || cu_k[0] != 0) return fail(RLK_ERR_INVALID_ARGUMENT, "cu_seqlens must start at 0");
  for (int s = 0; s < p->num_seqs; ++s) {
    const int64_t ql = static_cast<int64_t>(cu_q[s + 1]) - cu_q[s];
    const int64_t kl = static_cast<int64_t>(cu_k[s + 1]) - cu_k[s];
    if (ql < 0 || kl < 0) return fail(RLK_ERR_INVALID_ARGUMENT, "cu_seqlens not monotone at sequence %d", s);
    if (ql > kl) return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: q_len %lld > kv_len %lld", s,
                             static_cast<long long>(ql), static_cast<long long>(kl));
  }
  return RLK_OK;
}

// Batches of more sequences than one launch's tables hold (kMaxSeqs) run as
// consecutive ranges of at most kMaxSeqs sequences, each a complete call on
// rebased cu_seqlens and offset tensor pointers (per-sequence arithmetic does
// not depend on the other sequences of a batch, so the results are the
// same).  Every range is validated first (a dry run that stops before any
// device work), then the ranges launch in order on the caller's stream, so a
// bad argument anywhere still fails the call before its first launch.
template <class Fn>
rlk_status over_ranges(int num_seqs, Fn&& range_call) {
  g_dry_run = true;
  for (int s0 = 0; s0 < num_seqs; s0 += rlk::kMaxSeqs) {
    const rlk_status st = range_call(s0, std::min(num_seqs, s0 + rlk::kMaxSeqs));
    if (st) {
      g_dry_run = false;
      return st;
    }
  }
  g_dry_run = false;
  for (int s0 = 0; s0 < num_seqs; s0 += rlk::kMaxSeqs) {
    const rlk_status st = range_call(s0, std::min(num_seqs, s0 + rlk::kMaxSeqs));
    if (st) return st;
  }
  return ok();
}
// cu[s0..s1] - cu[s0]: the cumulative lengths of a sequence range
std::vector<int32_t> rebase(const int32_t* cu, int s0, int s1) {
  std::vector<int32_t> r(s1 - s0 + 1);
  for (int s = s0; s <= s1; ++s) r[s - s0] = cu[s] - cu[s0];
  return r;
}
// p advanced by n elements of `bytes` bytes (NULL stays NULL)
template <class T>
T* adv(T* p, int64_t n, int bytes) {
  using C = typename std::conditional<std::is_const<T>::value, const char, char>::type;
  return p ? reinterpret_cast<T*>(reinterpret_cast<C*>(p) + n * bytes) : nullptr;
}
rlk_attn_params range_params(const rlk_attn_params* p, int s0, int s1) {
  rlk_attn_params r = *p;
  r.num_seqs = s1 - s0;
  return r;
}

float scale_log2(const rlk_attn_params* p) {
  return static_cast<float>(static_cast<double>(p->softmax_scale) * 1.4426950408889634073599);
}

// Token chunks of a sequence of n tokens under the CP partition:
// (rank, begin, end) with bounds floor(c * n / chunks).
struct Chunk {
  int rank, begin, end;
};
std::vector<Chunk> partition(int n, int cp, int layout) {
  std::vector<Chunk> out;
  if (layout == 0) {
    for (int c = 0; c < cp; ++c)
      out.push_back({c, static_cast<int>(static_cast<int64_t>(c) * n / cp),
                     static_cast<int>(static_cast<int64_t>(c + 1) * n / cp)});
  } else {
    for (int c = 0; c < 2 * cp; ++c)
      out.push_back({c < cp ? c : 2 * cp - 1 - c, static_cast<int>(static_cast<int64_t>(c) * n / (2 * cp)),
                     static_cast<int>(static_cast<int64_t>(c + 1) * n / (2 * cp))});
  }
  return out;
}
int owner_rank(int pos, int n, int cp, int layout) {
  for (const Chunk& c : partition(n, cp, layout))
    if (pos >= c.begin && pos < c.end) return c.rank;
  return -1;
}

struct SlabPlan {
  std::vector<rlk_attn_slab> slabs;
  int64_t n_pairs = 0;
};

void plan_slabs(const rlk_attn_params* p, const int32_t* cu_q, const int32_t* cu_k, int cp_rank, int64_t base,
                SlabPlan* out) {
  const int B = p->kv_block_size;
  int64_t off = base;
  for (int s = 0; s < p->num_seqs; ++s) {
    const int ql = cu_q[s + 1] - cu_q[s];
    const int kl = cu_k[s + 1] - cu_k[s];
    if (ql == 0) continue;
    const int nb = (kl + B - 1) / B;
    const std::vector<Chunk> parts = partition(kl, p->cp_size, p->cp_layout);
    for (int b = 0; b < nb; ++b) {
      int prod = -1;
      for (const Chunk& c : parts)
        if (b * B >= c.begin && b * B < c.end) prod = c.rank;
      if (cp_rank >= 0 && prod != cp_rank) continue;
      rlk_attn_slab sl;
      sl.seq = s;
      sl.block = b;
      sl.row_begin = std::max(0, b * B - (kl - ql));
      sl.row_count = ql - sl.row_begin;
      sl.offset = off;
      sl.producer = prod;
      sl.reserved = 0;
      off += static_cast<int64_t>(sl.row_count) * p->num_q_heads;
      out->slabs.push_back(sl);
    }
  }
  out->n_pairs = off - base;
}

rlk_status launch_fwd_tiles(rlk::FwdParams* fp, const std::vector<rlk::FwdTile>& tiles, int items_per_tile,
                            const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DeviceInfo* dev, cudaStream_t stream) {
  for (size_t t0 = 0; t0 < tiles.size(); t0 += rlk::kMaxTilesPerLaunch) {
    const size_t n = std::min(tiles.size() - t0, static_cast<size_t>(rlk::kMaxTilesPerLaunch));
    std::copy(tiles.begin() + t0, tiles.begin() + t0 + n, fp->tiles);
    fp->num_tiles = static_cast<int32_t>(n);
    fp->num_items = static_cast<int32_t>(n) * items_per_tile;
    const int grid = std::min(fp->num_items, dev->num_sms);
    cudaError_t e = rlk::launch_fwd(*fp, tq, tk, tv, grid, stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
  }
  return RLK_OK;
}

void fill_seqs(rlk::FwdParams* fp, const rlk_attn_params* p, const int32_t* cu_q, const int32_t* cu_k) {
  for (int s = 0; s <= p->num_seqs; ++s) {
    fp->cu_q[s] = cu_q[s];
    fp->cu_k[s] = cu_k[s];
  }
}

void base_fwd(rlk::FwdParams* fp, const rlk_attn_params* p, const DeviceInfo* dev, int mode) {
  std::memset(fp, 0, sizeof(*fp));
  fp->err = dev->err;
  fp->mode = mode;
  fp->hq = p->num_q_heads;
  fp->hkv = p->num_kv_heads;
  fp->group = p->num_q_heads / p->num_kv_heads;
  fp->block = p->kv_block_size;
  fp->scale_log2 = scale_log2(p);
}

}  // namespace


extern "C" {

const char* rlk_attn_last_error(void) { return g_last_error.c_str(); }

const char* rlk_attn_core_id(void) {
  return "rlk_attn.deterministic_core.v1/sm_103a;merge_order=global_block_index;"
         "downcast_at=final_write;split_kv=fixed_global_blocks;accumulate=fp32;pv=bf16x2_split";
}

rlk_status rlk_attn_plan_states(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                const int32_t* cu_seqlens_k, int32_t cp_rank, int64_t pair_base,
                                rlk_attn_slab* slabs, int64_t max_slabs, int64_t* n_slabs, int64_t* n_pairs) {
  rlk_status st = check_params(params);
  if (st) return st;
  if ((st = check_cu(params, cu_seqlens_q, cu_seqlens_k))) return st;
  if (cp_rank < -1 || cp_rank >= params->cp_size) return fail(RLK_ERR_INVALID_ARGUMENT, "cp_rank %d", cp_rank);
  if (pair_base < 0) return fail(RLK_ERR_INVALID_ARGUMENT, "pair_base < 0");
  if (!n_slabs || !n_pairs) return fail(RLK_ERR_INVALID_ARGUMENT, "n_slabs / n_pairs is NULL");
  SlabPlan plan;
  plan_slabs(params, cu_seqlens_q, cu_seqlens_k, cp_rank, pair_base, &plan);
  *n_slabs = static_cast<int64_t>(plan.slabs.size());
  *n_pairs = plan.n_pairs;
  if (slabs) {
    if (max_slabs < *n_slabs) return fail(RLK_ERR_WORKSPACE_TOO_SMALL, "max_slabs %lld < %lld",
                                          static_cast<long long>(max_slabs), static_cast<long long>(*n_slabs));
    std::copy(plan.slabs.begin(), plan.slabs.end(), slabs);
  }
  return ok();
}

rlk_status rlk_attn_block_manifest_hash(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                        const int32_t* cu_seqlens_k, uint64_t* hash) {
  rlk_status st = check_params(params);
  if (st) return st;
  if ((st = check_cu(params, cu_seqlens_q, cu_seqlens_k))) return st;
  if (!hash) return fail(RLK_ERR_INVALID_ARGUMENT, "hash is NULL");
  uint64_t h = 1469598103934665603ull;
  auto mix = [&h](int64_t v) {
    for (int i = 0; i < 8; ++i) {
      h ^= static_cast<uint64_t>((v >> (8 * i)) & 0xFF);
      h *= 1099511628211ull;
    }
  };
  const int B = params->kv_block_size;
  for (int s = 0; s < params->num_seqs; ++s) {
    const int kl = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
    for (int b = 0; b * B < kl; ++b) {
      mix(s);
      mix(b);
      mix(static_cast<int64_t>(b) * B);
      mix(std::min(kl, (b + 1) * B) - 1);
      mix(owner_rank(b * B, kl, params->cp_size, params->cp_layout));
    }
  }
  *hash = h;
  return ok();
}

rlk_status rlk_attn_prefill_states(const rlk_attn_params* params, const void* q, const void* k, const void* v,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t cp_rank,
                                   int64_t pair_base, float* state_o, float* state_lse, rlk_stream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if ((st = check_cu(params, cu_seqlens_q, cu_seqlens_k))) return st;
  if (cp_rank < -1 || cp_rank >= params->cp_size) return fail(RLK_ERR_INVALID_ARGUMENT, "cp_rank %d", cp_rank);
  if (pair_base < 0) return fail(RLK_ERR_INVALID_ARGUMENT, "pair_base < 0");
  if (!q || !k || !v || !state_o || !state_lse) return fail(RLK_ERR_INVALID_ARGUMENT, "NULL tensor");
  if (params->num_seqs > rlk::kMaxSeqs) {
    // the plan is sequence-major, so a range's slabs start where the plan of
    // the sequences before it ends
    return over_ranges(params->num_seqs, [&](int s0, int s1) {
      const rlk_attn_params rp = range_params(params, s0, s1);
      SlabPlan before;
      const rlk_attn_params head = range_params(params, 0, s0);
      if (s0 > 0) plan_slabs(&head, cu_seqlens_q, cu_seqlens_k, cp_rank, pair_base, &before);
      const auto cq = rebase(cu_seqlens_q, s0, s1), ck = rebase(cu_seqlens_k, s0, s1);
      const int64_t tq = cu_seqlens_q[s0], tk = cu_seqlens_k[s0];
      return rlk_attn_prefill_states(&rp, adv(q, tq * params->num_q_heads * 128, 2),
                                     adv(k, tk * params->num_kv_heads * 128, 2), adv(v, tk * params->num_kv_heads * 128, 2),
                                     cq.data(), ck.data(), cp_rank, pair_base + before.n_pairs, state_o, state_lse,
                                     stream);
    });
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state_o))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  if (g_dry_run) return ok();
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  SlabPlan plan;
  plan_slabs(params, cu_seqlens_q, cu_seqlens_k, cp_rank, pair_base, &plan);
  if (plan.slabs.empty()) return ok();
  const int tq = cu_seqlens_q[params->num_seqs], tk = cu_seqlens_k[params->num_seqs];
  CUtensorMap mq, mk, mv;
  if ((st = make_map(&mq, q, params->num_q_heads, tq, 1, rlk::kTileRows))) return st;
  if ((st = make_map(&mk, k, params->num_kv_heads, tk, 1, params->kv_block_size))) return st;
  if ((st = make_map(&mv, v, params->num_kv_heads, tk, 1, params->kv_block_size))) return st;
  // Items: a 128-row tile of a sequence's query rows and a run of
  // consecutive blocks this rank produces (the slabs of a run follow each
  // other in the plan, so the kernel derives each block's slab from the
  // first); longest runs first.  Rows of a tile that precede a block's slab
  // see none of its keys and write nothing for it.
  const int B = params->kv_block_size;
  std::vector<std::vector<int64_t>> slab_of(params->num_seqs);  // slab offset per (seq, block), -1 if not produced
  for (int s = 0; s < params->num_seqs; ++s)
    slab_of[s].assign((cu_seqlens_k[s + 1] - cu_seqlens_k[s] + B - 1) / B, -1);
  for (const rlk_attn_slab& sl : plan.slabs) slab_of[sl.seq][sl.block] = sl.offset;
  std::vector<std::pair<int, rlk::FwdTile>> costed;
  for (int s = 0; s < params->num_seqs; ++s) {
    const int ql = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    const int kl = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
    for (int r0 = 0; r0 < ql; r0 += rlk::kTileRows) {
      const int rows = std::min(rlk::kTileRows, ql - r0);
      const int nbt = (kl - ql + r0 + rows - 1) / B + 1;  // blocks the tile's last row sees
      for (int b = 0; b < nbt;) {
        if (slab_of[s][b] < 0) {
          ++b;
          continue;
        }
        int e = b;
        while (e < nbt && slab_of[s][e] >= 0) ++e;
        rlk::FwdTile t;
        std::memset(&t, 0, sizeof(t));
        t.seq = s;
        t.row_begin = r0;
        t.row_count = rows;
        t.block = b;
        t.slab_offset = slab_of[s][b];
        t.slab_row_count = e - b;
        costed.push_back({e - b, t});
        b = e;
      }
    }
  }
  std::stable_sort(costed.begin(), costed.end(),
                   [](const std::pair<int, rlk::FwdTile>& a, const std::pair<int, rlk::FwdTile>& b) {
                     return a.first > b.first;
                   });
  std::vector<rlk::FwdTile> tiles;
  for (auto& c : costed) tiles.push_back(c.second);
  auto fp = std::make_unique<rlk::FwdParams>();
  base_fwd(fp.get(), params, dev, rlk::kModeStates);
  fill_seqs(fp.get(), params, cu_seqlens_q, cu_seqlens_k);
  fp->state_o = state_o;
  fp->state_lse = state_lse;
  if ((st = launch_fwd_tiles(fp.get(), tiles, params->num_q_heads, mq, mk, mv, dev, stream))) return st;
  return ok();
}

}  // extern "C"

namespace {

// The fused prefill, with the query rows rotated by RoPE when rope_table is
// given (at their absolute positions kv_len - q_len + i): by a pass into the
// output buffer for whole sequences, inside the kernel for one CP rank's
// rows (the buffer's other rows belong to the other ranks' calls).
rlk_status prefill_impl(const rlk_attn_params* params, const void* q, const void* k, const void* v,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t cp_rank,
                        const float* rope_table, int32_t rope_max_pos, float* out_f32, void* out_bf16, float* lse,
                        cudaStream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if ((st = check_cu(params, cu_seqlens_q, cu_seqlens_k))) return st;
  if (cp_rank < -1 || cp_rank >= params->cp_size) return fail(RLK_ERR_INVALID_ARGUMENT, "cp_rank %d", cp_rank);
  if (!q || !k || !v) return fail(RLK_ERR_INVALID_ARGUMENT, "NULL tensor");
  if (!out_f32 && !out_bf16) return fail(RLK_ERR_INVALID_ARGUMENT, "out_f32 and out_bf16 are both NULL");
  if (rope_table) {
    if (!aligned16(rope_table)) return fail(RLK_ERR_INVALID_ARGUMENT, "rope table must be 16-byte aligned");
    for (int s = 0; s < params->num_seqs; ++s)
      if (cu_seqlens_q[s + 1] > cu_seqlens_q[s] && cu_seqlens_k[s + 1] - cu_seqlens_k[s] > rope_max_pos)
        return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: position %d is past the RoPE table (%d positions)", s,
                    cu_seqlens_k[s + 1] - cu_seqlens_k[s] - 1, rope_max_pos);
  }
  if (params->num_seqs > rlk::kMaxSeqs)
    return over_ranges(params->num_seqs, [&](int s0, int s1) {
      const rlk_attn_params rp = range_params(params, s0, s1);
      const auto cq = rebase(cu_seqlens_q, s0, s1), ck = rebase(cu_seqlens_k, s0, s1);
      const int64_t tq = cu_seqlens_q[s0], tk = cu_seqlens_k[s0];
      const int64_t oq = tq * params->num_q_heads, ok_ = tk * params->num_kv_heads;
      return prefill_impl(&rp, adv(q, oq * 128, 2), adv(k, ok_ * 128, 2), adv(v, ok_ * 128, 2), cq.data(),
                          ck.data(), cp_rank, rope_table, rope_max_pos, adv(out_f32, oq * 128, 4),
                          adv(out_bf16, oq * 128, 2), adv(lse, oq, 4), stream);
    });
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (out_f32 && !aligned16(out_f32)) ||
      (out_bf16 && !aligned16(out_bf16)))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  if (g_dry_run) return ok();
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  const int B = params->kv_block_size;
  std::vector<std::pair<int, rlk::FwdTile>> costed;
  for (int s = 0; s < params->num_seqs; ++s) {
    const int ql = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    const int kl = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
    if (ql == 0) continue;
    std::vector<Chunk> parts;
    if (cp_rank < 0) parts.push_back({-1, 0, ql});
    else
      for (const Chunk& c : partition(ql, params->cp_size, params->cp_layout))
        if (c.rank == cp_rank && c.end > c.begin) parts.push_back(c);
    for (const Chunk& c : parts) {
      for (int r = c.begin; r < c.end; r += rlk::kTileRows) {
        rlk::FwdTile t;
        std::memset(&t, 0, sizeof(t));
        t.seq = s;
        t.row_begin = r;
        t.row_count = std::min(rlk::kTileRows, c.end - r);
        t.block = -1;
        const int pmax = kl - ql + r + t.row_count - 1;
        costed.push_back({pmax / B + 1, t});
      }
    }
  }
  if (costed.empty()) return ok();
  // longest first; ties by (sequence, row) so the schedule is a pure function of the inputs
  std::stable_sort(costed.begin(), costed.end(),
                   [](const std::pair<int, rlk::FwdTile>& a, const std::pair<int, rlk::FwdTile>& b) {
                     return a.first > b.first;
                   });
  std::vector<rlk::FwdTile> tiles;
  for (auto& c : costed) tiles.push_back(c.second);
  const int tq = cu_seqlens_q[params->num_seqs], tk = cu_seqlens_k[params->num_seqs];
  CUtensorMap mq, mk, mv;
  if (rope_table && cp_rank < 0) {
    // whole sequences: one pass rotates the queries into the output buffer
    // and the plain fused kernel reads them from there.  Row (token, head)
    // goes to that row's own output slot, which only the item of that token
    // tile and head reads (at its start) and writes (at its end), so no item
    // reads a slot another has overwritten.  The rotation is the canonical
    // one the kernel would apply, so the bits are the same; the pass streams
    // at HBM rate and takes the rotation off the items' critical path.
    uint16_t* rq = out_bf16 ? static_cast<uint16_t*>(out_bf16) : reinterpret_cast<uint16_t*>(out_f32);
    const int ystride = out_bf16 ? rlk::kHeadDim : 2 * rlk::kHeadDim;  // BF16 elements per (token, head) slot
    auto rp = std::make_unique<rlk::RopeParams>();
    std::memset(rp.get(), 0, sizeof(*rp));
    rp->x = static_cast<const uint16_t*>(q);
    rp->y = rq;
    rp->y_stride = ystride;
    rp->table = rope_table;
    rp->rows = static_cast<int64_t>(tq) * params->num_q_heads;
    rp->heads = params->num_q_heads;
    rp->num_seqs = params->num_seqs;
    for (int s = 0; s <= params->num_seqs; ++s) rp->cu[s] = cu_seqlens_q[s];
    for (int s = 0; s < params->num_seqs; ++s)
      rp->pos0[s] = (cu_seqlens_k[s + 1] - cu_seqlens_k[s]) - (cu_seqlens_q[s + 1] - cu_seqlens_q[s]);
    cudaError_t e = rlk::launch_rope(*rp, dev->num_sms, stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "rope launch: %s", cudaGetErrorString(e));
    if ((st = make_map(&mq, rq, params->num_q_heads, tq, 1, rlk::kTileRows, 2ull * ystride))) return st;
    rope_table = nullptr;
  } else if ((st = make_map(&mq, q, params->num_q_heads, tq, 1, rlk::kTileRows))) {
    return st;
  }
  if ((st = make_map(&mk, k, params->num_kv_heads, tk, 1, B))) return st;
  if ((st = make_map(&mv, v, params->num_kv_heads, tk, 1, B))) return st;
  auto fp = std::make_unique<rlk::FwdParams>();
  base_fwd(fp.get(), params, dev, rlk::kModeFused);
  fill_seqs(fp.get(), params, cu_seqlens_q, cu_seqlens_k);
  fp->out_f32 = out_f32;
  fp->out_bf16 = static_cast<uint16_t*>(out_bf16);
  fp->lse = lse;
  fp->rope_table = rope_table;
  if ((st = launch_fwd_tiles(fp.get(), tiles, params->num_q_heads, mq, mk, mv, dev, stream))) return st;
  return ok();
}

}  // namespace

extern "C" {

rlk_status rlk_attn_prefill(const rlk_attn_params* params, const void* q, const void* k, const void* v,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t cp_rank,
                            float* out_f32, void* out_bf16, float* lse, rlk_stream_t stream) {
  return prefill_impl(params, q, k, v, cu_seqlens_q, cu_seqlens_k, cp_rank, nullptr, 0, out_f32, out_bf16, lse,
                      stream);
}

rlk_status rlk_attn_prefill_rope(const rlk_attn_params* params, const void* q, const void* k, const void* v,
                                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t cp_rank,
                                 const float* rope_table, int32_t rope_max_pos, float* out_f32, void* out_bf16,
                                 float* lse, rlk_stream_t stream) {
  if (!rope_table) return fail(RLK_ERR_INVALID_ARGUMENT, "rope table is NULL");
  return prefill_impl(params, q, k, v, cu_seqlens_q, cu_seqlens_k, cp_rank, rope_table, rope_max_pos, out_f32,
                      out_bf16, lse, stream);
}

namespace {

rlk_status decode_paged_impl(const rlk_attn_params* params, const void* q, const void* k_pool, const void* v_pool,
                             int32_t n_pages, int32_t page_size, const int32_t* page_table, int32_t max_pages,
                             const int32_t* seqlens, const float* rope_table, int32_t rope_max_pos,
                             float* out_f32, void* out_bf16, float* lse, cudaStream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if (!q || !k_pool || !v_pool || !page_table || !seqlens) return fail(RLK_ERR_INVALID_ARGUMENT, "NULL argument");
  if (!out_f32 && !out_bf16) return fail(RLK_ERR_INVALID_ARGUMENT, "out_f32 and out_bf16 are both NULL");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || (out_f32 && !aligned16(out_f32)) ||
      (out_bf16 && !aligned16(out_bf16)))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  if (params->num_seqs > rlk::kMaxSeqs)
    return over_ranges(params->num_seqs, [&](int s0, int s1) {
      const rlk_attn_params rp = range_params(params, s0, s1);
      const int64_t o = static_cast<int64_t>(s0) * params->num_q_heads;
      return decode_paged_impl(&rp, adv(q, o * 128, 2), k_pool, v_pool, n_pages, page_size,
                               page_table + static_cast<int64_t>(s0) * max_pages, max_pages, seqlens + s0, rope_table,
                               rope_max_pos, adv(out_f32, o * 128, 4), adv(out_bf16, o * 128, 2), adv(lse, o, 4),
                               stream);
    });
  const int B = params->kv_block_size;
  if (page_size < 8 || page_size > B || B % page_size)
    return fail(RLK_ERR_UNSUPPORTED, "page_size %d must be >= 8 and divide kv_block_size %d", page_size, B);
  if (n_pages < 1 || max_pages < 1) return fail(RLK_ERR_INVALID_ARGUMENT, "n_pages / max_pages < 1");
  if (static_cast<int64_t>(n_pages + 1) * page_size >= (int64_t(1) << 31))
    return fail(RLK_ERR_UNSUPPORTED, "page pool too large for 32-bit token coordinates");
  for (int s = 0; s < params->num_seqs; ++s)
    if (seqlens[s] < 1 || static_cast<int64_t>(seqlens[s]) > static_cast<int64_t>(max_pages) * page_size)
      return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: context length %d not in 1..max_pages*page_size", s,
                  seqlens[s]);
  if (rope_table) {
    if (!aligned16(rope_table)) return fail(RLK_ERR_INVALID_ARGUMENT, "rope table must be 16-byte aligned");
    if (B != 128 || params->num_q_heads / params->num_kv_heads > rlk::kDecodeMaxGroup)
      return fail(RLK_ERR_UNSUPPORTED, "decode with RoPE needs kv_block_size 128 and at most %d query heads per KV head",
                  rlk::kDecodeMaxGroup);
    for (int s = 0; s < params->num_seqs; ++s)
      if (seqlens[s] > rope_max_pos)
        return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: position %d is past the RoPE table (%d positions)", s,
                    seqlens[s] - 1, rope_max_pos);
  }
  if (g_dry_run) return ok();
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  const int group = params->num_q_heads / params->num_kv_heads;
  std::vector<std::pair<int, rlk::FwdTile>> costed;
  for (int s = 0; s < params->num_seqs; ++s)
    for (int g = 0; g < params->num_kv_heads; ++g) {
      rlk::FwdTile t;
      std::memset(&t, 0, sizeof(t));
      t.seq = s;
      t.row_begin = g;
      t.row_count = group;
      t.block = -1;
      costed.push_back({(seqlens[s] + B - 1) / B, t});
    }
  std::stable_sort(costed.begin(), costed.end(),
                   [](const std::pair<int, rlk::FwdTile>& a, const std::pair<int, rlk::FwdTile>& b) {
                     return a.first > b.first;
                   });
  std::vector<rlk::FwdTile> tiles;
  for (auto& c : costed) tiles.push_back(c.second);
  CUtensorMap mq, mk, mv;
  // one query head per TMA box: the kernel places each head in its own lane quadrant
  if ((st = make_map(&mq, q, params->num_q_heads, params->num_seqs, 1, 1))) return st;
  if ((st = make_map(&mk, k_pool, params->num_kv_heads, static_cast<uint64_t>(n_pages) * page_size, 1, page_size)))
    return st;
  if ((st = make_map(&mv, v_pool, params->num_kv_heads, static_cast<uint64_t>(n_pages) * page_size, 1, page_size)))
    return st;
  auto fp = std::make_unique<rlk::FwdParams>();
  base_fwd(fp.get(), params, dev, rlk::kModeDecode);
  for (int s = 0; s < params->num_seqs; ++s) fp->cu_k[s] = seqlens[s];
  fp->out_f32 = out_f32;
  fp->out_bf16 = static_cast<uint16_t*>(out_bf16);
  fp->lse = lse;
  fp->page_table = page_table;
  fp->max_pages = max_pages;
  fp->page_size = page_size;
  fp->n_pages = n_pages;
  fp->rope_table = rope_table;
  if (!rlk::decode_transposed_supported(*fp)) {
    if ((st = launch_fwd_tiles(fp.get(), tiles, 1, mq, mk, mv, dev, stream))) return st;
    return ok();
  }
  // KV blocks of 128 keys and up to 8 query heads per KV head: the
  // transposed decode kernel (keys on the MMA's M side)
  for (size_t t0 = 0; t0 < tiles.size(); t0 += rlk::kMaxTilesPerLaunch) {
    const size_t n = std::min(tiles.size() - t0, static_cast<size_t>(rlk::kMaxTilesPerLaunch));
    std::copy(tiles.begin() + t0, tiles.begin() + t0 + n, fp->tiles);
    fp->num_tiles = static_cast<int32_t>(n);
    fp->num_items = static_cast<int32_t>(n);
    const int grid = std::min(fp->num_items, dev->num_sms);
    cudaError_t e = rlk::launch_decode(*fp, mq, mk, mv, grid, stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  }
  return ok();
}

}  // namespace

rlk_status rlk_attn_decode_paged(const rlk_attn_params* params, const void* q, const void* k_pool,
                                 const void* v_pool, int32_t n_pages, int32_t page_size,
                                 const int32_t* page_table, int32_t max_pages, const int32_t* seqlens,
                                 float* out_f32, void* out_bf16, float* lse, rlk_stream_t stream) {
  return decode_paged_impl(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens, nullptr, 0,
                           out_f32, out_bf16, lse, stream);
}

rlk_status rlk_attn_decode_paged_rope(const rlk_attn_params* params, const void* q, const void* k_pool,
                                      const void* v_pool, int32_t n_pages, int32_t page_size,
                                      const int32_t* page_table, int32_t max_pages, const int32_t* seqlens,
                                      const float* rope_table, int32_t rope_max_pos, float* out_f32,
                                      void* out_bf16, float* lse, rlk_stream_t stream) {
  if (!rope_table) return fail(RLK_ERR_INVALID_ARGUMENT, "rope table is NULL");
  return decode_paged_impl(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens,
                           rope_table, rope_max_pos, out_f32, out_bf16, lse, stream);
}

rlk_status rlk_attn_rope_table(double theta, int32_t max_pos, float* table) {
  if (!(theta > 1.0) || !std::isfinite(theta)) return fail(RLK_ERR_INVALID_ARGUMENT, "theta must be finite and > 1");
  if (max_pos < 1) return fail(RLK_ERR_INVALID_ARGUMENT, "max_pos %d < 1", max_pos);
  if (!table) return fail(RLK_ERR_INVALID_ARGUMENT, "table is NULL");
  constexpr int kHalf = rlk::kHeadDim / 2;
  for (int i = 0; i < kHalf; ++i) {
    // frequency theta^(-2i/D) and the angle in double, one rounding to FP32
    const double inv = std::pow(theta, (-2.0 * static_cast<double>(i)) / static_cast<double>(rlk::kHeadDim));
    for (int32_t p = 0; p < max_pos; ++p) {
      const double a = static_cast<double>(p) * inv;
      table[static_cast<int64_t>(p) * rlk::kHeadDim + i] = static_cast<float>(std::cos(a));
      table[static_cast<int64_t>(p) * rlk::kHeadDim + kHalf + i] = static_cast<float>(std::sin(a));
    }
  }
  return ok();
}

}  // extern "C"

namespace {

// The RoPE pass over x (num_heads heads) and, when x2 is given, over x2
// (num_heads2 heads) of the same tokens, in one launch.
rlk_status rope_impl(const rlk_attn_params* params, const void* x, void* y, int32_t num_heads, const void* x2,
                     void* y2, int32_t num_heads2, const int32_t* cu_seqlens, const int32_t* pos_offset,
                     const float* table, int32_t max_pos, cudaStream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if (!x || !y || !table || !cu_seqlens) return fail(RLK_ERR_INVALID_ARGUMENT, "NULL argument");
  if (!aligned16(x) || !aligned16(y) || !aligned16(table))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  if (num_heads < 1) return fail(RLK_ERR_INVALID_ARGUMENT, "num_heads %d < 1", num_heads);
  if (x2 && (!y2 || !aligned16(x2) || !aligned16(y2) || num_heads2 < 1))
    return fail(RLK_ERR_INVALID_ARGUMENT, "second tensor: NULL, unaligned or no heads");
  if (cu_seqlens[0] != 0) return fail(RLK_ERR_INVALID_ARGUMENT, "cu_seqlens must start at 0");
  if (params->num_seqs > rlk::kMaxSeqs)
    return over_ranges(params->num_seqs, [&](int s0, int s1) {
      const rlk_attn_params rp = range_params(params, s0, s1);
      const auto cu = rebase(cu_seqlens, s0, s1);
      const int64_t o = static_cast<int64_t>(cu_seqlens[s0]) * num_heads * 128;
      const int64_t o2 = static_cast<int64_t>(cu_seqlens[s0]) * num_heads2 * 128;
      return rope_impl(&rp, adv(x, o, 2), adv(y, o, 2), num_heads, x2 ? adv(x2, o2, 2) : nullptr,
                       x2 ? adv(y2, o2, 2) : nullptr, num_heads2, cu.data(), pos_offset ? pos_offset + s0 : nullptr,
                       table, max_pos, stream);
    });
  for (int s = 0; s < params->num_seqs; ++s) {
    const int64_t len = static_cast<int64_t>(cu_seqlens[s + 1]) - cu_seqlens[s];
    if (len < 0) return fail(RLK_ERR_INVALID_ARGUMENT, "cu_seqlens not monotone at sequence %d", s);
    const int64_t p0 = pos_offset ? pos_offset[s] : 0;
    if (p0 < 0) return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: negative position offset", s);
    if (len > 0 && p0 + len > max_pos)
      return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: positions up to %lld are past the table (%d positions)", s,
                  static_cast<long long>(p0 + len - 1), max_pos);
  }
  const int64_t rows = static_cast<int64_t>(cu_seqlens[params->num_seqs]) * num_heads;
  if (rows == 0) return ok();
  if (g_dry_run) return ok();
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  auto rp = std::make_unique<rlk::RopeParams>();
  std::memset(rp.get(), 0, sizeof(*rp));
  rp->x = static_cast<const uint16_t*>(x);
  rp->y = static_cast<uint16_t*>(y);
  rp->table = table;
  rp->rows = rows;
  rp->heads = num_heads;
  if (x2) {
    rp->x2 = static_cast<const uint16_t*>(x2);
    rp->y2 = static_cast<uint16_t*>(y2);
    rp->rows2 = static_cast<int64_t>(cu_seqlens[params->num_seqs]) * num_heads2;
    rp->heads2 = num_heads2;
  }
  rp->num_seqs = params->num_seqs;
  for (int s = 0; s <= params->num_seqs; ++s) rp->cu[s] = cu_seqlens[s];
  for (int s = 0; s < params->num_seqs; ++s) rp->pos0[s] = pos_offset ? pos_offset[s] : 0;
  cudaError_t e = rlk::launch_rope(*rp, dev->num_sms, stream);
  if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "rope launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

rlk_status rlk_attn_rope(const rlk_attn_params* params, const void* x, void* y, int32_t num_heads,
                         const int32_t* cu_seqlens, const int32_t* pos_offset, const float* table, int32_t max_pos,
                         rlk_stream_t stream) {
  return rope_impl(params, x, y, num_heads, nullptr, nullptr, 0, cu_seqlens, pos_offset, table, max_pos, stream);
}

rlk_status rlk_attn_rope_qk(const rlk_attn_params* params, const void* q, void* q_out, const void* k, void* k_out,
                            const int32_t* cu_seqlens, const int32_t* pos_offset, const float* table,
                            int32_t max_pos, rlk_stream_t stream) {
  if (!params) return fail(RLK_ERR_INVALID_ARGUMENT, "params is NULL");
  if (!k || !k_out) return fail(RLK_ERR_INVALID_ARGUMENT, "NULL argument");
  return rope_impl(params, q, q_out, params->num_q_heads, k, k_out, params->num_kv_heads, cu_seqlens, pos_offset,
                   table, max_pos, stream);
}


namespace {

// Split factor for split_k == 0.  Cost of a candidate k, in units of one KV
// block's processing time on one SM: the busiest CTA's load when the items
// (sorted by size, largest first) are dealt to min(items, SMs) CTAs in the
// decode kernel's snake order, each item adding a fixed start-up, plus -- for
// k > 1 -- the fold kernel, whose serial lse chain walks the longest
// sequence's blocks.  Candidates stay within one launch's item list; ties go
// to the smaller k (less state traffic).
constexpr double kSplitItemStartup = 1.0;  // blocks' worth of start-up per item
constexpr double kSplitFoldPerBlock = 0.08;  // fold chain step / KV block step

// split decode workspace: the state table (o_b then lse_b of every pair),
// rounded to 256 bytes, then one 8-byte fill flag per (sequence, KV head,
// item) for the on-chip fold
size_t split_table_bytes(int64_t pairs) {
  return static_cast<size_t>((pairs * (rlk::kHeadDim + 1) * 4 + 255) / 256 * 256);
}
size_t split_flag_bytes(int num_seqs, int hkv) {
  return static_cast<size_t>(num_seqs) * hkv * rlk::kMaxSplitK * sizeof(uint64_t);
}

// A value no earlier call of this process has used (an odd step walks all
// 2^64 values before repeating), from a random start, so that a flag an
// earlier call or another process left in a workspace does not hold it.
uint64_t next_fill_nonce() {
  static std::atomic<uint64_t> next{[] {
    std::random_device rd;
    return (static_cast<uint64_t>(rd()) << 32) ^ rd() ^
           static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count());
  }()};
  for (;;) {
    const uint64_t v = next.fetch_add(0x9E3779B97F4A7C15ull);
    if (v != 0 && v != ~0ull) return v;  // not the values a zero or all-ones fill leaves
  }
}

// The fold on chip: split_k producer items per (sequence, KV head) pair and
// fold CTAs (one warp per (sequence, query head), 16 a CTA) in one
// cooperative launch, the folds following their producers, so every CTA must
// be resident at once: one CTA per SM.
constexpr int kFoldChainsPerCta = 16;
int fold_ctas(int num_seqs, int hq) { return (num_seqs * hq + kFoldChainsPerCta - 1) / kFoldChainsPerCta; }
bool fold_on_chip(int num_seqs, int hkv, int hq, int k, int num_sms) {
  const int64_t items = static_cast<int64_t>(num_seqs) * hkv * k;
  return k >= 2 && items + fold_ctas(num_seqs, hq) <= num_sms && items <= rlk::kMaxTilesPerLaunch;
}

int choose_split(const int32_t* seqlens, int num_seqs, int hkv, int hq, int B, int num_sms) {
  std::vector<int> nbs(num_seqs);
  int nb_max = 0;
  for (int s = 0; s < num_seqs; ++s) {
    nbs[s] = (seqlens[s] + B - 1) / B;
    nb_max = std::max(nb_max, nbs[s]);
  }
  // few pairs: spread each over as many SMs as there are to share, with the
  // fold on chip (hidden behind the producers, so no fold term to weigh)
  {
    const int free_sms = num_sms - fold_ctas(num_seqs, hq);
    const int k = std::min({std::max(free_sms, 0) / std::max(num_seqs * hkv, 1), nb_max, 64});
    if (fold_on_chip(num_seqs, hkv, hq, k, num_sms)) return k;
  }
  int best_k = 1;
  double best = 0.0;
  std::vector<int> sizes;
  std::vector<double> load;
  for (int k = 1; k <= 64; ++k) {
    sizes.clear();
    for (int s = 0; s < num_seqs; ++s)
      for (int r = 0; r < k; ++r) {
        const int n = static_cast<int>(static_cast<int64_t>(r + 1) * nbs[s] / k - static_cast<int64_t>(r) * nbs[s] / k);
        if (n > 0)
          for (int g = 0; g < hkv; ++g) sizes.push_back(n);
      }
    if (k > 1 && sizes.size() > static_cast<size_t>(rlk::kMaxTilesPerLaunch)) break;
    std::sort(sizes.begin(), sizes.end(), [](int a, int b) { return a > b; });
    const int grid = std::min(static_cast<int>(sizes.size()), num_sms);
    load.assign(grid, 0.0);
    for (size_t i = 0; i < sizes.size(); ++i) {
      const int round = static_cast<int>(i / grid), c = static_cast<int>(i % grid);
      load[(round & 1) ? grid - 1 - c : c] += sizes[i] + kSplitItemStartup;
    }
    double cost = *std::max_element(load.begin(), load.end());
    if (k > 1) cost += nb_max * kSplitFoldPerBlock;
    if (k == 1 || cost < best) {
      best = cost;
      best_k = k;
    }
  }
  return best_k;
}

}  // namespace

int32_t rlk_attn_decode_auto_split(const rlk_attn_params* params, const int32_t* seqlens, int32_t num_sms) {
  if (check_params(params) || !seqlens || num_sms < 1) return -1;
  const int B = params->kv_block_size;
  for (int s = 0; s < params->num_seqs; ++s)
    if (seqlens[s] < 1) return -1;
  return choose_split(seqlens, params->num_seqs, params->num_kv_heads, params->num_q_heads, B, num_sms);
}

namespace {

rlk_status decode_splitk_impl(const rlk_attn_params* params, const void* q, const void* k_pool, const void* v_pool,
                              int32_t n_pages, int32_t page_size, const int32_t* page_table, int32_t max_pages,
                              const int32_t* seqlens, int32_t split_k, const float* rope_table,
                              int32_t rope_max_pos, float* out_f32, void* out_bf16, float* lse, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if (!q || !k_pool || !v_pool || !page_table || !seqlens) return fail(RLK_ERR_INVALID_ARGUMENT, "NULL argument");
  if (!out_f32 && !out_bf16) return fail(RLK_ERR_INVALID_ARGUMENT, "out_f32 and out_bf16 are both NULL");
  if (split_k < 0 || split_k > 64) return fail(RLK_ERR_INVALID_ARGUMENT, "split_k %d not in 0..64", split_k);
  if (params->num_seqs > rlk::kMaxSeqs)
    // each range reuses the workspace from its start (the ranges run in
    // order on the stream, and a range's state table is no larger than the
    // whole call's)
    return over_ranges(params->num_seqs, [&](int s0, int s1) {
      const rlk_attn_params rp = range_params(params, s0, s1);
      const int64_t o = static_cast<int64_t>(s0) * params->num_q_heads;
      return decode_splitk_impl(&rp, adv(q, o * 128, 2), k_pool, v_pool, n_pages, page_size,
                                page_table + static_cast<int64_t>(s0) * max_pages, max_pages, seqlens + s0, split_k,
                                rope_table, rope_max_pos, adv(out_f32, o * 128, 4), adv(out_bf16, o * 128, 2),
                                adv(lse, o, 4), workspace, workspace_bytes, stream);
    });
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || (out_f32 && !aligned16(out_f32)) ||
      (out_bf16 && !aligned16(out_bf16)) || !aligned16(workspace))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  const int B = params->kv_block_size;
  const int group = params->num_q_heads / params->num_kv_heads;
  if (B != 128 || group > rlk::kDecodeMaxGroup)
    return fail(RLK_ERR_UNSUPPORTED, "split decode needs kv_block_size 128 and at most %d query heads per KV head",
                rlk::kDecodeMaxGroup);
  if (page_size < 8 || page_size > B || B % page_size)
    return fail(RLK_ERR_UNSUPPORTED, "page_size %d must be >= 8 and divide kv_block_size %d", page_size, B);
  if (n_pages < 1 || max_pages < 1) return fail(RLK_ERR_INVALID_ARGUMENT, "n_pages / max_pages < 1");
  if (static_cast<int64_t>(n_pages + 1) * page_size >= (int64_t(1) << 31))
    return fail(RLK_ERR_UNSUPPORTED, "page pool too large for 32-bit token coordinates");
  for (int s = 0; s < params->num_seqs; ++s)
    if (seqlens[s] < 1 || static_cast<int64_t>(seqlens[s]) > static_cast<int64_t>(max_pages) * page_size)
      return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: context length %d not in 1..max_pages*page_size", s,
                  seqlens[s]);
  if (rope_table) {
    if (!aligned16(rope_table)) return fail(RLK_ERR_INVALID_ARGUMENT, "rope table must be 16-byte aligned");
    for (int s = 0; s < params->num_seqs; ++s)
      if (seqlens[s] > rope_max_pos)
        return fail(RLK_ERR_INVALID_ARGUMENT, "sequence %d: position %d is past the RoPE table (%d positions)", s,
                    seqlens[s] - 1, rope_max_pos);
  }
  const size_t need = rlk_attn_workspace_size(params, RLK_OP_DECODE_SPLIT, nullptr, seqlens);
  if (!workspace || workspace_bytes < need)
    return fail(RLK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", workspace_bytes, need);
  if (g_dry_run) return ok();
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  if (split_k == 0) {
    split_k = choose_split(seqlens, params->num_seqs, params->num_kv_heads, params->num_q_heads, B, dev->num_sms);
    // one range per sequence is the single-pass decode, which needs no state table
    if (split_k == 1)
      return decode_paged_impl(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens,
                               rope_table, rope_max_pos, out_f32, out_bf16, lse, stream);
  }
  // state table: pair (block_base[s] + b) * Hq + head; o_b FP32 [pair][128], then lse_b [pair]
  std::vector<int32_t> block_base(params->num_seqs + 1, 0);
  for (int s = 0; s < params->num_seqs; ++s) block_base[s + 1] = block_base[s] + (seqlens[s] + B - 1) / B;
  const int64_t pairs = static_cast<int64_t>(block_base[params->num_seqs]) * params->num_q_heads;
  bool on_chip = fold_on_chip(params->num_seqs, params->num_kv_heads, params->num_q_heads, split_k, dev->num_sms);
  std::vector<std::pair<int, rlk::FwdTile>> costed;
  if (on_chip) {
    // item r of a pair takes its blocks r, r + k, r + 2k, ...: the pair's
    // blocks are produced in ascending order across its k CTAs, and the fold
    // warps of item 0 follow them
    for (int s = 0; s < params->num_seqs; ++s) {
      const int nb = (seqlens[s] + B - 1) / B;
      for (int g = 0; g < params->num_kv_heads; ++g)
        for (int r = 0; r < split_k && r < nb; ++r) {
          rlk::FwdTile t;
          std::memset(&t, 0, sizeof(t));
          t.seq = s;
          t.row_begin = g;
          t.row_count = group;
          t.block = r;
          t.slab_row_count = (nb - r + split_k - 1) / split_k;
          costed.push_back({t.slab_row_count, t});
        }
    }
  }
  // contiguous ranges (the second kernel folds), longest first
  auto contiguous_items = [&]() {
    costed.clear();
    for (int s = 0; s < params->num_seqs; ++s) {
      const int nb = (seqlens[s] + B - 1) / B;
      for (int g = 0; g < params->num_kv_heads; ++g)
        for (int r = 0; r < split_k; ++r) {
          const int b0 = static_cast<int>(static_cast<int64_t>(r) * nb / split_k);
          const int b1 = static_cast<int>(static_cast<int64_t>(r + 1) * nb / split_k);
          if (b1 <= b0) continue;
          rlk::FwdTile t;
          std::memset(&t, 0, sizeof(t));
          t.seq = s;
          t.row_begin = g;
          t.row_count = group;
          t.block = b0;
          t.slab_row_count = b1 - b0;
          costed.push_back({b1 - b0, t});
        }
    }
    std::stable_sort(costed.begin(), costed.end(),
                     [](const std::pair<int, rlk::FwdTile>& a, const std::pair<int, rlk::FwdTile>& b) {
                       return a.first > b.first;
                     });
  };
  if (!on_chip) contiguous_items();
  CUtensorMap mq, mk, mv;
  // one query head per TMA box: the kernel places each head in its own operand row
  if ((st = make_map(&mq, q, params->num_q_heads, params->num_seqs, 1, 1))) return st;
  if ((st = make_map(&mk, k_pool, params->num_kv_heads, static_cast<uint64_t>(n_pages) * page_size, 1, page_size)))
    return st;
  if ((st = make_map(&mv, v_pool, params->num_kv_heads, static_cast<uint64_t>(n_pages) * page_size, 1, page_size)))
    return st;
  auto fp = std::make_unique<rlk::FwdParams>();
  base_fwd(fp.get(), params, dev, rlk::kModeDecode);
  for (int s = 0; s < params->num_seqs; ++s) {
    fp->cu_k[s] = seqlens[s];
    fp->cu_q[s] = block_base[s];
  }
  fp->state_o = static_cast<float*>(workspace);
  fp->state_lse = static_cast<float*>(workspace) + pairs * rlk::kHeadDim;
  fp->rope_table = rope_table;
  fp->page_table = page_table;
  fp->max_pages = max_pages;
  fp->page_size = page_size;
  fp->n_pages = n_pages;
  if (on_chip) {
    // the fold warps take a state as landed once it differs from the fill;
    // each item fills its own slots and publishes a flag, except inside a
    // graph capture, where a replay would find the flags of the previous
    // replay already set: there a fill of the table precedes the launch
    const size_t state_bytes = static_cast<size_t>(pairs) * (rlk::kHeadDim + 1) * 4;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
      (void)cudaGetLastError();
      cap = cudaStreamCaptureStatusActive;  // unknown: take the form that is safe in both
    }
    const bool self_fill = cap == cudaStreamCaptureStatusNone;
    fp->fill_flag = self_fill ? reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(workspace) + split_table_bytes(pairs))
                              : nullptr;
    fp->fill_nonce = self_fill ? next_fill_nonce() : 0;
    fp->split_stride = split_k;
    fp->fold_seqs = params->num_seqs;
    fp->out_f32 = out_f32;
    fp->out_bf16 = static_cast<uint16_t*>(out_bf16);
    fp->lse = lse;
    for (size_t i = 0; i < costed.size(); ++i) fp->tiles[i] = costed[i].second;
    fp->num_tiles = static_cast<int32_t>(costed.size());
    fp->num_items = fp->num_tiles;
    static_assert(rlk::kUnwritten == 0xFFFFFFFFu, "the table fill is all-ones bytes");
    cudaError_t e = self_fill ? cudaSuccess : cudaMemsetAsync(workspace, 0xFF, state_bytes, stream);
    const int grid = fp->num_items + fold_ctas(params->num_seqs, params->num_q_heads);
    if (e == cudaSuccess) e = rlk::launch_decode_cooperative(*fp, mq, mk, mv, grid, stream);
    if (e == cudaSuccess) return ok();
    if (e != cudaErrorCooperativeLaunchTooLarge && e != cudaErrorNotSupported)
      return fail(RLK_ERR_CUDA, "split decode launch: %s", cudaGetErrorString(e));
    // fewer SMs free than the device has (shared or partitioned), or no
    // cooperative launches: the same split in contiguous ranges, folded by
    // the second kernel
    (void)cudaGetLastError();
    on_chip = false;
    fp->split_stride = 0;
    fp->fold_seqs = 0;
    fp->fill_flag = nullptr;
    contiguous_items();
  }
  for (size_t t0 = 0; t0 < costed.size(); t0 += rlk::kMaxTilesPerLaunch) {
    const size_t n = std::min(costed.size() - t0, static_cast<size_t>(rlk::kMaxTilesPerLaunch));
    for (size_t i = 0; i < n; ++i) fp->tiles[i] = costed[t0 + i].second;
    fp->num_tiles = static_cast<int32_t>(n);
    fp->num_items = static_cast<int32_t>(n);
    const int grid = std::min(fp->num_items, dev->num_sms);
    cudaError_t e = rlk::launch_decode(*fp, mq, mk, mv, grid, stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "split decode launch: %s", cudaGetErrorString(e));
  }
  // fold: num_tiles carries the sequence count for the merge
  fp->num_tiles = params->num_seqs;
  fp->out_f32 = out_f32;
  fp->out_bf16 = static_cast<uint16_t*>(out_bf16);
  fp->lse = lse;
  cudaError_t e = rlk::launch_decode_merge(*fp, dev->num_sms, stream);
  if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "split decode merge launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

rlk_status rlk_attn_decode_paged_splitk(const rlk_attn_params* params, const void* q, const void* k_pool,
                                        const void* v_pool, int32_t n_pages, int32_t page_size,
                                        const int32_t* page_table, int32_t max_pages,
                                        const int32_t* seqlens, int32_t split_k, float* out_f32,
                                        void* out_bf16, float* lse, void* workspace,
                                        size_t workspace_bytes, rlk_stream_t stream) {
  return decode_splitk_impl(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens, split_k,
                            nullptr, 0, out_f32, out_bf16, lse, workspace, workspace_bytes, stream);
}

rlk_status rlk_attn_decode_paged_splitk_rope(const rlk_attn_params* params, const void* q, const void* k_pool,
                                             const void* v_pool, int32_t n_pages, int32_t page_size,
                                             const int32_t* page_table, int32_t max_pages,
                                             const int32_t* seqlens, int32_t split_k, const float* rope_table,
                                             int32_t rope_max_pos, float* out_f32, void* out_bf16, float* lse,
                                             void* workspace, size_t workspace_bytes, rlk_stream_t stream) {
  if (!rope_table) return fail(RLK_ERR_INVALID_ARGUMENT, "rope table is NULL");
  return decode_splitk_impl(params, q, k_pool, v_pool, n_pages, page_size, page_table, max_pages, seqlens, split_k,
                            rope_table, rope_max_pos, out_f32, out_bf16, lse, workspace, workspace_bytes, stream);
}

size_t rlk_attn_workspace_size(const rlk_attn_params* params, int32_t op, const int32_t* cu_seqlens_q,
                               const int32_t* cu_seqlens_k) {
  if (check_params(params) != RLK_OK) return 0;
  if (op == RLK_OP_DECODE_SPLIT) {
    if (!cu_seqlens_k) return 0;
    int64_t blocks = 0;
    for (int s = 0; s < params->num_seqs; ++s) {
      if (cu_seqlens_k[s] < 1) return 0;
      blocks += (cu_seqlens_k[s] + params->kv_block_size - 1) / params->kv_block_size;
    }
    const int64_t pairs = blocks * params->num_q_heads;
    return split_table_bytes(pairs) + split_flag_bytes(params->num_seqs, params->num_kv_heads);
  }
  if (op == RLK_OP_MERGE) {
    if (check_cu(params, cu_seqlens_q, cu_seqlens_k) != RLK_OK) return 0;
    int max_blocks = 1;
    for (int s = 0; s < params->num_seqs; ++s)
      max_blocks = std::max(max_blocks, (cu_seqlens_k[s + 1] - cu_seqlens_k[s] + params->kv_block_size - 1) /
                                            params->kv_block_size);
    const size_t bytes = static_cast<size_t>(params->num_seqs) * max_blocks * sizeof(int32_t);
    return (bytes + 255) / 256 * 256;
  }
  if (op == RLK_OP_BACKWARD) {
    if (check_cu(params, cu_seqlens_q, cu_seqlens_q) != RLK_OK) return 0;
    return rlk::backward_workspace_bytes(params, cu_seqlens_q);
  }
  return 0;
}

}  // extern "C"

namespace {

// The merge of one launch's sequence range [seq_base, seq_base + num_seqs)
// of a call over total_seqs sequences: cu_q / cu_k are the range's (rebased),
// out / lse point at the range's first row, and the slab table, state table
// and index scratch are the whole call's.
rlk_status merge_range(const rlk_attn_params* params, const int32_t* cu_q, const int32_t* cu_k, int seq_base,
                       int total_seqs, const rlk_attn_slab* slabs, int64_t n_slabs, const float* state_o,
                       const float* state_lse, int64_t n_state_pairs, float* out_f32, void* out_bf16, float* lse,
                       int32_t* index, const DeviceInfo* dev, cudaStream_t stream) {
  const int64_t total_rows = cu_q[params->num_seqs];
  if (total_rows == 0) return ok();
  auto mp = std::make_unique<rlk::MergeParams>();
  std::memset(mp.get(), 0, sizeof(*mp));
  mp->err = dev->err;
  mp->num_seqs = params->num_seqs;
  mp->hq = params->num_q_heads;
  mp->block = params->kv_block_size;
  int max_blocks = 1;
  for (int s = 0; s < params->num_seqs; ++s)
    max_blocks = std::max(max_blocks, (cu_k[s + 1] - cu_k[s] + params->kv_block_size - 1) / params->kv_block_size);
  mp->max_blocks = max_blocks;
  mp->seq_base = seq_base;
  mp->total_seqs = total_seqs;
  mp->total_rows = total_rows;
  mp->n_slabs = n_slabs;
  mp->slabs = reinterpret_cast<const rlk::Slab*>(slabs);
  mp->state_o = state_o;
  mp->state_lse = state_lse;
  mp->n_pairs = n_state_pairs;
  mp->index = index;
  mp->out_f32 = out_f32;
  mp->out_bf16 = static_cast<uint16_t*>(out_bf16);
  mp->lse = lse;
  for (int s = 0; s <= params->num_seqs; ++s) {
    mp->cu_q[s] = cu_q[s];
    mp->cu_k[s] = cu_k[s];
  }
  const cudaError_t e = rlk::launch_merge(*mp, dev->num_sms, stream);
  if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
  return ok();
}

// Both merge entry points after their own checks: the whole call, or its
// kMaxSeqs-sequence ranges in order (each range indexes only its own
// sequences' slabs, so the index scratch is reused range after range).
rlk_status merge_call(const rlk_attn_params* params, const int32_t* cu_q, const int32_t* cu_k,
                      const rlk_attn_slab* slabs, int64_t n_slabs, const float* state_o, const float* state_lse,
                      int64_t n_state_pairs, float* out_f32, void* out_bf16, float* lse, int32_t* index,
                      const DeviceInfo* dev, cudaStream_t stream) {
  if (params->num_seqs <= rlk::kMaxSeqs)
    return merge_range(params, cu_q, cu_k, 0, params->num_seqs, slabs, n_slabs, state_o, state_lse, n_state_pairs,
                       out_f32, out_bf16, lse, index, dev, stream);
  for (int s0 = 0; s0 < params->num_seqs; s0 += rlk::kMaxSeqs) {
    const int s1 = std::min(params->num_seqs, s0 + rlk::kMaxSeqs);
    const rlk_attn_params rp = range_params(params, s0, s1);
    const auto cq = rebase(cu_q, s0, s1), ck = rebase(cu_k, s0, s1);
    const int64_t o = static_cast<int64_t>(cu_q[s0]) * params->num_q_heads;
    const rlk_status st = merge_range(&rp, cq.data(), ck.data(), s0, params->num_seqs, slabs, n_slabs, state_o,
                                      state_lse, n_state_pairs, adv(out_f32, o * 128, 4), adv(out_bf16, o * 128, 2),
                                      adv(lse, o, 4), index, dev, stream);
    if (st) return st;
  }
  return ok();
}

}  // namespace

extern "C" {

rlk_status rlk_attn_merge_states(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                 const int32_t* cu_seqlens_k, const rlk_attn_slab* slabs, int64_t n_slabs,
                                 const float* state_o, const float* state_lse, int64_t n_state_pairs,
                                 float* out_f32, void* out_bf16, float* lse, void* workspace,
                                 size_t workspace_bytes, rlk_stream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if ((st = check_cu(params, cu_seqlens_q, cu_seqlens_k))) return st;
  if (n_slabs < 0 || n_state_pairs < 0 || (n_slabs > 0 && (!slabs || !state_o || !state_lse)))
    return fail(RLK_ERR_INVALID_ARGUMENT, "bad state table");
  if (!out_f32 && !out_bf16) return fail(RLK_ERR_INVALID_ARGUMENT, "out_f32 and out_bf16 are both NULL");
  if ((out_f32 && !aligned16(out_f32)) || (out_bf16 && !aligned16(out_bf16)) || (state_o && !aligned16(state_o)) ||
      (slabs && !aligned16(slabs)))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  const size_t need = rlk_attn_workspace_size(params, RLK_OP_MERGE, cu_seqlens_q, cu_seqlens_k);
  if (!workspace || workspace_bytes < need)
    return fail(RLK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  return merge_call(params, cu_seqlens_q, cu_seqlens_k, slabs, n_slabs, state_o, state_lse, n_state_pairs, out_f32,
                    out_bf16, lse, static_cast<int32_t*>(workspace), dev, stream);
}

rlk_status rlk_attn_merge_states_noalloc(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                         const int32_t* cu_seqlens_k, const rlk_attn_slab* slabs,
                                         int64_t n_slabs, const float* state_o, const float* state_lse,
                                         int64_t n_state_pairs, float* out_f32, void* out_bf16, float* lse,
                                         rlk_stream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if ((st = check_cu(params, cu_seqlens_q, cu_seqlens_k))) return st;
  if (n_slabs < 0 || n_state_pairs < 0 || (n_slabs > 0 && (!slabs || !state_o || !state_lse)))
    return fail(RLK_ERR_INVALID_ARGUMENT, "bad state table");
  if (!out_f32 && !out_bf16) return fail(RLK_ERR_INVALID_ARGUMENT, "out_f32 and out_bf16 are both NULL");
  if ((out_f32 && !aligned16(out_f32)) || (out_bf16 && !aligned16(out_bf16)) || (state_o && !aligned16(state_o)) ||
      (slabs && !aligned16(slabs)))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  int max_blocks = 1;
  for (int s = 0; s < params->num_seqs; ++s)
    max_blocks = std::max(max_blocks, (cu_seqlens_k[s + 1] - cu_seqlens_k[s] + params->kv_block_size - 1) /
                                          params->kv_block_size);
  // size limit first: nothing touches the device for a problem the scratch cannot hold
  if (static_cast<int64_t>(params->num_seqs) * max_blocks > rlk::kNoAllocIndexEntries)
    return fail(RLK_ERR_UNSUPPORTED,
                "no-alloc merge: num_seqs * max KV blocks per sequence = %lld exceeds the %lld-entry scratch",
                static_cast<long long>(params->num_seqs) * max_blocks,
                static_cast<long long>(rlk::kNoAllocIndexEntries));
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  return merge_call(params, cu_seqlens_q, cu_seqlens_k, slabs, n_slabs, state_o, state_lse, n_state_pairs, out_f32,
                    out_bf16, lse, dev->merge_scratch, dev, stream);
}

rlk_status rlk_attn_backward(const rlk_attn_params* params, const void* q, const void* k, const void* v,
                             const float* out_f32, const void* dout, const float* lse, const int32_t* cu_seqlens,
                             int32_t cp_rank, float* dq, float* dk, float* dv, void* workspace,
                             size_t workspace_bytes, rlk_stream_t stream) {
  rlk_status st = check_params(params);
  if (st) return st;
  if ((st = check_cu(params, cu_seqlens, cu_seqlens))) return st;
  if (cp_rank < -1 || cp_rank >= params->cp_size) return fail(RLK_ERR_INVALID_ARGUMENT, "cp_rank %d", cp_rank);
  if (!q || !k || !v || !out_f32 || !dout || !lse || !dq || !dk || !dv)
    return fail(RLK_ERR_INVALID_ARGUMENT, "NULL tensor");
  if (params->kv_block_size != 128) return fail(RLK_ERR_UNSUPPORTED, "the backward takes KV block 128");
  if (params->num_seqs > rlk::kMaxSeqs)
    return over_ranges(params->num_seqs, [&](int s0, int s1) {
      const rlk_attn_params rp = range_params(params, s0, s1);
      const auto cu = rebase(cu_seqlens, s0, s1);
      const int64_t t = cu_seqlens[s0];
      const int64_t oq = t * params->num_q_heads, ok_ = t * params->num_kv_heads;
      return rlk_attn_backward(&rp, adv(q, oq * 128, 2), adv(k, ok_ * 128, 2), adv(v, ok_ * 128, 2),
                               adv(out_f32, oq * 128, 4), adv(dout, oq * 128, 2), adv(lse, oq, 4), cu.data(), cp_rank,
                               adv(dq, oq * 128, 4), adv(dk, ok_ * 128, 4), adv(dv, ok_ * 128, 4), workspace,
                               workspace_bytes, stream);
    });
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out_f32) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(RLK_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  const size_t need = rlk::backward_workspace_bytes(params, cu_seqlens);
  if (!workspace || workspace_bytes < need)
    return fail(RLK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
  if (g_dry_run) return ok();
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev))) return st;
  st = rlk::run_backward(params, q, k, v, out_f32, dout, lse, cu_seqlens, cp_rank, dq, dk, dv, workspace,
                         workspace_bytes, dev->err, dev->num_sms, stream);
  if (st) return st;
  return ok();
}

namespace {

// One warp waits on a barrier that nothing completes, through the same
// bounded wait every kernel uses: after the wait's limit it reports a
// timeout (site 0x7e1) in the error word and returns.
__global__ void rlk_wait_selftest_kernel(rlk::ErrWord* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    rlk::mbar_init(&bar, 1);
    abort_flag = 0;
    rlk::fence_mbar_init();
  }
  __syncthreads();
  (void)rlk::mbar_wait(&bar, 0, &abort_flag, err, 0x7e1);
}

}  // namespace

rlk_status rlk_attn_selftest_wait_timeout(rlk_stream_t stream) {
  DeviceInfo* dev = nullptr;
  rlk_status st = device_info(&dev);
  if (st) return st;
  rlk_wait_selftest_kernel<<<1, 32, 0, stream>>>(dev->err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return ok();
}

rlk_status rlk_attn_check_device_error(rlk_stream_t stream) {
  DeviceInfo* dev = nullptr;
  rlk_status st = device_info(&dev);
  if (st) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
  rlk::ErrWord w{0, 0};
  e = cudaMemcpy(&w, dev->err, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(RLK_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
  if (w.bits == 0) return ok();
  const rlk::ErrWord zero{0, 0};
  cudaMemcpy(dev->err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (w.bits & rlk::kErrDeviceTimeout) return fail(RLK_ERR_DEVICE_TIMEOUT, "device wait timed out (site 0x%x)", w.site);
  // a slab that was not read also leaves its block missing: report the cause
  if (w.bits & rlk::kErrBadSlab) return fail(RLK_ERR_BAD_STATE_TABLE, "state table slab out of range");
  if (w.bits & rlk::kErrDuplicateBlock) return fail(RLK_ERR_DUPLICATE_BLOCK, "duplicate global block in state table");
  if (w.bits & rlk::kErrMissingBlock) return fail(RLK_ERR_MISSING_BLOCK, "missing global block in state table");
  if (w.bits & rlk::kErrBadPage) return fail(RLK_ERR_BAD_PAGE, "page id outside the pool");
  return fail(RLK_ERR_CUDA, "device error bits 0x%x", w.bits);
}

}  // extern "C"
