/*
 * rlk_oracle.c -- plain CPU oracle for deterministic context attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * execute this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes, and the passage each function follows:
 *
 *   rlko_attention_f64        causal GQA attention by its definition, FP64
 *                             ("WS2 Attention PR5 Drift Benchmark", Scope:
 *                             Hq=32, Hkv=8, D=128; full and chunked prefill).
 *   rlko_row_block_states_f64 the per-block partial state
 *                             state_i = (out_i, lse_i, global_block_index_i)
 *                             ("WS2 Attention PR5 Drift Benchmark",
 *                             Transformer Engine Reuse), FP64.
 *   rlko_fold_f32             sort states by global_block_index, then merge
 *                             with the online-softmax correction in FP32
 *                             (same section; "H100 validation and reproduction
 *                             guide", Status: FP32 accumulation, fixed
 *                             global_block_index merge order).  An arrival-order
 *                             variant is the negative control named by the
 *                             reduction_order knob of the cross-config PR #263.
 *   rlko_decode_paged_f64     one decode token per sequence read through a
 *                             paged KV pool and page table ("H100 validation
 *                             and reproduction guide", PR stack: decode KV-cache
 *                             replay, paged-KV adapter), FP64.
 *   rlko_backward_f64         dQ/dK/dV of the attention above by its
 *                             definition ("WS2 Attention PR5 Drift Benchmark",
 *                             Scope: optional backward dq, dk, dv), FP64.
 *   rlko_rope_f32             rotary position embedding of Q or K rows in
 *                             the canonical FP32 form, BF16 result
 *                             ("WS2 Attention PR5 Drift Benchmark", Scope:
 *                             optional RoPE composition before Attention,
 *                             Attention consuming post-RoPE Q/K; "H100
 *                             validation and reproduction guide", PR stack:
 *                             decode KV-cache replay and cache/position/RoPE
 *                             identity).
 *   rlko_rope_f64             the same rotation exactly, in double (for the
 *                             pins of rlko_rope_f32).
 *
 * Inputs are float32 arrays holding exact BF16 values; every arithmetic step
 * of the FP64 functions is done in double.  Build with -ffp-contract=off so
 * that no multiply-add is fused behind the reader's back.
 *
 * Pins: every function is checked on the CPU against closed forms, brute
 * force on tiny inputs, the log-sum-exp decomposition identity, finite
 * differences and invariants (tests/test_oracle.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define RLKO_OK 0
#define RLKO_EINVAL 1
#define RLKO_EDUP 2

/* Sequence containing packed token t: the s with cu[s] <= t < cu[s+1]. */
static int seq_of_token(int num_seqs, const int32_t* cu, int64_t t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

static int check_seqlens(int num_seqs, const int32_t* cu_q, const int32_t* cu_k) {
  if (num_seqs <= 0 || cu_q[0] != 0 || cu_k[0] != 0) return RLKO_EINVAL;
  for (int s = 0; s < num_seqs; ++s) {
    int ql = cu_q[s + 1] - cu_q[s], kl = cu_k[s + 1] - cu_k[s];
    if (ql < 0 || kl < 0 || ql > kl) return RLKO_EINVAL;
  }
  return RLKO_OK;
}

/*
 * Causal GQA attention, FP64, by definition.
 *
 * q [Tq, hq, d], k/v [Tk, hkv, d].  Query row i of sequence s sits at key
 * position p = kv_len - q_len + i (bottom-right alignment, so a chunk of new
 * queries sees the whole cache before it).  For query head h the KV head is
 * h / (hq / hkv).  With causal, keys j <= p are visible; otherwise all keys.
 *
 *   s_j   = scale * sum_d q_d k_jd
 *   lse   = log sum_j exp(s_j)            (natural log)
 *   out_d = sum_j exp(s_j - lse) v_jd
 *
 * rows == NULL: every token, out [Tq, hq, d], lse [Tq, hq].
 * rows != NULL: the n_rows listed tokens, out [n_rows, hq, d], lse [n_rows, hq].
 */
int rlko_attention_f64(int num_seqs, const int32_t* cu_q, const int32_t* cu_k,
                       int hq, int hkv, int d, double scale, int causal,
                       const float* q, const float* k, const float* v,
                       int64_t n_rows, const int64_t* rows,
                       double* out, double* lse) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || d <= 0) return RLKO_EINVAL;
  if (check_seqlens(num_seqs, cu_q, cu_k)) return RLKO_EINVAL;
  const int64_t tq = cu_q[num_seqs];
  const int64_t n = rows ? n_rows : tq;
  for (int64_t r = 0; r < n; ++r)
    if (rows && (rows[r] < 0 || rows[r] >= tq)) return RLKO_EINVAL;
  const int group = hq / hkv;
  int64_t max_kv = 0;
  for (int s = 0; s < num_seqs; ++s)
    if (cu_k[s + 1] - cu_k[s] > max_kv) max_kv = cu_k[s + 1] - cu_k[s];

#pragma omp parallel
  {
    double* sc = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t rh = 0; rh < n * hq; ++rh) {
      const int64_t r = rh / hq;
      const int h = (int)(rh % hq);
      const int64_t t = rows ? rows[r] : r;
      const int s = seq_of_token(num_seqs, cu_q, t);
      const int64_t i = t - cu_q[s];
      const int64_t q_len = cu_q[s + 1] - cu_q[s];
      const int64_t kv_len = cu_k[s + 1] - cu_k[s];
      const int64_t p = kv_len - q_len + i;
      const int64_t nkeys = causal ? p + 1 : kv_len;
      const int g = h / group;
      const float* qr = q + ((size_t)t * hq + h) * d;
      double m = -INFINITY;
      for (int64_t j = 0; j < nkeys; ++j) {
        const float* kr = k + ((size_t)(cu_k[s] + j) * hkv + g) * d;
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += (double)qr[e] * (double)kr[e];
        sc[j] = scale * acc;
        if (sc[j] > m) m = sc[j];
      }
      double sum = 0.0;
      for (int64_t j = 0; j < nkeys; ++j) sum += exp(sc[j] - m);
      const double l = m + log(sum);
      double* orow = out + ((size_t)r * hq + h) * d;
      for (int e = 0; e < d; ++e) orow[e] = 0.0;
      for (int64_t j = 0; j < nkeys; ++j) {
        const double w = exp(sc[j] - l);
        const float* vr = v + ((size_t)(cu_k[s] + j) * hkv + g) * d;
        for (int e = 0; e < d; ++e) orow[e] += w * (double)vr[e];
      }
      lse[(size_t)r * hq + h] = l;
    }
    free(sc);
  }
  return RLKO_OK;
}

/*
 * Per-block partial states of one (token, head), FP64.
 *
 * Global block b of a sequence holds the keys [b*block, (b+1)*block) counted
 * from the sequence's first key, cut at kv_len and at the causal limit p of
 * the row.  A block with no visible key produces no state.  For each block:
 *
 *   m_b   = max_j s_j
 *   l_b   = sum_j exp(s_j - m_b)
 *   o_b   = sum_j exp(s_j - m_b) v_j / l_b
 *   lse_b = m_b + log l_b
 *
 * o [max_nb, d], lse [max_nb]; *nb receives the number of states (blocks
 * 0 .. nb-1 in ascending global_block_index).
 */
int rlko_row_block_states_f64(int num_seqs, const int32_t* cu_q, const int32_t* cu_k,
                              int hq, int hkv, int d, double scale, int causal,
                              const float* q, const float* k, const float* v,
                              int block, int64_t token, int head,
                              double* o, double* lse, int max_nb, int* nb) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || d <= 0 || block <= 0) return RLKO_EINVAL;
  if (check_seqlens(num_seqs, cu_q, cu_k)) return RLKO_EINVAL;
  if (token < 0 || token >= cu_q[num_seqs] || head < 0 || head >= hq) return RLKO_EINVAL;
  const int s = seq_of_token(num_seqs, cu_q, token);
  const int64_t i = token - cu_q[s];
  const int64_t q_len = cu_q[s + 1] - cu_q[s];
  const int64_t kv_len = cu_k[s + 1] - cu_k[s];
  const int64_t p = kv_len - q_len + i;
  const int64_t nkeys = causal ? p + 1 : kv_len;
  const int g = head / (hq / hkv);
  const float* qr = q + ((size_t)token * hq + head) * d;
  const int64_t count = (nkeys + block - 1) / block;
  if (count > max_nb) return RLKO_EINVAL;
  double* sc = (double*)malloc(sizeof(double) * (size_t)block);
  for (int64_t b = 0; b < count; ++b) {
    const int64_t j0 = b * block;
    const int64_t j1 = (j0 + block < nkeys) ? j0 + block : nkeys;
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
      const float* kr = k + ((size_t)(cu_k[s] + j) * hkv + g) * d;
      double acc = 0.0;
      for (int e = 0; e < d; ++e) acc += (double)qr[e] * (double)kr[e];
      sc[j - j0] = scale * acc;
      if (sc[j - j0] > m) m = sc[j - j0];
    }
    double l = 0.0;
    for (int64_t j = j0; j < j1; ++j) l += exp(sc[j - j0] - m);
    double* ob = o + (size_t)b * d;
    for (int e = 0; e < d; ++e) ob[e] = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
      const double w = exp(sc[j - j0] - m);
      const float* vr = v + ((size_t)(cu_k[s] + j) * hkv + g) * d;
      for (int e = 0; e < d; ++e) ob[e] += w * (double)vr[e];
    }
    for (int e = 0; e < d; ++e) ob[e] /= l;
    lse[b] = m + log(l);
  }
  free(sc);
  *nb = (int)count;
  return RLKO_OK;
}

/*
 * Merge of n partial states of one (row, head), FP32.
 *
 * arrival_order == 0 (canonical): the states are first sorted by
 * global_block_index (a duplicate index is an error), then folded left to
 * right.  arrival_order != 0: folded in the order given (negative control).
 *
 * One fold step, merging running (O, L) with state (o_b, lse_b), is the
 * online-softmax correction written with one rounding per operation:
 *
 *   M     = max(L, lse_b),  mn = min(L, lse_b)
 *   L'    = M + log1p(exp(mn - M))          [= log(exp(L) + exp(lse_b))]
 *   alpha = exp(L - L'),  beta = exp(lse_b - L')
 *   O_d   = fma(o_b,d, beta, O_d * alpha)
 *
 * The first state initialises (O, L).  A state whose lse is -inf is empty and
 * skipped.  o [n, d], lse [n]; out [d], *lse_out.
 */
int rlko_fold_f32(int n, int d, const int32_t* gbi, const float* o, const float* lse,
                  int arrival_order, float* out, float* lse_out) {
  if (n <= 0 || d <= 0) return RLKO_EINVAL;
  int* idx = (int*)malloc(sizeof(int) * (size_t)n);
  for (int a = 0; a < n; ++a) idx[a] = a;
  if (!arrival_order) {
    /* insertion sort by global_block_index */
    for (int a = 1; a < n; ++a) {
      int key = idx[a], b = a - 1;
      while (b >= 0 && gbi[idx[b]] > gbi[key]) { idx[b + 1] = idx[b]; --b; }
      idx[b + 1] = key;
    }
    for (int a = 1; a < n; ++a)
      if (gbi[idx[a]] == gbi[idx[a - 1]]) { free(idx); return RLKO_EDUP; }
  }
  int started = 0;
  float L = -INFINITY;
  for (int a = 0; a < n; ++a) {
    const int st = idx[a];
    const float lb = lse[st];
    const float* ob = o + (size_t)st * d;
    if (isinf(lb) && lb < 0) continue;
    if (!started) {
      for (int e = 0; e < d; ++e) out[e] = ob[e];
      L = lb;
      started = 1;
      continue;
    }
    const float M = fmaxf(L, lb);
    const float mn = fminf(L, lb);
    const float Lp = M + log1pf(expf(mn - M));
    const float alpha = expf(L - Lp);
    const float beta = expf(lb - Lp);
    for (int e = 0; e < d; ++e) out[e] = fmaf(ob[e], beta, out[e] * alpha);
    L = Lp;
  }
  if (!started)
    for (int e = 0; e < d; ++e) out[e] = NAN;
  *lse_out = L;
  free(idx);
  return RLKO_OK;
}

/*
 * Paged-KV decode, FP64: one query token per sequence, at the last position
 * of its context, attends to all ctx keys.  Key t of sequence s lives in page
 * page_table[s * max_pages + t / page_size], slot t % page_size, of pools
 * shaped [n_pages, page_size, hkv, d].  Same formula as rlko_attention_f64.
 */
int rlko_decode_paged_f64(int n, int hq, int hkv, int d, double scale,
                          const float* q, const float* k_pool, const float* v_pool,
                          int n_pages, int page_size, const int32_t* page_table,
                          int max_pages, const int32_t* seqlens,
                          double* out, double* lse) {
  if (n <= 0 || hq <= 0 || hkv <= 0 || hq % hkv || d <= 0 || page_size <= 0) return RLKO_EINVAL;
  int32_t max_ctx = 0;
  for (int s = 0; s < n; ++s) {
    if (seqlens[s] <= 0 || seqlens[s] > (int64_t)max_pages * page_size) return RLKO_EINVAL;
    for (int pg = 0; pg < (seqlens[s] + page_size - 1) / page_size; ++pg) {
      int32_t e = page_table[(size_t)s * max_pages + pg];
      if (e < 0 || e >= n_pages) return RLKO_EINVAL;
    }
    if (seqlens[s] > max_ctx) max_ctx = seqlens[s];
  }
  const int group = hq / hkv;
#pragma omp parallel
  {
    double* sc = (double*)malloc(sizeof(double) * (size_t)max_ctx);
#pragma omp for schedule(dynamic, 1)
    for (int64_t sh = 0; sh < (int64_t)n * hq; ++sh) {
      const int s = (int)(sh / hq), h = (int)(sh % hq), g = h / group;
      const float* qr = q + ((size_t)s * hq + h) * d;
      const int ctx = seqlens[s];
      double m = -INFINITY;
      for (int t = 0; t < ctx; ++t) {
        const int32_t page = page_table[(size_t)s * max_pages + t / page_size];
        const float* kr = k_pool + (((size_t)page * page_size + t % page_size) * hkv + g) * d;
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += (double)qr[e] * (double)kr[e];
        sc[t] = scale * acc;
        if (sc[t] > m) m = sc[t];
      }
      double sum = 0.0;
      for (int t = 0; t < ctx; ++t) sum += exp(sc[t] - m);
      const double l = m + log(sum);
      double* orow = out + ((size_t)s * hq + h) * d;
      for (int e = 0; e < d; ++e) orow[e] = 0.0;
      for (int t = 0; t < ctx; ++t) {
        const int32_t page = page_table[(size_t)s * max_pages + t / page_size];
        const float* vr = v_pool + (((size_t)page * page_size + t % page_size) * hkv + g) * d;
        const double w = exp(sc[t] - l);
        for (int e = 0; e < d; ++e) orow[e] += w * (double)vr[e];
      }
      lse[(size_t)s * hq + h] = l;
    }
    free(sc);
  }
  return RLKO_OK;
}

/*
 * Backward of causal GQA attention, FP64, by definition (q_len == kv_len).
 * With P_ij = exp(s_ij - lse_i), out_i = sum_j P_ij v_j, loss = sum dout.out:
 *
 *   Delta_i = sum_d dout_id out_id
 *   dP_ij   = dout_i . v_j
 *   dS_ij   = P_ij (dP_ij - Delta_i)
 *   dq_i    = scale sum_j dS_ij k_j
 *   dk_j    = scale sum_{h in group} sum_i dS_ij q_i
 *   dv_j    = sum_{h in group} sum_i P_ij dout_i
 *
 * dq [T, hq, d], dk/dv [T, hkv, d], all written for the selected work.
 * only_seq / only_group >= 0 restrict the work to one sequence / one KV head
 * (and its query heads); the other entries are left untouched.
 */
int rlko_backward_f64(int num_seqs, const int32_t* cu, int hq, int hkv, int d,
                      double scale, const float* q, const float* k, const float* v,
                      const float* dout, int only_seq, int only_group,
                      double* dq, double* dk, double* dv) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || d <= 0) return RLKO_EINVAL;
  if (check_seqlens(num_seqs, cu, cu)) return RLKO_EINVAL;
  const int group = hq / hkv;
  int64_t max_len = 0;
  for (int s = 0; s < num_seqs; ++s)
    if (cu[s + 1] - cu[s] > max_len) max_len = cu[s + 1] - cu[s];
  const int64_t nwork = (int64_t)num_seqs * hkv;
#pragma omp parallel
  {
    double* sc = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* ds = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* orow = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < nwork; ++w) {
      const int s = (int)(w / hkv), g = (int)(w % hkv);
      if (only_seq >= 0 && s != only_seq) continue;
      if (only_group >= 0 && g != only_group) continue;
      const int64_t base = cu[s], len = cu[s + 1] - cu[s];
      for (int64_t j = 0; j < len; ++j)
        for (int e = 0; e < d; ++e) {
          dk[((size_t)(base + j) * hkv + g) * d + e] = 0.0;
          dv[((size_t)(base + j) * hkv + g) * d + e] = 0.0;
        }
      for (int h = g * group; h < (g + 1) * group; ++h) {
        for (int64_t i = 0; i < len; ++i) {
          const float* qi = q + ((size_t)(base + i) * hq + h) * d;
          const float* doi = dout + ((size_t)(base + i) * hq + h) * d;
          double m = -INFINITY;
          for (int64_t j = 0; j <= i; ++j) {
            const float* kj = k + ((size_t)(base + j) * hkv + g) * d;
            double acc = 0.0;
            for (int e = 0; e < d; ++e) acc += (double)qi[e] * (double)kj[e];
            sc[j] = scale * acc;
            if (sc[j] > m) m = sc[j];
          }
          double sum = 0.0;
          for (int64_t j = 0; j <= i; ++j) sum += exp(sc[j] - m);
          const double l = m + log(sum);
          for (int e = 0; e < d; ++e) orow[e] = 0.0;
          for (int64_t j = 0; j <= i; ++j) {
            sc[j] = exp(sc[j] - l); /* now P_ij */
            const float* vj = v + ((size_t)(base + j) * hkv + g) * d;
            for (int e = 0; e < d; ++e) orow[e] += sc[j] * (double)vj[e];
          }
          double delta = 0.0;
          for (int e = 0; e < d; ++e) delta += (double)doi[e] * orow[e];
          for (int64_t j = 0; j <= i; ++j) {
            const float* vj = v + ((size_t)(base + j) * hkv + g) * d;
            double dp = 0.0;
            for (int e = 0; e < d; ++e) dp += (double)doi[e] * (double)vj[e];
            ds[j] = sc[j] * (dp - delta);
          }
          double* dqi = dq + ((size_t)(base + i) * hq + h) * d;
          for (int e = 0; e < d; ++e) dqi[e] = 0.0;
          for (int64_t j = 0; j <= i; ++j) {
            const float* kj = k + ((size_t)(base + j) * hkv + g) * d;
            double* dkj = dk + ((size_t)(base + j) * hkv + g) * d;
            double* dvj = dv + ((size_t)(base + j) * hkv + g) * d;
            for (int e = 0; e < d; ++e) {
              dqi[e] += scale * ds[j] * (double)kj[e];
              dkj[e] += scale * ds[j] * (double)qi[e];
              dvj[e] += sc[j] * (double)doi[e];
            }
          }
        }
      }
    }
    free(sc);
    free(ds);
    free(orow);
  }
  return RLKO_OK;
}

/* ---------------------------------------------------------------- RoPE
 * The pages name RoPE only as a step composed before attention, with the
 * attention reading post-RoPE Q/K and decode replay keeping the cache,
 * position and RoPE identical to prefill.  Convention and precision are not
 * on the pages; the reading taken (rotate-half pairs (i, i + D/2), the
 * Qwen/NeoX layout, frequencies theta^(-2i/D)):
 *   angle = p * theta^(-2i/D)                  in double
 *   c = (float)cos(angle), s = (float)sin(angle)   one rounding each
 *   y_i       = bf16_rn(fmaf(x_i, c, -(x_{i+D/2} * s)))      product in float
 *   y_{i+D/2} = bf16_rn(fmaf(x_{i+D/2}, c, x_i * s))
 * x holds BF16 values (exact in float).  Rows are [n_tok][h][d]; pos[t] is
 * the position of row t. */
static double rope_angle(double theta, int d, int i, int32_t p) {
  const double inv = pow(theta, (-2.0 * (double)i) / (double)d);
  return (double)p * inv;
}

/* float -> nearest BF16 (ties to even), returned as the float it denotes. */
static float round_bf16(float v) {
  uint32_t b;
  memcpy(&b, &v, 4);
  if ((b & 0x7F800000u) == 0x7F800000u) return v;  /* inf / nan unchanged */
  b += 0x7FFFu + ((b >> 16) & 1u);
  b &= 0xFFFF0000u;
  float r;
  memcpy(&r, &b, 4);
  return r;
}

int rlko_rope_f32(int64_t n_tok, int h, int d, double theta, const int32_t* pos, const float* x,
                  float* y) {
  if (n_tok < 0 || h < 1 || d < 2 || (d & 1) || !(theta > 1.0) || (n_tok && (!pos || !x || !y)))
    return RLKO_EINVAL;
  const int half = d / 2;
  for (int64_t t = 0; t < n_tok; ++t)
    if (pos[t] < 0) return RLKO_EINVAL;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n_tok; ++t) {
    for (int i = 0; i < half; ++i) {
      const double a = rope_angle(theta, d, i, pos[t]);
      const float c = (float)cos(a), s = (float)sin(a);
      for (int hh = 0; hh < h; ++hh) {
        const float* xr = x + (t * h + hh) * (int64_t)d;
        float* yr = y + (t * h + hh) * (int64_t)d;
        const float x0 = xr[i], x1 = xr[i + half];
        const float p1 = x1 * s, p0 = x0 * s;
        yr[i] = round_bf16(fmaf(x0, c, -p1));
        yr[i + half] = round_bf16(fmaf(x1, c, p0));
      }
    }
  }
  return RLKO_OK;
}

int rlko_rope_f64(int64_t n_tok, int h, int d, double theta, const int32_t* pos, const float* x,
                  double* y) {
  if (n_tok < 0 || h < 1 || d < 2 || (d & 1) || !(theta > 1.0) || (n_tok && (!pos || !x || !y)))
    return RLKO_EINVAL;
  const int half = d / 2;
  for (int64_t t = 0; t < n_tok; ++t)
    if (pos[t] < 0) return RLKO_EINVAL;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n_tok; ++t) {
    for (int i = 0; i < half; ++i) {
      const double a = rope_angle(theta, d, i, pos[t]);
      const double c = cos(a), s = sin(a);
      for (int hh = 0; hh < h; ++hh) {
        const float* xr = x + (t * h + hh) * (int64_t)d;
        double* yr = y + (t * h + hh) * (int64_t)d;
        const double x0 = xr[i], x1 = xr[i + half];
        yr[i] = x0 * c - x1 * s;
        yr[i + half] = x1 * c + x0 * s;
      }
    }
  }
  return RLKO_OK;
}

/* Number of threads the oracle's parallel regions use. */
int rlko_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
