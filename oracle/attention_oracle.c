/*
 * CPU oracle for batched attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do. It shares no code with the CUDA path.
 *
 * It is the plain definition written out, in fp64, one (token, head) row at a
 * time, with its own paged indexing. The pages it follows are three pull
 * requests of the AMD-Ecosystem FlashInfer fork:
 *   [P1] "Route non-causal windowed prefill to AITER's masked kernel" (#339)
 *   [P2] "Support speculative-decode verify on ROCm, and stop auto routing
 *         short-query prefill to AITER" (#362)
 *   [P3] "Refuse attention inputs the ROCm kernels would compute wrongly" (#399)
 *
 * Definition, per request b, query row i in [0, Lq), query head h:
 *   key j in [0, Lk) sits in page kv_indices[kv_indptr[b] + j / P], slot j % P
 *   s_j   = sm_scale * <q[i,h,:], k[j, h / g, :]>          (g = Hq / Hk)
 *   valid = (!causal || j <= i + Lk - Lq)
 *           && (window_left < 0 || j + Lq + window_left >= Lk + i)
 *   lse   = ln sum_{valid j} exp(s_j)          (natural log; -inf if none)
 *   o     = sum_{valid j} exp(s_j - lse) v[j, h / g, :]   (0 if none)
 * Lk comes from the page metadata, not from the caller:
 *   Lk = (kv_indptr[b+1] - kv_indptr[b] - 1) * P + last_page_len[b].
 * With a custom (tree) mask, valid is further ANDed with bit (i * Lk + j) of
 * request b's bit-packed mask: tree drafts need a topology mask because the
 * causal one lets a draft attend to a sibling on another branch ([P2
 * "Architecture / design notes"]).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * Accumulation type. The parity oracle is the default build: fp64, single
 * thread. The same source is compiled a second time as the timed CPU
 * baseline with -DORC_ACC_FLOAT (fp32 accumulation, expf / logf) and OpenMP
 * over the selected rows; every row is still computed by one thread, in the
 * same order of operations, so the fp64 build's results are those of the
 * plain loops below.
 */
#ifdef ORC_ACC_FLOAT
typedef float orc_acc;
#define ORC_EXP expf
#define ORC_LOG logf
#else
typedef double orc_acc;
#define ORC_EXP exp
#define ORC_LOG log
#endif

/* Threads the row loop may use (the OpenMP build; 1 otherwise). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* 1 in the fp32-accumulate build, 0 in the fp64 parity build. */
int oracle_acc_is_float(void) { return (int)(sizeof(orc_acc) == sizeof(float)); }

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2 };

/* IEEE binary16 bits -> double, decoded field by field. */
static double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int mant = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)mant, -24); /* subnormal: mant * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)mant / 1024.0, expo - 15);
  }
  return sign ? -v : v;
}

/* bfloat16 bits are the top half of an IEEE binary32. */
static double orc_bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double orc_load(const void* base, int dtype, int64_t idx) {
  if (dtype == ORC_F16) return orc_half_to_double(((const uint16_t*)base)[idx]);
  if (dtype == ORC_BF16) return orc_bf16_to_double(((const uint16_t*)base)[idx]);
  return (double)((const float*)base)[idx];
}

/* [P2 "Review notes"]: the kernel derives kv_len from the paged metadata
 * (paged_kv_t::get_length), not from the caller's seq_lens. */
int64_t oracle_kv_len(const int32_t* kv_indptr, const int32_t* last_page_len,
                      int32_t b, int32_t page_size) {
  int64_t n_pages = (int64_t)kv_indptr[b + 1] - (int64_t)kv_indptr[b];
  if (n_pages <= 0) return 0;
  return (n_pages - 1) * (int64_t)page_size + (int64_t)last_page_len[b];
}

/* [P1 "Why window_size_right stays -1"]: the window is a left bound only,
 * anchored bottom-right and applied whether or not the mask is causal.
 * [P2 "Summary"]: the causal mask is bottom-right aligned. All compares are
 * signed 64-bit ([P1 "What changed"]: an unsigned kv_len strips the window). */
int oracle_key_valid(int64_t i, int64_t j, int64_t lq, int64_t lk, int causal,
                     int64_t window_left) {
  if (causal && !(j <= i + lk - lq)) return 0;
  if (window_left >= 0 && !(j + lq + window_left >= lk + i)) return 0;
  return 1;
}

/*
 * Bit (i * lk + j) of request b's custom mask. Request b's segment starts at
 * byte mask_indptr[b]; bit n of the segment is bit (n % 8) of byte n / 8,
 * least significant bit first.
 */
int oracle_custom_bit(const uint8_t* custom_mask, const int64_t* mask_indptr, int32_t b,
                      int64_t i, int64_t j, int64_t lk) {
  const int64_t n = i * lk + j;
  const uint8_t byte = custom_mask[mask_indptr[b] + n / 8];
  return (byte >> (n % 8)) & 1;
}

/*
 * Attention for selected (token, head) rows.
 *
 * q        [T, Hq, d] contiguous, dtype q_dtype
 * k_cache  [num_pages, P, Hk, d] contiguous, dtype kv_dtype (v_cache alike)
 * n_sel    number of rows; sel_token[r] in [0, T), sel_head[r] in [0, Hq)
 * o_out    [n_sel, d] fp64; lse_out [n_sel] fp64 (natural log)
 * custom_mask, mask_indptr: a bit-packed mask per request (see
 *          oracle_custom_bit) ANDed into the mask, or both NULL for none.
 * Returns 0, or -1 on an argument the definition does not cover.
 */
int oracle_attention_rows(const void* q, int q_dtype, const void* k_cache,
                          const void* v_cache, int kv_dtype,
                          const int32_t* kv_indices, const int32_t* qo_indptr,
                          const int32_t* kv_indptr,
                          const int32_t* last_page_len, int32_t batch,
                          int32_t page_size, int32_t num_qo_heads,
                          int32_t num_kv_heads, int32_t head_dim, int causal,
                          int32_t window_left, double sm_scale, int64_t n_sel,
                          const int64_t* sel_token, const int32_t* sel_head,
                          double* o_out, double* lse_out, const uint8_t* custom_mask,
                          const int64_t* mask_indptr) {
  if (num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 || page_size <= 0)
    return -1;
  const int32_t group = num_qo_heads / num_kv_heads;
  const int64_t d = head_dim;
  const int64_t tok_stride_kv = (int64_t)num_kv_heads * d;
  const int64_t page_stride_kv = (int64_t)page_size * tok_stride_kv;
  int64_t max_lk = 0;
  for (int32_t b = 0; b < batch; ++b) {
    int64_t lk = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
    if (lk > max_lk) max_lk = lk;
  }
  int bad = 0;

#pragma omp parallel
  {
  /* per-thread scratch: the scores of one row and its output accumulator */
  orc_acc* s = (orc_acc*)malloc(sizeof(orc_acc) * (size_t)(max_lk > 0 ? max_lk : 1));
  orc_acc* o = (orc_acc*)malloc(sizeof(orc_acc) * (size_t)(d > 0 ? d : 1));
  if (!s || !o) {
#pragma omp atomic write
    bad = 1;
  }

#pragma omp for schedule(dynamic, 4)
  for (int64_t r = 0; r < n_sel; ++r) {
    if (!s || !o) continue;
    const int64_t t = sel_token[r];
    const int32_t h = sel_head[r];
    /* the request that owns token t */
    int32_t b = -1;
    for (int32_t bb = 0; bb < batch; ++bb) {
      if (t >= qo_indptr[bb] && t < qo_indptr[bb + 1]) { b = bb; break; }
    }
    if (b < 0 || h < 0 || h >= num_qo_heads) {
#pragma omp atomic write
      bad = 1;
      continue;
    }
    const int64_t lq = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
    const int64_t lk = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
    const int64_t i = t - qo_indptr[b];
    const int32_t hk = h / group;
    const int64_t q_off = (t * num_qo_heads + h) * d;

    orc_acc m = -INFINITY;
    for (int64_t j = 0; j < lk; ++j) {
      s[j] = -INFINITY;
      if (!oracle_key_valid(i, j, lq, lk, causal, window_left)) continue;
      if (custom_mask && !oracle_custom_bit(custom_mask, mask_indptr, b, i, j, lk)) continue;
      const int64_t page = kv_indices[kv_indptr[b] + j / page_size];
      const int64_t k_off = page * page_stride_kv + (j % page_size) * tok_stride_kv + hk * d;
      orc_acc dot = 0;
      for (int64_t c = 0; c < d; ++c)
        dot += (orc_acc)orc_load(q, q_dtype, q_off + c) *
               (orc_acc)orc_load(k_cache, kv_dtype, k_off + c);
      s[j] = (orc_acc)sm_scale * dot;
      if (s[j] > m) m = s[j];
    }
    for (int64_t c = 0; c < d; ++c) o[c] = 0;
    double* o_row = o_out + r * d;
    if (m == -INFINITY) {
      for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
      lse_out[r] = -INFINITY;
      continue;
    }
    orc_acc sum = 0;
    for (int64_t j = 0; j < lk; ++j)
      if (s[j] != -INFINITY) sum += ORC_EXP(s[j] - m);
    const orc_acc lse = m + ORC_LOG(sum);
    lse_out[r] = (double)lse;
    for (int64_t j = 0; j < lk; ++j) {
      if (s[j] == -INFINITY) continue;
      const orc_acc w = ORC_EXP(s[j] - lse);
      const int64_t page = kv_indices[kv_indptr[b] + j / page_size];
      const int64_t v_off = page * page_stride_kv + (j % page_size) * tok_stride_kv + hk * d;
      for (int64_t c = 0; c < d; ++c) o[c] += w * (orc_acc)orc_load(v_cache, kv_dtype, v_off + c);
    }
    for (int64_t c = 0; c < d; ++c) o_row[c] = (double)o[c];
  }
  free(s);
  free(o);
  }
  return bad ? -1 : 0;
}

/*
 * Merge of attention states by their log-sum-exp ([P3 "What changed",
 * "Graph-mode partial_state merge"]; [P2 "What changed"], split-KV):
 *   s = m + ln sum_i exp(s_i - m),  o = sum_i exp(s_i - s) o_i,  m = max_i s_i.
 * All states at -inf give s = -inf and o = 0.
 *
 * v [n_rows, n_states, d] fp64, s [n_rows, n_states] fp64
 * -> v_out [n_rows, d], s_out [n_rows].
 */
void oracle_merge_states(const double* v, const double* s, int64_t n_rows,
                         int64_t n_states, int64_t d, double* v_out,
                         double* s_out) {
  for (int64_t r = 0; r < n_rows; ++r) {
    const double* vr = v + r * n_states * d;
    const double* sr = s + r * n_states;
    double* o = v_out + r * d;
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    double m = -INFINITY;
    for (int64_t k = 0; k < n_states; ++k)
      if (sr[k] > m) m = sr[k];
    if (m == -INFINITY) { s_out[r] = -INFINITY; continue; }
    double sum = 0.0;
    for (int64_t k = 0; k < n_states; ++k) sum += exp(sr[k] - m);
    const double lse = m + log(sum);
    s_out[r] = lse;
    for (int64_t k = 0; k < n_states; ++k) {
      const double w = exp(sr[k] - lse);
      for (int64_t c = 0; c < d; ++c) o[c] += w * vr[k * d + c];
    }
  }
}
