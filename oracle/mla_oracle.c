/*
 * fp64 CPU oracle for MLA tree-verify attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file: it exists so the tests, the smoke check and the CPU baseline of the benchmark
 * can check the CUDA kernels against a plain definition.  It shares no code with them.
 *
 * What it computes (speculative-decoding verify attention over an MLA latent cache):
 *   "The Architecture of Capture Safety: Designing a CUDA Graph-Compatible Verify
 *   Kernel for SGLang", sections "The Design Emerges" (split-K flash decode, second
 *   insight: prefix rows through kv_indices, draft rows through out_cache_loc; third
 *   insight: raw custom_mask + mask_indptr; fourth insight: prefix_len from
 *   kv_indptr) and "Input Knowledge Required" (online softmax m/l/o);
 *   "The Plan Document: A Pivot Point in Custom CUDA Kernel Development", section
 *   "Input Knowledge Required" (one compressed 512-dim latent shared by all heads).
 *
 * For request b with prefix P = kv_indptr[b+1]-kv_indptr[b], drafts
 * T = qo_indptr[b+1]-qo_indptr[b] and L = P + T key columns; draft i, head h:
 *   slot(c) = kv_indices[kv_indptr[b]+c]            for c <  P
 *           = out_cache_loc[qo_indptr[b]+c-P]        for c >= P
 *   vis(c)  = 1                                      for c <  P  (prefix fully visible)
 *           = custom_mask[mask_indptr[b]+i*L+c] != 0 for c >= P
 *   s_c     = sm_scale * sum_{d<576} q[r,h,d] * kv[slot(c), d],  r = qo_indptr[b]+i
 *   m = max_{vis} s_c,  l = sum_{vis} exp(s_c - m)
 *   out[r,h,d] = sum_{vis} exp(s_c - m) * kv[slot(c), d] / l    (d < 512: V = latent)
 *   lse[r,h]   = m + ln(l)
 * A row with no visible key gives out = 0, lse = -inf.
 *
 * The partial / combine pair restates the split-K reduction of the same sections:
 * a key range [c0, c1) yields (m, l, o) by the formulas above restricted to the
 * range (o unnormalised), and partials merge as
 *   M = max_s m_s,  l = sum_s l_s e^{m_s - M},  out = sum_s e^{m_s - M} o_s / l,
 *   lse = M + ln(l).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_QK 576
#define D_V 512

enum {
  ORACLE_OK = 0,
  ORACLE_BAD_ARG = -1,
  ORACLE_BAD_INDEX = -2,
  ORACLE_NO_MEMORY = -3,
};

typedef struct {
  const uint16_t *q;        /* bf16 bits [total_q][H][576] */
  const uint16_t *kv;       /* bf16 bits [num_slots][576] */
  const int32_t *kv_indices;
  const int32_t *kv_indptr; /* [bs+1] */
  const int64_t *out_cache_loc;
  const uint8_t *custom_mask;
  const int64_t *mask_indptr; /* [bs+1] */
  const int64_t *qo_indptr;   /* [bs+1] */
  int64_t bs, num_heads, num_slots;
  double sm_scale;
} oracle_inputs;

static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Slot of key column c of request b, or -1 if it is out of the pool. */
static int64_t key_slot(const oracle_inputs *in, int64_t b, int64_t c) {
  int64_t P = (int64_t)in->kv_indptr[b + 1] - (int64_t)in->kv_indptr[b];
  int64_t slot;
  if (c < P)
    slot = in->kv_indices[(int64_t)in->kv_indptr[b] + c];
  else
    slot = in->out_cache_loc[in->qo_indptr[b] + (c - P)];
  if (slot < 0 || slot >= in->num_slots) return -1;
  return slot;
}

static int key_visible(const oracle_inputs *in, int64_t b, int64_t i, int64_t c) {
  int64_t P = (int64_t)in->kv_indptr[b + 1] - (int64_t)in->kv_indptr[b];
  int64_t T = in->qo_indptr[b + 1] - in->qo_indptr[b];
  if (c < P) return 1;
  return in->custom_mask[in->mask_indptr[b] + i * (P + T) + c] != 0;
}

static double score(const oracle_inputs *in, int64_t r, int64_t h, int64_t slot) {
  const uint16_t *qv = in->q + (r * in->num_heads + h) * D_QK;
  const uint16_t *kv = in->kv + slot * D_QK;
  double acc = 0.0;
  for (int d = 0; d < D_QK; ++d) acc += bf16_value(qv[d]) * bf16_value(kv[d]);
  return in->sm_scale * acc;
}

/* Request that owns query row r (binary search on qo_indptr). */
static int64_t request_of_row(const oracle_inputs *in, int64_t r) {
  int64_t lo = 0, hi = in->bs;
  while (hi - lo > 1) {
    int64_t mid = (lo + hi) / 2;
    if (in->qo_indptr[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

/*
 * Partial over key columns [c0, c1) of (row r, head h): o (unnormalised, 512),
 * m and l.  No visible key in the range gives m = -inf, l = 0, o = 0.
 */
int mla_oracle_partial(const oracle_inputs *in, int64_t r, int64_t h, int64_t c0, int64_t c1,
                       double *o, double *m_out, double *l_out) {
  if (!in || !o || !m_out || !l_out) return ORACLE_BAD_ARG;
  int64_t b = request_of_row(in, r);
  int64_t i = r - in->qo_indptr[b];
  int64_t P = (int64_t)in->kv_indptr[b + 1] - (int64_t)in->kv_indptr[b];
  int64_t L = P + (in->qo_indptr[b + 1] - in->qo_indptr[b]);
  if (c0 < 0) c0 = 0;
  if (c1 > L) c1 = L;
  for (int d = 0; d < D_V; ++d) o[d] = 0.0;
  *m_out = -INFINITY;
  *l_out = 0.0;
  if (c1 <= c0) return ORACLE_OK;
  double *s = (double *)malloc(sizeof(double) * (size_t)(c1 - c0));
  if (!s) return ORACLE_NO_MEMORY;
  /* scores of the visible keys, and their maximum */
  double m = -INFINITY;
  for (int64_t c = c0; c < c1; ++c) {
    s[c - c0] = -INFINITY;
    if (!key_visible(in, b, i, c)) continue;
    int64_t slot = key_slot(in, b, c);
    if (slot < 0) { free(s); return ORACLE_BAD_INDEX; }
    s[c - c0] = score(in, r, h, slot);
    if (s[c - c0] > m) m = s[c - c0];
  }
  double l = 0.0;
  if (m != -INFINITY) {
    for (int64_t c = c0; c < c1; ++c) {
      if (s[c - c0] == -INFINITY) continue;
      double p = exp(s[c - c0] - m);
      const uint16_t *v = in->kv + key_slot(in, b, c) * D_QK;
      l += p;
      for (int d = 0; d < D_V; ++d) o[d] += p * bf16_value(v[d]);
    }
  }
  free(s);
  *m_out = m;
  *l_out = l;
  return ORACLE_OK;
}

/* Merge n partials (m_s, l_s, o_s) into the normalised output and its lse. */
void mla_oracle_combine(int64_t n, const double *m, const double *l, const double *o,
                        double *out, double *lse) {
  double M = -INFINITY;
  for (int64_t s = 0; s < n; ++s)
    if (l[s] > 0.0 && m[s] > M) M = m[s];
  for (int d = 0; d < D_V; ++d) out[d] = 0.0;
  if (M == -INFINITY) { *lse = -INFINITY; return; }
  double sum = 0.0;
  for (int64_t s = 0; s < n; ++s) {
    if (!(l[s] > 0.0)) continue;
    double w = exp(m[s] - M);
    sum += w * l[s];
    for (int d = 0; d < D_V; ++d) out[d] += w * o[s * D_V + d];
  }
  for (int d = 0; d < D_V; ++d) out[d] /= sum;
  *lse = M + log(sum);
}

/*
 * Attention for a list of (row, head) pairs: rows[2k] = query row r, rows[2k+1] =
 * head h; out [n][512], lse [n].  With rows == NULL every (row, head) of the batch
 * is computed, in row-major (r, h) order.  Pairs are independent, so they are
 * spread over `threads` OpenMP threads.
 */
int mla_oracle_attend(const oracle_inputs *in, const int64_t *rows, int64_t n, double *out,
                      double *lse, int threads) {
  if (!in || !out || !lse) return ORACLE_BAD_ARG;
  int64_t total_q = in->qo_indptr[in->bs];
  if (!rows) n = total_q * in->num_heads;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
  for (int64_t k = 0; k < n; ++k) {
    int64_t r = rows ? rows[2 * k] : k / in->num_heads;
    int64_t h = rows ? rows[2 * k + 1] : k % in->num_heads;
    if (r < 0 || r >= total_q || h < 0 || h >= in->num_heads) {
#pragma omp atomic write
      status = ORACLE_BAD_ARG;
      continue;
    }
    double m, l, o[D_V];
    int st = mla_oracle_partial(in, r, h, 0, INT64_MAX, o, &m, &l);
    if (st != ORACLE_OK) {
#pragma omp atomic write
      status = st;
      continue;
    }
    mla_oracle_combine(1, &m, &l, o, out + k * D_V, lse + k);
  }
  return status;
}

/*
 * Index enumeration, for comparing the kernel's gather and mask indexing bit for bit:
 * slots[kv_col_offset(b) + c] = slot(c) of request b (c < L_b; offsets are the
 * running sum of L_b), vis[mask_indptr[b] + i*L_b + c] = vis(c) for draft i.
 */
int mla_oracle_enumerate(const oracle_inputs *in, int64_t *slots, uint8_t *vis) {
  if (!in || !slots || !vis) return ORACLE_BAD_ARG;
  int64_t off = 0;
  for (int64_t b = 0; b < in->bs; ++b) {
    int64_t P = (int64_t)in->kv_indptr[b + 1] - (int64_t)in->kv_indptr[b];
    int64_t T = in->qo_indptr[b + 1] - in->qo_indptr[b];
    for (int64_t c = 0; c < P + T; ++c) {
      int64_t s = key_slot(in, b, c);
      if (s < 0) return ORACLE_BAD_INDEX;
      slots[off + c] = s;
    }
    for (int64_t i = 0; i < T; ++i)
      for (int64_t c = 0; c < P + T; ++c)
        vis[in->mask_indptr[b] + i * (P + T) + c] = (uint8_t)key_visible(in, b, i, c);
    off += P + T;
  }
  return ORACLE_OK;
}

/*
 * KV gather-copy ("The Plan Document: A Pivot Point in Custom CUDA Kernel Development",
 * sections "Context: The Bottleneck That Demanded a Custom Kernel" (K/V defragmentation
 * as the second avenue) and "Output Knowledge Created" (Phase 3: KV defragmentation).
 * Those sections give no algorithm; the plainest reading is taken: the scattered
 * page_size=1 prefix rows of a batch are copied into consecutive rows, in index order,
 * so that later reads of them are contiguous).  For every index entry i in [kv_indptr[0],
 * kv_indptr[bs]), with j = i - kv_indptr[0]:
 *   dst[j] = kv[kv_indices[i]]          (all 576 bf16 values, bit for bit)
 *          = 0                          if kv_indices[i] is outside [0, num_slots)
 *   new_indices[i] = dst_slot0 + j
 * so that request b's rows land, in order, at dst rows [kv_indptr[b] - kv_indptr[0],
 * kv_indptr[b+1] - kv_indptr[0]).  Returns the number of out-of-pool entries, or -1
 * for bad arguments (indptr decreasing or negative, more rows than dst_rows).
 */
int64_t mla_oracle_kv_gather(const uint16_t *kv, int64_t num_slots, const int32_t *kv_indices,
                             const int32_t *kv_indptr, int64_t bs, uint16_t *dst,
                             int64_t dst_rows, int32_t dst_slot0, int32_t *new_indices) {
  if (!kv || !kv_indptr || !dst || !new_indices || bs < 0) return -1;
  const int64_t i0 = kv_indptr[0], i1 = kv_indptr[bs];
  if (i0 < 0 || i1 < i0 || i1 - i0 > dst_rows) return -1;
  for (int64_t b = 0; b < bs; ++b)
    if (kv_indptr[b + 1] < kv_indptr[b]) return -1;
  int64_t bad = 0;
  for (int64_t i = i0; i < i1; ++i) {
    const int64_t j = i - i0;
    const int64_t s = kv_indices[i];
    uint16_t *row = dst + j * D_QK;
    if (s < 0 || s >= num_slots) {
      for (int d = 0; d < D_QK; ++d) row[d] = 0;
      ++bad;
    } else {
      for (int d = 0; d < D_QK; ++d) row[d] = kv[s * D_QK + d];
    }
    new_indices[i] = (int32_t)(dst_slot0 + j);
  }
  return bad;
}

int mla_oracle_abi_version(void) { return 2; }
