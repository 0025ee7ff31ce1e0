// Shared device-side definitions for the MLA tree-verify kernels: problem constants,
// workspace layout, the balanced work plan, and the per-column index rules.
//
// The method (speculative-decoding verify attention over an MLA latent cache) is the
// one of "The Architecture of Capture Safety: Designing a CUDA Graph-Compatible
// Verify Kernel for SGLang" (section "The Design Emerges") and "The Plan Document: A
// Pivot Point in Custom CUDA Kernel Development" (sections "Variant 3", "Input
// Knowledge Required").
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mtv {

constexpr int kHeads = 64;     // MMA columns of the kernel: 64 heads of one draft token, or
                               // 8 heads of each of 8 consecutive draft tokens (heads = 8)
constexpr int kDqk = 576;      // 512 latent + 64 rope dims
constexpr int kDv = 512;       // V = the latent part of each row
constexpr int kNsplit = 64;    // at most this many partials per query token
// Work units of one query token: its key tiles plus kSegCost empty units that stand for
// the cost of starting and finishing a segment (loading q, the epilogue), about one
// tile's time; with them, the even split of units balances CTAs that walk many short
// tokens against CTAs that walk a few long ones.
constexpr int kSegCost = 1;
constexpr int kRowBytes = kDqk * 2;

// Device-side error bits, OR-ed into WsHeader::error_flags (never a trap).
constexpr uint32_t kErrBadSlot = 1u;    // a gathered slot is outside [0, num_slots)
constexpr uint32_t kErrBadIndptr = 2u;  // kv/qo indptr out of range or decreasing, T_b > max_q
constexpr uint32_t kErrBadMask = 4u;    // mask_indptr inconsistent with T_b*(P_b+T_b) or mask_len

// The workspace starts with this header; the rest is laid out by WsLayout.
struct WsHeader {
  uint32_t error_flags;
  int32_t grid;          // CTAs of the split kernel
  int64_t total_units;   // U = sum_b T_b * tiles_b
  int64_t capacity;      // units per split CTA
  int64_t max_tiles;     // max_b tiles_b
  int32_t tile;          // key columns per unit
  int32_t bs;
  int64_t reserved[11];
};
static_assert(sizeof(WsHeader) == 128, "header size");

struct Problem {
  const uint16_t* q;          // bf16 [total_q][64][576]
  const uint16_t* kv;         // bf16 [num_slots][576]
  const int32_t* kv_indices;  // [num_kv_indices]
  const int32_t* kv_indptr;   // [bs+1]
  const int64_t* out_cache_loc;  // [total_q]
  const uint8_t* custom_mask;    // [mask_len]
  const int64_t* mask_indptr;    // [bs+1]
  const int64_t* qo_indptr;      // [bs+1]
  uint16_t* out;                 // bf16 [total_q][64][512]
  float* lse;                    // [total_q][64]
  float sm_scale;
  int32_t bs;
  int32_t max_q_per_req;
  int32_t heads;          // query heads per token: 64, or 8 (tensor-parallel shard)
  int32_t group_tokens;   // 64 / heads: draft tokens whose heads fill the 64 columns
  int64_t num_slots;
  int64_t total_q;
  int64_t num_kv_indices;
  int64_t mask_len;
  // workspace views
  WsHeader* hdr;
  int64_t* cum_units;   // [bs+1]
  float* part_lse;      // [num_seg][64]
  float* part_o;        // [num_seg][64][512]
  int32_t* tok_done;    // [bs * max_q_per_req] finished segments per query token
  int64_t num_seg;
  // optional index dump (null unless the debug entry point is used)
  int64_t* dump_slots;  // [sum_b L_b]
  uint8_t* dump_vis;    // [mask_len]
};

struct WsLayout {
  size_t cum_off, cnt_off, lse_off, o_off, total;
  int64_t num_seg;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int64_t bs, int64_t max_q, int64_t grid) {
  WsLayout w;
  w.num_seg = bs * max_q + grid;
  w.cum_off = sizeof(WsHeader);
  w.cnt_off = align_up(w.cum_off + sizeof(int64_t) * (size_t)(bs + 1), 256);
  w.lse_off = align_up(w.cnt_off + sizeof(int32_t) * (size_t)(bs * max_q), 256);
  w.o_off = align_up(w.lse_off + sizeof(float) * (size_t)w.num_seg * kHeads, 256);
  w.total = align_up(w.o_off + sizeof(float) * (size_t)w.num_seg * kHeads * kDv, 256);
  return w;
}

// Per-request sizes, straight from the indptr arrays (fourth insight of "The Design
// Emerges": prefix_len_b = kv_indptr[b+1] - kv_indptr[b], derived on the device).
struct ReqInfo {
  int64_t P, T, L;  // prefix keys, draft tokens, key columns
  int64_t kv_base;  // kv_indptr[b]
  int64_t q_base;   // qo_indptr[b]
  int64_t m_base;   // mask_indptr[b]
};

__device__ __forceinline__ ReqInfo req_info(const Problem& p, int64_t b) {
  ReqInfo r;
  r.kv_base = p.kv_indptr[b];
  r.P = (int64_t)p.kv_indptr[b + 1] - r.kv_base;
  r.q_base = p.qo_indptr[b];
  r.T = p.qo_indptr[b + 1] - r.q_base;
  r.L = r.P + r.T;
  r.m_base = p.mask_indptr[b];
  return r;
}

// Slot of key column c (second insight: prefix rows through kv_indices, draft rows
// through out_cache_loc, no concatenated index buffer).  Returns -1 when the slot is
// outside the pool.
__device__ __forceinline__ int64_t key_slot(const Problem& p, const ReqInfo& r, int64_t c) {
  int64_t s = (c < r.P) ? (int64_t)p.kv_indices[r.kv_base + c]
                        : p.out_cache_loc[r.q_base + (c - r.P)];
  return (s >= 0 && s < p.num_slots) ? s : -1;
}

// Visibility of key column c to draft t (third insight: the raw custom_mask read
// inline at mask_indptr[b] + t*L + c).  Prefix columns are always visible.
__device__ __forceinline__ bool key_visible(const Problem& p, const ReqInfo& r, int64_t t,
                                            int64_t c) {
  if (c < r.P) return true;
  return p.custom_mask[r.m_base + t * r.L + c] != 0;
}

__device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Request owning unit u: the largest b with cum_units[b] <= u (cum is nondecreasing).
__device__ __forceinline__ int64_t unit_request(const int64_t* cum, int64_t bs, int64_t u) {
  int64_t lo = 0, hi = bs;
  while (hi - lo > 1) {
    int64_t mid = (lo + hi) >> 1;
    if (cum[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void raise_error(const Problem& p, uint32_t bits) {
  atomicOr(&p.hdr->error_flags, bits);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// fp32 -> bf16, round to nearest even (finite inputs; NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// Where the partials of query row r live: nseg segments starting at seg0 (0 when the
// request got no units).  Segment slots follow the work plan: CTA k writes token
// index tok's partial to slot tok + k.
__device__ __forceinline__ void token_segments(const Problem& p, int64_t b, const ReqInfo& ri,
                                               int64_t t, int64_t tok, int64_t tile,
                                               int64_t capacity, int64_t& seg0, int64_t& nseg) {
  nseg = 0;
  seg0 = 0;
  if (t < 0 || t >= ri.T || p.cum_units[b + 1] <= p.cum_units[b]) return;
  const int64_t tiles = ceil_div64(ri.L, tile);
  const int64_t u0 = p.cum_units[b] + t * (tiles + kSegCost);
  const int64_t k0 = u0 / capacity, k1 = (u0 + tiles - 1) / capacity;
  nseg = k1 - k0 + 1;
  seg0 = tok + k0;
}

constexpr int kMergeGroup = 16;

// One step of the partial merge, shared by every merge path so that the result does not
// depend on which CTA merges or how: acc + (w0 v0 + w1 v1), rounding fixed.  Segments
// are taken in index order in pairs (0, 1), (2, 3), ...; an odd last one pairs with a
// zero weight.
__device__ __forceinline__ float merge_step(float acc, float w0, float v0, float w1, float v1) {
  return __fadd_rn(acc, __fmaf_rn(w1, v1, __fmul_rn(w0, v0)));
}

// Merge statistics of one group of 64 columns over its nseg partial lse values (thread t
// of 256: four threads per column): M_h = max_s lse_s into scratch[h], 1 / sum_s
// e^{lse_s - M_h} into scratch[64 + h] (0 when no partial is finite), and the lse
// M_h + ln(sum) of columns h < ncols to lse row lrow0 + h.
__device__ __forceinline__ void merge_stats(const Problem& p, int64_t lrow0, int ncols,
                                            int64_t seg0, int64_t nseg, int t, float* scratch) {
  float* M_s = scratch;
  float* inv_s = scratch + 64;
  // four threads per head, each over segments part, part+4, ...
  const int h = t >> 2, part = t & 3;
  float lv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int64_t sg = part + 4 * i;
    lv[i] = sg < nseg ? __ldcg(p.part_lse + (seg0 + sg) * kHeads + h) : -INFINITY;
  }
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < 16; ++i) M = fmaxf(M, lv[i]);
  M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
  M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
  float S = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int i = 0; i < 16; ++i) S += (lv[i] == -INFINITY) ? 0.f : expf(lv[i] - M);
  }
  S += __shfl_xor_sync(0xffffffffu, S, 1);
  S += __shfl_xor_sync(0xffffffffu, S, 2);
  if (part == 0) {
    M_s[h] = M;
    inv_s[h] = (M == -INFINITY) ? 0.f : 1.f / S;
    if (h < ncols) p.lse[lrow0 + h] = (M == -INFINITY) ? -INFINITY : M + logf(S);
  }
}

// Normalised weights w_s / sum_s w_s of segments [g0, g0 + kMergeGroup) of a row into
// wbuf[s - g0][h] (after merge_stats and a barrier): thread t (of 256) covers head t & 63
// and segments g0 + t/64 + 4k.
__device__ __forceinline__ void merge_weights(const Problem& p, int64_t seg0, int64_t nseg,
                                              int t, int64_t g0, const float* scratch,
                                              float* wbuf) {
  const int h = t & 63;
#pragma unroll
  for (int k = 0; k < kMergeGroup / 4; ++k) {
    const int j = (t >> 6) + 4 * k;
    float w = 0.f;
    if (g0 + j < nseg) {
      const float l = __ldcg(p.part_lse + (seg0 + g0 + j) * kHeads + h);
      w = (l == -INFINITY) ? 0.f : expf(l - scratch[h]) * scratch[64 + h];
    }
    wbuf[j * kHeads + h] = w;
  }
}

// Merges the nseg (1..64) partials of one group of 64 columns (the 64 heads of a draft
// token, or 8 heads of each of 8 draft tokens), weighted by their log-sum-exp (the
// reduce of the split-K pattern, "Input Knowledge Required":
//   M = max_s lse_s,  w_s = e^{lse_s - M},  out = sum_s w_s o_s / sum_s w_s,
//   lse = M + ln sum_s w_s),
// and writes the bf16 output rows (round to nearest even) and the lse of columns
// h < ncols to out / lse row lrow0 + h.  A column with no finite partial lse gets
// out = 0, lse = -inf.  Run by `nthreads` = 256 consecutive
// threads starting at `first`, which synchronise on named barrier `bar`; `scratch`
// holds 128 floats of shared memory and `wbuf` kMergeGroup x 64 floats, the weights
// w_s / sum_s w_s of up to kMergeGroup segments per head, computed once per segment and
// head.  Partials are read from L2 (other CTAs wrote them): each thread keeps sixteen
// 16-byte loads (two segments) in flight, and the inner loop is loads and FMAs only.
template <int kThreadsM>
__device__ __forceinline__ void merge_token(const Problem& p, int64_t lrow0, int ncols,
                                            int64_t seg0, int64_t nseg, int first, uint32_t bar,
                                            float* scratch, float* wbuf) {
  static_assert(kThreadsM == 256, "256 merging threads");
  const int t = (int)threadIdx.x - first;
  merge_stats(p, lrow0, ncols, seg0, nseg, t, scratch);
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
  auto weights = [&](int64_t g0) { merge_weights(p, seg0, nseg, t, g0, scratch, wbuf); };
  const bool one_group = nseg <= kMergeGroup;
  if (one_group) {
    weights(0);
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
  }
  // The token's partials are [nseg][64 heads][128 float4]; float4 i of a segment is
  // head i >> 7.  Four rounds of eight float4 per thread cover the 8192 of a segment.
  uint2* out_tok = (uint2*)(p.out + lrow0 * kDv);
#pragma unroll 1
  for (int rd = 0; rd < 4; ++rd) {
    float4 acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int64_t g0 = 0; g0 < nseg; g0 += kMergeGroup) {
      if (!one_group) {   // the previous group's weights are no longer read
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
        weights(g0);
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
      }
      const int64_t gn = min((int64_t)kMergeGroup, nseg - g0);
      // two segments per round trip: every load of the pair is issued before any use
#pragma unroll 1
      for (int64_t sg = 0; sg < gn; sg += 2) {
        const bool two = sg + 1 < gn;
        const float4* src0 = (const float4*)(p.part_o + (seg0 + g0 + sg) * kHeads * kDv);
        const float4* src1 = src0 + (two ? kHeads * kDv / 4 : 0);
        const float* w0s = wbuf + sg * kHeads;
        const float* w1s = w0s + (two ? kHeads : 0);
        float4 v0[8], v1[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int i = (rd * 8 + e) * kThreadsM + t;
          v0[e] = __ldcg(src0 + i);
          v1[e] = __ldcg(src1 + i);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int h = ((rd * 8 + e) * kThreadsM + t) >> 7;
          const float w0 = w0s[h];
          const float w1 = two ? w1s[h] : 0.f;
          acc[e].x = merge_step(acc[e].x, w0, v0[e].x, w1, v1[e].x);
          acc[e].y = merge_step(acc[e].y, w0, v0[e].y, w1, v1[e].y);
          acc[e].z = merge_step(acc[e].z, w0, v0[e].z, w1, v1[e].z);
          acc[e].w = merge_step(acc[e].w, w0, v0[e].w, w1, v1[e].w);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = (rd * 8 + e) * kThreadsM + t;
      uint2 pk;
      pk.x = (uint32_t)f32_to_bf16(acc[e].x) | ((uint32_t)f32_to_bf16(acc[e].y) << 16);
      pk.y = (uint32_t)f32_to_bf16(acc[e].z) | ((uint32_t)f32_to_bf16(acc[e].w) << 16);
      if ((i >> 7) < ncols) out_tok[i] = pk;
    }
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
}

}  // namespace mtv
