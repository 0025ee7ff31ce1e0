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
// Lanes: split CTAs that walk one unit range together, each on a different column group
// (or a different part of one column group's key tiles) of the same request, so that a
// request's draft tokens read the same key tiles at the same time.  The workspace is sized
// for up to kMaxLanes.
constexpr int kMaxLanes = 8;
// A column group cut into more pieces than kMergeGroup merges in two levels: the last of
// each group of kMergeFan consecutive pieces merges the group into one partial, and the
// last group merges those (at most kNsplit / kMergeFan of them) into the output.
constexpr int kMergeFan = 8;

// Device-side error bits, OR-ed into WsHeader::error_flags (never a trap).
constexpr uint32_t kErrBadSlot = 1u;    // a gathered slot is outside [0, num_slots)
constexpr uint32_t kErrBadIndptr = 2u;  // kv/qo indptr out of range or decreasing, T_b > max_q
constexpr uint32_t kErrBadMask = 4u;    // mask_indptr inconsistent with T_b*(P_b+T_b) or mask_len

// One job of the work plan (JobGeo below), as the planner writes it: all that a lane needs
// to walk the job, with no division and no further index load.
struct alignas(16) JobRec {
  int64_t js;        // first unit
  int64_t m_base;    // mask_indptr[b]
  int32_t tok0;      // lane-token index of the job's lane 0 (SegMap)
  int32_t b;         // request
  int32_t kv_base;   // kv_indptr[b]
  int32_t P, T;      // prefix keys, draft tokens of the request
  int32_t q_base;    // qo_indptr[b]
  int32_t cg0;       // the job's first column group within the request
  int32_t tiles;     // key tiles of the request
  int32_t sl;        // tiles per sub-range
  int32_t nt, k;     // column groups, sub-ranges per column group
  int32_t g_lo;      // lane group of unit js
  int32_t n_full;    // pieces of each sub-range but the last
  int32_t ns;        // non-empty sub-ranges
  int32_t nseg;      // pieces of each column group
  int32_t pad;
};
static_assert(sizeof(JobRec) == 80, "job record");

// The workspace starts with this header; the rest is laid out by WsLayout.
struct WsHeader {
  uint32_t error_flags;
  int32_t grid;          // CTAs of the split kernel
  int64_t total_units;   // U = sum_b units_b (see JobGeo)
  int64_t capacity;      // units per lane group
  int64_t max_tiles;     // max_b tiles_b
  int32_t tile;          // key columns per unit
  int32_t bs;
  int32_t lanes;         // CTAs per lane group (1, 2, 4 or 8)
  int32_t groups;        // lane groups: grid / lanes
  uint32_t merges_tmem;  // split tokens merged from TMEM by the CTA of their last piece
  uint32_t merges_ws;    // split tokens merged from the workspace after the last ticket
  int64_t reserved[9];
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
  int64_t* cum_tok;     // [bs+1] first lane-token index of each request (SegMap)
  int64_t* cum_job;     // [bs+1] first job of each request
  JobRec* jobs;         // [max jobs] the plan's jobs, in unit order
  int32_t* grp_job;     // [grid] job of each lane group's first unit
  float* part_lse;      // [num_seg][64]
  float* part_o;        // [num_seg][64][512]
  int32_t* tok_done;    // [bs * max_q_per_req] finished segments (or groups) per query token
  int32_t* grp_done;    // [bs * max_q_per_req][kMergeFan] finished segments per group of
                        // kMergeFan pieces (two-level merges only)
  int64_t num_seg;
  int32_t lanes;        // CTAs per lane group, chosen by the host (the planner records it)
  int32_t merge_mode;   // 0: as timing allows; 1: never from TMEM; 2: from TMEM when it can
  uint64_t wait_ns;     // limit of every bounded wait in the split kernel
  // optional index dump (null unless the debug entry point is used)
  int64_t* dump_slots;  // [sum_b L_b]
  uint8_t* dump_vis;    // [mask_len]
};

struct WsLayout {
  size_t cum_off, tok_off, job_cum_off, job_off, grp_off, cnt_off, gdone_off, lse_off, o_off, total;
  int64_t num_seg;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Partial slots (SegMap): below (lane-token indices) + grid.  A request has ceil(T_b / gt)
// column groups, which jobs of `lanes` column groups cover with at most lanes - 1 lane-token
// indices to spare: at most bs * (ceil(max_q / gt) + kMaxLanes - 1) of them.
__host__ __device__ inline WsLayout ws_layout(int64_t bs, int64_t max_q, int64_t grid,
                                              int64_t gt) {
  WsLayout w;
  w.num_seg = bs * ((max_q + gt - 1) / gt + kMaxLanes - 1) + grid;
  w.cum_off = sizeof(WsHeader);
  w.tok_off = align_up(w.cum_off + sizeof(int64_t) * (size_t)(bs + 1), 256);
  w.job_cum_off = align_up(w.tok_off + sizeof(int64_t) * (size_t)(bs + 1), 256);
  w.job_off = align_up(w.job_cum_off + sizeof(int64_t) * (size_t)(bs + 1), 256);
  // at most ceil(ceil(T_b / gt) / lanes) <= ceil(max_q / gt) jobs per request
  w.grp_off = align_up(w.job_off + sizeof(JobRec) * (size_t)(bs * ((max_q + gt - 1) / gt)), 256);
  w.cnt_off = align_up(w.grp_off + sizeof(int32_t) * (size_t)grid, 256);
  w.gdone_off = align_up(w.cnt_off + sizeof(int32_t) * (size_t)(bs * max_q), 256);
  w.lse_off = align_up(w.gdone_off + sizeof(int32_t) * (size_t)(bs * max_q) * kMergeFan, 256);
  w.o_off = align_up(w.lse_off + sizeof(float) * (size_t)w.num_seg * kHeads, 256);
  w.total = align_up(w.o_off + sizeof(float) * (size_t)w.num_seg * kHeads * kDv, 256);
  return w;
}

// Per-request sizes, straight from the indptr arrays (fourth insight of "The Design
// Emerges": prefix_len_b = kv_indptr[b+1] - kv_indptr[b], derived on the device).
struct ReqInfo {
  int32_t P, T;      // prefix keys, draft tokens
  int32_t kv_base;   // kv_indptr[b] (int32 by the ABI)
  int32_t q_base;    // qo_indptr[b] (below total_q, which the host keeps below 2^31 / 64)
  int64_t L;         // key columns P + T
  int64_t m_base;    // mask_indptr[b]
};

__device__ __forceinline__ ReqInfo req_info(const Problem& p, int64_t b) {
  ReqInfo r;
  r.kv_base = p.kv_indptr[b];
  r.P = p.kv_indptr[b + 1] - r.kv_base;
  r.q_base = (int32_t)p.qo_indptr[b];
  r.T = (int32_t)(p.qo_indptr[b + 1] - p.qo_indptr[b]);
  r.L = (int64_t)r.P + r.T;
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

// a / b for a >= 0, b > 0, in 32 bits when both fit (a 64-bit division is a long
// emulated sequence; the work plan's numbers fit 32 bits at any realistic size).
__host__ __device__ inline int64_t udiv(int64_t a, int64_t b) {
  if ((((uint64_t)a | (uint64_t)b) >> 32) == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
  return a / b;
}

// ---- the work plan ----
// A column group is the set of draft tokens whose heads fill the kernel's 64 columns (one
// token with 64 heads, or gt = 8 tokens with 8 heads).  Request b has ncg = ceil(T_b / gt)
// of them and tiles = ceil(L_b / tile) key tiles.  Its jobs each take `lanes` consecutive
// column groups, one per lane; the last job takes the nt <= lanes that remain, and then
// splits each column group's tiles into k = lanes / nt sub-ranges of sl = ceil(tiles / k)
// tiles, so that lane r works on column group r % nt, sub-range r / nt (lanes r >= nt k
// idle).  A job occupies sl + kSegCost units (sl = tiles for a full job); lane r processes
// its sub-range's tile o at the job's unit o.  Units are numbered request by request and
// job by job; lane group g (CTAs g * lanes .. g * lanes + lanes - 1) owns units
// [g C, (g + 1) C).
struct JobGeo {
  int64_t tiles;    // key tiles of the request
  int64_t hf;       // units of a full job: tiles + kSegCost
  int64_t jobs;     // ceil(ncg / lanes)
  int64_t sl_last;  // tiles per sub-range of the last job
  int32_t nt_last;  // column groups of the last job
  int32_t k_last;   // sub-ranges per column group in the last job
};

__host__ __device__ inline JobGeo job_geo(int64_t L, int64_t T, int64_t gt, int64_t lanes,
                                          int64_t tile) {
  JobGeo g;
  const int64_t ncg = udiv(T + gt - 1, gt);
  g.tiles = udiv(L + tile - 1, tile);
  g.hf = g.tiles + kSegCost;
  g.jobs = udiv(ncg + lanes - 1, lanes);
  g.nt_last = (int32_t)(ncg - (g.jobs - 1) * lanes);
  g.k_last = (int32_t)(lanes / g.nt_last);
  g.sl_last = udiv(g.tiles + g.k_last - 1, g.k_last);
  return g;
}

// Units of a request with T > 0: full jobs, then the last one.
__host__ __device__ inline int64_t req_units(const JobGeo& g) {
  return (g.jobs - 1) * g.hf + g.sl_last + kSegCost;
}

// Column groups nt, sub-ranges k and tiles per sub-range sl of job j.
__host__ __device__ inline void job_shape(const JobGeo& g, int64_t j, int64_t lanes, int32_t& nt,
                                          int32_t& k, int64_t& sl) {
  const bool last = j == g.jobs - 1;
  nt = last ? g.nt_last : (int32_t)lanes;
  k = last ? g.k_last : 1;
  sl = last ? g.sl_last : g.tiles;
}

// Tiles of sub-range s (sl tiles each) of a request with `tiles` tiles.
__host__ __device__ inline int64_t sub_len(int64_t tiles, int64_t s, int64_t sl) {
  const int64_t n = tiles - s * sl;
  return n <= 0 ? 0 : (n < sl ? n : sl);
}

// Active lanes of a request's jobs: W for each full job, nt k for the last.  Each active
// lane of each job gets a lane-token index tok, request after request, job after job:
// cum_tok[b] + j W + r.
__host__ __device__ inline int64_t req_toks(const JobGeo& g, int64_t lanes) {
  return (g.jobs - 1) * lanes + (int64_t)g.nt_last * g.k_last;
}

// Where the partials of one column group live.  Its pieces are its sub-ranges cut by the
// lane groups, taken in order of sub-range, then lane group: sub-range s (of ns non-empty
// ones; all but the last have n_full pieces) is computed by lane r = cgl + s nt, whose
// piece in lane group g sits in slot tok + W g, tok = tok0 + s nt.  Walking its units, a
// lane's (tok, g) pairs only grow, and the toks of one job are W consecutive values, so
// no two pieces share a slot, and every slot is below (lane-token indices) + grid.
struct SegMap {
  int64_t tok0;    // lane-token index of sub-range 0 of the column group
  int64_t g_lo;    // lane group of the job's first unit
  int32_t nt;      // column groups of the job: lane-token stride between sub-ranges
  int32_t W;       // lanes per group
  int32_t n_full;  // pieces of each sub-range but the last
  int32_t ns;      // non-empty sub-ranges
  __host__ __device__ int64_t slot(int32_t i) const {
    int32_t s = n_full > 0 ? i / n_full : 0;
    if (s > ns - 1) s = ns - 1;
    return tok0 + (int64_t)s * nt + (int64_t)W * (g_lo + i - (int64_t)s * n_full);
  }
};

// The slot map of column group cgl of job j (first unit js, shape nt, k, sl) of a
// request with `tiles` tiles whose first lane-token index is tok_b, and its piece count.
__host__ __device__ inline SegMap seg_map(int64_t tok_b, int64_t j, int64_t lanes, int64_t cgl,
                                          int64_t js, int64_t tiles, int32_t nt, int64_t sl,
                                          int64_t C, int32_t& nseg) {
  SegMap m;
  m.tok0 = tok_b + j * lanes + cgl;
  m.g_lo = udiv(js, C);
  m.nt = nt;
  m.W = (int32_t)lanes;
  m.ns = (int32_t)udiv(tiles + sl - 1, sl);
  const int64_t len_last = tiles - (int64_t)(m.ns - 1) * sl;
  m.n_full = (int32_t)(udiv(js + sl - 1, C) - m.g_lo + 1);
  const int32_t n_last = (int32_t)(udiv(js + len_last - 1, C) - m.g_lo + 1);
  nseg = (m.ns - 1) * m.n_full + n_last;
  return m;
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
// M_h + ln(sum) of columns h < ncols to lse_out[h].
__device__ __forceinline__ void merge_stats(const Problem& p, float* lse_out, int ncols,
                                            const int32_t* slots, int64_t nseg, int t,
                                            float* scratch) {
  float* M_s = scratch;
  float* inv_s = scratch + 64;
  // four threads per head, each over segments part, part+4, ...
  const int h = t >> 2, part = t & 3;
  float lv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int64_t sg = part + 4 * i;
    lv[i] = sg < nseg ? __ldcg(p.part_lse + (int64_t)slots[sg] * kHeads + h) : -INFINITY;
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
    if (h < ncols) lse_out[h] = (M == -INFINITY) ? -INFINITY : M + logf(S);
  }
}

// Normalised weights w_s / sum_s w_s of segments [g0, g0 + kMergeGroup) of a row into
// wbuf[s - g0][h] (after merge_stats and a barrier): thread t (of 256) covers head t & 63
// and segments g0 + t/64 + 4k.
__device__ __forceinline__ void merge_weights(const Problem& p, const int32_t* slots, int64_t nseg,
                                              int t, int64_t g0, const float* scratch,
                                              float* wbuf) {
  const int h = t & 63;
#pragma unroll
  for (int k = 0; k < kMergeGroup / 4; ++k) {
    const int j = (t >> 6) + 4 * k;
    float w = 0.f;
    if (g0 + j < nseg) {
      const float l = __ldcg(p.part_lse + (int64_t)slots[g0 + j] * kHeads + h);
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
// h < ncols to out / lse row lrow0 + h; or, with kToPartial (the first level of a
// two-level merge), the normalised fp32 o and the lse of all 64 columns to partial slot
// dst_slot, which may be one of the merged slots (each element is read before it is
// written, by the same thread; the lse goes through `lse_tmp`, 64 floats of shared
// memory, after every read).  A column with no finite partial lse gets out = 0, lse =
// -inf.  Run by `nthreads` = 256 consecutive
// threads starting at `first`, which synchronise on named barrier `bar`; `scratch`
// holds 128 floats of shared memory and `wbuf` kMergeGroup x 64 floats, the weights
// w_s / sum_s w_s of up to kMergeGroup segments per head, computed once per segment and
// head.  Partials are read from L2 (other CTAs wrote them): each thread keeps sixteen
// 16-byte loads (two segments) in flight, and the inner loop is loads and FMAs only.
template <int kThreadsM, bool kToPartial = false>
__device__ __forceinline__ void merge_token(const Problem& p, int64_t lrow0, int ncols,
                                            const int32_t* slots, int64_t nseg, int first,
                                            uint32_t bar,
                                            float* scratch, float* wbuf,
                                            int32_t dst_slot = 0, float* lse_tmp = nullptr) {
  static_assert(kThreadsM == 256, "256 merging threads");
  const int t = (int)threadIdx.x - first;
  if constexpr (kToPartial) merge_stats(p, lse_tmp, kHeads, slots, nseg, t, scratch);
  else merge_stats(p, p.lse + lrow0, ncols, slots, nseg, t, scratch);
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
  auto weights = [&](int64_t g0) { merge_weights(p, slots, nseg, t, g0, scratch, wbuf); };
  const bool one_group = nseg <= kMergeGroup;
  if (one_group) {
    weights(0);
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
  }
  // The token's partials are [nseg][64 heads][128 float4]; float4 i of a segment is
  // head i >> 7.  Four rounds of eight float4 per thread cover the 8192 of a segment.
  uint2* out_tok = (uint2*)(p.out + lrow0 * kDv);
  float4* out_part = (float4*)(p.part_o + (int64_t)dst_slot * kHeads * kDv);
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
        const float4* src0 = (const float4*)(p.part_o + (int64_t)slots[g0 + sg] * kHeads * kDv);
        const float4* src1 =
            two ? (const float4*)(p.part_o + (int64_t)slots[g0 + sg + 1] * kHeads * kDv) : src0;
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
      if constexpr (kToPartial) {
        __stcg(out_part + i, acc[e]);
      } else {
        uint2 pk;
        pk.x = (uint32_t)f32_to_bf16(acc[e].x) | ((uint32_t)f32_to_bf16(acc[e].y) << 16);
        pk.y = (uint32_t)f32_to_bf16(acc[e].z) | ((uint32_t)f32_to_bf16(acc[e].w) << 16);
        if ((i >> 7) < ncols) out_tok[i] = pk;
      }
    }
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kThreadsM) : "memory");
  if constexpr (kToPartial) {   // every read of the merged slots' lse is done
    if (t < kHeads) __stcg(p.part_lse + (int64_t)dst_slot * kHeads + t, lse_tmp[t]);
  }
}

}  // namespace mtv
