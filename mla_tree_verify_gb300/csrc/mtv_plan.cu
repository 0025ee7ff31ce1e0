// Planner kernel of the MLA tree-verify path.
//
// Planner: one CTA turns kv_indptr / qo_indptr / mask_indptr into the balanced work
// plan that the split kernel walks, without any host round trip (the capture-safety
// requirement of "The Architecture of Capture Safety", section "The Design Emerges":
// fixed grid, sizes derived on the device, no .item()).
//
// Work plan (JobGeo in mtv_common.cuh).  A unit is one key tile of one job; the split
// CTAs form lane groups of `lanes` CTAs, and the lanes of a group walk the same units,
// each on its own column group (draft tokens) of the job, so that the draft tokens of a
// request read each key tile at about the same time and all but the first read hit L2.
// Each job also owns kSegCost empty units (the cost of a segment's start and end, about
// one tile).  Lane group g owns units [g C, (g + 1) C), where C is the larger of
// ceil(U / groups) and ceil(max_tiles / (NSPLIT - 2 lanes)), so that no column group is
// cut into more than NSPLIT = 64 partials ("The Architecture of Capture Safety" fixes
// NSPLIT at 64: section "The Design Emerges", first insight).  Each active lane of each job
// gets a lane-token index (cum_tok[b] + j lanes + r), and its piece in lane group g is
// written to partial slot tok + lanes g (SegMap in mtv_common.cuh).
//
// The merge of the partials runs at the end of the split kernel (merge_token() in
// mtv_common.cuh).
#include "mtv_common.cuh"

namespace mtv {

// Inclusive block scan of one int64 per thread (blockDim.x a multiple of 32, <= 1024).
__device__ int64_t block_inclusive_scan(int64_t v, int64_t* s_warp, int64_t* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    int64_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < nwarps ? s_warp[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nwarps) s_warp[lane] = w;
    if (lane == 31) *s_total = w;
  }
  __syncthreads();
  if (warp > 0) v += s_warp[warp - 1];
  return v;
}

__global__ void __launch_bounds__(256) plan_kernel(Problem p, int32_t grid, int32_t tile) {
  __shared__ int64_t s_warp[32];
  __shared__ int64_t s_total;
  __shared__ int64_t s_maxt[32];
  __shared__ int32_t s_bad[32];      // requests whose mask block is inconsistent
  __shared__ int32_t s_nbad;
  // The split kernel may start its prologue now; it waits for this grid's results.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  if (tid == 0) {
    p.hdr->error_flags = 0u;
    p.hdr->merges_tmem = 0u;
    p.hdr->merges_ws = 0u;
    s_nbad = 0;
  }
  // One request per thread: its six indptr entries are loaded once (one round of
  // loads when bs <= blockDim; after an L2 flush each round is a trip to DRAM).
  struct Req { int64_t kv0, kv1, q0, q1, m0, m1; };
  auto load_req = [&](int64_t b) {
    Req r;
    r.kv0 = p.kv_indptr[b]; r.kv1 = p.kv_indptr[b + 1];
    r.q0 = p.qo_indptr[b]; r.q1 = p.qo_indptr[b + 1];
    r.m0 = p.mask_indptr[b]; r.m1 = p.mask_indptr[b + 1];
    return r;
  };
  const bool one_pass = p.bs <= (int32_t)blockDim.x;
  Req mine{0, 0, 0, 0, 0, 0};
  if (one_pass && tid < p.bs) mine = load_req(tid);
  for (int64_t i = tid; i < (int64_t)p.bs * p.max_q_per_req; i += blockDim.x) p.tok_done[i] = 0;
  __syncthreads();

  // 1. indptr arrays must be in range and nondecreasing, else nothing is computed.
  auto indptr_bad = [&](const Req& r) {
    return r.kv0 < 0 || r.kv1 < r.kv0 || r.kv1 > p.num_kv_indices || r.q0 < 0 || r.q1 < r.q0 ||
           r.q1 > p.total_q || r.q1 - r.q0 > p.max_q_per_req;
  };
  int bad = 0;
  for (int64_t b = tid; b < p.bs; b += blockDim.x) bad |= indptr_bad(one_pass ? mine : load_req(b));
  bad = __syncthreads_or(bad);
  if (bad) {
    for (int64_t b = tid; b <= p.bs; b += blockDim.x) p.cum_units[b] = p.cum_tok[b] = 0;
    if (tid == 0) {
      atomicOr(&p.hdr->error_flags, kErrBadIndptr);
      p.hdr->total_units = 0;
      p.hdr->capacity = 1;
      p.hdr->max_tiles = 0;
      p.hdr->grid = grid;
      p.hdr->tile = tile;
      p.hdr->bs = p.bs;
      p.hdr->lanes = p.lanes;
      p.hdr->groups = grid / p.lanes;
    }
    return;
  }

  // 2. units per request (a request whose mask block is inconsistent gets none), and
  //    their exclusive prefix sum.
  int64_t carry = 0, maxt = 0;
  for (int64_t base = 0; base < p.bs; base += blockDim.x) {
    int64_t b = base + tid;
    int64_t units = 0;
    if (b < p.bs) {
      const Req r = one_pass ? mine : load_req(b);
      int64_t P = r.kv1 - r.kv0;
      int64_t T = r.q1 - r.q0;
      int64_t L = P + T;
      if (r.m0 < 0 || r.m1 - r.m0 != T * L || r.m1 > p.mask_len) {
        if (T > 0) {
          atomicOr(&p.hdr->error_flags, kErrBadMask);
          const int slot = atomicAdd(&s_nbad, 1);
          if (slot < 32) s_bad[slot] = (int32_t)b;
        }
      } else if (T > 0) {
        const JobGeo g = job_geo(L, T, p.group_tokens, p.lanes, tile);
        units = req_units(g);
        maxt = max(maxt, g.tiles);
      }
    }
    int64_t incl = block_inclusive_scan(units, s_warp, &s_total);
    if (b < p.bs) p.cum_units[b] = carry + incl - units;
    carry += s_total;
    __syncthreads();
  }
  for (int o = 16; o > 0; o >>= 1) maxt = max(maxt, __shfl_xor_sync(0xffffffffu, maxt, o));
  if ((tid & 31) == 0) s_maxt[tid >> 5] = maxt;
  __syncthreads();
  // Rows of requests with an inconsistent mask block get out = 0, lse = -inf (no split
  // CTA visits them).
  {
    const int nbad = s_nbad;
    for (int64_t bi = 0; bi < p.bs; ++bi) {
      int64_t b;
      if (nbad <= 32) {
        if (bi >= nbad) break;
        b = s_bad[bi];
      } else {  // more than 32: test every request
        b = bi;
        const int64_t T = p.qo_indptr[b + 1] - p.qo_indptr[b];
        const int64_t L = ((int64_t)p.kv_indptr[b + 1] - p.kv_indptr[b]) + T;
        const int64_t m0 = p.mask_indptr[b], m1 = p.mask_indptr[b + 1];
        if (T == 0 || !(m0 < 0 || m1 - m0 != T * L || m1 > p.mask_len)) continue;
      }
      const int64_t q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
      for (int64_t i = tid; i < (q1 - q0) * p.heads * (kDv / 8); i += blockDim.x)
        ((uint4*)(p.out + q0 * p.heads * kDv))[i] = make_uint4(0, 0, 0, 0);
      for (int64_t i = tid; i < (q1 - q0) * p.heads; i += blockDim.x)
        p.lse[q0 * p.heads + i] = -INFINITY;
    }
  }
  __shared__ int64_t s_cap;
  if (tid == 0) {
    int64_t mt = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mt = max(mt, s_maxt[w]);
    p.cum_units[p.bs] = carry;
    const int64_t groups = grid / p.lanes;
    // Units per lane group: an even share, at most 64 partials per column group, and at
    // least min(max_tiles, 3) + kSegCost, so that a small batch is not spread one tile per
    // CTA (every token would then need a merge that costs more than the tiles it saves).
    int64_t cap = max(ceil_div64(carry, groups), ceil_div64(mt, kNsplit - 2 * p.lanes));
    cap = max(cap, min(mt, (int64_t)3) + kSegCost);
    cap = max(cap, (int64_t)1);
    s_cap = cap;
    p.hdr->total_units = carry;
    p.hdr->capacity = cap;
    p.hdr->max_tiles = mt;
    p.hdr->grid = grid;
    p.hdr->tile = tile;
    p.hdr->bs = p.bs;
    p.hdr->lanes = p.lanes;
    p.hdr->groups = (int32_t)groups;
  }
  __syncthreads();
  // 3. first lane-token index of each request: the exclusive prefix sum of its active
  //    lanes.
  carry = 0;
  for (int64_t base = 0; base < p.bs; base += blockDim.x) {
    const int64_t b = base + tid;
    int64_t pieces = 0;
    if (b < p.bs) {
      const int64_t u0 = p.cum_units[b];
      if (p.cum_units[b + 1] > u0) {   // the request has units: T > 0 and a valid mask block
        const Req r = one_pass ? mine : load_req(b);
        const int64_t T = r.q1 - r.q0;
        const JobGeo g = job_geo((r.kv1 - r.kv0) + T, T, p.group_tokens, p.lanes, tile);
        pieces = req_toks(g, p.lanes);
      }
    }
    const int64_t incl = block_inclusive_scan(pieces, s_warp, &s_total);
    if (b < p.bs) p.cum_tok[b] = carry + incl - pieces;
    carry += s_total;
    __syncthreads();
  }
  if (tid == 0) p.cum_tok[p.bs] = carry;
}

void launch_plan(const Problem& p, int grid, int tile, cudaStream_t stream) {
  plan_kernel<<<1, 256, 0, stream>>>(p, grid, tile);
}

}  // namespace mtv
