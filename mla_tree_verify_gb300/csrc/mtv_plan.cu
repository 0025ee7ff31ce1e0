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

// Inclusive block scans of three int64 per thread at once (blockDim.x a multiple of 32,
// <= 1024): v[i] becomes the sum of v[i] over threads 0..tid, total[i] the block's sum.
__device__ void block_inclusive_scan3(int64_t (&v)[3], int64_t (*s_warp)[32], int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
#pragma unroll
  for (int i = 0; i < 3; ++i)
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, v[i], o);
      if (lane >= o) v[i] += y;
    }
  if (lane == 31)
    for (int i = 0; i < 3; ++i) s_warp[i][warp] = v[i];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      int64_t w = lane < nwarps ? s_warp[i][lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nwarps) s_warp[i][lane] = w;
      if (lane == 31) total[i] = w;
    }
  }
  __syncthreads();
  if (warp > 0)
    for (int i = 0; i < 3; ++i) v[i] += s_warp[i][warp - 1];
}

__global__ void __launch_bounds__(256) plan_kernel(Problem p, int32_t grid, int32_t tile) {
  __shared__ int64_t s_warp[3][32];
  __shared__ int64_t s_total[3];
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
  for (int64_t i = tid; i < (int64_t)p.bs * p.max_q_per_req * kMergeFan; i += blockDim.x)
    p.grp_done[i] = 0;
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
    for (int64_t b = tid; b <= p.bs; b += blockDim.x) p.cum_units[b] = p.cum_tok[b] = p.cum_job[b] = 0;
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

  // 2. units, active lanes and jobs per request (a request whose mask block is
  //    inconsistent gets none), and their exclusive prefix sums; with one pass, each
  //    thread keeps its request's sums for step 3.
  int64_t carry[3] = {0, 0, 0}, maxt = 0, mine_cum[3] = {0, 0, 0};
  JobGeo mine_geo{};
  for (int64_t base = 0; base < p.bs; base += blockDim.x) {
    int64_t b = base + tid;
    int64_t v[3] = {0, 0, 0};   // units, lane tokens, jobs
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
        v[0] = req_units(g);
        v[1] = req_toks(g, p.lanes);
        v[2] = g.jobs;
        maxt = max(maxt, g.tiles);
        if (one_pass) mine_geo = g;
      }
    }
    const int64_t own[3] = {v[0], v[1], v[2]};
    block_inclusive_scan3(v, s_warp, s_total);
    if (b < p.bs) {
      p.cum_units[b] = carry[0] + v[0] - own[0];
      p.cum_tok[b] = carry[1] + v[1] - own[1];
      p.cum_job[b] = carry[2] + v[2] - own[2];
      if (one_pass)
        for (int i = 0; i < 3; ++i) mine_cum[i] = carry[i] + v[i] - own[i];
    }
    for (int i = 0; i < 3; ++i) carry[i] += s_total[i];
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
    p.cum_units[p.bs] = carry[0];
    p.cum_tok[p.bs] = carry[1];
    p.cum_job[p.bs] = carry[2];
    const int64_t groups = grid / p.lanes;
    // Units per lane group: an even share, at most 64 partials per column group, and at
    // least min(max_tiles, 3) + kSegCost, so that a small batch is not spread one tile per
    // CTA (every token would then need a merge that costs more than the tiles it saves).
    int64_t cap = max(ceil_div64(carry[0], groups), ceil_div64(mt, kNsplit - 2 * p.lanes));
    cap = max(cap, min(mt, (int64_t)3) + kSegCost);
    cap = max(cap, (int64_t)1);
    s_cap = cap;
    p.hdr->total_units = carry[0];
    p.hdr->capacity = cap;
    p.hdr->max_tiles = mt;
    p.hdr->grid = grid;
    p.hdr->tile = tile;
    p.hdr->bs = p.bs;
    p.hdr->lanes = p.lanes;
    p.hdr->groups = (int32_t)groups;
  }
  __syncthreads();
  // 3. each request's job records (the divisions by C happen here, so that the split
  //    kernel's walk has none), and the first job of each lane group whose first unit
  //    falls in the request.
  const int64_t cap = s_cap, groups = grid / p.lanes;
  for (int64_t b = tid; b < p.bs; b += blockDim.x) {
    const int64_t cu = one_pass ? mine_cum[0] : p.cum_units[b];
    const Req r = one_pass ? mine : load_req(b);
    const int64_t T = r.q1 - r.q0, L = (r.kv1 - r.kv0) + T;
    const bool ok = T > 0 && !(r.m0 < 0 || r.m1 - r.m0 != T * L || r.m1 > p.mask_len);
    if (!ok) continue;
    const int64_t ct = one_pass ? mine_cum[1] : p.cum_tok[b];
    const int64_t cj = one_pass ? mine_cum[2] : p.cum_job[b];
    const JobGeo g = one_pass ? mine_geo : job_geo(L, T, p.group_tokens, p.lanes, tile);
    for (int64_t j = 0; j < g.jobs; ++j) {
      int32_t nt, k;
      int64_t sl;
      job_shape(g, j, p.lanes, nt, k, sl);
      JobRec rec;
      rec.js = cu + j * g.hf;
      rec.m_base = r.m0;
      rec.tok0 = (int32_t)(ct + j * p.lanes);
      rec.b = (int32_t)b;
      rec.kv_base = (int32_t)r.kv0;
      rec.P = (int32_t)(r.kv1 - r.kv0);
      rec.T = (int32_t)T;
      rec.q_base = (int32_t)r.q0;
      rec.cg0 = (int32_t)(j * p.lanes);
      rec.tiles = (int32_t)g.tiles;
      rec.sl = (int32_t)sl;
      rec.nt = nt;
      rec.k = k;
      int32_t nseg;
      const SegMap m = seg_map(0, 0, p.lanes, 0, rec.js, g.tiles, nt, sl, cap, nseg);
      rec.g_lo = (int32_t)m.g_lo;
      rec.n_full = m.n_full;
      rec.ns = m.ns;
      rec.nseg = nseg;
      rec.pad = 0;
      p.jobs[cj + j] = rec;
    }
    // lane groups whose first unit u = g C lies in [cu, cu + units)
    const int64_t units = req_units(g);
    for (int64_t gi = udiv(cu + cap - 1, cap); gi * cap < cu + units && gi < groups; ++gi)
      p.grp_job[gi] = (int32_t)(cj + min(udiv(gi * cap - cu, g.hf), g.jobs - 1));
  }
  // lane groups that start past the last unit have no work
  for (int64_t gi = udiv(carry[0] + cap - 1, cap) + tid; gi < groups; gi += blockDim.x)
    p.grp_job[gi] = 0;
}

void launch_plan(const Problem& p, int grid, int tile, cudaStream_t stream) {
  plan_kernel<<<1, 256, 0, stream>>>(p, grid, tile);
}

}  // namespace mtv
