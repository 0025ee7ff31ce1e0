// Planner and split-combine kernels of the MLA tree-verify path.
//
// Planner: one CTA turns kv_indptr / qo_indptr / mask_indptr into the balanced work
// plan that the split kernel walks, without any host round trip (the capture-safety
// requirement of "The Architecture of Capture Safety", section "The Design Emerges":
// fixed grid, sizes derived on the device, no .item()).
//
// Work plan.  A unit is one query token x one tile of `tile` key columns; request b
// has T_b * ceil(L_b / tile) units, numbered request by request, token by token, tile
// by tile.  Split CTA k owns units [k*C, (k+1)*C).  C is the larger of ceil(U / grid)
// and ceil(max_tiles / (NSPLIT-1)), so no query token is cut into more than NSPLIT=64
// partials (the pages fix NSPLIT at 64, first insight of "The Design Emerges").  The
// partial that CTA k writes for token index tok (row minus qo_indptr[0]) lives in
// segment slot tok + k: walking the units in order moves either tok or k forward by at
// least one, so these slots never collide and stay below total_q_max + grid.
//
// Combine: merges the partials of one query token, per head, weighted by their
// log-sum-exp (the reduce of the split-K flash-decode pattern, "Input Knowledge
// Required": the m/l/o online-softmax state):
//   M = max_s lse_s,  w_s = e^{lse_s - M},  out = sum_s w_s o_s / sum_s w_s,
//   lse = M + ln sum_s w_s.
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

__global__ void __launch_bounds__(1024) plan_kernel(Problem p, int32_t grid, int32_t tile) {
  __shared__ int64_t s_warp[32];
  __shared__ int64_t s_total;
  __shared__ int64_t s_maxt[32];
  const int tid = threadIdx.x;
  if (tid == 0) p.hdr->error_flags = 0u;
  __syncthreads();

  // 1. indptr arrays must be in range and nondecreasing, else nothing is computed.
  int bad = 0;
  for (int64_t b = tid; b < p.bs; b += blockDim.x) {
    int64_t kv0 = p.kv_indptr[b], kv1 = p.kv_indptr[b + 1];
    int64_t q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
    if (kv0 < 0 || kv1 < kv0 || kv1 > p.num_kv_indices || q0 < 0 || q1 < q0 ||
        q1 > p.total_q || q1 - q0 > p.max_q_per_req)
      bad = 1;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    for (int64_t b = tid; b <= p.bs; b += blockDim.x) p.cum_units[b] = 0;
    if (tid == 0) {
      atomicOr(&p.hdr->error_flags, kErrBadIndptr);
      p.hdr->total_units = 0;
      p.hdr->capacity = 1;
      p.hdr->max_tiles = 0;
      p.hdr->grid = grid;
      p.hdr->tile = tile;
      p.hdr->bs = p.bs;
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
      int64_t P = (int64_t)p.kv_indptr[b + 1] - p.kv_indptr[b];
      int64_t T = p.qo_indptr[b + 1] - p.qo_indptr[b];
      int64_t L = P + T;
      int64_t m0 = p.mask_indptr[b], m1 = p.mask_indptr[b + 1];
      if (m0 < 0 || m1 - m0 != T * L || m1 > p.mask_len) {
        if (T > 0) atomicOr(&p.hdr->error_flags, kErrBadMask);
      } else if (T > 0) {
        int64_t tiles = ceil_div64(L, tile);
        units = T * tiles;
        maxt = max(maxt, tiles);
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
  if (tid == 0) {
    int64_t mt = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mt = max(mt, s_maxt[w]);
    p.cum_units[p.bs] = carry;
    int64_t cap = max(ceil_div64(carry, grid), ceil_div64(mt, kNsplit - 1));
    p.hdr->total_units = carry;
    p.hdr->capacity = max(cap, (int64_t)1);
    p.hdr->max_tiles = mt;
    p.hdr->grid = grid;
    p.hdr->tile = tile;
    p.hdr->bs = p.bs;
  }
}

// One warp per (query token, head): 8 warps per CTA cover 8 heads of one token; the
// grid covers bs * max_q_per_req tokens (token i is row qo_indptr[0] + i).  Rows
// outside [qo_indptr[0], qo_indptr[bs]) are not written; when the planner rejected
// the indptr arrays nothing is written.
__global__ void __launch_bounds__(256) combine_kernel(Problem p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const WsHeader& hdr = *p.hdr;
  if (hdr.error_flags & kErrBadIndptr) return;
  const int64_t tok = blockIdx.x >> 3;
  const int h = (blockIdx.x & 7) * 8 + warp;
  const int64_t r = p.qo_indptr[0] + tok;
  if (r >= p.qo_indptr[p.bs]) return;

  int64_t nseg = 0, seg0 = 0;
  {
    const int64_t b = row_request(p.qo_indptr, p.bs, r);
    const ReqInfo ri = req_info(p, b);
    const int64_t t = r - ri.q_base;
    if (t >= 0 && t < ri.T && p.cum_units[b + 1] > p.cum_units[b]) {
      const int64_t tiles = ceil_div64(ri.L, hdr.tile);
      const int64_t u0 = p.cum_units[b] + t * tiles;
      const int64_t k0 = u0 / hdr.capacity, k1 = (u0 + tiles - 1) / hdr.capacity;
      nseg = k1 - k0 + 1;
      seg0 = tok + k0;
    }
  }
  uint16_t* orow = p.out + (r * kHeads + h) * kDv;
  // per-lane partial LSEs (nseg <= 64)
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < nseg) l0 = p.part_lse[(seg0 + lane) * kHeads + h];
  if (lane + 32 < nseg) l1 = p.part_lse[(seg0 + lane + 32) * kHeads + h];
  float M = fmaxf(l0, l1);
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (nseg <= 0 || M == -INFINITY) {
    for (int d = lane * 8; d < kDv; d += 256) *(uint4*)(orow + d) = make_uint4(0, 0, 0, 0);
    if (lane == 0) p.lse[r * kHeads + h] = -INFINITY;
    return;
  }
  const float w0 = (l0 == -INFINITY) ? 0.f : expf(l0 - M);
  const float w1 = (l1 == -INFINITY) ? 0.f : expf(l1 - M);
  float S = w0 + w1;
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sg = 0; sg < nseg; ++sg) {
    const float w = __shfl_sync(0xffffffffu, sg < 32 ? w0 : w1, sg & 31);
    if (w == 0.f) continue;
    const float4* src = (const float4*)(p.part_o + ((seg0 + sg) * kHeads + h) * kDv);
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = src[lane + 32 * i];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i].x += w * v[i].x; acc[i].y += w * v[i].y; acc[i].z += w * v[i].z; acc[i].w += w * v[i].w;
    }
  }
  const float inv = 1.f / S;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int d = 4 * (lane + 32 * i);
    uint2 pk;
    pk.x = (uint32_t)f32_to_bf16(acc[i].x * inv) | ((uint32_t)f32_to_bf16(acc[i].y * inv) << 16);
    pk.y = (uint32_t)f32_to_bf16(acc[i].z * inv) | ((uint32_t)f32_to_bf16(acc[i].w * inv) << 16);
    *(uint2*)(orow + d) = pk;
  }
  if (lane == 0) p.lse[r * kHeads + h] = M + logf(S);
}

void launch_plan(const Problem& p, int grid, int tile, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(p, grid, tile);
}

void launch_combine(const Problem& p, cudaStream_t stream) {
  int64_t rows = (int64_t)p.bs * p.max_q_per_req;
  if (rows <= 0) return;
  combine_kernel<<<(unsigned)(rows * 8), 256, 0, stream>>>(p);
}

}  // namespace mtv
