// Split-K partial kernel, plain CUDA-core version (fp32 FMA).  It walks the same
// balanced work plan as the tensor-core kernel and writes the same partials; it is
// kept as the simple, obviously-indexed implementation of the split step.
//
// Per segment (one query token, a run of key tiles): the token's 64 heads x 576 query
// dims stay in shared memory; each tile of kTile key columns is gathered row by row
// (prefix slots via kv_indices, draft slots via out_cache_loc), scored against all
// heads, masked inline, folded into the online softmax state (m, l, o) and
// accumulated against the tile's first 512 dims (the MLA latent is both key and
// value).  "The Plan Document", section "Variant 3": one block reads each key row
// once for all of its heads.
#include "mtv_common.cuh"

namespace mtv {
namespace simt {

constexpr int kTile = 32;
constexpr int kThreads = 256;
constexpr int kRowPad = kDqk + 8;  // bf16 elements per shared row (bank spread)
constexpr size_t kSmemQ = (size_t)kHeads * kRowPad * 2;
constexpr size_t kSmemK = (size_t)kTile * kRowPad * 2;
constexpr size_t kSmemP = (size_t)kHeads * (kTile + 1) * 4;
constexpr size_t kSmemBytes = kSmemQ + kSmemK + kSmemP + kTile * 4;

__device__ __forceinline__ float2 bf2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__global__ void __launch_bounds__(kThreads, 1) split_kernel(Problem p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* q_s = (uint16_t*)smem;
  uint16_t* k_s = (uint16_t*)(smem + kSmemQ);
  float* p_s = (float*)(smem + kSmemQ + kSmemK);
  float* vis_s = (float*)(smem + kSmemQ + kSmemK + kSmemP);

  const int tid = threadIdx.x;
  const int h = tid >> 2;   // head owned for scores, softmax state and output
  const int sub = tid & 3;  // key columns sub + 4j; output dims 8i + 2sub + {0,1}
  const int64_t U = p.hdr->total_units, C = p.hdr->capacity;
  const int64_t k = blockIdx.x;
  int64_t u = k * C;
  const int64_t u_end = min(U, u + C);
  const float scale_log2 = p.sm_scale * 1.4426950408889634f;
  const int64_t q_first = p.qo_indptr[0];

  while (u < u_end) {
    const int64_t b = unit_request(p.cum_units, p.bs, u);
    const ReqInfo ri = req_info(p, b);
    const int64_t tiles = ceil_div64(ri.L, kTile);
    const int64_t t = (u - p.cum_units[b]) / tiles;
    const int64_t tile0 = (u - p.cum_units[b]) % tiles;
    const int64_t seg_end = min(u_end, p.cum_units[b] + (t + 1) * tiles);
    const int64_t tile1 = tile0 + (seg_end - u);
    const int64_t r = ri.q_base + t;
    const int64_t seg = (r - q_first) + k;

    // query rows of this token: [64][576] bf16
    __syncthreads();
    for (int i = tid; i < kHeads * (kDqk / 8); i += kThreads) {
      int hh = i / (kDqk / 8), c8 = i % (kDqk / 8);
      uint4 v = *(const uint4*)(p.q + ((r * kHeads + hh) * kDqk) + c8 * 8);
      *(uint4*)(q_s + hh * kRowPad + c8 * 8) = v;
    }

    float m = -INFINITY, l = 0.f;  // base-2 running max and sum for head h
    float o[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) o[i] = 0.f;

    for (int64_t tl = tile0; tl < tile1; ++tl) {
      const int64_t c0 = tl * kTile;
      __syncthreads();  // previous tile fully consumed
      // gather the tile's key rows (zero rows past the end or with a bad slot)
      for (int i = tid; i < kTile * (kDqk / 8); i += kThreads) {
        int row = i / (kDqk / 8), c8 = i % (kDqk / 8);
        int64_t c = c0 + row;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (c < ri.L) {
          int64_t slot = key_slot(p, ri, c);
          if (slot >= 0) {
            v = *(const uint4*)(p.kv + slot * kDqk + c8 * 8);
          } else if (c8 == 0) {
            raise_error(p, kErrBadSlot);
          }
          if (c8 == 0 && p.dump_slots) {
            int64_t col_off = (ri.kv_base - p.kv_indptr[0]) + (ri.q_base - q_first);
            p.dump_slots[col_off + c] = slot;
          }
        }
        *(uint4*)(k_s + row * kRowPad + c8 * 8) = v;
      }
      if (tid < kTile) {
        int64_t c = c0 + tid;
        bool vis = c < ri.L && key_visible(p, ri, t, c);
        vis_s[tid] = vis ? 1.f : 0.f;
        if (c < ri.L && p.dump_vis) p.dump_vis[ri.m_base + t * ri.L + c] = vis ? 1 : 0;
      }
      __syncthreads();

      // scores for head h, key columns sub + 4j
      float s[kTile / 4];
#pragma unroll
      for (int j = 0; j < kTile / 4; ++j) s[j] = 0.f;
      const uint32_t* qrow = (const uint32_t*)(q_s + h * kRowPad);
      for (int d2 = 0; d2 < kDqk / 2; ++d2) {
        float2 qv = bf2(qrow[d2]);
#pragma unroll
        for (int j = 0; j < kTile / 4; ++j) {
          float2 kv = bf2(((const uint32_t*)(k_s + (sub + 4 * j) * kRowPad))[d2]);
          s[j] = fmaf(qv.x, kv.x, s[j]);
          s[j] = fmaf(qv.y, kv.y, s[j]);
        }
      }
      // online softmax (base 2), masked columns contribute nothing
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTile / 4; ++j) {
        s[j] = vis_s[sub + 4 * j] != 0.f ? s[j] * scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, s[j]);
      }
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float m_new = fmaxf(m, tmax);
      const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m - m_new);
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < kTile / 4; ++j) {
        float pj = (s[j] == -INFINITY) ? 0.f : exp2f(s[j] - m_new);
        psum += pj;
        p_s[h * (kTile + 1) + sub + 4 * j] = pj;
      }
      psum += __shfl_xor_sync(0xffffffffu, psum, 1);
      psum += __shfl_xor_sync(0xffffffffu, psum, 2);
      l = l * alpha + psum;
      m = m_new;
      __syncwarp();
      // o = alpha * o + sum_c p[h][c] * v[c][:]
#pragma unroll
      for (int i = 0; i < 128; ++i) o[i] *= alpha;
      for (int c = 0; c < kTile; ++c) {
        float pc = p_s[h * (kTile + 1) + c];
        if (pc == 0.f) continue;
        const uint32_t* vrow = (const uint32_t*)(k_s + c * kRowPad);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float2 v = bf2(vrow[4 * i + sub]);
          o[2 * i] = fmaf(pc, v.x, o[2 * i]);
          o[2 * i + 1] = fmaf(pc, v.y, o[2 * i + 1]);
        }
      }
    }

    // partial: normalised o and natural-log lse (no visible key: o = 0, lse = -inf)
    float* dst = p.part_o + (seg * kHeads + h) * kDv;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i)
      *(float2*)(dst + 8 * i + 2 * sub) = make_float2(o[2 * i] * inv, o[2 * i + 1] * inv);
    if (sub == 0)
      p.part_lse[seg * kHeads + h] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    u = seg_end;
  }
}

}  // namespace simt

int split_tile() { return simt::kTile; }

cudaError_t split_prepare() {
  return cudaFuncSetAttribute(simt::split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)simt::kSmemBytes);
}

void launch_split(const Problem& p, int grid, cudaStream_t stream) {
  simt::split_kernel<<<grid, simt::kThreads, simt::kSmemBytes, stream>>>(p);
}

}  // namespace mtv
