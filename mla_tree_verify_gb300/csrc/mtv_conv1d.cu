// Conv-state update of chain speculative verify with a deduplicated intermediate window
// (conv width 4): the kernel behind causal_conv1d_update_dedup() (include/causal_conv1d_dedup.h).
//
// What it computes is stated in that header (the pull request "jianc99/sglang#1",
// sections "Motivation", "Modifications" and "Accuracy Tests"): per request and channel,
// the full row f = [3 state values, T inputs]; out[t] = act(bias + sum_k w[k] f[t + k]);
// the window row f[1 .. T + 2], written once; the state becomes f[T .. T + 2].
//
// Layout on the GPU.  The call is a stream over HBM (about 64 bytes per request and
// channel at T = 8 against 4 multiply-adds per output), so it is written for bandwidth:
// one thread owns 4 consecutive channels of one request, so that its x and out values of a
// token, its weights, its 3-column state block and its 4 window rows are each one
// contiguous, 8-byte aligned span; x, the state, weights and out move with 8- or 16-byte
// accesses, x with streaming loads issued for all T tokens before any arithmetic.  The
// window rows are assembled in registers (T is a template parameter, so the assembly is
// static).  A thread's window rows (4 * (T + 2) values) and state block are one contiguous
// run, and so are a warp's: each warp stages them in shared memory and writes the run with
// consecutive 16-byte stores, so that every 32-byte sector is written whole, once.  When
// the window's columns are channel-contiguous instead (column c of every channel of a slot
// in one run, as in a [T + 2][num_slots][dim] buffer seen transposed), column c of a
// thread's 4 channels is one 8-byte vector, stored directly: for c >= 2 it is input c - 2
// exactly as loaded.  Four
// channels rather than eight keep the registers low enough for 7 blocks of 128 threads an
// SM at T = 8.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "causal_conv1d_dedup.h"

namespace conv1d {
namespace {

constexpr int kCh = 4;   // channels per thread: one 8-byte vector of bf16

__device__ __forceinline__ uint2 ld_stream(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint32_t half16(const uint2& v, int i) {   // element i of 4
  const uint32_t w = i < 2 ? v.x : v.y;
  return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

__device__ __forceinline__ uint32_t to_bf16(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Element e of a thread's 4 channels x kW window columns (channel-major): channel e / kW,
// column e % kW, i.e. f[column + 1] of that channel.
template <int kT>
__device__ __forceinline__ uint32_t window_elem(int e, const uint32_t (&s1)[kCh],
                                                const uint32_t (&s2)[kCh], const uint2 (&xv)[kT]) {
  constexpr int kW = kT + 2;
  const int c = e / kW, j = e % kW;
  return j == 0 ? s1[c] : j == 1 ? s2[c] : half16(xv[j - 2], c);
}

// The arithmetic of one thread's 4 channels: loads, outputs (stored directly), and the
// window rows and (state_len 3) state block staged in the warp's shared buffers.
template <int kT, bool kColMajor>
__device__ __forceinline__ void compute_channels(
    const uint16_t* __restrict__ x, uint16_t* state, const uint16_t* __restrict__ weight,
    const uint16_t* __restrict__ bias, uint16_t* out, uint2* s_win, uint2* s_st, int b, int d,
    int32_t dim, int32_t slot, int32_t state_len, int32_t o, int32_t silu, bool valid,
    uint16_t* window, int64_t ws_slot, int64_t ws_col) {
  constexpr int kW = kT + 2;
  const int lane = threadIdx.x & 31;
  if (!valid) return;
  // the T tokens' inputs of these 4 channels, all in flight at once
  const uint16_t* xr = x + (int64_t)b * kT * dim + d;
  uint2 xv[kT];
#pragma unroll
  for (int t = 0; t < kT; ++t) xv[t] = ld_stream(xr + (int64_t)t * dim);
  // weights [d][4] of 4 channels = 32 contiguous bytes; bias
  uint4 wv[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) wv[i] = __ldg((const uint4*)(weight + (int64_t)d * 4) + i);
  const uint2 bv = bias ? __ldg((const uint2*)(bias + d)) : make_uint2(0u, 0u);
  // state columns o, o+1, o+2 of the 4 channels (bits)
  uint16_t* st = state + ((int64_t)slot * dim + d) * state_len;
  uint32_t s0[kCh], s1[kCh], s2[kCh];
  if (state_len == 3) {   // the block is 12 contiguous values: three 8-byte vectors
    const uint2 a = *(const uint2*)st, m = *((const uint2*)st + 1), z = *((const uint2*)st + 2);
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
      const int e = 3 * c;
      const uint2& v0 = e < 4 ? a : e < 8 ? m : z;
      const uint2& v1 = e + 1 < 4 ? a : e + 1 < 8 ? m : z;
      const uint2& v2 = e + 2 < 4 ? a : e + 2 < 8 ? m : z;
      s0[c] = half16(v0, e & 3);
      s1[c] = half16(v1, (e + 1) & 3);
      s2[c] = half16(v2, (e + 2) & 3);
    }
  } else {
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
      s0[c] = st[c * state_len + o];
      s1[c] = st[c * state_len + o + 1];
      s2[c] = st[c * state_len + o + 2];
    }
  }
  // outputs, token by token (f[t .. t+3] = prev three values and x_t)
  uint16_t* orow = out + (int64_t)b * kT * dim + d;
  float fa[kCh], fb[kCh], fc[kCh];
#pragma unroll
  for (int c = 0; c < kCh; ++c) {
    fa[c] = bf(s0[c]);
    fb[c] = bf(s1[c]);
    fc[c] = bf(s2[c]);
  }
#pragma unroll
  for (int t = 0; t < kT; ++t) {
    uint32_t ob[kCh];
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
      const float xf = bf(half16(xv[t], c));
      const uint4& wc = wv[c >> 1];
      const uint32_t wlo = (c & 1) ? wc.z : wc.x, whi = (c & 1) ? wc.w : wc.y;
      float acc = bf(half16(bv, c));
      acc = fmaf(bf(wlo & 0xFFFFu), fa[c], acc);
      acc = fmaf(bf(wlo >> 16), fb[c], acc);
      acc = fmaf(bf(whi & 0xFFFFu), fc[c], acc);
      acc = fmaf(bf(whi >> 16), xf, acc);
      if (silu) acc = __fdividef(acc, 1.f + __expf(-acc));
      ob[c] = to_bf16(acc);
      fa[c] = fb[c];
      fb[c] = fc[c];
      fc[c] = xf;
    }
    *(uint2*)(orow + (int64_t)t * dim) = make_uint2(ob[0] | (ob[1] << 16), ob[2] | (ob[3] << 16));
  }
  if constexpr (kColMajor) {
    // window columns channel-contiguous: column c of the 4 channels is one 8-byte vector,
    // and columns 2 .. T + 1 are the inputs exactly as loaded
    uint16_t* gw = window + (int64_t)slot * ws_slot + d;
    *(uint2*)gw = make_uint2(s1[0] | (s1[1] << 16), s1[2] | (s1[3] << 16));
    *(uint2*)(gw + ws_col) = make_uint2(s2[0] | (s2[1] << 16), s2[2] | (s2[3] << 16));
#pragma unroll
    for (int t = 0; t < kT; ++t) *(uint2*)(gw + (t + 2) * ws_col) = xv[t];
  } else {
    // the window rows of the 4 channels: 4 * kW values, staged for the warp's store
#pragma unroll
    for (int q = 0; q < kW; ++q) {   // 4 * kW / 4 vectors
      uint32_t e[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) e[i] = window_elem<kT>(4 * q + i, s1, s2, xv);
      s_win[lane * kW + q] = make_uint2(e[0] | (e[1] << 16), e[2] | (e[3] << 16));
    }
  }
  // the state after the last token: f[T], f[T+1], f[T+2] into columns 0..2
  uint32_t n0[kCh], n1[kCh], n2[kCh];
#pragma unroll
  for (int c = 0; c < kCh; ++c) {
    n0[c] = kT >= 3 ? half16(xv[kT >= 3 ? kT - 3 : 0], c) : (kT == 2 ? s2[c] : s1[c]);
    n1[c] = kT >= 2 ? half16(xv[kT >= 2 ? kT - 2 : 0], c) : s2[c];
    n2[c] = half16(xv[kT - 1], c);
  }
  if (state_len == 3) {
    uint32_t e[12];
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
      e[3 * c] = n0[c];
      e[3 * c + 1] = n1[c];
      e[3 * c + 2] = n2[c];
    }
#pragma unroll
    for (int q = 0; q < 3; ++q)
      s_st[lane * 3 + q] =
          make_uint2(e[4 * q] | (e[4 * q + 1] << 16), e[4 * q + 2] | (e[4 * q + 3] << 16));
  } else {
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
      st[c * state_len] = (uint16_t)n0[c];
      st[c * state_len + 1] = (uint16_t)n1[c];
      st[c * state_len + 2] = (uint16_t)n2[c];
    }
  }
}

// Resident blocks of 128 threads an SM that the registers of a kT instantiation allow
// without spills (more blocks keep more of the stream in flight).
constexpr int min_blocks(int t) { return t <= 5 ? 8 : t <= 8 ? 7 : t <= 10 ? 6 : 4; }

template <int kT, bool kColMajor>
__global__ void __launch_bounds__(128, min_blocks(kT))
    conv1d_dedup_kernel(const uint16_t* __restrict__ x, uint16_t* state,
                        const uint16_t* __restrict__ weight, const uint16_t* __restrict__ bias,
                        const int32_t* __restrict__ slots, const int32_t* __restrict__ num_accept,
                        uint16_t* window, uint16_t* out, uint32_t* status, int32_t dim,
                        int32_t state_len, int64_t num_slots, int32_t silu, int64_t ws_slot,
                        int64_t ws_col) {
  constexpr int kW = kT + 2;
  // each warp stages its window rows and state blocks here, then writes them as one
  // contiguous run of 16-byte stores
  __shared__ uint2 s_win[4][32 * kW];
  __shared__ uint2 s_st[4][32 * 3];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int d_warp = (blockIdx.x * blockDim.x + wid * 32) * kCh;
  const int d = d_warp + lane * kCh;
  const int nv = max(0, min(32, (dim - d_warp) / kCh));   // lanes of this warp with channels
  const bool valid = lane < nv;
  const int32_t slot = slots[b];
  if (slot == CONV1D_PAD_SLOT) return;   // (b, and so every test below, is the block's)
  if (slot < 0 || slot >= num_slots) {
    if (d == 0) atomicOr(status, CONV1D_STATUS_BAD_SLOT);
    return;
  }
  const int32_t o = num_accept ? num_accept[b] - 1 : 0;
  if (o < 0 || o > state_len - 3) {
    if (d == 0) atomicOr(status, CONV1D_STATUS_BAD_ACCEPT);
    return;
  }
  if (nv == 0) return;                    // the whole warp is past the last channel
  compute_channels<kT, kColMajor>(x, state, weight, bias, out, s_win[wid], s_st[wid], b, d, dim,
                                  slot, state_len, o, silu, valid, window, ws_slot, ws_col);
  __syncwarp();
  // the warp's window rows: nv * kW 8-byte pieces, contiguous in global memory and
  // 16-byte aligned (d_warp is a multiple of 128 and dim of 8)
  if constexpr (!kColMajor) {
    uint2* gw = (uint2*)(window + ((int64_t)slot * dim + d_warp) * kW);
    const int n8 = nv * kW;
    for (int i = lane; i < n8 / 2; i += 32) ((uint4*)gw)[i] = ((const uint4*)s_win[wid])[i];
    if ((n8 & 1) && lane == 0) gw[n8 - 1] = s_win[wid][n8 - 1];
  }
  if (state_len == 3) {   // the warp's state blocks: nv * 3 pieces, 16-byte aligned
    uint2* gs = (uint2*)(state + ((int64_t)slot * dim + d_warp) * 3);
    const int n8 = nv * 3;
    for (int i = lane; i < n8 / 2; i += 32) ((uint4*)gs)[i] = ((const uint4*)s_st[wid])[i];
    if ((n8 & 1) && lane == 0) gs[n8 - 1] = s_st[wid][n8 - 1];
  }
}

template <int kT>
cudaError_t launch_t(const void* x, void* conv_state, const void* weight, const void* bias,
                     const int32_t* slots, const int32_t* num_accept, void* window, void* out,
                     uint32_t* status, int32_t bs, int32_t dim, int32_t state_len,
                     int64_t num_slots, int32_t silu, int64_t ws_slot, int64_t ws_col,
                     cudaStream_t stream) {
  // 128 threads a block, fewer when a small batch would leave SMs idle
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads_needed = (dim + kCh - 1) / kCh;
  int threads = 128;
  while (threads > 32 && (int64_t)bs * ((threads_needed + threads - 1) / threads) < 2 * sms)
    threads >>= 1;
  dim3 grid((threads_needed + threads - 1) / threads, bs);
  if (ws_col > 0)
    conv1d_dedup_kernel<kT, true><<<grid, threads, 0, stream>>>(
        (const uint16_t*)x, (uint16_t*)conv_state, (const uint16_t*)weight,
        (const uint16_t*)bias, slots, num_accept, (uint16_t*)window, (uint16_t*)out, status, dim,
        state_len, num_slots, silu, ws_slot, ws_col);
  else
    conv1d_dedup_kernel<kT, false><<<grid, threads, 0, stream>>>(
        (const uint16_t*)x, (uint16_t*)conv_state, (const uint16_t*)weight,
        (const uint16_t*)bias, slots, num_accept, (uint16_t*)window, (uint16_t*)out, status, dim,
        state_len, num_slots, silu, 0, 0);
  return cudaGetLastError();
}

}  // namespace
}  // namespace conv1d

namespace conv1d {
// The bf16 kernel for T tokens; ws_col > 0 selects window columns that are channel-
// contiguous (column c of channel d of slot s at s * ws_slot + d + c * ws_col), else the
// rows are contiguous [num_slots][dim][T + 2].  The callers have checked the arguments.
int launch_fast(const void* x, void* conv_state, const void* weight, const void* bias,
                const int32_t* slots, const int32_t* num_accept, void* window, void* out,
                uint32_t* status, int32_t bs, int32_t T, int32_t dim, int32_t state_len,
                int64_t num_slots, int32_t silu, int64_t ws_slot, int64_t ws_col,
                cudaStream_t stream) {
  cudaError_t e = cudaErrorInvalidValue;
#define CONV1D_CASE(n)                                                                           \
  case n:                                                                                        \
    e = launch_t<n>(x, conv_state, weight, bias, slots, num_accept, window, out, status, bs,     \
                    dim, state_len, num_slots, silu, ws_slot, ws_col, stream);                   \
    break;
  switch (T) {
    CONV1D_CASE(1) CONV1D_CASE(2) CONV1D_CASE(3) CONV1D_CASE(4) CONV1D_CASE(5) CONV1D_CASE(6)
    CONV1D_CASE(7) CONV1D_CASE(8) CONV1D_CASE(9) CONV1D_CASE(10) CONV1D_CASE(11)
    CONV1D_CASE(12) CONV1D_CASE(13) CONV1D_CASE(14) CONV1D_CASE(15) CONV1D_CASE(16)
  }
#undef CONV1D_CASE
  return e == cudaSuccess ? 0 : -7;
}
}  // namespace conv1d

extern "C" int causal_conv1d_update_dedup(const void* x, void* conv_state, const void* weight,
                                          const void* bias, const int32_t* slots,
                                          const int32_t* num_accept, void* window, void* out,
                                          uint32_t* status, int32_t bs, int32_t T, int32_t dim,
                                          int32_t state_len, int64_t num_slots, int32_t silu,
                                          cudaStream_t stream) {
  if (!x || !conv_state || !weight || !slots || !window || !out || !status) return -1;
  if (bs < 1 || bs > 65535 || T < 1 || T > CONV1D_MAX_T || dim < 8 || dim % 8 != 0 ||
      state_len < 3 || state_len > CONV1D_MAX_STATE_LEN || num_slots < 1 || num_slots > INT32_MAX)
    return -3;
  auto mis = [](const void* p) { return ((uintptr_t)p & 15u) != 0; };
  if (mis(x) || mis(conv_state) || mis(weight) || (bias && mis(bias)) || mis(window) || mis(out))
    return -4;
  return conv1d::launch_fast(x, conv_state, weight, bias, slots, num_accept, window, out, status,
                             bs, T, dim, state_len, num_slots, silu, 0, 0, stream);
}
