// Conv-state update of chain speculative verify with a deduplicated intermediate window
// (conv width 4), general form: fp32 or bf16 inputs and state, in any mix, any channel
// count, and strided views of the conv state and of the window rows.  The kernel behind
// causal_conv1d_update_dedup_ex() (include/causal_conv1d_dedup.h).
//
// What it computes is the same as the bf16 path in mtv_conv1d.cu (the pull request
// "jianc99/sglang#1", sections "Motivation", "Modifications" and "Accuracy Tests", which
// lists fp32 and bf16, mixed input and state dtypes, transposed window views and a channel
// count that leaves a partial block): per request and channel the row
// f = [3 state values, T inputs]; out[t] = act(bias + sum_k w[k] f[t + k]), computed in
// fp32 and stored in the input type; the window row f[1 .. T + 2] and the new state
// f[T .. T + 2], stored in the state type.
//
// One thread owns one channel of one request, so x and out move as coalesced rows of the
// block's 128 channels whatever the element type.  The window rows are written through
// their strides; when they are contiguous ([slot][dim][T + 2]) the block's rows form one
// span, which the block stages in shared memory and writes with consecutive stores.  When
// both types are bf16, the conv state contiguous, the channel count a multiple of 8 and
// the window rows contiguous or their columns channel-contiguous (MambaPool's axis-0
// layout seen transposed), the entry point takes the 4-channels-a-thread kernel of
// mtv_conv1d.cu instead.
#include <cstdint>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "causal_conv1d_dedup.h"

namespace conv1d {
// the bf16 kernel of mtv_conv1d.cu (contiguous window rows, or ws_col > 0: channel-
// contiguous window columns)
int launch_fast(const void* x, void* conv_state, const void* weight, const void* bias,
                const int32_t* slots, const int32_t* num_accept, void* window, void* out,
                uint32_t* status, int32_t bs, int32_t T, int32_t dim, int32_t state_len,
                int64_t num_slots, int32_t silu, int64_t ws_slot, int64_t ws_col,
                cudaStream_t stream);
}  // namespace conv1d

namespace conv1d_general {
namespace {

constexpr int kThreads = 128;

// element access by type: bf16 travels as its 16 bits, fp32 as itself
template <typename E> struct Elem;
template <> struct Elem<uint16_t> {
  static __device__ __forceinline__ float load(const uint16_t* p) {
    return __uint_as_float((uint32_t)__ldg(p) << 16);
  }
  static __device__ __forceinline__ float load_rw(const uint16_t* p) {
    return __uint_as_float((uint32_t)*p << 16);
  }
  static __device__ __forceinline__ uint16_t from(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
};
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return __ldg(p); }
  static __device__ __forceinline__ float load_rw(const float* p) { return *p; }
  static __device__ __forceinline__ float from(float f) { return f; }
};

struct Params {
  const void* x;
  void* state;
  const void* weight;
  const void* bias;
  const int32_t* slots;
  const int32_t* num_accept;
  void* window;
  void* out;
  uint32_t* status;
  int32_t T, dim, state_len, silu;
  int64_t num_slots;
  int64_t ss_slot, ss_dim, ss_col;   // conv state strides, elements
  int64_t ws_slot, ws_dim, ws_col;   // window strides, elements
  int32_t staged;                    // window rows contiguous: stage and write as one span
};

// T is a template parameter, so that the token loops, the window row and the new state
// are all static: the kernel issues no more instructions than its T needs
template <typename TX, typename TS, int kT>
__global__ void __launch_bounds__(kThreads) general_kernel(Params p) {
  constexpr int W = kT + 2;
  __shared__ TS s_win[kThreads * W];
  const int b = blockIdx.y;
  const int d0 = blockIdx.x * kThreads;
  const int d = d0 + threadIdx.x;
  const int32_t slot = p.slots[b];
  if (slot == CONV1D_PAD_SLOT) return;   // b, and so each test here, is the block's
  if (slot < 0 || slot >= p.num_slots) {
    if (d == 0) atomicOr(p.status, CONV1D_STATUS_BAD_SLOT);
    return;
  }
  const int32_t o = p.num_accept ? p.num_accept[b] - 1 : 0;
  if (o < 0 || o > p.state_len - 3) {
    if (d == 0) atomicOr(p.status, CONV1D_STATUS_BAD_ACCEPT);
    return;
  }
  const bool valid = d < p.dim;
  float xv[kT];
  float f0 = 0.f, f1 = 0.f, f2 = 0.f;
  TS* st = (TS*)p.state + slot * p.ss_slot + (int64_t)d * p.ss_dim;
  if (valid) {
    // all T inputs in flight first, then the weights, bias and the three state values
    const TX* xr = (const TX*)p.x + (int64_t)b * kT * p.dim + d;
#pragma unroll
    for (int t = 0; t < kT; ++t) xv[t] = Elem<TX>::load(xr + (int64_t)t * p.dim);
    const TX* wr = (const TX*)p.weight + (int64_t)d * 4;
    const float w0 = Elem<TX>::load(wr), w1 = Elem<TX>::load(wr + 1);
    const float w2 = Elem<TX>::load(wr + 2), w3 = Elem<TX>::load(wr + 3);
    const float bias = p.bias ? Elem<TX>::load((const TX*)p.bias + d) : 0.f;
    f0 = Elem<TS>::load_rw(st + o * p.ss_col);
    f1 = Elem<TS>::load_rw(st + (o + 1) * p.ss_col);
    f2 = Elem<TS>::load_rw(st + (o + 2) * p.ss_col);
    // outputs token by token; fa, fb, fc are f[t], f[t + 1], f[t + 2]
    TX* orow = (TX*)p.out + (int64_t)b * kT * p.dim + d;
    float fa = f0, fb = f1, fc = f2;
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      float acc = bias;
      acc = fmaf(w0, fa, acc);
      acc = fmaf(w1, fb, acc);
      acc = fmaf(w2, fc, acc);
      acc = fmaf(w3, xv[t], acc);
      if (p.silu) acc = __fdividef(acc, 1.f + __expf(-acc));
      orow[(int64_t)t * p.dim] = Elem<TX>::from(acc);
      fa = fb;
      fb = fc;
      fc = xv[t];
    }
  }
  // the window row f[1 .. T + 2] in the state type: column 0 is f[1], 1 is f[2], c >= 2 is
  // input c - 2
  if (p.staged) {
    if (valid) {
#pragma unroll
      for (int c = 0; c < W; ++c)
        s_win[threadIdx.x * W + c] =
            Elem<TS>::from(c == 0 ? f1 : c == 1 ? f2 : xv[c >= 2 ? c - 2 : 0]);
    }
    __syncthreads();
    const int nvalid = min(kThreads, p.dim - d0);
    TS* gw = (TS*)p.window + slot * p.ws_slot + (int64_t)d0 * W;
    for (int i = threadIdx.x; i < nvalid * W; i += kThreads) gw[i] = s_win[i];
  } else if (valid) {
    TS* gw = (TS*)p.window + slot * p.ws_slot + (int64_t)d * p.ws_dim;
#pragma unroll
    for (int c = 0; c < W; ++c)
      gw[c * p.ws_col] = Elem<TS>::from(c == 0 ? f1 : c == 1 ? f2 : xv[c >= 2 ? c - 2 : 0]);
  }
  if (!valid) return;
  // the state after the last token: columns 0 .. 2 become f[T], f[T + 1], f[T + 2]
  const float n0 = kT >= 3 ? xv[kT >= 3 ? kT - 3 : 0] : (kT == 2 ? f2 : f1);
  const float n1 = kT >= 2 ? xv[kT >= 2 ? kT - 2 : 0] : f2;
  const float n2 = xv[kT - 1];
  st[0] = Elem<TS>::from(n0);
  st[p.ss_col] = Elem<TS>::from(n1);
  st[2 * p.ss_col] = Elem<TS>::from(n2);
}

template <typename TX, typename TS, int kT>
cudaError_t launch_t(const Params& p, int32_t bs, cudaStream_t stream) {
  dim3 grid((p.dim + kThreads - 1) / kThreads, bs);
  general_kernel<TX, TS, kT><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// the instantiation for p.T (1 .. CONV1D_MAX_T)
template <typename TX, typename TS, int... Ts>
cudaError_t launch_seq(const Params& p, int32_t bs, cudaStream_t stream,
                       std::integer_sequence<int, Ts...>) {
  cudaError_t e = cudaErrorInvalidValue;
  ((p.T == Ts + 1 ? (void)(e = launch_t<TX, TS, Ts + 1>(p, bs, stream)) : (void)0), ...);
  return e;
}

template <typename TX, typename TS>
cudaError_t launch(const Params& p, int32_t bs, cudaStream_t stream) {
  return launch_seq<TX, TS>(p, bs, stream, std::make_integer_sequence<int, CONV1D_MAX_T>{});
}

}  // namespace
}  // namespace conv1d_general

extern "C" int causal_conv1d_update_dedup_ex(
    const void* x, void* conv_state, const void* weight, const void* bias, const int32_t* slots,
    const int32_t* num_accept, void* window, void* out, uint32_t* status, int32_t bs, int32_t T,
    int32_t dim, int32_t state_len, int64_t num_slots, int32_t silu, int32_t input_dtype,
    int32_t state_dtype, const int64_t* state_strides, const int64_t* window_strides,
    cudaStream_t stream) {
  if (!x || !conv_state || !weight || !slots || !window || !out || !status) return -1;
  if (bs < 1 || bs > 65535 || T < 1 || T > CONV1D_MAX_T || dim < 1 || state_len < 3 ||
      state_len > CONV1D_MAX_STATE_LEN || num_slots < 1 || num_slots > INT32_MAX)
    return -3;
  auto known = [](int32_t t) { return t == CONV1D_DTYPE_BF16 || t == CONV1D_DTYPE_F32; };
  if (!known(input_dtype) || !known(state_dtype)) return -3;
  const int64_t ss_def[3] = {(int64_t)dim * state_len, state_len, 1};
  const int64_t ws_def[3] = {(int64_t)dim * (T + 2), T + 2, 1};
  int64_t ss[3], ws[3];
  bool contiguous = true;
  for (int i = 0; i < 3; ++i) {
    ss[i] = state_strides ? state_strides[i] : ss_def[i];
    ws[i] = window_strides ? window_strides[i] : ws_def[i];
    if (ss[i] < 1 || ws[i] < 1) return -3;
    contiguous = contiguous && ss[i] == ss_def[i] && ws[i] == ws_def[i];
  }
  const uintptr_t xa = input_dtype == CONV1D_DTYPE_BF16 ? 2 : 4;
  const uintptr_t sa = state_dtype == CONV1D_DTYPE_BF16 ? 2 : 4;
  auto mis = [](const void* ptr, uintptr_t a) { return ((uintptr_t)ptr & (a - 1)) != 0; };
  if (mis(x, xa) || mis(weight, xa) || (bias && mis(bias, xa)) || mis(out, xa) ||
      mis(conv_state, sa) || mis(window, sa))
    return -4;
  const bool all16 = !mis(x, 16) && !mis(weight, 16) && !(bias && mis(bias, 16)) &&
                     !mis(out, 16) && !mis(conv_state, 16) && !mis(window, 16);
  const bool state_contiguous = ss[0] == ss_def[0] && ss[1] == ss_def[1] && ss[2] == ss_def[2];
  // window columns channel-contiguous (MambaPool's axis-0 layout seen transposed), each
  // 4-channel piece 8-byte aligned
  const bool col_major = ws[1] == 1 && ws[0] % 4 == 0 && ws[2] % 4 == 0 && !mis(window, 8);
  if (input_dtype == CONV1D_DTYPE_BF16 && state_dtype == CONV1D_DTYPE_BF16 && dim % 8 == 0) {
    if (contiguous && all16)
      return causal_conv1d_update_dedup(x, conv_state, weight, bias, slots, num_accept, window,
                                        out, status, bs, T, dim, state_len, num_slots, silu,
                                        stream);
    if (state_contiguous && col_major && !mis(x, 16) && !mis(weight, 16) &&
        !(bias && mis(bias, 16)) && !mis(out, 16) && !mis(conv_state, 16))
      return conv1d::launch_fast(x, conv_state, weight, bias, slots, num_accept, window, out,
                                 status, bs, T, dim, state_len, num_slots, silu, ws[0], ws[2],
                                 stream);
  }
  conv1d_general::Params p{x,  conv_state, weight, bias,      slots, num_accept, window,
                           out, status,    T,      dim,       state_len, silu, num_slots,
                           ss[0], ss[1],   ss[2],  ws[0],     ws[1], ws[2],
                           ws[2] == 1 && ws[1] == T + 2};
  cudaError_t e;
  if (input_dtype == CONV1D_DTYPE_BF16)
    e = state_dtype == CONV1D_DTYPE_BF16
            ? conv1d_general::launch<uint16_t, uint16_t>(p, bs, stream)
            : conv1d_general::launch<uint16_t, float>(p, bs, stream);
  else
    e = state_dtype == CONV1D_DTYPE_BF16 ? conv1d_general::launch<float, uint16_t>(p, bs, stream)
                                         : conv1d_general::launch<float, float>(p, bs, stream);
  return e == cudaSuccess ? 0 : -7;
}
