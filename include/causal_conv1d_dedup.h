/*
 * Conv-state update of chain speculative verify with a deduplicated intermediate window
 * (conv width K = 4), as a C ABI.
 *
 * What it computes: the pull request "jianc99/sglang#1" (deduplicated conv window).
 *   - Section "Motivation": a chain verify calls causal_conv1d_update with an intermediate
 *     conv window, from which the conv state of the accepted prefix is restored; the
 *     deduplicated layout keeps one [dim][T + K - 2] row per state slot, read as
 *     overlapping [T][dim][K - 1] windows whose step stride equals the window stride.
 *   - Section "Modifications": step t's window is columns t .. t + 2 of the row
 *     [state[1], state[2], x_0, ..., x_{T-1}]; the row is written once, not three values
 *     per step; padded rows store nothing; the path is for conv width 4.
 *   - Section "Accuracy Tests": a num_accept_tokens offset into the state.
 * For request b with slot s = slots[b] and o = num_accept[b] - 1 (0 without accept
 * counts), per channel d, with f = [S[s][d][o], S[s][d][o+1], S[s][d][o+2],
 * x[b][0][d], ..., x[b][T-1][d]] (S the conv state):
 *   out[b][t][d]     = act(bias[d] + sum_{k<4} w[d][k] * f[t + k])    (fp32, stored bf16 RNE)
 *   window[s][d][c]  = f[c + 1], c < T + 2                            (bit copies)
 *   S[s][d][i]       = f[T + i], i < 3                                (state after the call)
 * act is SiLU (v / (1 + e^-v)) when `silu` is nonzero, else the identity.
 *
 * Layouts (bf16 = 16-bit bfloat16, all row-major and contiguous, device pointers):
 *   x          bf16 [bs][T][dim]            the draft tokens' conv inputs
 *   conv_state bf16 [num_slots][dim][state_len], read and updated in place
 *   weight     bf16 [dim][4]
 *   bias       bf16 [dim], or NULL
 *   slots      int32 [bs]: distinct slots in [0, num_slots), or CONV1D_PAD_SLOT
 *   num_accept int32 [bs] in [1, state_len - 2], or NULL
 *   window     bf16 [num_slots][dim][T + 2]  the deduplicated window rows
 *   out        bf16 [bs][T][dim]
 *   status     uint32, device, zeroed by the caller; bits CONV1D_STATUS_* are OR-ed in
 * Constraints: 1 <= T <= 16, 3 <= state_len <= 32, dim a positive multiple of 8,
 * every pointer 16-byte aligned.  The caller owns every buffer; the call allocates
 * nothing, never synchronises and is capturable in a CUDA graph (sizes are fixed by the
 * arguments; slots and accept counts are read on the device).
 *
 * Errors: the function returns 0 when the kernel was enqueued, else
 *   -1 a required pointer is NULL, -3 a size is out of range, -4 misalignment,
 *   -7 the launch failed.
 * On the device, a request whose slot is outside [0, num_slots) (and not the pad value)
 * or whose accept count is out of range stores nothing and sets a status bit.  Rows of
 * padded requests, and slots no request names, are left untouched.
 */
#ifndef CAUSAL_CONV1D_DEDUP_H
#define CAUSAL_CONV1D_DEDUP_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CONV1D_K 4
#define CONV1D_PAD_SLOT (-1)
#define CONV1D_MAX_T 16
#define CONV1D_MAX_STATE_LEN 32
#define CONV1D_STATUS_BAD_SLOT 1u
#define CONV1D_STATUS_BAD_ACCEPT 2u
#define CONV1D_DTYPE_BF16 0
#define CONV1D_DTYPE_F32 1

int causal_conv1d_update_dedup(const void* x, void* conv_state, const void* weight,
                               const void* bias, const int32_t* slots,
                               const int32_t* num_accept, void* window, void* out,
                               uint32_t* status, int32_t bs, int32_t T, int32_t dim,
                               int32_t state_len, int64_t num_slots, int32_t silu,
                               cudaStream_t stream);

/*
 * The general form: the same update, with element types and strided views of the conv
 * state and the window rows.  The page's section "Accuracy Tests" lists fp32 and bf16,
 * mixed input and state dtypes, transposed window views and a channel count that leaves
 * a partial block.
 *   input_dtype  CONV1D_DTYPE_BF16 or CONV1D_DTYPE_F32: the type of x, weight, bias and out
 *   state_dtype  the same choice, for conv_state and window
 *   state_strides   host array of 3 element strides (slot, channel, column) of conv_state,
 *                   or NULL for the contiguous [num_slots][dim][state_len]
 *   window_strides  host array of 3 element strides (slot, channel, column) of the window
 *                   rows, or NULL for the contiguous [num_slots][dim][T + 2]; column c of
 *                   a row is step c's first window entry, so the per-step view [T][dim][3]
 *                   has step stride equal to window stride, as the page requires
 * Arithmetic is fp32 whatever the types; out is stored in the input type (bf16 rounding
 * to nearest even); the window and state entries are the row's values in the state type:
 * a bf16 value widens exactly, an fp32 input narrows to bf16 rounding to nearest even.
 * x, weight, bias and out are contiguous; dim is any positive count; every pointer is
 * aligned to its element size.  Every stride is at least 1, and the caller guarantees
 * that distinct (slot, channel, column) entries of each view are distinct elements of
 * its buffer.  When both types are bf16, both views contiguous, dim a multiple of 8 and
 * every pointer 16-byte aligned, this is causal_conv1d_update_dedup above.
 * Errors as above; -3 also for an unknown type code or a stride below 1.
 */
int causal_conv1d_update_dedup_ex(const void* x, void* conv_state, const void* weight,
                                  const void* bias, const int32_t* slots,
                                  const int32_t* num_accept, void* window, void* out,
                                  uint32_t* status, int32_t bs, int32_t T, int32_t dim,
                                  int32_t state_len, int64_t num_slots, int32_t silu,
                                  int32_t input_dtype, int32_t state_dtype,
                                  const int64_t* state_strides, const int64_t* window_strides,
                                  cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif
