// Host side of the C ABI declared in include/mla_tree_verify.h: argument checks, the
// workspace layout, and the three launches (planner, split, combine) on the caller's
// stream.  No allocation, no synchronisation, no device reads on this path ("The
// Architecture of Capture Safety", section "The Design Emerges": fixed grid,
// preallocated workspace, raw pointers plus scalars).
#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla_tree_verify.h"
#include "mtv_common.cuh"

namespace mtv {
void launch_plan(const Problem& p, int grid, int tile, cudaStream_t stream);
void launch_combine(const Problem& p, cudaStream_t stream);
int split_tile();
cudaError_t split_prepare();
int launch_split(const Problem& p, int grid, cudaStream_t stream);
}  // namespace mtv

namespace {

constexpr int kMaxDevices = 64;
std::once_flag g_prep_once[kMaxDevices];
int g_prep_status[kMaxDevices];
int g_sm_count[kMaxDevices];

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_TV_ERR_DEVICE;
  }
  return MLA_TV_OK;
}

int prepare_device(int dev) {
  std::call_once(g_prep_once[dev], [dev]() {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
      cudaGetLastError();
      g_prep_status[dev] = MLA_TV_ERR_DEVICE;
      return;
    }
    g_sm_count[dev] = sms;
    g_prep_status[dev] = (mtv::split_prepare() == cudaSuccess) ? MLA_TV_OK : MLA_TV_ERR_DEVICE;
    cudaGetLastError();
  });
  return g_prep_status[dev];
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

int run(const void* q, const void* kv_cache, const int32_t* kv_indices, const int32_t* kv_indptr,
        const int64_t* out_cache_loc, const uint8_t* custom_mask, const int64_t* mask_indptr,
        const int64_t* qo_indptr, float sm_scale, void* out, float* lse, void* workspace,
        size_t workspace_bytes, int32_t bs, int32_t max_q_per_req, int32_t num_heads,
        int64_t num_slots, int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
        int64_t* slot_dump, uint8_t* vis_dump, cudaEvent_t* events, cudaStream_t stream) {
  if (num_heads != MLA_TV_HEADS) return MLA_TV_ERR_HEADS;
  if (bs < 1 || max_q_per_req < 1 || max_q_per_req > MLA_TV_MAX_Q_PER_REQ || num_slots < 1 ||
      num_slots > INT32_MAX || total_q > INT32_MAX / MLA_TV_HEADS ||
      total_q < 0 || num_kv_indices < 0 || mask_len < 0)
    return MLA_TV_ERR_SHAPE;
  if (!kv_cache || !kv_indptr || !mask_indptr || !qo_indptr || !workspace ||
      (total_q > 0 && (!q || !out || !lse || !out_cache_loc)) ||
      (num_kv_indices > 0 && !kv_indices) || (mask_len > 0 && !custom_mask))
    return MLA_TV_ERR_NULL;
  if (!std::isfinite(sm_scale)) return MLA_TV_ERR_SCALE;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(workspace, 256) || !aligned(kv_indices, 4) || !aligned(kv_indptr, 4) ||
      !aligned(out_cache_loc, 8) || !aligned(mask_indptr, 8) || !aligned(qo_indptr, 8))
    return MLA_TV_ERR_ALIGN;
  int dev;
  if (current_device(&dev) != MLA_TV_OK) return MLA_TV_ERR_DEVICE;
  int st = prepare_device(dev);
  if (st != MLA_TV_OK) return st;
  const int grid = g_sm_count[dev];
  const mtv::WsLayout w = mtv::ws_layout(bs, max_q_per_req, grid);
  if (workspace_bytes < w.total) return MLA_TV_ERR_WORKSPACE;

  mtv::Problem p;
  p.q = (const uint16_t*)q;
  p.kv = (const uint16_t*)kv_cache;
  p.kv_indices = kv_indices;
  p.kv_indptr = kv_indptr;
  p.out_cache_loc = out_cache_loc;
  p.custom_mask = custom_mask;
  p.mask_indptr = mask_indptr;
  p.qo_indptr = qo_indptr;
  p.out = (uint16_t*)out;
  p.lse = lse;
  p.sm_scale = sm_scale;
  p.bs = bs;
  p.max_q_per_req = max_q_per_req;
  p.num_slots = num_slots;
  p.total_q = total_q;
  p.num_kv_indices = num_kv_indices;
  p.mask_len = mask_len;
  unsigned char* ws = (unsigned char*)workspace;
  p.hdr = (mtv::WsHeader*)ws;
  p.cum_units = (int64_t*)(ws + w.cum_off);
  p.part_lse = (float*)(ws + w.lse_off);
  p.part_o = (float*)(ws + w.o_off);
  p.num_seg = w.num_seg;
  p.dump_slots = slot_dump;
  p.dump_vis = vis_dump;

  cudaGetLastError();  // launches below report only their own errors
  if (events) cudaEventRecord(events[0], stream);
  mtv::launch_plan(p, grid, mtv::split_tile(), stream);
  if (events) cudaEventRecord(events[1], stream);
  const int split_status = mtv::launch_split(p, grid, stream);
  if (events) cudaEventRecord(events[2], stream);
  mtv::launch_combine(p, stream);
  if (events) cudaEventRecord(events[3], stream);
  if (cudaGetLastError() != cudaSuccess || split_status != 0) return MLA_TV_ERR_LAUNCH;
  return MLA_TV_OK;
}

}  // namespace

extern "C" {

size_t mla_tree_verify_workspace_bytes(int32_t bs, int32_t max_q_per_req, int32_t num_heads) {
  if (num_heads != MLA_TV_HEADS || bs < 1 || max_q_per_req < 1 ||
      max_q_per_req > MLA_TV_MAX_Q_PER_REQ)
    return 0;
  int dev;
  if (current_device(&dev) != MLA_TV_OK || prepare_device(dev) != MLA_TV_OK) return 0;
  return mtv::ws_layout(bs, max_q_per_req, g_sm_count[dev]).total;
}

int mla_tree_verify(const void* q, const void* kv_cache, const int32_t* kv_indices,
                    const int32_t* kv_indptr, const int64_t* out_cache_loc,
                    const uint8_t* custom_mask, const int64_t* mask_indptr,
                    const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                    void* workspace, size_t workspace_bytes, int32_t bs, int32_t max_q_per_req,
                    int32_t num_heads, int64_t num_slots, int64_t total_q,
                    int64_t num_kv_indices, int64_t mask_len, cudaStream_t stream) {
  return run(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
             qo_indptr, sm_scale, out, lse, workspace, workspace_bytes, bs, max_q_per_req,
             num_heads, num_slots, total_q, num_kv_indices, mask_len, nullptr, nullptr, nullptr,
             stream);
}

int mla_tree_verify_debug(const void* q, const void* kv_cache, const int32_t* kv_indices,
                          const int32_t* kv_indptr, const int64_t* out_cache_loc,
                          const uint8_t* custom_mask, const int64_t* mask_indptr,
                          const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, int32_t bs,
                          int32_t max_q_per_req, int32_t num_heads, int64_t num_slots,
                          int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
                          int64_t* slot_dump, uint8_t* vis_dump, cudaStream_t stream) {
  if (!slot_dump || !vis_dump) return MLA_TV_ERR_NULL;
  return run(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
             qo_indptr, sm_scale, out, lse, workspace, workspace_bytes, bs, max_q_per_req,
             num_heads, num_slots, total_q, num_kv_indices, mask_len, slot_dump, vis_dump,
             nullptr, stream);
}

int mla_tree_verify_profiled(const void* q, const void* kv_cache, const int32_t* kv_indices,
                             const int32_t* kv_indptr, const int64_t* out_cache_loc,
                             const uint8_t* custom_mask, const int64_t* mask_indptr,
                             const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t bs,
                             int32_t max_q_per_req, int32_t num_heads, int64_t num_slots,
                             int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
                             cudaEvent_t* events, cudaStream_t stream) {
  if (!events || !events[0] || !events[1] || !events[2] || !events[3]) return MLA_TV_ERR_NULL;
  return run(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
             qo_indptr, sm_scale, out, lse, workspace, workspace_bytes, bs, max_q_per_req,
             num_heads, num_slots, total_q, num_kv_indices, mask_len, nullptr, nullptr, events,
             stream);
}

int mla_tree_verify_prepare(void) {
  int dev;
  if (current_device(&dev) != MLA_TV_OK) return MLA_TV_ERR_DEVICE;
  return prepare_device(dev);
}

int mla_tree_verify_read_device_status(const void* workspace, uint32_t* flags,
                                       cudaStream_t stream) {
  if (!workspace || !flags) return MLA_TV_ERR_NULL;
  if (cudaMemcpyAsync(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_TV_ERR_LAUNCH;
  }
  return MLA_TV_OK;
}

int32_t mla_tree_verify_split_grid(void) {
  int dev;
  if (current_device(&dev) != MLA_TV_OK || prepare_device(dev) != MLA_TV_OK) return 0;
  return g_sm_count[dev];
}

const char* mla_tree_verify_status_string(int status) {
  switch (status) {
    case MLA_TV_OK: return "ok";
    case MLA_TV_ERR_NULL: return "a required pointer is NULL";
    case MLA_TV_ERR_HEADS: return "num_heads must be 64";
    case MLA_TV_ERR_SHAPE: return "invalid batch size, max_q_per_req or array length";
    case MLA_TV_ERR_ALIGN: return "misaligned buffer (q/kv_cache/out 16 B, workspace 256 B)";
    case MLA_TV_ERR_WORKSPACE: return "workspace smaller than mla_tree_verify_workspace_bytes()";
    case MLA_TV_ERR_LAUNCH: return "kernel launch failed";
    case MLA_TV_ERR_DEVICE: return "no current CUDA device, or it is not sm_103";
    case MLA_TV_ERR_SCALE: return "sm_scale is not finite";
    default: return "unknown status";
  }
}

}  // extern "C"
