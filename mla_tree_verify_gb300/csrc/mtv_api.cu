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
int kv_gather_ctas_per_sm();
int launch_kv_gather(const void* kv, int64_t num_slots, const int32_t* kv_indices,
                     int64_t num_kv_indices, const int32_t* kv_indptr, int32_t bs, void* dst, int64_t dst_rows,
                     int32_t dst_slot0, int32_t* new_indices, uint32_t* status, int grid,
                     cudaStream_t stream);
void launch_plan(const Problem& p, int grid, int tile, cudaStream_t stream);
int split_tile();
cudaError_t split_prepare();
int launch_split(const Problem& p, int grid, cudaStream_t stream);
}  // namespace mtv

namespace {

int static_ws_setup(int dev);   // the scratch of mla_tree_verify_static_ws(), at the end

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

// What a call does beyond the computation itself: index dumps, timing events, and the
// debug settings of mla_tree_verify_debug_ex().
struct RunOpts {
  int64_t* slot_dump = nullptr;
  uint8_t* vis_dump = nullptr;
  cudaEvent_t* events = nullptr;
  uint64_t wait_ns = 0;        // 0: kDefaultWaitNs
  int32_t merge_mode = 0;
  int32_t lanes = 0;           // 0: default_lanes()
};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// CTAs per lane group: the largest power of two up to kMaxLanes that divides the grid and
// does not exceed a request's column groups (so that a full job can exist).
int default_lanes(int grid, int32_t max_q_per_req, int32_t gt) {
  const int ncg = (max_q_per_req + gt - 1) / gt;
  int w = 1;
  while (2 * w <= mtv::kMaxLanes && 2 * w <= ncg && grid % (2 * w) == 0) w *= 2;
  return w;
}

int run(const void* q, const void* kv_cache, const int32_t* kv_indices, const int32_t* kv_indptr,
        const int64_t* out_cache_loc, const uint8_t* custom_mask, const int64_t* mask_indptr,
        const int64_t* qo_indptr, float sm_scale, void* out, float* lse, void* workspace,
        size_t workspace_bytes, int32_t bs, int32_t max_q_per_req, int32_t num_heads,
        int64_t num_slots, int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
        const RunOpts& opt, cudaStream_t stream) {
  if (num_heads != MLA_TV_HEADS && num_heads != MLA_TV_HEADS_TP8) return MLA_TV_ERR_HEADS;
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
  const int32_t gt = MLA_TV_HEADS / num_heads;
  const int lanes = opt.lanes ? opt.lanes : default_lanes(grid, max_q_per_req, gt);
  if (lanes < 1 || lanes > mtv::kMaxLanes || (lanes & (lanes - 1)) || grid % lanes)
    return MLA_TV_ERR_SHAPE;
  const mtv::WsLayout w = mtv::ws_layout(bs, max_q_per_req, grid, gt);
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
  p.heads = num_heads;
  p.group_tokens = gt;
  p.lanes = lanes;
  p.merge_mode = opt.merge_mode;
  p.wait_ns = opt.wait_ns ? opt.wait_ns : kDefaultWaitNs;
  p.num_slots = num_slots;
  p.total_q = total_q;
  p.num_kv_indices = num_kv_indices;
  p.mask_len = mask_len;
  unsigned char* ws = (unsigned char*)workspace;
  p.hdr = (mtv::WsHeader*)ws;
  p.cum_units = (int64_t*)(ws + w.cum_off);
  p.cum_tok = (int64_t*)(ws + w.tok_off);
  p.cum_job = (int64_t*)(ws + w.job_cum_off);
  p.jobs = (mtv::JobRec*)(ws + w.job_off);
  p.grp_job = (int32_t*)(ws + w.grp_off);
  p.tok_done = (int32_t*)(ws + w.cnt_off);
  p.grp_done = (int32_t*)(ws + w.gdone_off);
  p.part_lse = (float*)(ws + w.lse_off);
  p.part_o = (float*)(ws + w.o_off);
  p.num_seg = w.num_seg;
  p.dump_slots = opt.slot_dump;
  p.dump_vis = opt.vis_dump;
  cudaEvent_t* events = opt.events;

  cudaGetLastError();  // launches below report only their own errors
  if (events) cudaEventRecordWithFlags(events[0], stream, cudaEventRecordExternal);
  mtv::launch_plan(p, grid, mtv::split_tile(), stream);
  if (events) cudaEventRecordWithFlags(events[1], stream, cudaEventRecordExternal);
  const int split_status = mtv::launch_split(p, grid, stream);
  if (events) cudaEventRecordWithFlags(events[2], stream, cudaEventRecordExternal);
  if (cudaGetLastError() != cudaSuccess || split_status != 0) return MLA_TV_ERR_LAUNCH;
  return MLA_TV_OK;
}

}  // namespace

extern "C" {

size_t mla_tree_verify_workspace_bytes(int32_t bs, int32_t max_q_per_req, int32_t num_heads) {
  if ((num_heads != MLA_TV_HEADS && num_heads != MLA_TV_HEADS_TP8) || bs < 1 || max_q_per_req < 1 ||
      max_q_per_req > MLA_TV_MAX_Q_PER_REQ)
    return 0;
  int dev;
  if (current_device(&dev) != MLA_TV_OK || prepare_device(dev) != MLA_TV_OK) return 0;
  return mtv::ws_layout(bs, max_q_per_req, g_sm_count[dev], MLA_TV_HEADS / num_heads).total;
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
             num_heads, num_slots, total_q, num_kv_indices, mask_len, RunOpts(), stream);
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
  RunOpts opt;
  opt.slot_dump = slot_dump;
  opt.vis_dump = vis_dump;
  return run(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
             qo_indptr, sm_scale, out, lse, workspace, workspace_bytes, bs, max_q_per_req,
             num_heads, num_slots, total_q, num_kv_indices, mask_len, opt, stream);
}

int mla_tree_verify_debug_ex(const void* q, const void* kv_cache, const int32_t* kv_indices,
                             const int32_t* kv_indptr, const int64_t* out_cache_loc,
                             const uint8_t* custom_mask, const int64_t* mask_indptr,
                             const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t bs,
                             int32_t max_q_per_req, int32_t num_heads, int64_t num_slots,
                             int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
                             const mla_tree_verify_debug_opts* opts, cudaStream_t stream) {
  if (!opts || (!opts->slot_dump) != (!opts->vis_dump)) return MLA_TV_ERR_NULL;
  if (opts->merge_mode < MLA_TV_MERGE_AUTO || opts->merge_mode > MLA_TV_MERGE_PREFER_TMEM ||
      opts->lanes < 0)
    return MLA_TV_ERR_SHAPE;
  RunOpts opt;
  opt.slot_dump = opts->slot_dump;
  opt.vis_dump = opts->vis_dump;
  opt.wait_ns = opts->wait_limit_ns;
  opt.merge_mode = opts->merge_mode;
  opt.lanes = opts->lanes;
  return run(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
             qo_indptr, sm_scale, out, lse, workspace, workspace_bytes, bs, max_q_per_req,
             num_heads, num_slots, total_q, num_kv_indices, mask_len, opt, stream);
}

int mla_tree_verify_profiled(const void* q, const void* kv_cache, const int32_t* kv_indices,
                             const int32_t* kv_indptr, const int64_t* out_cache_loc,
                             const uint8_t* custom_mask, const int64_t* mask_indptr,
                             const int64_t* qo_indptr, float sm_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t bs,
                             int32_t max_q_per_req, int32_t num_heads, int64_t num_slots,
                             int64_t total_q, int64_t num_kv_indices, int64_t mask_len,
                             cudaEvent_t* events, cudaStream_t stream) {
  if (!events || !events[0] || !events[1] || !events[2]) return MLA_TV_ERR_NULL;
  RunOpts opt;
  opt.events = events;
  return run(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
             qo_indptr, sm_scale, out, lse, workspace, workspace_bytes, bs, max_q_per_req,
             num_heads, num_slots, total_q, num_kv_indices, mask_len, opt, stream);
}

int mla_tree_verify_prepare(void) {
  int dev;
  if (current_device(&dev) != MLA_TV_OK) return MLA_TV_ERR_DEVICE;
  const int st = prepare_device(dev);
  if (st != MLA_TV_OK) return st;
  return static_ws_setup(dev);
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

int mla_tree_verify_kv_gather(const void* kv_cache, int64_t num_slots, const int32_t* kv_indices,
                              int64_t num_kv_indices, const int32_t* kv_indptr, int32_t bs, void* dst, int64_t dst_rows,
                              int32_t dst_slot0, int32_t* new_indices, uint32_t* status,
                              cudaStream_t stream) {
  if (!kv_cache || !kv_indices || !kv_indptr || !dst || !new_indices || !status)
    return MLA_TV_ERR_NULL;
  if (bs < 1 || num_slots < 1 || num_slots > INT32_MAX || num_kv_indices < 0 || dst_rows < 0 ||
      dst_slot0 < 0 ||
      (int64_t)dst_slot0 + dst_rows > INT32_MAX)
    return MLA_TV_ERR_SHAPE;
  if (!aligned(kv_cache, 16) || !aligned(dst, 16) || !aligned(kv_indices, 4) ||
      !aligned(kv_indptr, 4) || !aligned(new_indices, 4) || !aligned(status, 4))
    return MLA_TV_ERR_ALIGN;
  int dev;
  if (current_device(&dev) != MLA_TV_OK) return MLA_TV_ERR_DEVICE;
  const int st = prepare_device(dev);
  if (st != MLA_TV_OK) return st;
  cudaGetLastError();
  const int grid = g_sm_count[dev] * mtv::kv_gather_ctas_per_sm();
  if (mtv::launch_kv_gather(kv_cache, num_slots, kv_indices, num_kv_indices, kv_indptr, bs, dst, dst_rows,
                            dst_slot0, new_indices, status, grid, stream) != 0)
    return MLA_TV_ERR_LAUNCH;
  return MLA_TV_OK;
}

const char* mla_tree_verify_status_string(int status) {
  switch (status) {
    case MLA_TV_OK: return "ok";
    case MLA_TV_ERR_NULL: return "a required pointer is NULL";
    case MLA_TV_ERR_HEADS: return "num_heads must be 64, or 8 (MLA_TV_HEADS_TP8)";
    case MLA_TV_ERR_SHAPE: return "invalid batch size, max_q_per_req or array length";
    case MLA_TV_ERR_ALIGN: return "misaligned buffer (q/kv_cache/out 16 B, workspace 256 B)";
    case MLA_TV_ERR_WORKSPACE: return "workspace smaller than mla_tree_verify_workspace_bytes()";
    case MLA_TV_ERR_LAUNCH: return "kernel launch failed";
    case MLA_TV_ERR_DEVICE: return "no current CUDA device, or it is not sm_103";
    case MLA_TV_ERR_SCALE: return "sm_scale is not finite";
    case MLA_TV_ERR_STATIC_LIMIT:
      return "batch needs more scratch than the built-in static workspace holds";
    default: return "unknown status";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// Built-in scratch for callers that cannot allocate device memory.
//
// Some callers have no device allocator of their own: an engine may hand this library
// raw tensor pointers while keeping its memory pool private, or C code may run where
// cudaMalloc is not allowed after start-up (it can synchronise the device, and it is
// forbidden while a CUDA graph is being captured).  For them the library carries one
// scratch array in device memory, sized at build time; every GPU that loads the
// library holds it until the process exits.  The array is shared by all calls on a
// device and keeps the previous call's contents.  The planner kernel rewrites the
// header (including the error bits, the only part that must start at zero) and the
// work plan at the start of every call, and every partial result is written before it
// is read, so nothing is cleared by hand.  Calls that can overlap on the GPU (two
// streams without ordering, or several host threads) race on the array.
static __device__ __align__(256) unsigned char g_static_ws[MLA_TV_STATIC_WS_BYTES];

namespace {

std::once_flag g_static_once[kMaxDevices];
void* g_static_ptr[kMaxDevices];
int g_static_status[kMaxDevices];

// With `dev` current: the device address of g_static_ws (the host-side name is only a
// stand-in for it and must never be handed to a kernel).
int static_ws_setup(int dev) {
  std::call_once(g_static_once[dev], [dev]() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      g_static_status[dev] = MLA_TV_ERR_DEVICE;
      return;
    }
    g_static_ptr[dev] = ptr;
    g_static_status[dev] = MLA_TV_OK;
  });
  return g_static_status[dev];
}

}  // namespace

extern "C" int mla_tree_verify_static_ws(
    const void* q, const void* kv_cache, const int32_t* kv_indices, const int32_t* kv_indptr,
    const int64_t* out_cache_loc, const uint8_t* custom_mask, const int64_t* mask_indptr,
    const int64_t* qo_indptr, float sm_scale, void* out, float* lse, int32_t bs,
    int32_t max_q_per_req, int32_t num_heads, int64_t num_slots, int64_t total_q,
    int64_t num_kv_indices, int64_t mask_len, cudaStream_t stream) {
  if (num_heads != MLA_TV_HEADS && num_heads != MLA_TV_HEADS_TP8) return MLA_TV_ERR_HEADS;
  if (bs < 1 || max_q_per_req < 1 || max_q_per_req > MLA_TV_MAX_Q_PER_REQ)
    return MLA_TV_ERR_SHAPE;
  int dev;
  if (current_device(&dev) != MLA_TV_OK) return MLA_TV_ERR_DEVICE;
  int st = prepare_device(dev);
  if (st != MLA_TV_OK) return st;
  if (mtv::ws_layout(bs, max_q_per_req, g_sm_count[dev], MLA_TV_HEADS / num_heads).total >
      (size_t)MLA_TV_STATIC_WS_BYTES)
    return MLA_TV_ERR_STATIC_LIMIT;
  st = static_ws_setup(dev);
  if (st != MLA_TV_OK) return st;
  return run(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
             qo_indptr, sm_scale, out, lse, g_static_ptr[dev], (size_t)MLA_TV_STATIC_WS_BYTES,
             bs, max_q_per_req, num_heads, num_slots, total_q, num_kv_indices, mask_len,
             RunOpts(), stream);
}
