// Split-K partial kernel on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes is the split step of the verify attention ("The Architecture of
// Capture Safety", section "The Design Emerges": a split of the key sequence yields
// an online-softmax partial (m, l, o); prefix rows come through kv_indices, draft rows
// through out_cache_loc, visibility is read inline from custom_mask; "The Plan
// Document", section "Variant 3": each key row is read once per block for all of the
// block's heads).
//
// Layout on the SM.  One CTA per SM walks its share of (query token, key tile) units.
// For the current token, the 64 heads x 576 dims of q sit in shared memory as nine
// 128-byte-swizzled K-major chunks of [64 heads][64 dims] (TMA tile loads).  A key tile
// is 128 gathered cache rows, held as nine chunk slots of [128 rows][64 dims], filled
// by three producer warps with 16-byte cp.async copies (rows past the end of the request
// are zero-filled).  The MMAs run transposed, with key rows and value dims on the TMEM
// lanes, because the fp32 output of one token (64 x 512) already fills half of TMEM:
//   S^T[128 keys][64 heads]   = K_tile . Q^T          (M=128, N=64, K=576: 36 MMAs)
//   O^T[512 dims][64 heads]  += V_tile^T . P^T         (4 x M=128, N=64, K=128)
// The same shared-memory tile serves as K-major A for the first product and as
// MN-major A (V^T) for the second.  P^T is written in bf16 over the tile's rope chunk,
// which the first product no longer needs.
//
// Softmax.  Eight softmax warps: warp pair (w, w+4) shares one quarter of the TMEM
// lanes (32 key rows) and splits the 64 heads in halves.  Each thread holds 32 scores
// of its key row.  The running maximum per head is exact: every tile takes the
// column maximum over its 128 rows (warp max reduction, then four quarters through
// shared memory), and O^T and the per-thread partial sums l are rescaled when it rises,
// so the largest term of each head enters the bf16 P exactly as 1.  l is reduced across
// rows once per segment.
//
// Warp roles: warps 0-2 load (cp.async for key tiles, TMA for q) and issue the QK
// product of the chunks they loaded, each into its own partial S^T (the softmax adds the
// three in a fixed order); warp 3 (one thread) issues the PV product and owns TMEM;
// warps 4-11 run the softmax, the rescale and the epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mtv_common.cuh"
#include "mtv_ptx.cuh"

namespace mtv {
namespace tc {

constexpr int kTile = 128;
constexpr int kChunks = 9;               // 576 dims = 9 x 64
constexpr int kProducerWarps = 3;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = 32 * (kProducerWarps + 1 + kSoftmaxWarps);   // 384
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kFirstSoftmaxThread = 32 * (kProducerWarps + 1);
constexpr uint32_t kQChunk = 64 * 128;   // [64 heads][64 dims] bf16
constexpr uint32_t kKvChunk = 128 * 128; // [128 rows][64 dims] bf16
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKvOff = kQOff + kChunks * kQChunk;       // 73728
constexpr uint32_t kBarOff = kKvOff + kChunks * kKvChunk;     // 221184
constexpr uint32_t kRedOff = kBarOff + 256;                    // float [2][64][4]
constexpr uint32_t kRed2Off = kRedOff + 2 * 64 * 4 * 4;        // float [64][4]
constexpr uint32_t kStatOff = kRed2Off + 64 * 4 * 4;           // 1/l[64]
constexpr uint32_t kMOff = kStatOff + 64 * 4;                  // float [2][64]
constexpr uint32_t kAlphaOff = kMOff + 2 * 64 * 4;             // float [2][64]
constexpr uint32_t kMPrevOff = kAlphaOff + 2 * 64 * 4;         // float [64]
constexpr uint32_t kMiscOff = kMPrevOff + 64 * 4;              // tmem slot, abort flag
constexpr uint32_t kWOff = kMiscOff + 64;                      // merge weights [16][64]
constexpr uint32_t kSegOff = kWOff + kMergeGroup * 64 * 4;     // SegInfo of the segment
constexpr uint32_t kSlotOff = kSegOff + 64;                    // int32 [64] partial slots
constexpr uint32_t kSmemUsed = kSlotOff + kNsplit * 4;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;              // + alignment slack
static_assert(kSmemBytes <= 232448, "dynamic shared memory of one CTA");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;          // partial S^T of producer warp w at 256 + 64w; O^T at 0..255
constexpr uint32_t kIdescQK = ptx::idesc_bf16(128, 64, 0, 0);
constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, 64, 1, 1);
constexpr uint32_t kErrTimeout = 8u;
constexpr uint64_t kMergeWaitNs = 20000000ull;   // merge mode 2: wait for the other pieces
constexpr uint32_t kSoftmaxBar = 1;      // named barrier of the softmax warps

// Chunk slots are released in pairs: PV block m reads value dims [128m, 128m+128),
// i.e. slots 2m and 2m+1; slot 8 (rope, then P^T) is released after the last block.
__host__ __device__ constexpr int release_group(int c) { return c < 8 ? c >> 1 : 4; }

struct Bars {
  uint64_t q_full, q_empty, s_full, p_full, o_done, o_free, drain;
  uint64_t kv_empty[5], drain_p[kProducerWarps];
  uint64_t kv_full[kChunks];   // TMA tile loads of a run of consecutive slots, per chunk slot
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Seg {
  ReqInfo ri;
  int64_t r;                   // the column group's first token row
  SegMap map;                  // partial slots of the column group's pieces
  int32_t nseg;                // its pieces
  int32_t piece;               // this CTA's piece among them
  int32_t seg;                 // the partial slot of this piece
  int32_t b, t, tile0, tile1;  // request, column group of the request, tile range
  int32_t ncols;               // columns of the group that are real (token, head) pairs
  bool lead;                   // the first lane on this tile range (it prefetches the rows)
};

// The partial slots of the softmax warps' current segment, parked in shared memory from the
// segment's start to its epilogue (they are not needed in between).
struct SegInfo {
  SegMap map;
  int32_t nseg, piece, seg;
};
static_assert(sizeof(SegInfo) <= 64, "segment info block");

// Where a CTA walks the plan: its lane group's units [u, u_end), the group g, its lane in
// the group, the lanes per group W, and J, the job that owns unit u or an earlier one.
struct Walk {
  int64_t u, u_end;
  int32_t g, lane, W, J;
};

// The lane's next segment in its group's units [u, u_end): the run of tiles that this
// lane processes in the next job it has work in (JobGeo and JobRec in mtv_common.cuh).
// The jobs are walked in order, from the planner's records.
__device__ __forceinline__ bool next_segment(const Problem& p, Walk& wk, Seg& s) {
  for (;;) {
    if (wk.u >= wk.u_end) return false;
    const JobRec r = p.jobs[wk.J];
    const int64_t je = r.js + r.sl + kSegCost;
    if (wk.u >= je) {                          // this lane has passed the job
      ++wk.J;
      continue;
    }
    const int64_t o0 = wk.u - r.js;
    const int64_t o1 = min(wk.u_end, je) - r.js;
    wk.u = r.js + o1;                          // the next call starts at the next job
    if (wk.lane >= r.nt * r.k) continue;       // no work for this lane in the job
    const int32_t sub = wk.lane / r.nt, cgl = wk.lane - sub * r.nt;
    const int64_t len = sub_len(r.tiles, sub, r.sl);
    if (o0 >= len) continue;                   // its sub-range ends before the range begins
    s.ri.P = r.P;
    s.ri.T = r.T;
    s.ri.kv_base = r.kv_base;
    s.ri.q_base = r.q_base;
    s.ri.L = (int64_t)r.P + r.T;
    s.ri.m_base = r.m_base;
    s.b = r.b;
    s.t = r.cg0 + cgl;
    s.tile0 = (int32_t)((int64_t)sub * r.sl + o0);
    s.tile1 = (int32_t)((int64_t)sub * r.sl + min(o1, len));
    s.r = (int64_t)r.q_base + (int64_t)s.t * p.group_tokens;
    s.ncols = min(p.group_tokens, r.T - s.t * p.group_tokens) * p.heads;
    s.lead = cgl == 0;
    s.map.tok0 = r.tok0 + cgl;
    s.map.g_lo = r.g_lo;
    s.map.nt = r.nt;
    s.map.W = wk.W;
    s.map.n_full = r.n_full;
    s.map.ns = r.ns;
    s.nseg = r.nseg;
    s.piece = sub * r.n_full + (wk.g - r.g_lo);
    s.seg = (int32_t)s.map.slot(s.piece);
    return true;
  }
}

__device__ __forceinline__ void fail(const Problem& p, volatile int* abort) {
  *abort = 1;
  atomicOr(&p.hdr->error_flags, kErrTimeout);
}

// Reduces v[i] over the 32 lanes of a warp for all 32 i at once (transpose butterfly,
// 31 shuffles): afterwards v[0] on lane l holds the reduction of v[l] over the lanes.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < off; ++k) {
      const float send = upper ? v[k] : v[k + off];
      const float keep = upper ? v[k + off] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// 128B-swizzled offset of 16-byte granule g in row r of an [rows][128 B] chunk.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t g) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((g ^ (r & 7u)) << 4);
}

// ------------------------------------------------------------------ producers (warps 0-2)
// Producer warp pw gathers chunk slots c = pw, pw + 3, pw + 6 of each tile (all 128
// rows) and issues the QK product of those chunks itself, into its own partial
// S^T_pw (TMEM columns 256 + 64 pw): lane 0 issues a chunk's four MMAs as soon as the
// warp's copies of it have landed and been fenced for the async proxy, so no other
// thread has to be told that the chunk is there.  The softmax adds the three partials in
// a fixed order.  One instruction moves four rows x 128 bytes: lane l copies granule l%8
// of row 4i + l/8.  Each warp keeps two chunks in flight.
__device__ void producer(const Problem& p, const CUtensorMap* tm_q, const CUtensorMap* tm_kv,
                         unsigned char* sm, Bars* bars, volatile int* abort, uint32_t tmem,
                         Walk wk) {
  const int lane = threadIdx.x & 31, pw = threadIdx.x >> 5;
  const uint32_t q_base = ptx::smem_addr(sm + kQOff);
  const uint32_t kv_base = ptx::smem_addr(sm + kKvOff);
  // K-major operands: 8-row groups 1024 B apart; a K step of 16 dims is +32 B.
  const uint64_t dq0 = ptx::sdesc_sw128(q_base, 16, 1024);
  const uint64_t dk0 = ptx::sdesc_sw128(kv_base, 16, 1024);
  const uint32_t d_s = tmem + kSCol + 64 * pw;
  const uint32_t g = lane & 7, sub = lane >> 3;
  const unsigned char* kv = (const unsigned char*)p.kv;
  uint32_t tl = 0, sc = 0;
  uint32_t nt = 0;          // tiles this warp loaded with TMA (phase of its kv_full barriers)
  uint32_t pending = 0;     // chunk slots with a TMA load not yet waited for
  bool ok = true;
  Seg s;
  while (ok && next_segment(p, wk, s)) {
    // Tiles load as TMA tile copies only where the request's prefix may be one run of
    // consecutive slots (its first and last slots P - 1 apart); other requests skip the
    // per-tile test, whose slot reads would otherwise come before the slot wait.
    bool may_run = false;
    if (s.ri.P >= kTile) {
      const int64_t first = p.kv_indices[s.ri.kv_base];
      const int64_t last = p.kv_indices[s.ri.kv_base + s.ri.P - 1];
      may_run = last - first == s.ri.P - 1;
    }
    if (pw == 0) {
      if (sc > 0) {
        int w = lane == 0 ? ptx::mbar_wait(&bars->q_empty, (sc - 1) & 1, abort, p.wait_ns) : 0;
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) break;
      }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&bars->q_full, kChunks * kQChunk);
        for (int c = 0; c < kChunks; ++c)
          ptx::tma_load_2d(q_base + c * kQChunk, tm_q, c * 64, (int32_t)(s.r * p.heads),
                           &bars->q_full);
      }
    }
    ++sc;
    for (int64_t j = s.tile0; ok && j < s.tile1; ++j, ++tl) {
      // slots of the tile's 128 rows: lane holds rows lane + 32h, h = 0..3
      int32_t slot4[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int64_t c = j * kTile + 32 * h + lane;
        slot4[h] = (int32_t)(c < s.ri.L ? key_slot(p, s.ri, c) : -1);
      }
      // The next tile's rows go to L2 now: its copies can only start once this tile's
      // value blocks are done, and then they should hit L2.
      if (s.lead && j + 1 < s.tile1) {
        for (int r = 32 * pw + lane; r < kTile; r += 32 * kProducerWarps) {
          const int64_t c = (j + 1) * kTile + r;
          const int64_t sl = c < s.ri.L ? key_slot(p, s.ri, c) : -1;
          if (sl >= 0) {
            const unsigned char* rowp = kv + sl * kRowBytes;
#pragma unroll
            for (int ln = 0; ln < kRowBytes / 128; ++ln) ptx::prefetch_l2(rowp + 128 * ln);
          }
        }
      }
      // QK of chunk c (this warp's copies of it have landed): publish the copies to the
      // async proxy, then lane 0 issues its four MMAs; the warp's first chunk of the tile
      // starts the partial sum.  A segment's first tile first waits for q.
      auto qk_chunk = [&](int c, bool first_chunk) -> bool {
        ptx::fence_proxy_async();
        __syncwarp();
        int st = 1;
        if (lane == 0) {
          if (first_chunk && j == s.tile0) st = ptx::mbar_wait(&bars->q_full, (sc - 1) & 1, abort, p.wait_ns);
          if (st) {
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t koff = (c * kKvChunk + kk * 32) >> 4, qoff = (c * kQChunk + kk * 32) >> 4;
              ptx::mma_bf16(d_s, dk0 + koff, dq0 + qoff, kIdescQK, !(first_chunk && kk == 0));
            }
          }
        }
        return __shfl_sync(0xffffffffu, st, 0) != 0;
      };
      // A tile whose 128 rows sit in consecutive, valid slots (a defragmented prefix) is
      // loaded with one TMA tile copy per chunk: the tensor map's 128-byte swizzle gives
      // the same shared-memory layout as the row copies below.
      int32_t s0 = 0;
      bool use_tma = false;
      if (may_run) {   // warp-uniform
        s0 = __shfl_sync(0xffffffffu, slot4[0], 0);
        bool run = true;
#pragma unroll
        for (int h = 0; h < 4; ++h) run &= slot4[h] >= 0 && slot4[h] == s0 + lane + 32 * h;
        use_tma = __all_sync(0xffffffffu, run);
      }
      if (use_tma) {
        for (int c = pw; c < kChunks; c += kProducerWarps) {
          if (tl > 0) {
            int w = lane == 0 ? ptx::mbar_wait(&bars->kv_empty[release_group(c)], (tl - 1) & 1, abort, p.wait_ns)
                              : 0;
            ok = __shfl_sync(0xffffffffu, w, 0) != 0;
            if (!ok) break;
          }
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&bars->kv_full[c], kKvChunk);
            ptx::tma_load_2d(kv_base + c * kKvChunk, tm_kv, c * 64, s0, &bars->kv_full[c]);
          }
          pending |= 1u << c;
        }
        for (int c = pw; ok && c < kChunks; c += kProducerWarps) {
          int w = lane == 0 ? ptx::mbar_wait(&bars->kv_full[c], nt & 1, abort, p.wait_ns) : 0;
          ok = __shfl_sync(0xffffffffu, w, 0) != 0;
          if (!ok) break;
          pending &= ~(1u << c);
          ok = qk_chunk(c, c == pw);
        }
        ++nt;
        if (!ok) break;
        if (lane == 0) {
          ptx::mma_commit(&bars->s_full);
          if (j + 1 == s.tile1) ptx::mma_commit(&bars->q_empty);
        }
        __syncwarp();
        continue;
      }
      int prev = -1;
      for (int c = pw; c < kChunks; c += kProducerWarps) {
        if (tl > 0) {
          int w = lane == 0 ? ptx::mbar_wait(&bars->kv_empty[release_group(c)], (tl - 1) & 1, abort, p.wait_ns)
                            : 0;
          ok = __shfl_sync(0xffffffffu, w, 0) != 0;
          if (!ok) break;
        }
        const uint32_t dst0 = kv_base + c * kKvChunk;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t row = 4 * i + sub;                 // 0..127
          const int32_t sl = __shfl_sync(0xffffffffu, slot4[row >> 5], row & 31);
          const unsigned char* from =
              kv + (sl >= 0 ? (int64_t)sl * kRowBytes + c * 128 + g * 16 : 0);
          ptx::cp_async16(dst0 + swz(row, g), from, sl >= 0 ? 16 : 0);
        }
        ptx::cp_async_commit();
        if (prev >= 0) {
          ptx::cp_async_wait<1>();
          ok = qk_chunk(prev, prev == pw);
          if (!ok) break;
        }
        prev = c;
      }
      if (!ok) break;
      ptx::cp_async_wait<0>();
      ok = qk_chunk(prev, prev == pw);
      if (!ok) break;
      if (lane == 0) {
        ptx::mma_commit(&bars->s_full);
        if (j + 1 == s.tile1) ptx::mma_commit(&bars->q_empty);
      }
      __syncwarp();
    }
  }
  if (!ok && lane == 0) fail(p, abort);
  // Before the CTA exits every copy this thread issued must have landed, and every MMA
  // lane 0 issued must be done (bounded waits).
  ptx::cp_async_wait<0>();
  if (lane == 0) {
    volatile int never = 0;
    ptx::mma_commit(&bars->drain_p[pw]);
    ptx::mbar_wait(&bars->drain_p[pw], 0, &never, 100000000ull);
    if (pw == 0 && sc > 0) ptx::mbar_wait(&bars->q_full, (sc - 1) & 1, &never, 100000000ull);
    for (int c = pw; c < kChunks; c += kProducerWarps)
      if (pending & (1u << c)) ptx::mbar_wait(&bars->kv_full[c], (nt - 1) & 1, &never, 100000000ull);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issuer (warp 3, lane 0)
// Issues the PV product of each tile once the softmax has written P^T (and, for a
// segment's first tile, once the epilogue of the previous segment has read O^T).  Each
// value block releases its two chunk slots; the rope slot (P^T) is released after the
// last block.
__device__ void mma_issuer(const Problem& p, unsigned char* sm, Bars* bars, volatile int* abort,
                           uint32_t tmem, Walk wk) {
  const uint32_t kv_base = ptx::smem_addr(sm + kKvOff);
  // MN-major operands: 64-element chunks 16 KB apart (LBO), 8-row groups 1024 B apart
  // (SBO); a K step of 16 key rows is +2048 B.
  const uint64_t dv0 = ptx::sdesc_sw128(kv_base, kKvChunk, 1024);
  const uint64_t dp0 = ptx::sdesc_sw128(kv_base + 8 * kKvChunk, kKvChunk, 1024);
  uint32_t tl = 0, sc = 0;
  Seg s;
  while (next_segment(p, wk, s)) {
    for (int64_t j = s.tile0; j < s.tile1; ++j, ++tl) {
      if (!ptx::mbar_wait(&bars->p_full, tl & 1, abort, p.wait_ns)) goto failed;
      ptx::tc_fence_after();
      const bool first = (j == s.tile0);
      if (first && sc > 0) {
        if (!ptx::mbar_wait(&bars->o_free, (sc - 1) & 1, abort, p.wait_ns)) goto failed;
        ptx::tc_fence_after();
      }
      for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t voff = (2 * m * kKvChunk + ks * 2048) >> 4, poff = (ks * 2048) >> 4;
          ptx::mma_bf16(tmem + 64 * m, dv0 + voff, dp0 + poff, kIdescPV, !(first && ks == 0));
        }
        ptx::mma_commit(&bars->kv_empty[m]);
      }
      ptx::mma_commit(&bars->kv_empty[4]);
      if (j + 1 == s.tile1) ptx::mma_commit(&bars->o_done);
    }
    ++sc;
  }
  return;
failed:
  fail(p, abort);
  {  // every MMA issued so far must finish before TMEM is released (bounded wait)
    volatile int never = 0;
    ptx::mma_commit(&bars->drain);
    ptx::mbar_wait(&bars->drain, 0, &never, 100000000ull);
  }
}

// ------------------------------------------------------------------ softmax (warps 4-11)
// 4x4 transpose of 32-bit words across the four lanes of a quad: afterwards a[b] holds
// what lane (quad base + b) had in a[lane & 3].
__device__ __forceinline__ void quad_transpose(uint32_t (&a)[4]) {
  const int q = threadIdx.x & 3;
  uint32_t x0 = (q & 1) ? a[0] : a[1], x1 = (q & 1) ? a[2] : a[3];
  uint32_t y0 = __shfl_xor_sync(0xffffffffu, x0, 1), y1 = __shfl_xor_sync(0xffffffffu, x1, 1);
  if (q & 1) { a[0] = y0; a[2] = y1; } else { a[1] = y0; a[3] = y1; }
  x0 = (q & 2) ? a[0] : a[2];
  x1 = (q & 2) ? a[1] : a[3];
  y0 = __shfl_xor_sync(0xffffffffu, x0, 2);
  y1 = __shfl_xor_sync(0xffffffffu, x1, 2);
  if (q & 2) { a[0] = y0; a[1] = y1; } else { a[2] = y0; a[3] = y1; }
}

// A lane holds v[i] = value of column i (of 32) at one value dim; the four lanes of a quad
// hold four consecutive dims starting at dst (column 0, first dim of the quad; rows of
// 512).  Stores columns i < nvalid (a multiple of 8, or >= 32; only checked when kMask) as
// bf16 (round to nearest even), four dims of one column per 8-byte store.
template <bool kMask>
__device__ __forceinline__ void store_heads_bf16(uint16_t* dst, const float (&v)[32], int32_t nvalid) {
  const int q = threadIdx.x & 3;
#pragma unroll
  for (int g = 0; g < 4; ++g) {   // heads 8g .. 8g+7: word k = heads (8g+2k, 8g+2k+1)
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = ptx::pack_bf16x2(v[8 * g + 2 * k], v[8 * g + 2 * k + 1]);
    quad_transpose(w);            // w[b] = heads (8g+2q, 8g+2q+1) at dim b
    const int h = 8 * g + 2 * q;
    if (!kMask || h < nvalid) {   // h even and nvalid a multiple of 8: h + 1 is valid too
      *(uint2*)(dst + h * kDv) = make_uint2(__byte_perm(w[0], w[1], 0x5410), __byte_perm(w[2], w[3], 0x5410));
      *(uint2*)(dst + (h + 1) * kDv) = make_uint2(__byte_perm(w[0], w[1], 0x7632), __byte_perm(w[2], w[3], 0x7632));
    }
  }
}

// The fp32 counterpart: four dims of one head per 16-byte store.
__device__ __forceinline__ void store_heads_f32(float* dst, const float (&v)[32]) {
  const int q = threadIdx.x & 3;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = __float_as_uint(v[4 * g + k]);
    quad_transpose(w);            // w[b] = head 4g+q at dim b
    *(uint4*)(dst + (4 * g + q) * kDv) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The fast merge of one query row: out[h][d] = sum_s w_s,h o_s[h][d] over all nseg
// partials, where this CTA's own o (segment jo) is O^T / l read from TMEM (column base
// `ta` holds this thread's 32 heads of value dim `row` in block 0) and the others come
// from the workspace.  Same pairs, order and rounding as merge_token (merge_step), so the
// output is bit-identical whichever CTA merges.  kMB value blocks per round trip.
template <int kMB, bool kMask>
__device__ __forceinline__ void fast_merge(const Problem& p, uint32_t ta, int64_t lrow0,
                                           int32_t ncols, const int32_t* slots, int64_t nseg,
                                           int64_t jo,
                                           uint32_t hb, uint32_t row, const float* inv_l,
                                           const float* wb) {
  uint16_t* dst = p.out + (lrow0 + hb) * kDv + (row & ~3u);
  const int32_t nvalid = ncols - (int32_t)hb;
#pragma unroll 1
  for (int mb0 = 0; mb0 < 4; mb0 += kMB) {
    float own[kMB][32], acc[kMB][32];
#pragma unroll
    for (int b = 0; b < kMB; ++b) {
      uint32_t r16[2][16];
      ptx::tmem_ld16(ta + 64 * (mb0 + b), r16[0]);
      ptx::tmem_ld16(ta + 64 * (mb0 + b) + 16, r16[1]);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        own[b][i] = __fmul_rn(__uint_as_float(r16[i >> 4][i & 15]), inv_l[hb + i]);
        acc[b][i] = 0.f;
      }
    }
#pragma unroll 1
    for (int64_t j0 = 0; j0 < nseg; j0 += 2) {
      const bool two = j0 + 1 < nseg;
      const int64_t j1 = two ? j0 + 1 : j0;
      float v0[kMB][32], v1[kMB][32];
      const float* src0 = p.part_o + ((int64_t)slots[j0] * kHeads + hb) * kDv + row;
      const float* src1 = p.part_o + ((int64_t)slots[j1] * kHeads + hb) * kDv + row;
#pragma unroll
      for (int b = 0; b < kMB; ++b)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v0[b][i] = j0 == jo ? own[b][i] : __ldcg(src0 + i * kDv + 128 * (mb0 + b));
          v1[b][i] = j1 == jo ? own[b][i] : __ldcg(src1 + i * kDv + 128 * (mb0 + b));
        }
#pragma unroll
      for (int b = 0; b < kMB; ++b)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float w0 = wb[j0 * kHeads + hb + i];
          const float w1 = two ? wb[j1 * kHeads + hb + i] : 0.f;
          acc[b][i] = merge_step(acc[b][i], w0, v0[b][i], w1, v1[b][i]);
        }
    }
#pragma unroll
    for (int b = 0; b < kMB; ++b) store_heads_bf16<kMask>(dst + 128 * (mb0 + b), acc[b], nvalid);
  }
}

// kGT: draft tokens per group of 64 columns (1 for 64 heads per token, 8 for 8 heads).
template <int kGT>
__device__ void softmax_role(const Problem& p, unsigned char* sm, Bars* bars, volatile int* abort,
                             uint32_t tmem, Walk wk) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
  const uint32_t half = (warp - kProducerWarps - 1) >> 2;   // heads [32*half, 32*half + 32)
  const uint32_t hb = 32 * half;
  const uint32_t row = 32 * quarter + lane;        // key row of the tile / value dim in a block
  const uint32_t tl_lane = (32u * quarter) << 16;
  float* red = (float*)(sm + kRedOff);             // [2][64 heads][4 quarters]
  float* red2 = (float*)(sm + kRed2Off);           // [64 heads][4 quarters]
  float* inv_l = (float*)(sm + kStatOff);          // [64]
  float* m_s = (float*)(sm + kMOff);                // [2][64] running max per tile parity
  float* alpha_s = (float*)(sm + kAlphaOff);       // [2][64] rescale factors
  float* mprev_s = (float*)(sm + kMPrevOff);       // [64] running max (base 2)
  volatile int* ticket_s = (volatile int*)(sm + kMiscOff + 16);
  unsigned char* p_slot = sm + kKvOff + 8 * kKvChunk;
  const float scale_log2 = p.sm_scale * 1.4426950408889634f;
  const int64_t q_first = p.qo_indptr[0];
  uint32_t tl = 0, sc = 0;
  Seg s;
  SegInfo* si = (SegInfo*)(sm + kSegOff);
  int32_t* slots_s = (int32_t*)(sm + kSlotOff);
  while (next_segment(p, wk, s)) {
    if (threadIdx.x == kFirstSoftmaxThread) {   // read back in the epilogue, after barriers
      si->map = s.map;
      si->nseg = s.nseg;
      si->piece = s.piece;
      si->seg = s.seg;
    }
    float lp[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) lp[i] = 0.f;
    if (quarter == 0) mprev_s[hb + lane] = -INFINITY;
    const int64_t col_off = (s.ri.kv_base - p.kv_indptr[0]) + (s.ri.q_base - q_first);
    for (int64_t j = s.tile0; j < s.tile1; ++j, ++tl) {
      const int64_t c = j * kTile + row;
      const bool in_range = c < s.ri.L;
      const int64_t slot = in_range ? key_slot(p, s.ri, c) : -1;
      // Visibility of key c to the tokens of this thread's 32 columns: one token for 64
      // heads per token; with 8 heads per token, columns hb + 8q .. hb + 8q + 7 belong to
      // draft token kGT * s.t + (hb + 8q) / 8 (bit q of vq; columns past the group's real
      // ones see nothing).
      bool vis = false;
      uint32_t vq = 0u;
      if constexpr (kGT == 1) {
        vis = slot >= 0 && key_visible(p, s.ri, s.t, c);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int32_t col = (int32_t)hb + 8 * q;
          if (slot >= 0 && col < s.ncols && key_visible(p, s.ri, kGT * s.t + (col >> 3), c))
            vq |= 1u << q;
        }
      }
      auto colvis = [&](int i) -> bool {   // column hb + i
        if constexpr (kGT == 1) return vis;
        else return ((vq >> (i >> 3)) & 1u) != 0u;
      };
      if (in_range) {
        if (half == 0 && slot < 0) raise_error(p, kErrBadSlot);
        if (p.dump_slots) {
          if (half == 0) p.dump_slots[col_off + c] = slot;
          if constexpr (kGT == 1) {
            if (half == 0) p.dump_vis[s.ri.m_base + s.t * s.ri.L + c] = vis ? 1 : 0;
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int32_t col = (int32_t)hb + 8 * q;
              if (col < s.ncols)
                p.dump_vis[s.ri.m_base + (kGT * s.t + (col >> 3)) * s.ri.L + c] = (vq >> q) & 1u;
            }
          }
        }
      }
      {
        const bool ok = ptx::mbar_wait(&bars->s_full, tl & 1, abort, p.wait_ns);
        if (ptx::bar_any(kSoftmaxBar, kSoftmaxThreads, !ok)) { if (threadIdx.x == kFirstSoftmaxThread) fail(p, abort); return; }
      }
      ptx::tc_fence_after();
      float x[32];
      {
        // S^T = the three producer warps' partial sums, added in a fixed order
        uint32_t ra[16], rb2[16], rc[16], rd[16];
        const uint32_t ts = tmem + tl_lane + kSCol + hb;
        ptx::tmem_ld16(ts, ra);
        ptx::tmem_ld16(ts + 16, rb2);
        ptx::tmem_ld16(ts + 64, rc);
        ptx::tmem_ld16(ts + 64 + 16, rd);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x[i] = __uint_as_float(ra[i]) + __uint_as_float(rc[i]);
          x[16 + i] = __uint_as_float(rb2[i]) + __uint_as_float(rd[i]);
        }
        ptx::tmem_ld16(ts + 128, ra);
        ptx::tmem_ld16(ts + 128 + 16, rb2);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x[i] = colvis(i) ? (x[i] + __uint_as_float(ra[i])) * scale_log2 : -INFINITY;
          x[16 + i] = colvis(16 + i) ? (x[16 + i] + __uint_as_float(rb2[i])) * scale_log2 : -INFINITY;
        }
      }
      // exact column maximum over the tile's 128 rows, per head: each warp reduces its
      // 32 rows, lane i of the quarter-0 warp of each half folds the four quarters and
      // the running maximum of head hb+i, and every thread reads the results back
      float* rb = red + (tl & 1) * 256;
      {
        // one warp-wide max reduction per head; lane i keeps the one of head hb + i
        float mine = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float r = ptx::warp_max(x[i]);
          mine = lane == i ? r : mine;
        }
        rb[(hb + lane) * 4 + quarter] = mine;
      }
      ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
      float* mw = m_s + (tl & 1) * 64;          // running maximum after this tile
      float* aw = alpha_s + (tl & 1) * 64;      // its rescale factor, 0 < a <= 1
      if (quarter == 0) {
        const float4 t4 = *(const float4*)(rb + (hb + lane) * 4);
        const float mt = fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w));
        const float mo = mprev_s[hb + lane];
        const float mn = fmaxf(mo, mt);
        mw[hb + lane] = mn;
        aw[hb + lane] = (mn > mo) ? ptx::ex2(mo - mn) : 1.f;   // 0 when mo was -inf
        mprev_s[hb + lane] = mn;
      }
      ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
      float m[32];
      bool rescale[2] = {false, false};   // per group of 16 heads
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const float4 mm = *(const float4*)(mw + hb + 4 * i4);
        const float4 aa = *(const float4*)(aw + hb + 4 * i4);
        m[4 * i4] = mm.x; m[4 * i4 + 1] = mm.y; m[4 * i4 + 2] = mm.z; m[4 * i4 + 3] = mm.w;
        lp[4 * i4] *= aa.x; lp[4 * i4 + 1] *= aa.y; lp[4 * i4 + 2] *= aa.z; lp[4 * i4 + 3] *= aa.w;
        rescale[i4 >> 2] |= (aa.x < 1.f) | (aa.y < 1.f) | (aa.z < 1.f) | (aa.w < 1.f);
      }
      // P^T row, heads [hb, hb+32), bf16, over the rope chunk; l from the fp32 P
#pragma unroll
      for (int gq = 0; gq < 4; ++gq) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 8 * gq + 2 * e;
          const float p0 = colvis(i) ? ptx::ex2(x[i] - m[i]) : 0.f;
          const float p1 = colvis(i + 1) ? ptx::ex2(x[i + 1] - m[i + 1]) : 0.f;
          pk[e] = ptx::pack_bf16x2(p0, p1);
          lp[i] += p0;
          lp[i + 1] += p1;
        }
        *(uint4*)(p_slot + swz(row, 4 * half + gq)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      // O^T columns of these heads follow a rising maximum (the previous tile's PV is
      // complete: its MMAs were issued before this tile's S^T was committed).  The
      // decision is warp-uniform: every lane holds the same per-head maxima.
      if (j != s.tile0) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (!rescale[q]) continue;
          {   // all four value blocks in one round trip
            uint32_t o[4][16];
            const uint32_t ta = tmem + tl_lane + hb + 16 * q;
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) ptx::tmem_ld16(ta + 64 * mb, o[mb]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a = aw[hb + 16 * q + i];
#pragma unroll
              for (int mb = 0; mb < 4; ++mb) o[mb][i] = __float_as_uint(__uint_as_float(o[mb][i]) * a);
            }
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) ptx::tmem_st16(ta + 64 * mb, o[mb]);
          }
        }
        ptx::tmem_wait_st();
      }
      ptx::fence_proxy_async();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->p_full);
    }
    // epilogue: l across the 128 rows, normalised O^T, lse
    red2[(hb + lane) * 4 + quarter] = warp_transpose_reduce<false>(lp);
    ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
    const int64_t nseg = si->nseg;
    const int32_t seg = si->seg, piece = si->piece;
    {   // the column group's partial slots, read by the merge paths after later barriers
      const int t = (int)threadIdx.x - kFirstSoftmaxThread;
      if (t < nseg) slots_s[t] = (int32_t)si->map.slot(t);
    }
    if (quarter == 0) {  // lane i of the quarter-0 warp of each half finalises head hb + i
      const float4 t4 = *(const float4*)(red2 + (hb + lane) * 4);
      const float l = (t4.x + t4.y) + (t4.z + t4.w);
      inv_l[hb + lane] = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (mprev_s[hb + lane] + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      if (nseg == 1) {
        if ((int32_t)(hb + lane) < s.ncols) p.lse[s.r * p.heads + hb + lane] = lse;
      } else {
        p.part_lse[seg * kHeads + hb + lane] = lse;
      }
    }
    // Fast merge: when every other segment of the token has already taken its ticket,
    // their partials are published and this CTA is the last; it merges them with its own
    // output straight from TMEM, without writing its partial or taking a ticket.  Merge
    // mode 1 never takes this path; mode 2 makes the CTA with the last piece wait for the
    // others (bounded, then the ticket path), so that the path is taken wherever it can be.
    if (nseg > 1 && threadIdx.x == kFirstSoftmaxThread) {
      const int* done = p.tok_done + (s.r - q_first);
      int fast = 0;
      if (p.merge_mode != 1 && nseg <= kMergeGroup) {
        fast = ptx::ld_acquire_gpu(done) == nseg - 1;
        if (!fast && p.merge_mode == 2 && piece == nseg - 1) {
          const uint64_t t0 = ptx::globaltimer();
          while (!(fast = ptx::ld_acquire_gpu(done) == nseg - 1) &&
                 ptx::globaltimer() - t0 < kMergeWaitNs)
            __nanosleep(256);
        }
      }
      *ticket_s = fast;
    }
    {
      const bool ok = ptx::mbar_wait(&bars->o_done, sc & 1, abort, p.wait_ns);
      if (ptx::bar_any(kSoftmaxBar, kSoftmaxThreads, !ok)) { if (threadIdx.x == kFirstSoftmaxThread) fail(p, abort); return; }
    }
    ptx::tc_fence_after();
    if (nseg > 1 && *ticket_s) {
      float* wb = (float*)(sm + kWOff);
      const int t = (int)threadIdx.x - kFirstSoftmaxThread;
      if (t == 0) atomicAdd(&p.hdr->merges_tmem, 1u);
      merge_stats(p, p.lse + s.r * p.heads, s.ncols, slots_s, nseg, t, m_s);
      ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
      merge_weights(p, slots_s, nseg, t, 0, m_s, wb);
      ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
      const int64_t jo = piece;          // this CTA's segment among the token's
      fast_merge<1, (kGT > 1)>(p, tmem + tl_lane + hb, s.r * p.heads, s.ncols, slots_s, nseg, jo,
                               hb, row, inv_l, wb);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->o_free);
      ++sc;
      continue;
    }
    if (nseg == 1) {
      // the whole token sat in this CTA: its normalised output is final (bf16, RNE)
      uint16_t* dst = p.out + (s.r * p.heads + hb) * kDv + (row & ~3u);
      const int32_t nvalid = s.ncols - (int32_t)hb;   // of this thread's 32 columns
#pragma unroll
      for (int mp = 0; mp < 4; mp += 2) {   // two value blocks (64 values) per TMEM round trip
        uint32_t r16[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) ptx::tmem_ld16(tmem + tl_lane + 64 * (mp + (q >> 1)) + hb + 16 * (q & 1), r16[q]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r16[2 * b + (i >> 4)][i & 15]) * inv_l[hb + i];
          store_heads_bf16<(kGT > 1)>(dst + 128 * (mp + b), v, nvalid);
        }
      }
    } else {
      float* dst = p.part_o + (seg * kHeads + hb) * kDv + (row & ~3u);
#pragma unroll
      for (int mp = 0; mp < 4; mp += 2) {
        uint32_t r16[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) ptx::tmem_ld16(tmem + tl_lane + 64 * (mp + (q >> 1)) + hb + 16 * (q & 1), r16[q]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(__uint_as_float(r16[2 * b + (i >> 4)][i & 15]), inv_l[hb + i]);
          store_heads_f32(dst + 128 * (mp + b), v);
        }
      }
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&bars->o_free);
    if (nseg > 1) {
      // Ticket: the CTA that finishes the token's last segment merges its partials.
      // Writers publish (fence) before the ticket; the merger fences after it.  With more
      // than kMergeGroup pieces the merge has two levels: the last piece of each group of
      // kMergeFan merges the group into the group's first slot, then takes the token's
      // ticket, and the last group merges the group results.
      const bool two_level = nseg > kMergeGroup;
      const int32_t grp = piece / kMergeFan;
      const int32_t gsz = min((int32_t)kMergeFan, (int32_t)nseg - kMergeFan * grp);
      __threadfence();
      ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
      if (threadIdx.x == kFirstSoftmaxThread)
        *ticket_s = two_level ? atomicAdd(p.grp_done + (s.r - q_first) * kMergeFan + grp, 1)
                              : atomicAdd(p.tok_done + (s.r - q_first), 1);
      ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
      bool last = *ticket_s == (two_level ? gsz - 1 : nseg - 1);
      int64_t nmerge = nseg;
      if (last && two_level) {
        __threadfence();
        merge_token<kSoftmaxThreads, true>(p, 0, kHeads, slots_s + kMergeFan * grp, gsz,
                                           kFirstSoftmaxThread, kSoftmaxBar, m_s,
                                           (float*)(sm + kWOff), slots_s[kMergeFan * grp],
                                           alpha_s);
        __threadfence();
        ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
        if (threadIdx.x == kFirstSoftmaxThread) {
          *ticket_s = atomicAdd(p.tok_done + (s.r - q_first), 1);
          // the group results sit in each group's first slot
          for (int i = 1; i * kMergeFan < nseg; ++i) slots_s[i] = slots_s[kMergeFan * i];
        }
        ptx::bar_sync(kSoftmaxBar, kSoftmaxThreads);
        nmerge = (nseg + kMergeFan - 1) / kMergeFan;
        last = *ticket_s == nmerge - 1;
      }
      if (last) {
        __threadfence();
        if (threadIdx.x == kFirstSoftmaxThread) atomicAdd(&p.hdr->merges_ws, 1u);
        merge_token<kSoftmaxThreads>(p, s.r * p.heads, s.ncols, slots_s, nmerge, kFirstSoftmaxThread, kSoftmaxBar, m_s,
                                     (float*)(sm + kWOff));
      }
    }
    ++sc;
  }
}

// kGT: draft tokens per group of 64 columns (1: 64 heads per token; 8: 8 heads per token).
template <int kGT>
__global__ void __launch_bounds__(kThreads, 1)
    split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                 const Problem p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* bars = (Bars*)(sm + kBarOff);
  uint32_t* tmem_slot = (uint32_t*)(sm + kMiscOff);
  volatile int* abort = (volatile int*)(sm + kMiscOff + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    ptx::mbar_init(&bars->q_empty, kProducerWarps);
    ptx::mbar_init(&bars->s_full, kProducerWarps);
    ptx::mbar_init(&bars->p_full, kSoftmaxThreads);
    ptx::mbar_init(&bars->o_done, 1);
    ptx::mbar_init(&bars->o_free, kSoftmaxThreads);
    ptx::mbar_init(&bars->drain, 1);
    for (int g = 0; g < 5; ++g) ptx::mbar_init(&bars->kv_empty[g], 1);
    for (int w = 0; w < kProducerWarps; ++w) ptx::mbar_init(&bars->drain_p[w], 1);
    for (int c = 0; c < kChunks; ++c) ptx::mbar_init(&bars->kv_full[c], 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarps) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The prologue above overlaps the planner; its results are read only after it is done.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  Walk wk;
  wk.W = p.lanes;
  wk.g = (int32_t)blockIdx.x / wk.W;
  wk.lane = (int32_t)blockIdx.x - wk.g * wk.W;
  const int64_t C = p.hdr->capacity;
  wk.u = (int64_t)wk.g * C;
  wk.u_end = min(p.hdr->total_units, wk.u + C);
  wk.J = wk.g < p.hdr->groups ? p.grp_job[wk.g] : 0;

  if (wk.g >= p.hdr->groups || wk.u >= wk.u_end) {
    // no work for this CTA
  } else if (warp < kProducerWarps) {
    producer(p, &tm_q, &tm_kv, sm, bars, abort, tmem, wk);
  } else if (warp == kProducerWarps) {
    if (lane == 0) mma_issuer(p, sm, bars, abort, tmem, wk);
    __syncwarp();
  } else {
    softmax_role<kGT>(p, sm, bars, abort, tmem, wk);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kProducerWarps) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
  }
  return fn;
}

// 2-D bf16 view [rows][576] with 1152-byte rows, box [box_rows][64], 128B swizzle.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDqk, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kRowBytes};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

int split_tile() { return tc::kTile; }

cudaError_t split_prepare() {
  if (!tc::encode_fn()) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(tc::split_kernel<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc::split_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc::kSmemBytes);
}

int launch_split(const Problem& p, int grid, cudaStream_t stream) {
  if (p.total_q <= 0) return 0;
  CUtensorMap tm_q;
  // q as [total_q * heads][576]: 64 rows are one token's 64 heads or 8 tokens' 8 heads
  if (!tc::encode_rows(&tm_q, p.q, p.total_q * p.heads, 64)) return -1;
  // the cache as [num_slots][576]: one 128-row box per chunk of a run of consecutive slots
  CUtensorMap tm_kv;
  if (!tc::encode_rows(&tm_kv, p.kv, p.num_slots, tc::kTile)) return -1;
  // Programmatic dependent launch: the kernel's prologue may overlap the planner.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(tc::kThreads);
  cfg.dynamicSmemBytes = tc::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = p.group_tokens == 1
                            ? cudaLaunchKernelEx(&cfg, tc::split_kernel<1>, tm_q, tm_kv, p)
                            : cudaLaunchKernelEx(&cfg, tc::split_kernel<8>, tm_q, tm_kv, p);
  return e == cudaSuccess ? 0 : -1;
}

}  // namespace mtv
