// The persistent decode megakernel: an on-GPU interpreter of a static task DAG.
//
// One CTA per SM walks a static queue of 64-byte task descriptors.  Before a
// task runs, one thread waits (acquire) until the task's counter reaches
// epoch * remaining_deps; after it runs, one warp adds 1 (release) to the
// counter of every dependent.  There is no grid-wide barrier between ops:
// each tile starts when its own producers finish ("Megakernels",
// runhoid.com, "Hoid's approach to megakernels" and Fig. 5; the edge array
// and descriptor of "mega kernel initial", 1y33.com).  Because weights never
// change during a step, a producer warp streams the weights (and the cached
// KV rows) of the CTA's upcoming tasks into a shared-memory ring with bulk
// async copies before their dependencies resolve ("Megakernels", the note
// that managing dependencies by hand allows prefetching any input, and
// Fig. 3 on overlapping one kernel's loads with another's compute).
//
// Warp roles: warps 0-7 consume (compute), warp 8 produces (bulk copies).
// Task bodies:
//   GEMV: one output-column tile (or one K split of a row block), on CUDA
//     cores for one or two activation rows, on the tensor cores from three
//     (up to eight, rows past B zero); epilogues
//     RMS_NORM_INPUT, SILU_MUL, ADD_RESIDUAL, ARGMAX_EPI ("mega kernel
//     initial", lowering part: the fusions are epilogue flags of one GEMV
//     pass, and the final norm is fused into the lm_head GEMV).
//   ATTENTION_APPEND: RoPE on k, bf16 k/v written at row pos (OpId table).
//   ATTENTION_PARTIAL: online softmax over one KV chunk -> (m, l, o).
//   ATTENTION_COMBINE: log-sum-exp merge of the partials -> O.
//   MEMCPY: embedding row gather.   SAMPLE: argmax over the tile pairs.
// Every wait is bounded by timeout_ns; on expiry the CTA records an error
// in the status word, raises the abort flag that all CTAs poll, lets its
// in-flight copies land and exits.  Nothing traps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>

#include "kernel.h"
#include "ptx.cuh"

namespace mk {

using namespace ptx;

// ------------------------------------------------------------------ status
__device__ __forceinline__ bool aborted(const KParams& p) {
  return ld_relaxed(p.status + kStatusAbort) != 0;
}

__device__ void raise_error(const KParams& p, int code, int task) {
  if (atomicCAS(p.status + kStatusCode, 0, code) == 0) atomicExch(p.status + kStatusTask, task);
  atomicExch(p.status + kStatusAbort, 1);
}

// Bounded wait on an mbarrier phase.  Returns false on abort or timeout
// (and records the timeout); the caller then continues without the data.
__device__ bool bar_wait(const KParams& p, uint64_t* bar, uint32_t parity, int task, bool honor_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (honor_abort && aborted(p)) return false;
      if (globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, MK_DEV_RING_TIMEOUT, task);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ task order
struct Seq {
  int i = 0, hi = 0, lvl = 0;
};

__device__ __forceinline__ void seq_init(Seq& s, const KParams& p) {
  if (p.mode == MK_MODE_MEGA) {
    s.i = p.queue_off[blockIdx.x];
    s.hi = p.queue_off[blockIdx.x + 1];
  } else if (p.mode == MK_MODE_LEVELS) {
    s.lvl = 0;
    s.i = p.level_off[0] + blockIdx.x;
    s.hi = p.level_off[1];
  } else {
    s.i = 0;
    s.hi = 1;
  }
}

__device__ __forceinline__ bool seq_next(Seq& s, const KParams& p, int& task, int& lvl) {
  if (p.mode == MK_MODE_MEGA) {
    if (s.i >= s.hi) return false;
    task = p.queue[s.i++];
    lvl = 0;
    return true;
  }
  if (p.mode == MK_MODE_LEVELS) {
    while (s.i >= s.hi) {
      if (++s.lvl >= p.num_levels) return false;
      s.i = p.level_off[s.lvl] + blockIdx.x;
      s.hi = p.level_off[s.lvl + 1];
    }
    task = p.level_tasks[s.i];
    s.i += gridDim.x;
    lvl = s.lvl;
    return true;
  }
  if (s.i >= s.hi) return false;
  s.i = s.hi;
  task = p.first_task + blockIdx.x;
  lvl = 0;
  return true;
}

// ------------------------------------------------------------------ GEMV plan
// A GEMV tile streams its weight rows [c0, c0+cn) (and the matching up rows
// for SILU_MUL) in k-segments of KS columns.  A ring slot holds rs whole
// row-segments.  Consumer warp w reads columns [wcol*KS/WCOL, ...) of rows
// r = wrow (mod WROW) of each slot, with x in registers (B*NV*8 floats).
struct GemvGeom {
  int B, BT, K, n, c0, cn, seg, KS, nks, WCOL, WROW, lgW, NV, rs, RG;
};

__device__ __forceinline__ void gemv_geom(const mk_task_descriptor& d, GemvGeom& g) {
  g.B = d.m;
  g.BT = g.B == 1 ? 1 : g.B == 2 ? 2 : 8;  // instantiated batch width
  g.K = d.k;
  g.n = d.n;
  g.c0 = (int)d.reserved[0];
  g.cn = (int)d.reserved[1];
  g.seg = (d.flags & MK_F_SILU_MUL) ? 2 : 1;
  const int u = g.K / 256;
  g.KS = 256; g.nks = u; g.WCOL = 1; g.WROW = 8; g.NV = 1;
  for (int q = 1; q <= u; ++q) {
    if (u % q) continue;
    const int uk = u / q;
    if (uk > 64) continue;
    int wcol = 1;
    while (wcol < 8 && (uk % (wcol * 2)) == 0) wcol *= 2;
    const int nv = uk / wcol;
    if (g.BT == 1 ? (nv == 3 || nv == 5 || nv == 6 || nv > 7) : nv > 1) continue;
    g.KS = uk * 256; g.nks = q; g.WCOL = wcol; g.WROW = 8 / wcol; g.NV = nv;
    break;
  }
  g.lgW = g.WROW == 8 ? 3 : g.WROW == 4 ? 2 : g.WROW == 2 ? 1 : 0;
  // whole rows per slot, no more than the warps cover ((8 / NV) rows of
  // every warp row: at NV = 7 and one warp column, 8 of the 9 that fit)
  g.rs = min(kStageElems / g.KS, (8 / g.NV) * g.WROW);
  int rg = kSlotFloats / (g.seg * g.BT * g.WCOL);
  rg = min(rg, kAccFloats / (g.seg * g.BT));
  g.RG = min(rg, g.cn);
}

// Tensor-core tile plan (three or more rows): row groups of RG rows (the TMA box).  The
// MMA's N holds the group's rows of every segment (gate and up rows stacked
// for SILU_MUL): segment sg occupies rows [sg * Nr, sg * Nr + RG) of the
// weight tile and accumulator columns [sg * Nr, ...), N = seg * Nr <= 256.
// A K-split tile (kv_len = j | S << 16, S >= 2) covers K columns [k0, k0 +
// kn) only; otherwise k0 = 0, kn = K.  nkb K blocks of 64 columns per ring
// slot, nkr K ranges.
struct TcGeom {
  int RG, Nr, N, nkb, nkr, seg, K, k0, kn, S, j;
};

__device__ __forceinline__ void tc_geom(int rows, const mk_task_descriptor& d, TcGeom& t) {
  t.RG = rows;
  t.seg = (d.flags & MK_F_SILU_MUL) ? 2 : 1;
  t.Nr = t.seg == 2 ? (t.RG + 7) & ~7 : (t.RG + 15) & ~15;
  t.N = t.seg * t.Nr;
  t.K = d.k;
  t.S = (int)((uint32_t)d.kv_len >> 16);
  if (t.S >= 2) {
    t.j = d.kv_len & 0xFFFF;
    t.k0 = (int)(d.reserved[3] & 0xFFFFu);
    t.kn = (int)(d.reserved[3] >> 16);
  } else {
    t.S = 1;
    t.j = 0;
    t.k0 = 0;
    t.kn = d.k;
  }
  const int nkbt = t.kn / 64;
  t.nkb = 4;  // K blocks per slot: the staged activations of 4 blocks fill one 12 KB tile
  while (t.nkb > 1 && (t.nkb * t.N * 128 > kStageBytes || nkbt % t.nkb)) t.nkb >>= 1;
  t.nkr = nkbt / t.nkb;
}

// ------------------------------------------------------------------ PARTIAL plan
// A chunk step of T tokens per sequence (T = 1: a decode step): token t
// sits at pos + t and sees keys 0 .. pos + t.  The chunks split the keys of
// the last token, [0, pos + T); keys below pos are cached rows of earlier
// steps (streamed through the ring), keys from pos on are this step's rows,
// taken from qkv.
struct PartGeom {
  int s, g, Hkv, T, c, P, slot, D, Hq, G, cap, pos, j0, j1, jst, nb0, nn, R, nstage, nblk;
  bool has_new;
  bool bad;
};

// Tensor-core partials: the chunk's cached keys in blocks of kKeyBlock, each
// block's K rows brought by 2-D TMA in the 128-byte swizzle (boxes of 64
// dims x kKeyBlock rows) and its V rows by a bulk copy; used when the K
// cache has a tensor map, the query rows (T tokens x G heads) number at most
// four and the chunk holds at least kMinTcBlocks blocks of cached keys (for
// short chunks the tensor-core round trips cost more than the CUDA-core
// partial saves: measured on 129- and 216-key chunks).
constexpr int kKeyBlock = kKeyBlockRows;
constexpr int kMinTcBlocks = 4;

__device__ __forceinline__ bool tc_partial(const mk_task_descriptor& d, int tm_rows, int nblk) {
  const int Hkv = (int)(d.reserved[2] & 0xFFFFu), T = (int)(d.reserved[2] >> 16) + 1;
  return tm_rows == kKeyBlock && (d.k / Hkv) * T <= 4 && nblk >= kMinTcBlocks;
}

__device__ __forceinline__ void part_geom(const int32_t* state, const mk_task_descriptor& d, PartGeom& q) {
  q.s = (int)d.reserved[0];
  q.g = (int)d.reserved[1];
  q.Hkv = (int)(d.reserved[2] & 0xFFFFu);
  q.T = (int)(d.reserved[2] >> 16) + 1;
  q.c = (int)(d.reserved[3] & 0xFFFFu);
  q.P = (int)(d.reserved[3] >> 16);
  q.slot = (int)d.reserved[4] + q.c;
  q.D = d.n;
  q.Hq = d.k;
  q.G = q.Hq / q.Hkv;
  q.cap = d.kv_len;
  q.pos = ld_relaxed(state + 2 * q.s + 1);
  q.bad = q.pos < 0 || q.pos + q.T > q.cap;
  if (q.bad) {
    q.j0 = q.j1 = q.jst = q.nb0 = q.nn = 0;
    q.nstage = 0;
    q.nblk = 0;
    q.R = 1;
    q.has_new = false;
    return;
  }
  const int L = q.pos + q.T;
  const int e = (L + q.P - 1) / q.P;
  q.j0 = min(q.c * e, L);
  q.j1 = min(q.j0 + e, L);
  q.jst = min(q.j1, q.pos);
  q.nb0 = max(q.j0, q.pos);           // this step's keys in the chunk: [nb0, j1)
  q.nn = max(0, q.j1 - q.nb0);
  q.R = (kStageBytes / 4) / q.D;  // rows of K and of V per slot
  const int nrows = max(0, q.jst - q.j0);
  q.nstage = (nrows + q.R - 1) / q.R;
  q.nblk = (nrows + kKeyBlock - 1) / kKeyBlock;
  q.has_new = q.nn > 0;
}

// ------------------------------------------------------------------ control block
// Shared-memory words and mbarriers after the ring's full/empty barriers.
struct TcCtl {
  volatile int32_t run;            // consumers: 1 while the current task may run
  uint32_t tmem;                   // tensor-memory base address
  volatile int32_t mb_task;        // mailbox to the MMA warp: task index, -1 = no more tasks
  volatile uint32_t mb_slot;       //   ring slot and phase parity of its first weight / key slot
  volatile uint32_t mb_phase;
  volatile uint32_t mb_nblk;       //   split-KV partial: blocks of 128 cached keys
  volatile uint32_t mb_qt;         //   split-KV partial: shared address of the query tile
  uint32_t pad;
  uint64_t mma_bar[2];             // GEMV: commit of each K range (alternating)
  uint64_t x_full[2];              // GEMV: a K range's activations are staged (one arrival per consumer warp)
  uint64_t acc_full;               // GEMV: commit after a row group's last MMA
  uint64_t acc_empty;              // GEMV: the consumers have read the accumulators
  uint64_t task_go;                // the mailbox holds a task
  uint64_t s_full[2];              // partial: commit of a key block's scores (alternating buffers)
  uint64_t s_empty[2];             // partial: the softmax warps have read a score buffer
  uint64_t q_full;                 // partial: the query tile is staged (one arrival per consumer warp)
  uint64_t p_full[2];              // partial: a block's probabilities are written (softmax warps)
  uint64_t p_empty[2];             // partial: the P V warps have read them
  uint64_t pad2;
};
static_assert(sizeof(TcCtl) == 168, "control block layout");
constexpr int kCtlBytes = 192;

// ------------------------------------------------------------------ task records
// A warp of the producer group walks the CTA's task order ahead of the
// consumers and leaves, per task, its descriptor with everything the
// descriptor only names resolved: buffer pointers, mirrors, the dependency
// plan's ranges and first entries.  The consumers then start a task from
// shared memory instead of a chain of dependent global loads (queue entry,
// descriptor, buffer table, plan offsets).  kRecs entries, each guarded by
// a full and an empty mbarrier.
enum { kPIn0 = 0, kPIn1 = 1, kPIn2 = 2, kPOut = 3, kMirX = 4, kMirAux = 5, kMirOut = 6, kPPairs = 7 };
struct TaskRec {
  mk_task_descriptor d;
  uint64_t ptr[8];     // in_buf[0..2] and out_buf resolved; mirrors of in_buf[0], in_buf[2], out_buf;
                       // the argmax pairs of a GEMV with ARGMAX_EPI (null where absent)
  int32_t task, lvl;   // task index (-1: no more tasks), level (LEVELS)
  uint32_t w0, nw;     // MEGA: wait entries [w0, w0 + nw)
  uint32_t s0, ns;     //   and signal entries [s0, s0 + ns)
  uint2 wi[4];         //   the first four wait entries
  uint32_t si[4];      //   the first four signal entries
  int32_t tm_rows;     // rows of in_buf[1]'s tensor map box (0: none)
  uint32_t pad[13];
};
static_assert(sizeof(TaskRec) == kRecBytes, "task record layout");

// ------------------------------------------------------------------ ring position
// Slot index and mbarrier phase parity of the next ring use, advanced
// without division (this runs once per slot in every warp).
struct RingPos {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void advance(int nst) {
    if (++slot == (uint32_t)nst) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// ------------------------------------------------------------------ producer
// Paced L2 warm-up at one or two rows.  During the attention phase HBM
// idles while the partials and the combine run.  After a partial's slots
// the copy thread plans the weight tiles of the next two GEMV tasks whose
// records are made (the output projection and the gate and up projection),
// up to kL2AheadBytes beyond what the ring will hold.  Once the consumers
// have released the partial's first slot (its query and new key are
// staged), it prefetches one kStageBytes chunk at a time, at most one per
// kL2GapNs (about 1.5 times this SM's share of HBM), and only while it
// waits for a free ring slot.  A burst of prefetches queued in front of the
// polls of the partials and the combine and delayed them; so did a pace
// much faster than this one, while a much slower one ran on into the
// GEMVs' own streaming.
constexpr uint32_t kL2AheadBytes = 768u * 1024u;
constexpr uint32_t kL2GapNs = 500u;

struct L2Warm {
  const char* src[3];  // the ranges left, current first
  uint32_t left[3];
  const uint64_t* start;  // its phase start_par opens the warm-up (null: open)
  uint32_t start_par;
  uint64_t next;  // globaltimer of the earliest next prefetch
};

__device__ __forceinline__ void l2_plan(const TaskRec* recs, uint64_t* rfull, uint32_t k, L2Warm& w) {
  uint32_t budget = kL2AheadBytes + (uint32_t)kMaxStages * kStageBytes;
  w.left[0] = w.left[1] = w.left[2] = 0u;
  w.next = 0;
  int gemvs = 0, n = 0;
  for (uint32_t a = 1; a < (uint32_t)kRecs && budget > 0 && gemvs < 2; ++a) {
    const uint32_t kk = k + a, e = kk & (kRecs - 1);
    if (!mbar_test_wait(&rfull[e], (kk / kRecs) & 1u)) break;  // not made yet
    const TaskRec* r = recs + e;
    if (r->task < 0) break;
    const mk_task_descriptor& d = r->d;
    if (d.op_id != MK_OP_GEMV || d.config_id != 0) continue;
    ++gemvs;
    const int seg = (d.flags & MK_F_SILU_MUL) ? 2 : 1;
    const char* W = reinterpret_cast<const char*>(r->ptr[kPIn1]);
    const uint64_t rowb = (uint64_t)d.k * 2u;
    for (int sg = 0; sg < seg && budget > 0 && n < 3; ++sg, ++n) {
      const uint32_t len = (uint32_t)min((uint64_t)d.reserved[1] * rowb, (uint64_t)budget);
      const char* src = W + ((uint64_t)(sg ? d.n : 0) + d.reserved[0]) * rowb;
      // appended at position n (0..2) through selects: no run-time array index
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (q == n) {
          w.src[q] = src;
          w.left[q] = len;
        }
      budget -= len;
    }
  }
}

// One paced prefetch of the plan, if it is open and due.
__device__ __forceinline__ void l2_step(L2Warm& w) {
  if (w.left[0] == 0u) return;
  if (w.start) {
    if (!mbar_test_wait(const_cast<uint64_t*>(w.start), w.start_par)) return;
    w.start = nullptr;
  }
  const uint64_t now = globaltimer();
  if (now < w.next) return;
  const uint32_t c = min(w.left[0], kStageBytes);
  prefetch_l2(w.src[0], c);
  w.src[0] += c;
  w.left[0] -= c;
  if (w.left[0] == 0u) {  // next range
    w.src[0] = w.src[1];
    w.left[0] = w.left[1];
    w.src[1] = w.src[2];
    w.left[1] = w.left[2];
    w.left[2] = 0u;
  }
  w.next = now + kL2GapNs;
}

// Claim the next ring slot once the consumers have freed it and announce the
// bytes the coming copies will deliver; *fb receives the slot's full
// barrier.  Null on abort or timeout.
__device__ __forceinline__ uint8_t* produce_slot(const KParams& p, uint8_t* ring, uint64_t* full, uint64_t* empty,
                                                 RingPos& rp, uint32_t& issued, int task, uint32_t bytes,
                                                 uint64_t** fb, L2Warm* w = nullptr) {
  const uint32_t slot = rp.slot;
  if (w && w->left[0] != 0u) {  // a warm-up is planned: step it while the slot is busy
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1; !mbar_test_wait(&empty[slot], rp.phase ^ 1u); ++it) {
      l2_step(*w);
      if ((it & 255u) == 0) {
        if (aborted(p)) return nullptr;
        if (globaltimer() - t0 > p.timeout_ns) {
          raise_error(p, MK_DEV_RING_TIMEOUT, task);
          return nullptr;
        }
      }
    }
  } else if (!bar_wait(p, &empty[slot], rp.phase ^ 1u, task, true)) {
    return nullptr;
  }
  if (w && w->start == &empty[slot]) w->start = nullptr;  // reusing the slot: the opening phase completed
  mbar_arrive_expect_tx(&full[slot], bytes);
  rp.advance(p.nstages);
  ++issued;
  *fb = &full[slot];
  return ring + (size_t)slot * kStageBytes;
}

// Producer (one thread): walks the task records and streams every task's
// operand tiles into the ring, at most nstages slots ahead of the consumers.
template <int BCLASS>
__device__ void producer(const KParams& p, uint8_t* ring, uint64_t* full, uint64_t* empty, const TaskRec* recs,
                         uint64_t* rfull, uint64_t* rempty) {
  if ((threadIdx.x & 31) != 0) return;
  const uint64_t pol = policy_evict_first();
  const int nst = p.nstages;
  RingPos rp;
  uint32_t issued = 0;
  bool stop = false;
  const int32_t* state = static_cast<const int32_t*>(p.bufs[MK_BUF_STATE]);
  __shared__ L2Warm warm;  // the copy thread's plan (its registers are few)
  L2Warm* wp = nullptr;
  if (BCLASS == 0) {
    warm.left[0] = warm.left[1] = warm.left[2] = 0u;
    warm.start = nullptr;
    warm.next = 0;
    wp = &warm;
  }
  for (uint32_t k = 0; !stop; ++k) {
    const uint32_t e = k & (kRecs - 1);
    const TaskRec* r = recs + e;
    if (!bar_wait(p, &rfull[e], (k / kRecs) & 1u, -1, true)) break;
    const int task = r->task;
    if (task < 0) break;
    const mk_task_descriptor& d = r->d;
    const int tmr = r->tm_rows;
    if (d.op_id == MK_OP_GEMV && d.config_id == 1 && tmr > 0) {
      // tensor-core tile: per K range and segment one slot of nkb K blocks,
      // each a TMA box of 64 columns x RG rows in the 128-byte swizzle
      TcGeom T;
      tc_geom(tmr, d, T);
      const uint8_t* tmap = p.tmaps + (size_t)d.in_buf[1] * kTmapBytes;
      const int c0 = (int)d.reserved[0], cn = (int)d.reserved[1];
      if (d.flags & MK_F_RMS_NORM_INPUT) prefetch_l2(reinterpret_cast<const void*>(r->ptr[kPIn2]), (uint32_t)d.k * 2u);
      // one slot per K range: nkb K blocks of every segment's RG rows
      for (int g0 = 0; g0 < cn && !stop; g0 += T.RG)
        for (int kr = 0; kr < T.nkr && !stop; ++kr) {
          uint64_t* fb;
          uint8_t* dst = produce_slot(p, ring, full, empty, rp, issued, task,
                                      (uint32_t)(T.nkb * T.seg * T.RG * 128), &fb);
          if (!dst) { stop = true; break; }
          for (int kb = 0; kb < T.nkb; ++kb)
            for (int sg = 0; sg < T.seg; ++sg)
              tma_load_2d(dst + (size_t)(kb * T.N + sg * T.Nr) * 128, tmap, T.k0 + (kr * T.nkb + kb) * 64,
                          (sg ? d.n : 0) + c0 + g0, fb, pol);
        }
    } else if (d.op_id == MK_OP_GEMV) {
      GemvGeom G;
      gemv_geom(d, G);
      const uint16_t* W = reinterpret_cast<const uint16_t*>(r->ptr[kPIn1]);
      // the norm gain is read right after the dependency wait: warm the L2
      if (d.flags & MK_F_RMS_NORM_INPUT) prefetch_l2(reinterpret_cast<const void*>(r->ptr[kPIn2]), (uint32_t)G.K * 2u);
      for (int g0 = 0; g0 < G.cn && !stop; g0 += G.RG) {
        const int rows_g = min(G.RG, G.cn - g0);
        for (int ks = 0; ks < G.nks && !stop; ++ks)
          for (int sg = 0; sg < G.seg && !stop; ++sg)
            for (int r0 = 0; r0 < rows_g; r0 += G.rs) {
              const int nr = min(G.rs, rows_g - r0);
              const uint32_t bytes = (uint32_t)nr * G.KS * 2u;
              uint64_t* fb;
              uint8_t* dst = produce_slot(p, ring, full, empty, rp, issued, task, bytes, &fb, wp);
              if (!dst) { stop = true; break; }
              const int64_t row = (int64_t)(sg ? G.n : 0) + G.c0 + g0 + r0;
              const uint16_t* src = W + row * G.K + (int64_t)ks * G.KS;
              if (G.nks == 1) {
                bulk_g2s(dst, src, bytes, fb, pol);
              } else {
                for (int rr = 0; rr < nr; ++rr)
                  bulk_g2s(dst + (size_t)rr * G.KS * 2, src + (int64_t)rr * G.K, (uint32_t)G.KS * 2u, fb, pol);
              }
            }
      }
    } else if (d.op_id == MK_OP_ATTENTION_PARTIAL) {
      PartGeom q;
      part_geom(state, d, q);
      const uint16_t* Kc = reinterpret_cast<const uint16_t*>(r->ptr[kPIn1]);
      const uint16_t* Vc = reinterpret_cast<const uint16_t*>(r->ptr[kPIn2]);
      const int64_t rowbase = ((int64_t)q.s * q.Hkv + q.g) * q.cap;
      if (!q.bad && (p.rope_half * 4) % 16 == 0) {  // the RoPE rows of pos
        prefetch_l2(p.rope_cos + (size_t)q.pos * p.rope_half, (uint32_t)p.rope_half * 4u);
        prefetch_l2(p.rope_sin + (size_t)q.pos * p.rope_half, (uint32_t)p.rope_half * 4u);
      }
      if (tc_partial(d, tmr, q.nblk)) {
        // per block of kKeyBlock cached keys: the K rows through the tensor
        // map (D / 64 boxes), then the V rows (D = 128: a slot each; D = 64:
        // K in the first half of one slot, V in the second)
        const uint8_t* kmap = p.tmaps + (size_t)d.in_buf[1] * kTmapBytes;
        const uint32_t kbytes = (uint32_t)(q.D / 64) * kKeyBlock * 128u;
        for (int b = 0; b < q.nblk && !stop; ++b) {
          const int j = q.j0 + b * kKeyBlock;
          const int nr = min(kKeyBlock, q.jst - j);
          const uint32_t vbytes = (uint32_t)nr * q.D * 2u;
          uint64_t* fb;
          uint8_t* dst = produce_slot(p, ring, full, empty, rp, issued, task, q.D == 128 ? kbytes : kbytes + vbytes, &fb);
          if (!dst) { stop = true; break; }
          for (int kb = 0; kb < q.D / 64; ++kb)
            tma_load_2d(dst + (size_t)kb * kKeyBlock * 128, kmap, kb * 64, (int32_t)(rowbase + j), fb, pol);
          if (q.D == 128) {
            dst = produce_slot(p, ring, full, empty, rp, issued, task, vbytes, &fb);
            if (!dst) { stop = true; break; }
            bulk_g2s(dst, Vc + (rowbase + j) * q.D, vbytes, fb, pol);
          } else {
            bulk_g2s(dst + kbytes, Vc + (rowbase + j) * q.D, vbytes, fb, pol);
          }
        }
        mbar_arrive(&rempty[e]);
        continue;
      }
      const uint32_t s0 = rp.slot, ph0 = rp.phase;  // the chunk's first slot
      for (int i = 0; i < q.nstage && !stop; ++i) {
        const int j = q.j0 + i * q.R;
        const int nr = min(q.R, q.jst - j);
        const uint32_t bytes = (uint32_t)nr * q.D * 2u;
        uint64_t* fb;
        uint8_t* dst = produce_slot(p, ring, full, empty, rp, issued, task, 2u * bytes, &fb, wp);
        if (!dst) { stop = true; break; }
        bulk_g2s(dst, Kc + (rowbase + j) * q.D, bytes, fb, pol);
        bulk_g2s(dst + kStageBytes / 2, Vc + (rowbase + j) * q.D, bytes, fb, pol);
      }
      if (wp && !stop && q.nstage > 0) {
        l2_plan(recs, rfull, k, *wp);
        wp->start = &empty[s0];
        wp->start_par = ph0;
      }
    }
    mbar_arrive(&rempty[e]);  // done with the record (the consumers arrive too)
  }
  // Let every copy still in flight land before the CTA can exit.
  const uint32_t inflight = issued < (uint32_t)nst ? issued : (uint32_t)nst;
  for (uint32_t k = 0; k < inflight; ++k) {
    const uint32_t st = issued - 1 - k;
    bar_wait(p, &full[st % nst], (st / nst) & 1u, -1, false);
  }
}

// The record warp: per task, lanes 0-15 copy the descriptor, lanes 0-7
// resolve its pointers, lanes 8-11 read its plan ranges and lane 12 its
// tensor-map rows; then the first plan entries.  Runs at most kRecs tasks
// ahead of the producer and the consumers, which both release a record.
__device__ void record_warp(const KParams& p, TaskRec* recs, uint64_t* rfull, uint64_t* rempty) {
  const int lane = threadIdx.x & 31;
  const uint32_t all = 0xffffffffu;
  Seq sq;
  seq_init(sq, p);
  int task = 0, lvl = 0;
  for (uint32_t k = 0;; ++k) {
    const uint32_t e = k & (kRecs - 1);
    TaskRec* r = recs + e;
    if (k >= (uint32_t)kRecs) {  // the consumers are done with this entry's previous task
      const int ok = bar_wait(p, &rempty[e], ((k / kRecs) - 1) & 1u, -1, true) ? 1 : 0;  // every lane waits
      if (!__shfl_sync(all, ok, 0)) return;
    }
    if (!seq_next(sq, p, task, lvl)) {
      if (lane == 0) {
        r->task = -1;
        mbar_arrive(&rfull[e]);
      }
      return;
    }
    if (lane < 16) reinterpret_cast<uint32_t*>(&r->d)[lane] = __ldg(reinterpret_cast<const uint32_t*>(p.tasks + task) + lane);
    __syncwarp();
    const bool mega = p.mode == MK_MODE_MEGA;
    const mk_task_descriptor& d = r->d;
    if (lane < 8) {
      const bool argmax = d.op_id == MK_OP_GEMV && (d.flags & MK_F_ARGMAX_EPI);
      const uint32_t idx = lane < 3 ? d.in_buf[lane] : lane == 3 ? d.out_buf : lane == 4 ? d.in_buf[0]
                         : lane == 5 ? d.in_buf[2] : lane == 6 ? d.out_buf : argmax ? d.reserved[3] : (uint32_t)MK_NO_BUF;
      uint64_t v = 0;
      if (idx < (uint32_t)p.num_bufs) {
        if (lane < 4 || lane == 7) v = reinterpret_cast<uint64_t>(p.bufs[idx]);
        else if (mega) v = reinterpret_cast<uint64_t>(p.mirrors[idx]);
      }
      r->ptr[lane] = v;
    } else if (lane < 12) {
      const uint32_t ov = mega ? __ldg((lane < 10 ? p.wait_off : p.sig_off) + task + (lane & 1)) : 0u;
      (&r->w0)[lane - 8] = ov;  // w0, nw, s0, ns hold the four offsets for now
    } else if (lane == 12) {
      const uint32_t in1 = d.in_buf[1];
      r->tm_rows = ((d.op_id == MK_OP_GEMV && d.config_id == 1) || d.op_id == MK_OP_ATTENTION_PARTIAL) &&
                           in1 < (uint32_t)p.num_bufs
                       ? p.tm_rows[in1]
                       : 0;
    }
    __syncwarp();
    const uint32_t wb = r->w0, we = r->nw, sb = r->s0, se = r->ns;
    __syncwarp();
    if (lane == 0) {
      r->task = task;
      r->lvl = lvl;
      r->nw = we - wb;
      r->ns = se - sb;
    }
    if (lane < 4 && (uint32_t)lane < we - wb) r->wi[lane] = __ldg(p.wait + wb + lane);
    if (lane >= 4 && lane < 8 && (uint32_t)(lane - 4) < se - sb) r->si[lane - 4] = __ldg(p.sig + sb + lane - 4);
    __syncwarp();
    if (lane == 0) mbar_arrive(&rfull[e]);  // release: publishes every lane's writes (ordered by the syncwarp)
  }
}

// ------------------------------------------------------------------ consumer context
struct Ctx {
  const KParams* p;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  float* scratch;
  RingPos rp;  // next ring slot to wait for (consume_begin)
  int nst;
  int task;
  uint64_t mark[3];  // optional trace marks inside a task body (thread 0)
  uint32_t ring_waits;  // traced: ring slots thread 0 found not yet landed
  uint8_t* xbuf;        // class-2 kernel: activation staging tiles (tensor-core A operand)
  TcCtl* ctl;
  uint32_t taddr;       // tensor-memory accumulator base
  uint32_t tc_ph;       // completed phases seen: mma_bar[0] (bit 0), mma_bar[1] (bit 1), acc_full (bit 2)
  const TaskRec* rec;   // the current task's record
  int32_t* state;       // the decode state (token, position) per sequence
  uint32_t pcol;        // tensor-memory column of the partials' score buffers
};

template <class T>
__device__ __forceinline__ T* rec_ptr(const Ctx& c, int i) {
  return reinterpret_cast<T*>(c.rec->ptr[i]);
}

__device__ __forceinline__ void trace_mark(Ctx& c, int i) {
  if (c.p->trace && threadIdx.x == 0) c.mark[i] = globaltimer();
}

// Every lane waits for the slot (acquiring the bytes the copies wrote);
// no divergent single-lane wait and warp barrier before the loads.
// Slots are waited for and handed back in order; a consumer may wait for
// the next slot before handing back the current one.
__device__ __forceinline__ uint32_t consume_begin(Ctx& c) {
  const uint32_t slot = c.rp.slot, ph = c.rp.phase;
  c.rp.advance(c.nst);
  if (c.p->trace && threadIdx.x == 0 && !mbar_try_wait(&c.full[slot], ph)) ++c.ring_waits;
  bar_wait(*c.p, &c.full[slot], ph, c.task, true);
  return slot;
}

__device__ __forceinline__ void consume_end(Ctx& c, uint32_t slot) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&c.empty[slot]);
}

__device__ __forceinline__ void cbar() { named_bar_sync(1, kConsumerThreads); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index) max with ties to the lower index, across the 256 consumer
// threads; result valid in thread 0.  red: 16 floats of shared scratch.
__device__ void block_argmax(float& v, int& idx, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ov > v || (ov == v && oi < idx)) {
      v = ov;
      idx = oi;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[warp] = v;
    reinterpret_cast<int*>(red)[8 + warp] = idx;
  }
  cbar();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kConsumerWarps; ++w) {
      const float ov = red[w];
      const int oi = reinterpret_cast<int*>(red)[8 + w];
      if (ov > v || (ov == v && oi < idx)) {
        v = ov;
        idx = oi;
      }
    }
  }
  cbar();
}

// ------------------------------------------------------------------ tagged hand-offs
// At one or two rows the activations that GEMVs read, and the qkv rows that
// appends and partials read, also travel as (step tag, value) pairs in
// mirrors of their buffers: one 8-byte word, tag in the high half (MEGA mode
// only; every launch has a new tag, so pairs of earlier steps never match).
// A task whose inputs all have mirrors waits on no counter: it loads its
// pairs and polls those whose tag is not yet this step's.
__device__ __forceinline__ uint64_t ll_pack(float v, uint32_t tag) {
  return ((uint64_t)tag << 32) | __float_as_uint(v);
}

__device__ __forceinline__ bool ll_ready(uint64_t v, uint32_t tag) { return (uint32_t)(v >> 32) == tag; }

// Poll the pair at m (found stale) until it carries this step's tag, and
// return it; on abort or timeout (raised here) return the stale pair, and
// the caller carries on with it as after any failed wait.
__device__ uint64_t ll_wait(const KParams& p, const uint64_t* m, int task) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    const uint64_t v = ld_relaxed_u64(m);
    if (ll_ready(v, p.tag)) return v;
    if ((it & 15u) == 0) {
      if (aborted(p)) return v;
      if (globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, MK_DEV_DEP_TIMEOUT, task);
        return v;
      }
    }
  }
}

// Warp-uniform poll: every lane polls the pair the leader names (one
// request per poll for the warp, no divergent single-lane loop); lane 0's
// answer decides for the warp.
__device__ __forceinline__ bool ll_poll_warp(const KParams& p, const uint64_t* pm, int leader, int task) {
  pm = reinterpret_cast<const uint64_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(pm), leader));
  const int ready = ll_ready(ll_wait(p, pm, task), p.tag) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ready, 0) != 0;
}

__device__ __forceinline__ float ll_load1(const KParams& p, const uint64_t* m, int task) {
  uint64_t v = ld_relaxed_u64(m);
  if (!ll_ready(v, p.tag)) v = ll_wait(p, m, task);
  return __uint_as_float((uint32_t)v);
}

// Warp-collective: lane loads the pairs at m[i] where use[i]; while some
// lane holds a stale pair, the lowest such lane polls it and every lane
// then reloads its stale pairs.
template <int N>
__device__ __forceinline__ void ll_gather(const KParams& p, int task, const uint64_t* const (&m)[N],
                                          const bool (&use)[N], float (&out)[N]) {
  uint64_t q[N];
#pragma unroll
  for (int i = 0; i < N; ++i) q[i] = use[i] ? ld_relaxed_u64(m[i]) : ll_pack(0.f, p.tag);
  for (;;) {
    int first = -1;
#pragma unroll
    for (int i = N - 1; i >= 0; --i)
      if (!ll_ready(q[i], p.tag)) first = i;
    const uint32_t want = __ballot_sync(0xffffffffu, first >= 0);
    if (!want) break;
    const int leader = __ffs(want) - 1;
    const uint64_t* pm = m[0];
#pragma unroll
    for (int i = 1; i < N; ++i)
      if (first == i) pm = m[i];
    if (!ll_poll_warp(p, pm, leader, task)) break;
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (!ll_ready(q[i], p.tag)) q[i] = ld_relaxed_u64(m[i]);
  }
#pragma unroll
  for (int i = 0; i < N; ++i) out[i] = __uint_as_float((uint32_t)q[i]);
}

// Eight consecutive pairs (m 64-byte aligned) into o; returns the mask of
// those already tagged.  Two 32-byte loads: every L2 sector is requested
// once (16-byte loads asked for each sector twice, and every SM reads the
// same vector, so the L2's sector rate bounded the load).
__device__ __forceinline__ uint32_t ll_piece(const uint64_t* m, uint32_t tag, float (&o)[8]) {
  uint64_t lo[4], hi[4];
  ld_relaxed_v4u64(m, lo);
  ld_relaxed_v4u64(m + 4, hi);
  const uint64_t q[8] = {lo[0], lo[1], lo[2], lo[3], hi[0], hi[1], hi[2], hi[3]};
  uint32_t ok = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    o[k] = __uint_as_float((uint32_t)q[k]);
    ok |= (ll_ready(q[k], tag) ? 1u : 0u) << k;
  }
  return ok;
}

// x for this lane's pieces (b, v) of 8 columns from the mirror xm: all
// pieces are loaded at once; while some lane holds stale pairs, one lane
// (the lowest with a stale pair) polls that pair until it turns and the
// warp then reloads its pending pieces.  One poller per warp keeps the
// polling traffic on the producers' lines low.  Warp-collective.
template <int B, int NV>
__device__ __forceinline__ void ll_load_x(const KParams& p, int task, float (&xr)[B][NV][8], const uint64_t* xm,
                                          int K, int col0, int Bact) {
  const int lane = threadIdx.x & 31;
  uint32_t pend = 0;
  const uint64_t* probe = nullptr;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (b < Bact) {
        const uint64_t* m = xm + (size_t)b * K + col0 + v * 256;
        const uint32_t ok = ll_piece(m, p.tag, xr[b][v]);
        if (ok != 0xFFu) {
          pend |= 1u << (v * B + b);
          if (!probe) probe = m + (__ffs(~ok) - 1);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) xr[b][v][k] = 0.f;
      }
    }
  }
  for (;;) {
    const uint32_t want = __ballot_sync(0xffffffffu, pend != 0);
    if (!want) break;
    const int leader = __ffs(want) - 1;
    if (!ll_poll_warp(p, probe, leader, task)) break;  // abort or timeout: carry on with what is loaded
    probe = nullptr;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (pend & (1u << (v * B + b))) {
          const uint64_t* m = xm + (size_t)b * K + col0 + v * 256;
          const uint32_t ok = ll_piece(m, p.tag, xr[b][v]);
          if (ok == 0xFFu) pend &= ~(1u << (v * B + b));
          else if (!probe) probe = m + (__ffs(~ok) - 1);
        }
      }
    }
  }
}

// ------------------------------------------------------------------ GEMV body
// Shared-memory scratch of a GEMV task: per-(row, batch, warp column) slots,
// per-(row, batch) accumulators, then a small reduction area:
//   red[0,64) sum-of-squares partials, red[64,72) 1/rms per batch row,
//   red[80,96) argmax scratch, red[96,104) tile max, red[104,112) tile argmax.
__device__ __forceinline__ float* gemv_slots(Ctx& c) { return c.scratch; }
__device__ __forceinline__ float* gemv_acc(Ctx& c) { return c.scratch + kSlotFloats; }
__device__ __forceinline__ float* gemv_red(Ctx& c) { return c.scratch + kSlotFloats + kAccFloats; }

// x (times gamma when normalising) for this lane's columns col0 + v*256 + [0,8),
// and the sum of squares of the raw x values loaded (for the RMS norm); from
// the mirror xm when the task reads tagged pairs.
template <int B, int NV>
__device__ __forceinline__ void gemv_load_x(const KParams& p, int task, float (&xr)[B][NV][8], float (&ss)[B],
                                            const float* __restrict__ x, const uint64_t* xm,
                                            const uint16_t* __restrict__ gamma, int K, int col0, int Bact) {
  // the gains do not depend on x: with few pieces (every normalised GEMV
  // has NV <= 2) their loads go out before x's, and before any wait for it
  uint4 gv[NV <= 2 ? NV : 1];
  if constexpr (NV <= 2) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
      gv[v] = gamma ? __ldg(reinterpret_cast<const uint4*>(gamma + col0 + v * 256)) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (xm) {
    ll_load_x<B, NV>(p, task, xr, xm, K, col0, Bact);
  } else {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (b < Bact) {
          ldcg_v8f(x + (size_t)b * K + col0 + v * 256, xr[b][v]);  // one request per sector
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) xr[b][v][k] = 0.f;
        }
      }
    }
  }
#pragma unroll
  for (int b = 0; b < B; ++b) ss[b] = 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int col = col0 + v * 256;
    float gm[8];
    if (gamma) {
      uint4 g4;
      if constexpr (NV <= 2) g4 = gv[v];
      else g4 = __ldg(reinterpret_cast<const uint4*>(gamma + col));
      gm[0] = bf_lo(g4.x); gm[1] = bf_hi(g4.x); gm[2] = bf_lo(g4.y); gm[3] = bf_hi(g4.y);
      gm[4] = bf_lo(g4.z); gm[5] = bf_hi(g4.z); gm[6] = bf_lo(g4.w); gm[7] = bf_hi(g4.w);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) gm[k] = 1.f;
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ss[b] = fmaf(xr[b][v][k], xr[b][v][k], ss[b]);
        xr[b][v][k] *= gm[k];
      }
    }
  }
}

// The tile's running argmax, and 1/rms = 1 when the input is not
// normalised (a normalised input gets it from gemv_fold).  Once per task.
__device__ __forceinline__ void gemv_prologue(const mk_task_descriptor& d, const GemvGeom& G, float* red) {
  const int tid = threadIdx.x;
  if (!(d.flags & MK_F_RMS_NORM_INPUT) && tid < G.B) red[64 + tid] = 1.f;
  if ((d.flags & MK_F_ARGMAX_EPI) && tid < G.B) {
    red[96 + tid] = -FLT_MAX;
    reinterpret_cast<int*>(red)[104 + tid] = INT_MAX;
  }
}

// Sum N values (N a power of two, at most 32) across the warp.  Afterwards
// lane l holds the warp-wide sum of value l >> (5 - log2 N); the first
// log2 N steps halve the values each lane carries, the rest are butterflies.
template <int N>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane) {
  static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
#pragma unroll
  for (int t = 0; t < 5; ++t) {
    const int o = 16 >> t;
    const int n = N >> t;  // values each lane still carries (a constant once unrolled)
    if (n > 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = up ? v[i] : v[i + n / 2];
        const float keep = up ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

// Every ring slot of one (row group, k-segment).  A warp takes rows
// wrow, wrow + WROW, ... of each slot over its column block, with x in
// registers: all shared loads of a slot first, independent FMA chains per
// row, then one transposed reduction of the slot's (row, batch) sums.
// Below batch 8 the loads are unconditional: rows past the slot's last
// valid row read stale bytes of the same slot, and their sums are never
// stored.
// Results go to slots[(row, b, warp column)].
template <int B, int NV>
__device__ __forceinline__ void gemv_stages(Ctx& c, const mk_task_descriptor& d, const GemvGeom& G, int rows_g,
                                            int ks, bool first_group, const uint64_t* xm) {
  const KParams& p = *c.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wcol = warp % G.WCOL, wrow = warp / G.WCOL;
  const int colw = G.KS / G.WCOL;
  const float* x = rec_ptr<const float>(c, kPIn0);
  const uint16_t* gamma = (d.flags & MK_F_RMS_NORM_INPUT) ? rec_ptr<const uint16_t>(c, kPIn2) : nullptr;
  float* slots = gemv_slots(c);
  float xr[B][NV][8], ss[B];
  gemv_load_x<B, NV>(p, c.task, xr, ss, x, xm, gamma, G.K, ks * G.KS + wcol * colw + lane * 8, G.B);
  if (gamma && first_group) {
    // sum of squares of x over this warp's columns; warps of the first warp
    // row cover every column once (the others contribute zero)
    float* red = gemv_red(c);
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float t = warp_sum(wrow == 0 ? ss[b] : 0.f);
      if (lane == 0 && b < 8) red[warp * 8 + b] = (ks == 0 ? 0.f : red[warp * 8 + b]) + t;
    }
  }
  constexpr int RWM = 8 / NV;                // most rows a warp takes from one full slot
  constexpr int VPS = RWM * B;               // (row, batch) sums per slot
  constexpr int NR = VPS > 32 ? 32 : VPS;    // values per transposed reduction
  constexpr int SH = NR >= 32 ? 0 : (NR >= 16 ? 1 : (NR >= 8 ? 2 : (NR >= 4 ? 3 : (NR >= 2 ? 4 : 5))));
  for (int sg = 0; sg < G.seg; ++sg) {
    for (int r0 = 0; r0 < rows_g; r0 += G.rs) {
      const int nr = min(G.rs, rows_g - r0);
      const uint32_t slot = consume_begin(c);
      if (first_group && ks == 0 && sg == 0 && r0 == 0) trace_mark(c, 0);
      const uint32_t base = smem_addr(c.ring + (size_t)slot * kStageBytes) + (wcol * colw + lane * 8) * 2;
      const int rw = nr > wrow ? (nr - wrow + G.WROW - 1) >> G.lgW : 0;
      uint4 w[RWM][NV];
#pragma unroll
      for (int r = 0; r < RWM; ++r) {
        const uint32_t ra = base + (uint32_t)(wrow + r * G.WROW) * G.KS * 2;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          if constexpr (B >= 8) w[r][v] = r < rw ? lds128(ra + v * 512) : make_uint4(0u, 0u, 0u, 0u);  // no spills
          else w[r][v] = lds128(ra + v * 512);
        }
      }
      float acc[VPS];
#pragma unroll
      for (int i = 0; i < VPS; ++i) acc[i] = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
#pragma unroll
          for (int r = 0; r < RWM; ++r) {
            const uint32_t u = k2 == 0 ? w[r][v].x : k2 == 1 ? w[r][v].y : k2 == 2 ? w[r][v].z : w[r][v].w;
            const float lo = bf_lo(u), hi = bf_hi(u);
#pragma unroll
            for (int b = 0; b < B; ++b) {
              acc[r * B + b] = fmaf(lo, xr[b][v][2 * k2], acc[r * B + b]);
              acc[r * B + b] = fmaf(hi, xr[b][v][2 * k2 + 1], acc[r * B + b]);
            }
          }
        }
      }
      consume_end(c, slot);
#pragma unroll
      for (int h = 0; h < VPS / NR; ++h) {
        float vv[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) vv[i] = acc[h * NR + i];
        const float tot = transpose_reduce<NR>(vv, lane);
        if ((lane & ((1 << SH) - 1)) == 0) {
          const int i = h * NR + (lane >> SH);
          const int r = i / B, b = i % B;
          if (r < rw) {
            const int row = sg * rows_g + r0 + wrow + r * G.WROW;
            slots[(row * B + b) * G.WCOL + wcol] = tot;
          }
        }
      }
    }
  }
}

// Fold one k-segment's per-warp partials into the accumulators, in a fixed
// order (deterministic; no float atomics).
__device__ __forceinline__ void gemv_fold(const mk_task_descriptor& d, const GemvGeom& G, int rows_g, int ks,
                                       bool first_group, float* slots, float* acc, float* red) {
  cbar();
  for (int i = threadIdx.x; i < G.seg * rows_g * G.BT; i += kConsumerThreads) {
    float s = 0.f;
    for (int w = 0; w < G.WCOL; ++w) s += slots[i * G.WCOL + w];
    acc[i] = (ks == 0) ? s : acc[i] + s;
  }
  if ((d.flags & MK_F_RMS_NORM_INPUT) && first_group && ks == G.nks - 1 && threadIdx.x < G.B) {
    float t = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) t += red[w * 8 + threadIdx.x];
    red[64 + threadIdx.x] = 1.0f / sqrtf(t / (float)G.K + __uint_as_float(d.reserved[2]));
  }
  cbar();
}

// Epilogue of one row group: normalisation scale, SiLU*mul, residual,
// store, and the tile's running argmax.
__device__ __forceinline__ void gemv_epilogue(const KParams& p, const mk_task_descriptor& d, const GemvGeom& G,
                                           int g0, int rows_g, const float* acc, float* red,
                                           const float* staged_res, float* out, const float* res,
                                           const uint64_t* rm, uint64_t* om, int task) {
  const int tid = threadIdx.x;
  const bool silu = d.flags & MK_F_SILU_MUL;
  const bool argmax = d.flags & MK_F_ARGMAX_EPI;
  const int BT = G.BT;
  for (int b = 0; b < G.B; ++b) {
    const float inv = red[64 + b];
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    for (int j = tid; j < rows_g; j += kConsumerThreads) {
      float y = acc[j * BT + b] * inv;
      if (silu) {
        const float u = acc[(rows_g + j) * BT + b] * inv;
        y = y / (1.0f + expf(-y)) * u;
      }
      const int col = G.c0 + g0 + j;
      if (staged_res) y += staged_res[j * BT + b];
      else if (rm) y += ll_load1(p, rm + (size_t)b * G.n + col, task);
      else if (res) y += __ldcg(res + (size_t)b * G.n + col);
      out[(size_t)b * G.n + col] = y;
      if (om) st_relaxed_u64(om + (size_t)b * G.n + col, ll_pack(y, p.tag));
      if (y > bv) {
        bv = y;
        bi = col;
      }
    }
    if (argmax) {
      block_argmax(bv, bi, red + 80);
      if (tid == 0) {
        const float cv = red[96 + b];
        const int ci = reinterpret_cast<int*>(red)[104 + b];
        if (bv > cv || (bv == cv && bi < ci)) {
          red[96 + b] = bv;
          reinterpret_cast<int*>(red)[104 + b] = bi;
        }
      }
    }
  }
  cbar();
}

// Batch class 0 serves one or two activation rows (CUDA-core GEMVs), class
// 2 three to eight (tensor-core GEMVs; CUDA cores at batch width 8 only for
// a weight without a tensor map); each class is its own kernel so register
// allocations are not shared.
template <int BCLASS>
__device__ void gemv_task(Ctx& c, const mk_task_descriptor& d) {
  GemvGeom G;
  gemv_geom(d, G);
  float* red = gemv_red(c);
  gemv_prologue(d, G, red);
  // A residual read by the epilogue is loaded now, so its latency hides
  // behind the slots; it is parked in the (then free) slot area afterwards.
  // tagged pairs (one or two rows only): the output's mirror, and the inputs' when
  // both x and the residual have one (the task then waited on no counter)
  const KParams& p = *c.p;
  const uint64_t *xm = nullptr, *rm = nullptr;
  uint64_t* om = nullptr;
  if (BCLASS < 2) {  // the record holds mirrors in MEGA mode only
    om = rec_ptr<uint64_t>(c, kMirOut);
    xm = rec_ptr<const uint64_t>(c, kMirX);
    if (d.flags & MK_F_ADD_RESIDUAL) {
      rm = rec_ptr<const uint64_t>(c, kMirAux);
      if (!rm) xm = nullptr;
    }
    if (!xm) rm = nullptr;
  }
  float* out = rec_ptr<float>(c, kPOut);
  const float* res = (d.flags & MK_F_ADD_RESIDUAL) ? rec_ptr<const float>(c, kPIn2) : nullptr;
  const bool stage_res = (d.flags & MK_F_ADD_RESIDUAL) && G.cn <= kConsumerThreads && G.RG >= G.cn;
  float rv[8];
  // tagged residual pairs (at most two rows): issued now, examined once the
  // slots are consumed, so their round trip overlaps x's instead of
  // preceding it (the residual was complete long before)
  constexpr int RB = BCLASS < 2 ? 2 : 1;
  uint64_t rq[RB];
  const uint64_t* rc = nullptr;
  if (stage_res && rm) {
    rc = rm + G.c0 + threadIdx.x;
#pragma unroll
    for (int b = 0; b < RB; ++b)
      rq[b] = threadIdx.x < G.cn && b < G.B ? ld_relaxed_u64(rc + (size_t)b * G.n) : ll_pack(0.f, p.tag);
  } else if (stage_res && threadIdx.x < G.cn) {
#pragma unroll
    for (int b = 0; b < 8; ++b) rv[b] = b < G.B ? __ldcg(res + (size_t)b * G.n + G.c0 + threadIdx.x) : 0.f;
  }
  for (int g0 = 0; g0 < G.cn; g0 += G.RG) {
    const int rows_g = min(G.RG, G.cn - g0);
    for (int ks = 0; ks < G.nks; ++ks) {
      if constexpr (BCLASS == 0) {
        switch (G.BT * 16 + G.NV) {
          case 16 + 1: gemv_stages<1, 1>(c, d, G, rows_g, ks, g0 == 0, xm); break;
          case 16 + 2: gemv_stages<1, 2>(c, d, G, rows_g, ks, g0 == 0, xm); break;
          case 16 + 4: gemv_stages<1, 4>(c, d, G, rows_g, ks, g0 == 0, xm); break;
          case 16 + 7: gemv_stages<1, 7>(c, d, G, rows_g, ks, g0 == 0, xm); break;
          default: gemv_stages<2, 1>(c, d, G, rows_g, ks, g0 == 0, xm); break;
        }
      } else {
        gemv_stages<8, 1>(c, d, G, rows_g, ks, g0 == 0, xm);
      }
      gemv_fold(d, G, rows_g, ks, g0 == 0, gemv_slots(c), gemv_acc(c), red);
    }
    trace_mark(c, 1);
    if (rc) {  // warp-collective: a stale pair is polled, then every stale one reloaded
      for (;;) {
        int first = -1;
#pragma unroll
        for (int b = RB - 1; b >= 0; --b)
          if (!ll_ready(rq[b], p.tag)) first = b;
        const uint32_t want = __ballot_sync(0xffffffffu, first >= 0);
        if (!want) break;
        const int leader = __ffs(want) - 1;
        if (!ll_poll_warp(p, rc + (size_t)(first < 0 ? 0 : first) * G.n, leader, c.task)) break;
#pragma unroll
        for (int b = 0; b < RB; ++b)
          if (!ll_ready(rq[b], p.tag)) rq[b] = ld_relaxed_u64(rc + (size_t)b * G.n);
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) rv[b] = b < RB ? __uint_as_float((uint32_t)rq[b < RB ? b : 0]) : 0.f;
      rc = nullptr;
    }
    float* staged = nullptr;
    if (stage_res) {  // the fold's closing barrier has freed the slot area
      staged = gemv_slots(c);
      if (threadIdx.x < G.cn) {
#pragma unroll
        for (int b = 0; b < 8; ++b)
          if (b < G.B) staged[threadIdx.x * G.BT + b] = rv[b];
      }
    }
    gemv_epilogue(p, d, G, g0, rows_g, gemv_acc(c), red, staged, out, res, rm, om, c.task);
    trace_mark(c, 2);
  }
  if ((d.flags & MK_F_ARGMAX_EPI) && threadIdx.x < G.B) {
    mk_argmax_pair* pairs = rec_ptr<mk_argmax_pair>(c, kPPairs);
    mk_argmax_pair pr;
    pr.value = red[96 + threadIdx.x];
    pr.index = reinterpret_cast<int*>(red)[104 + threadIdx.x];
    pairs[(size_t)d.reserved[4] * G.B + threadIdx.x] = pr;
  }
}

// ------------------------------------------------------------------ GEMV on tensor cores (B = 8)
// From three rows a tile is a dense contraction (up to 8 columns of x against the
// tile's weight rows), so it runs on the 5th-generation tensor cores:
// D[128 x N] (+)= A[128 x K] * B[K x N] with
//   B = the tile's weight rows (N = rows rounded up to 16), K-major, brought
//       in by TMA tensor copies in the 128-byte-swizzled layout, 64 K per row;
//   A = the activations, split into three bf16 parts hi + mid + lo that
//       carry x to about f32 precision (A rows 0-7, 8-15, 16-23 hold the
//       parts of batch rows 0-7; the other 104 rows read whatever follows
//       and are never used);
//   D = f32 accumulators in tensor memory, y[b] = D[b] + D[8+b] + D[16+b].
// One thread issues the MMAs; a commit per K range arrives on an mbarrier,
// which releases that range's ring slots and staging tile.
// This thread's share of one K range of x: batch row = warp, kpt = 2 * nkb
// consecutive columns from k0 (rows past the batch read as zero).
// This lane's kpt columns of x from k0 (row b; zero past the batch) and,
// for a normalised input, the gains of those columns (bf16 pairs).
__device__ __forceinline__ void tc_load_x(float (&xv)[8], uint32_t (&gv)[4], const float* x, const uint16_t* gamma,
                                          int K, int b, int Bact, int k0, int kpt) {
  // the widest load that covers the lane's kpt (2, 4 or 8) columns: every
  // L2 sector is requested once
#pragma unroll
  for (int e = 0; e < 8; ++e) xv[e] = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) gv[e] = 0u;
  const float* px = x + (size_t)b * K + k0;
  const bool live = b < Bact;
  if (kpt == 8) {
    if (live) ldcg_v8f(px, xv);
    if (gamma) {
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(gamma + k0));
      gv[0] = g.x; gv[1] = g.y; gv[2] = g.z; gv[3] = g.w;
    }
  } else if (kpt == 4) {
    if (live) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(px));
      xv[0] = v.x; xv[1] = v.y; xv[2] = v.z; xv[3] = v.w;
    }
    if (gamma) {
      const uint2 g = __ldg(reinterpret_cast<const uint2*>(gamma + k0));
      gv[0] = g.x; gv[1] = g.y;
    }
  } else {
    if (live) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(px));
      xv[0] = v.x; xv[1] = v.y;
    }
    if (gamma) gv[0] = __ldg(reinterpret_cast<const uint32_t*>(gamma + k0));
  }
}

// Consumer side of a tensor-core tile: hand the task to the MMA warp, stage
// each K range's activations (three bf16 parts, 128-byte swizzle) into one
// of two staging tiles, read the accumulators from tensor memory at the
// end of each row group, run the usual epilogue.  No CTA-wide barrier per K
// range: the staging tile of range kr waits only for the MMAs of kr - 2.
// A K-split tile (one K range of a row block) stores its partial sums and
// sums of squares in its scratch record and counts itself in; the block's
// last split waits for the others, adds their records in split order to its
// own sums and runs the epilogue.
__device__ void tc_gemv_task(Ctx& c, const mk_task_descriptor& d) {
  const KParams& p = *c.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  TcCtl* ctl = c.ctl;
  GemvGeom G;
  gemv_geom(d, G);
  G.BT = 8;  // the accumulators hold 8 batch rows whatever B (rows past B are zero)
  TcGeom T;
  tc_geom(c.rec->tm_rows, d, T);
  float* red = gemv_red(c);
  float* acc = c.scratch;  // [seg * rows][8] results (the GEMV slot area is unused here)
  gemv_prologue(d, G, red);
  const float* x = rec_ptr<const float>(c, kPIn0);
  const uint16_t* gamma = (d.flags & MK_F_RMS_NORM_INPUT) ? rec_ptr<const uint16_t>(c, kPIn2) : nullptr;
  const int kpt = 2 * T.nkb;  // columns of x per lane and K range
  const uint32_t xb0 = smem_addr(c.xbuf);
  if (tid == 0) {  // the mbarrier arrive publishes the mailbox (release)
    ctl->mb_task = c.task;
    ctl->mb_slot = c.rp.slot;
    ctl->mb_phase = c.rp.phase;
    mbar_arrive(&ctl->task_go);
  }
  float ss = 0.f;  // sum of squares of this lane's raw x (first row group)
  for (int g0 = 0; g0 < G.cn; g0 += T.RG) {
    const int rows_g = min(T.RG, G.cn - g0);
    // x (and the gains) of the next two K ranges are in flight while a
    // range is staged
    float xa[8], xb[8];
    uint32_t ga[4], gb[4];
    tc_load_x(xa, ga, x, gamma, T.K, warp, G.B, T.k0 + lane * kpt, kpt);
    if (T.nkr > 1) tc_load_x(xb, gb, x, gamma, T.K, warp, G.B, T.k0 + T.nkb * 64 + lane * kpt, kpt);
    for (int kr = 0; kr < T.nkr; ++kr) {
      float xc[8];
      uint32_t gc[4];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        xc[e] = xa[e];
        xa[e] = xb[e];
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        gc[e] = ga[e];
        ga[e] = gb[e];
      }
      const int k0 = T.k0 + kr * T.nkb * 64 + lane * kpt;  // this lane's first column
      if (kr + 2 < T.nkr) tc_load_x(xb, gb, x, gamma, T.K, warp, G.B, k0 + 2 * T.nkb * 64, kpt);
      const int j = kr & 1;
      if (kr >= 2) {  // the MMAs of kr - 2 have read this staging tile
        bar_wait(p, &ctl->mma_bar[j], (c.tc_ph >> j) & 1u, c.task, false);  // every lane waits
        c.tc_ph ^= 1u << j;
      }
      const uint32_t xt = xb0 + (uint32_t)j * (kXbufBytes / 2);  // K block b at xt + b * 3072
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        if (e < kpt) {
          const int kl = lane * kpt + e;  // column within the K range
          const int kb = kl >> 6, kk = kl & 63;
          float v0 = xc[e], v1 = xc[e + 1];
          if (g0 == 0) ss += v0 * v0 + v1 * v1;
          if (gamma) {
            v0 *= bf_lo(gc[e >> 1]);
            v1 *= bf_hi(gc[e >> 1]);
          }
          // exact three-part split: each part is the bf16 rounding of what
          // the previous parts leave (f32 subtractions of nearby values)
          uint32_t part[3];
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            const __nv_bfloat162 a = __float22bfloat162_rn(make_float2(v0, v1));
            part[q] = *reinterpret_cast<const uint32_t*>(&a);
            v0 -= bf_lo(part[q]);
            v1 -= bf_hi(part[q]);
          }
          // row r of a K block sits at r * 128 bytes; its 16-byte chunk c is
          // stored at chunk c ^ (row within the 1024-byte group), as the
          // 128-byte swizzle reads it
          const uint32_t ch = (uint32_t)(kk >> 3), cb = (uint32_t)(kk & 7) * 2u;
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            const uint32_t ra = xt + (uint32_t)kb * 3072u + (uint32_t)q * 1024u + (uint32_t)warp * 128u;
            sts32(ra + ((ch ^ ((ra >> 7) & 7u)) << 4) + cb, part[q]);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->x_full[j]);
    }
    const float ssw = g0 == 0 ? warp_sum(ss) : 0.f;  // batch row `warp`: this tile's columns of x
    if (g0 == 0 && gamma && T.S == 1 && lane == 0)  // 1/rms per batch row (warp b holds row b's columns)
      red[64 + warp] = 1.0f / sqrtf(ssw / (float)T.K + __uint_as_float(d.reserved[2]));
    // the row group's MMAs are done (acc_full follows every earlier commit)
    bar_wait(p, &ctl->acc_full, (c.tc_ph >> 2) & 1u, c.task, false);  // every lane waits
    c.tc_ph ^= 4u;
    for (int kr = max(T.nkr - 2, 0); kr < T.nkr; ++kr)
      c.tc_ph ^= 1u << (kr & 1);  // the last two ranges' commits (only the MMA warp waited on them)
    if (warp == 0) {  // TMEM lanes 0-31 = A rows: the batch's hi, mid, lo parts in 0-7, 8-15, 16-23
      tc_fence_after();
      for (int sg = 0; sg < T.seg; ++sg)
        for (int j0 = 0; j0 < rows_g; j0 += 16) {
          float v[16];
          tmem_ld16(c.taddr + (uint32_t)(sg * T.Nr + j0), v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float mid = __shfl_down_sync(0xffffffffu, v[i], 8);
            const float lo = __shfl_down_sync(0xffffffffu, v[i], 16);
            if (lane < 8 && j0 + i < rows_g) acc[(sg * rows_g + j0 + i) * 8 + lane] = v[i] + mid + lo;
          }
        }
      tc_fence_before();
    }
    cbar();
    if (tid == 0) mbar_arrive(&ctl->acc_empty);  // tensor memory is free for the next row group
    if (T.S > 1) {
      // K split (one row group): partial sums through the scratch records
      const int rec0 = (int)d.reserved[4] - T.j, n8 = T.seg * rows_g * 8;
      uint32_t* arr = p.karr + rec0 + T.S - 1;  // the block's arrival counter
      if (T.j + 1 < T.S) {
        float* rec = p.ksplit + (size_t)d.reserved[4] * kKsplitRec;
        for (int i = tid * 4; i < n8; i += kConsumerThreads * 4)  // n8 is a multiple of 8
          *reinterpret_cast<float4*>(rec + i) = *reinterpret_cast<const float4*>(acc + i);
        if (lane == 0) rec[256 * 8 + warp] = ssw;
        cbar();
        if (tid == 0) {  // release: the record before the arrival
          fence_acq_rel_gpu();
          red_relaxed_add(arr, 1u);
        }
        break;  // the block's last split writes the outputs
      }
      if (lane == 0) red[warp] = ssw;  // this split's own sums of squares, per batch row
      if (tid == 0) {  // wait for the other splits (bounded; abort on failure)
        const uint32_t target = p.kmul * (uint32_t)(T.S - 1);
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 0; (int32_t)(ld_acquire(arr) - target) < 0; ++it) {
          if ((it & 63u) == 63u) {
            if (aborted(p)) break;
            if (globaltimer() - t0 > p.timeout_ns) {
              raise_error(p, MK_DEV_DEP_TIMEOUT, c.task);
              break;
            }
          }
        }
      }
      cbar();
      // the other splits' sums, added in split order; up to eight records'
      // float4 loads are in flight at once (a dependent chain of L2 reads
      // per element cost several microseconds)
      for (int i = tid * 4; i < n8; i += kConsumerThreads * 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q0 = 0; q0 < T.S - 1; q0 += 8) {
          float4 r[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            r[u] = q0 + u < T.S - 1
                       ? __ldcg(reinterpret_cast<const float4*>(p.ksplit + (size_t)(rec0 + q0 + u) * kKsplitRec + i))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (q0 + u < T.S - 1) {
              v.x += r[u].x;
              v.y += r[u].y;
              v.z += r[u].z;
              v.w += r[u].w;
            }
          }
        }
        const float4 o = *reinterpret_cast<const float4*>(acc + i);
        *reinterpret_cast<float4*>(acc + i) = make_float4(v.x + o.x, v.y + o.y, v.z + o.z, v.w + o.w);
      }
      if (gamma && tid < G.B) {
        float t = 0.f;
        for (int q = 0; q < T.S - 1; ++q) t += __ldcg(p.ksplit + (size_t)(rec0 + q) * kKsplitRec + 256 * 8 + tid);
        t += red[tid];  // this split's own, last
        red[64 + tid] = 1.0f / sqrtf(t / (float)T.K + __uint_as_float(d.reserved[2]));
      }
      cbar();
    }
    gemv_epilogue(p, d, G, g0, rows_g, acc, red, nullptr, rec_ptr<float>(c, kPOut),
                  (d.flags & MK_F_ADD_RESIDUAL) ? rec_ptr<const float>(c, kPIn2) : nullptr, nullptr, nullptr, c.task);
  }
  for (int g0 = 0; g0 < G.cn; g0 += T.RG)
    for (int i = 0; i < T.nkr; ++i) c.rp.advance(c.nst);
  if ((d.flags & MK_F_ARGMAX_EPI) && threadIdx.x < G.B) {
    mk_argmax_pair* pairs = rec_ptr<mk_argmax_pair>(c, kPPairs);
    mk_argmax_pair pr;
    pr.value = red[96 + threadIdx.x];
    pr.index = reinterpret_cast<int*>(red)[104 + threadIdx.x];
    pairs[(size_t)d.reserved[4] * G.B + threadIdx.x] = pr;
  }
}

// MMA warp of the class-2 kernel (lane 0 of the producer warpgroup's second
// warp): takes tensor-core tiles from the mailbox in the consumers' order;
// per K range it waits for the staged activations and the landed weight
// slots, issues the MMAs and commits; the commit of range kr - 2 hands that
// range's ring slots back to the producer.  Every wait is bounded; after a
// failed wait no more MMAs are issued but every commit still is, so the
// consumers' waits end.
// Split-KV partials (any batch class) come through the same mailbox: per
// block of kKeyBlock cached keys the warp waits for the block's K slot,
// issues S^T[keys x 16] = K [keys x D] * Q^T (the query tile: three bf16
// parts of each query row, K-major, 128-byte swizzle) into score buffer b % 2
// at column pcol, and commits to s_full[b % 2]; before reusing a buffer it
// waits until the softmax warps have read it (s_empty).
__device__ void tc_mma_warp(const KParams& p, uint8_t* ring, uint64_t* full, uint64_t* empty, TcCtl* ctl,
                            uint32_t xb0, uint32_t taddr, uint32_t pcol) {
  if ((threadIdx.x & 31) != 0) return;
  const int nst = p.nstages;
  // completed phases seen: task_go 0, x_full 1-2, mma_bar 3-4, acc_empty 5,
  // s_empty 6-7, q_full 8, s_full 9-10
  uint32_t ph = 0;
  bool first = true, ok = true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    // next task (or the end); idle waits are long, so only abort or a very
    // long silence end them
    for (uint32_t it = 0; !mbar_try_wait(&ctl->task_go, ph & 1u); ++it) {
      __nanosleep(256);
      if ((it & 255u) == 0 && (aborted(p) || globaltimer() - t0 > 64ull * p.timeout_ns)) return;
    }
    ph ^= 1u;
    const int task = ctl->mb_task;
    if (task < 0) return;
    RingPos rp, rel;
    rp.slot = rel.slot = ctl->mb_slot;
    rp.phase = rel.phase = ctl->mb_phase;
    if (__ldg(&p.tasks[task].op_id) == MK_OP_ATTENTION_PARTIAL) {
      const int D = __ldg(&p.tasks[task].n), nblk = (int)ctl->mb_nblk;
      const uint32_t qt = ctl->mb_qt;
      constexpr uint32_t NQ = 16;  // query tile rows: 3 parts x up to 4 query rows, padded
      const uint32_t idesc = idesc_bf16_f32(kKeyBlock, NQ);
      if (!bar_wait(p, &ctl->q_full, (ph >> 8) & 1u, task, false)) ok = false;
      ph ^= 1u << 8;
      for (int b = 0; b < nblk; ++b) {
        const int j = b & 1;
        if (b >= 2) {  // the softmax warps have read buffer j (block b - 2)
          if (!bar_wait(p, &ctl->s_empty[j], (ph >> (6 + j)) & 1u, task, false)) ok = false;
          ph ^= 1u << (6 + j);
        }
        if (ok && !bar_wait(p, &full[rp.slot], rp.phase, task, true)) ok = false;
        tc_fence_after();
        if (ok) {
          const uint32_t ka = smem_addr(ring + (size_t)rp.slot * kStageBytes);
#pragma unroll 1
          for (int q = 0; q < D / 16; ++q) {  // 64-dim box q / 4, K step q % 4
            const uint32_t kb = (uint32_t)q >> 2, ks = (uint32_t)q & 3u;
            tc_mma_bf16(taddr + pcol + (uint32_t)j * NQ, smem_desc_sw128(ka + kb * (kKeyBlock * 128u), 1024u) + ks * 2u,
                        smem_desc_sw128(qt + kb * (NQ * 128u), 1024u) + ks * 2u, idesc, q != 0 ? 1u : 0u);
          }
        }
        tc_commit(&ctl->s_full[j]);  // also when a wait failed, so the consumers' waits end
        if (D == 128) {
          // the K slot is free once the block's score MMAs are done: hand it
          // back now (for all eight consumer warps), so the copies of the
          // blocks ahead need not wait for the block's softmax and P V
          if (!bar_wait(p, &ctl->s_full[j], (ph >> (9 + j)) & 1u, task, false)) ok = false;
          mbar_arrive_cnt(&empty[rp.slot], kConsumerWarps);
        }
        ph ^= 1u << (9 + j);  // one phase per commit, waited for or not
        rp.advance(nst);
        if (D == 128) rp.advance(nst);  // the block's V slot
      }
      continue;
    }
    // only the fields the schedule needs (this warp runs on few registers)
    const mk_task_descriptor* td = p.tasks + task;
    const int cn = (int)__ldg(&td->reserved[1]);
    const int seg = (__ldg(&td->flags) & MK_F_SILU_MUL) ? 2 : 1;
    const int RG = p.tm_rows[__ldg(&td->in_buf[1])];
    const int N = seg * (seg == 2 ? (RG + 7) & ~7 : (RG + 15) & ~15);
    const int S = (int)((uint32_t)__ldg(&td->kv_len) >> 16);
    const int kn = S >= 2 ? (int)(__ldg(&td->reserved[3]) >> 16) : __ldg(&td->k);
    int nkb = 4;
    while (nkb > 1 && (nkb * N * 128 > kStageBytes || (kn / 64) % nkb)) nkb >>= 1;
    const int nkr = kn / 64 / nkb;
    const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)N);
    const uint32_t bstep = (uint32_t)(N * 128) >> 4;  // one K block of the weight tile, in 16 bytes
    for (int g0 = 0; g0 < cn; g0 += RG) {
      if (!first) {  // the consumers have read the previous accumulators
        if (!bar_wait(p, &ctl->acc_empty, (ph >> 5) & 1u, task, false)) ok = false;
        ph ^= 1u << 5;
      }
      first = false;
      for (int kr = 0; kr < nkr; ++kr) {
        const int j = kr & 1;
        if (!bar_wait(p, &ctl->x_full[j], (ph >> (1 + j)) & 1u, task, false)) ok = false;
        ph ^= 1u << (1 + j);
        if (kr >= 2) {  // range kr - 2 is done: its slot goes back to the producer
          if (!bar_wait(p, &ctl->mma_bar[j], (ph >> (3 + j)) & 1u, task, false)) ok = false;
          ph ^= 1u << (3 + j);
          mbar_arrive_cnt(&empty[rel.slot], kConsumerWarps);
          rel.advance(nst);
        }
        tc_fence_after();
        const uint64_t ad0 = smem_desc_sw128(xb0 + (uint32_t)j * (kXbufBytes / 2), 1024u);
        if (ok && !bar_wait(p, &full[rp.slot], rp.phase, task, true)) ok = false;
        if (ok) {
          // descriptors of the first K step; later steps add their byte
          // offset / 16 to the start-address field (no carry: < 256 KB).
          // One MMA covers every segment's rows (N = seg * Nr).
          const uint64_t bd0 = smem_desc_sw128(smem_addr(ring + (size_t)rp.slot * kStageBytes), 1024u);
#pragma unroll 1
          for (int q = 0; q < nkb * 4; ++q) {  // K block q / 4, K step q % 4
            const uint32_t kb = (uint32_t)q >> 2, ks = (uint32_t)q & 3u;
            tc_mma_bf16(taddr, ad0 + (uint64_t)(kb * (3072u >> 4) + ks * 2u), bd0 + (uint64_t)(kb * bstep + ks * 2u),
                        idesc, (kr | q) != 0 ? 1u : 0u);
          }
        }
        rp.advance(nst);
        tc_commit(&ctl->mma_bar[j]);
      }
      tc_commit(&ctl->acc_full);
      for (int kr = max(nkr - 2, 0); kr < nkr; ++kr) {  // the last ranges' slots
        const int j = kr & 1;
        if (!bar_wait(p, &ctl->mma_bar[j], (ph >> (3 + j)) & 1u, task, false)) ok = false;
        ph ^= 1u << (3 + j);
        mbar_arrive_cnt(&empty[rel.slot], kConsumerWarps);
        rel.advance(nst);
      }
    }
  }
}

// ------------------------------------------------------------------ attention bodies
// Token t (= the descriptor's step) of sequence s: its rotated key and its
// value go to row pos + t of the (s, g) cache block.
__device__ void append_task(Ctx& c, const mk_task_descriptor& d) {
  const KParams& p = *c.p;
  const int s = d.reserved[0], g = d.reserved[1], Hkv = d.reserved[2] & 0xFFFFu;
  const int T = (int)(d.reserved[2] >> 16) + 1, t_ = d.step;
  const int D = d.n, Hq = d.k, cap = d.kv_len, half = D / 2;
  const int pos = ld_relaxed(c.state + 2 * s + 1) + t_;
  if (pos < 0 || pos >= cap || t_ >= T) {
    if (threadIdx.x == 0) raise_error(p, MK_DEV_CAPACITY, c.task);
    return;
  }
  const size_t seq = (size_t)(s * T + t_) * (Hq + 2 * Hkv) * D;
  const float* qkv = rec_ptr<const float>(c, kPIn0) + seq;
  const uint64_t* qm = rec_ptr<const uint64_t>(c, kMirX);  // tagged qkv (MEGA, one or two rows), else null
  __nv_bfloat16* Kc = rec_ptr<__nv_bfloat16>(c, kPIn1);
  __nv_bfloat16* Vc = rec_ptr<__nv_bfloat16>(c, kPIn2);
  const size_t row = (((size_t)s * Hkv + g) * cap + pos) * D;
  const int t = threadIdx.x;
  const size_t ko = (size_t)Hq * D + (size_t)g * D + (t < half ? t : 0);
  const size_t vo = (size_t)(Hq + Hkv) * D + (size_t)g * D + (t < D ? t : 0);
  const float cs = t < half ? __ldg(p.rope_cos + (size_t)pos * p.rope_half + t) : 1.f;
  const float sn = t < half ? __ldg(p.rope_sin + (size_t)pos * p.rope_half + t) : 0.f;
  float k1 = 0.f, k2 = 0.f, vv = 0.f;
  if (qm) {
    const uint64_t* const mm[3] = {qm + seq + ko, qm + seq + ko + half, qm + seq + vo};
    const bool use[3] = {t < half, t < half, t < D};
    float v[3];
    ll_gather<3>(p, c.task, mm, use, v);
    k1 = v[0];
    k2 = v[1];
    vv = v[2];
  } else {
    if (t < half) {
      k1 = __ldcg(qkv + ko);
      k2 = __ldcg(qkv + ko + half);
    }
    if (t < D) vv = __ldcg(qkv + vo);
  }
  if (t < half) {
    Kc[row + t] = __float2bfloat16_rn(k1 * cs - k2 * sn);
    Kc[row + t + half] = __float2bfloat16_rn(k2 * cs + k1 * sn);
  }
  if (t < D) Vc[row + t] = __float2bfloat16_rn(vv);
}

// Eight keys of the online softmax (base 2) for four query rows (a KV
// group's heads, or (token, head) rows of a chunk step).  Lane = 8 * row +
// slice: the lane holds dims {c * 64 + slice * 8 + [0, 8) : c < DS / 8} of
// its row's query (qr) and output (o), element c * 8 + e at dim c * 64 +
// slice * 8 + e, so that the 8 slices of a 16-byte load cover 128
// consecutive bytes (every bank once); m is its row's running max (equal in
// the row's 8 lanes) and l the running sum of the probabilities of the keys
// the lane scored (key `slice` of each group; the row's sum is the sum of
// its 8 lanes' l, taken once at the end).  Keys k0 .. k0 + 7 (nvalid of them
// real) are read from shared memory (rows of DS * 8 bf16 at kb and vb):
// each lane reads its slices of every key, so the four rows' lanes share
// each address.  A score needs a sum over the row's 8 lanes only: a
// transposed reduction leaves key `slice`'s score in that lane.  The row
// sees only its first nlive of the keys (causal masking in a chunk step;
// nvalid else).
template <int DS>
__device__ __forceinline__ void partial_group8(const float (&qr)[DS], float (&o)[DS], float& m, float& l,
                                               uint32_t kb, uint32_t vb, int k0, int nvalid, int nlive,
                                               bool hlive, int lane) {
  constexpr int D = DS * 8;
  const int sl = lane & 7;
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a = kb + (uint32_t)((k0 + (j < nvalid ? j : 0)) * D) * 2 + (uint32_t)sl * 16;
    float sc = 0.f;
#pragma unroll
    for (int c4 = 0; c4 < DS / 8; ++c4) {
      const uint4 w = lds128(a + c4 * 128);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        sc = fmaf(qr[c4 * 8 + 2 * t], bf_lo(u[t]), sc);
        sc = fmaf(qr[c4 * 8 + 2 * t + 1], bf_hi(u[t]), sc);
      }
    }
    v[j] = sc;
  }
  // transposed sum over the 8 lanes of the head: afterwards lane sl holds key sl's score
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    const int o2 = 4 >> t, n = 8 >> t;
    const bool up = (lane & o2) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o2);
    }
  }
  const bool live = hlive && sl < nlive;
  float gmax = live ? v[0] : -INFINITY;
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
  const float mnew = fmaxf(m, gmax);
  const float pr = live ? exp2f(v[0] - mnew) : 0.f;
  const float sa = exp2f(m - mnew);  // 0 while m is -inf and mnew finite; exp2(nan) never: mnew >= m
  const float sc = mnew == -INFINITY ? 1.f : sa;
  l = fmaf(l, sc, pr);  // this lane's key only: the row's eight lanes are added once, at the end
#pragma unroll
  for (int e = 0; e < DS; ++e) o[e] *= sc;
  m = mnew;
  const int hb = lane & ~7;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float pj = __shfl_sync(0xffffffffu, pr, hb | j);
    const uint32_t a = vb + (uint32_t)((k0 + (j < nvalid ? j : 0)) * D) * 2 + (uint32_t)sl * 16;
#pragma unroll
    for (int c4 = 0; c4 < DS / 8; ++c4) {
      const uint4 w = lds128(a + c4 * 128);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        o[c4 * 8 + 2 * t] = fmaf(pj, bf_lo(u[t]), o[c4 * 8 + 2 * t]);
        o[c4 * 8 + 2 * t + 1] = fmaf(pj, bf_hi(u[t]), o[c4 * 8 + 2 * t + 1]);
      }
    }
  }
}

// Online softmax over one KV chunk for the G query heads of a KV group and
// the T tokens of a chunk step (T = 1: a decode step), NR = T * G query rows
// (token t, head h) = row t * G + h (log2 domain: scores are scaled by
// log2(e)/sqrt(D) and exponentials taken base 2).  Rows go in groups of four
// to WPG = 8 / ceil(NR / 4) warps, which split each ring slot's keys; row
// (t, h) sees keys up to pos + t.  This step's keys (positions pos ..) come
// from qkv, rotated and rounded to bf16 exactly as ATTENTION_APPEND stores
// them, so the partial does not wait for the appends.  Writes (m, l, o[D])
// per row to the chunk's scratch slot.
// The partial's inputs from qkv: qs [NR][D] the rotated query rows, scaled
// by log2(e) / sqrt(D) (row t * G + h: token t, head h of the KV group), and
// nkv this step's keys in the chunk [nn][D] then their values (from row T
// on), rotated and rounded to bf16 exactly as ATTENTION_APPEND stores them.
// CH: a chunk step (T >= 1 tokens); else a decode step, T = 1, specialised
// at compile time.  Ends before the barrier that publishes qs and nkv.
template <int DS, bool CH>
__device__ __forceinline__ void partial_stage(Ctx& c, const PartGeom& q, float* qs, uint16_t* nkv) {
  constexpr int D = DS * 8;
  const KParams& p = *c.p;
  const int tid = threadIdx.x;
  const int G = q.G, T = CH ? q.T : 1, NR = CH ? G * T : G, half = D / 2;
  const size_t rowlen = (size_t)(q.Hq + 2 * q.Hkv) * D;
  const size_t row0 = (size_t)q.s * q.T * rowlen;  // the sequence's first activation row
  const float* qkv = rec_ptr<const float>(c, kPIn0) + row0;
  const uint64_t* qm = rec_ptr<const uint64_t>(c, kMirX);  // tagged qkv (MEGA, one or two rows), else null
  if (qm) qm += row0;
  const float scale = 1.4426950408889634f / sqrtf((float)D);
  if constexpr (!CH) {
    // one pass, every load in flight at once: thread tid rotates query pair
    // (tid / half, tid % half) of the group's heads and, in the chunk that
    // holds the new token, stages dim tid of its key and value
    const bool act = tid < G * half, nact = q.has_new && tid < D;
    const int h = act ? tid / half : 0, j = tid - h * half;
    const int dd = tid, jj = dd < half ? dd : dd - half;
    const size_t o = (size_t)(q.g * G + h) * D + j;
    const size_t ko = (size_t)q.Hq * D + (size_t)q.g * D, vo = (size_t)(q.Hq + q.Hkv) * D + (size_t)q.g * D;
    // the table rows do not depend on qkv: their loads go out before the wait
    const size_t tr = (size_t)q.pos * p.rope_half;
    const float cs = act ? __ldg(p.rope_cos + tr + j) : 1.f, sn = act ? __ldg(p.rope_sin + tr + j) : 0.f;
    const float ncs = nact ? __ldg(p.rope_cos + tr + jj) : 1.f, nsn = nact ? __ldg(p.rope_sin + tr + jj) : 0.f;
    float v[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
    if (qm) {
      const uint64_t* const mm[5] = {qm + o, qm + o + half, qm + ko + jj, qm + ko + jj + half, qm + vo + dd};
      const bool use[5] = {act, act, nact, nact, nact};
      ll_gather<5>(p, c.task, mm, use, v);
    } else {
      if (act) {
        v[0] = __ldcg(qkv + o);
        v[1] = __ldcg(qkv + o + half);
      }
      if (nact) {
        v[2] = __ldcg(qkv + ko + jj);
        v[3] = __ldcg(qkv + ko + jj + half);
        v[4] = __ldcg(qkv + vo + dd);
      }
    }
    if (act) {
      qs[h * D + j] = (v[0] * cs - v[1] * sn) * scale;
      qs[h * D + j + half] = (v[1] * cs + v[0] * sn) * scale;
    }
    if (nact) {
      const float kr = dd < half ? v[2] * ncs - v[3] * nsn : v[3] * ncs + v[2] * nsn;
      nkv[dd] = __bfloat16_as_ushort(__float2bfloat16_rn(kr));
      nkv[D + dd] = __bfloat16_as_ushort(__float2bfloat16_rn(v[4]));
    }
  } else {
  // RoPE on the rows' queries: item (row, j) rotates the pair (j, j + D/2)
  for (int base = 0; base < NR * half; base += kConsumerThreads) {
    const int i = base + tid;
    const bool act = i < NR * half;
    const int r = act ? i / half : 0, j = i - r * half;
    const int t = r / G, h = r - t * G;
    const size_t o = (size_t)t * rowlen + (size_t)(q.g * G + h) * D + j;
    // the table rows do not depend on qkv: their loads go out before the wait
    const size_t tr = (size_t)(q.pos + t) * p.rope_half + j;
    const float cs = act ? __ldg(p.rope_cos + tr) : 1.f;
    const float sn = act ? __ldg(p.rope_sin + tr) : 0.f;
    float a, b;
    if (qm) {
      const uint64_t* const mm[2] = {qm + o, qm + o + half};
      const bool use[2] = {act, act};
      float v[2];
      ll_gather<2>(p, c.task, mm, use, v);
      a = v[0];
      b = v[1];
    } else {
      a = act ? __ldcg(qkv + o) : 0.f;
      b = act ? __ldcg(qkv + o + half) : 0.f;
    }
    if (act) {
      qs[r * D + j] = (a * cs - b * sn) * scale;
      qs[r * D + j + half] = (b * cs + a * sn) * scale;
    }
  }
  // this step's keys in the chunk, positions nb0 .. nb0 + nn - 1: key kk
  // is token nb0 + kk - pos's row of qkv
  for (int base = 0; base < q.nn * D; base += kConsumerThreads) {
    const int i = base + tid;
    const bool act = i < q.nn * D;
    const int kk = act ? i / D : 0, dd = i - kk * D;
    const int pk = q.nb0 + kk, jj = dd < half ? dd : dd - half;
    const size_t rb = (size_t)(pk - q.pos) * rowlen;
    const size_t ko = rb + (size_t)q.Hq * D + (size_t)q.g * D, vo = rb + (size_t)(q.Hq + q.Hkv) * D + (size_t)q.g * D;
    const float cs = act ? p.rope_cos[(size_t)pk * p.rope_half + jj] : 1.f;
    const float sn = act ? p.rope_sin[(size_t)pk * p.rope_half + jj] : 0.f;
    float k1 = 0.f, k2 = 0.f, vv = 0.f;
    if (qm) {
      const uint64_t* const mm[3] = {qm + ko + jj, qm + ko + jj + half, qm + vo + dd};
      const bool use[3] = {act, act, act};
      float v[3];
      ll_gather<3>(p, c.task, mm, use, v);
      k1 = v[0];
      k2 = v[1];
      vv = v[2];
    } else if (act) {
      k1 = __ldcg(qkv + ko + jj);
      k2 = __ldcg(qkv + ko + jj + half);
      vv = __ldcg(qkv + vo + dd);
    }
    if (act) {
      const float kr = dd < half ? k1 * cs - k2 * sn : k2 * cs + k1 * sn;
      nkv[kk * D + dd] = __bfloat16_as_ushort(__float2bfloat16_rn(kr));
      nkv[(T + kk) * D + dd] = __bfloat16_as_ushort(__float2bfloat16_rn(vv));
    }
  }
  }
}

// CH: a chunk step (T >= 1 tokens, loops over rows and keys); else a decode
// step, T = 1, specialised at compile time.
template <int DS, bool CH>  // dims per lane: D / 8
__device__ void partial_body(Ctx& c, const mk_task_descriptor& d, const PartGeom& q) {
  constexpr int D = DS * 8;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = q.G, T = CH ? q.T : 1, NR = CH ? G * T : G;
  const int NGR = CH ? (NR + 3) >> 2 : 1;                  // groups of four rows
  const int WPG = CH ? kConsumerWarps / NGR : kConsumerWarps;  // warps per group
  const int grp = CH ? warp / WPG : 0, sub = warp - grp * WPG;
  const bool wlive = grp < NGR;
  const int rr = grp * 4 + (lane >> 3), sl = lane & 7;
  const bool hlive = wlive && rr < NR;
  const int tq = CH && hlive ? rr / G : 0;  // the row's token
  // shared scratch: qs [NR][D] rotated, scaled queries; nkv this step's keys
  // [T][D] then values [T][D] (bf16); mrg [8 warps][4][D + 2] after them,
  // or over them (after a barrier) when the three do not fit side by side
  float* qs = c.scratch;
  uint16_t* nkv = reinterpret_cast<uint16_t*>(c.scratch + NR * D);
  const bool mrg_apart = (NR * D * 4 + 2 * T * D * 2 + kConsumerWarps * 4 * (D + 2) * 4) <= kScratchBytes;
  float* mrg = mrg_apart ? c.scratch + NR * D + T * D : c.scratch;  // nkv takes T * D floats
  partial_stage<DS, CH>(c, q, qs, nkv);
  cbar();
  float qr[DS], o[DS], m = -INFINITY, l = 0.f;
#pragma unroll
  for (int e = 0; e < DS; ++e) {  // element e: dim (e / 8) * 64 + sl * 8 + e % 8
    qr[e] = hlive ? qs[rr * D + (e >> 3) * 64 + sl * 8 + (e & 7)] : 0.f;
    o[e] = 0.f;
  }
  const int kpw = q.R / WPG;  // keys per warp per slot (a multiple of 8)
  for (int i = 0; i < q.nstage; ++i) {
    const int nr = min(q.R, q.jst - (q.j0 + i * q.R));
    const uint32_t slot = consume_begin(c);
    if (i == 0) trace_mark(c, 0);
    const uint32_t kb = smem_addr(c.ring + (size_t)slot * kStageBytes);
    const uint32_t vb = kb + kStageBytes / 2;
    if (wlive)  // cached keys precede every row's own position
      for (int k0 = sub * kpw; k0 < min(nr, (sub + 1) * kpw); k0 += 8)
        partial_group8<DS>(qr, o, m, l, kb, vb, k0, min(8, nr - k0), min(8, nr - k0), hlive, lane);
    consume_end(c, slot);
  }
  if (q.has_new && wlive && sub == WPG - 1) {
    // this step's keys last: row (t, h) sees those at positions <= pos + t
    const uint32_t nb = smem_addr(nkv);
    const int nlive = max(0, min(q.nn, q.pos + tq + 1 - q.nb0));
    partial_group8<DS>(qr, o, m, l, nb, nb + T * D * 2, 0, q.nn, nlive, hlive, lane);
  }
  trace_mark(c, 1);
  // each of a row's eight lanes summed the probabilities of its own keys
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (!mrg_apart) cbar();  // every warp is done with qs and nkv, which the merge area overlays
  // merge the warps of each row group
  if (hlive) {
    float* r = mrg + (warp * 4 + (lane >> 3)) * (D + 2);
    if (sl == 0) {
      r[0] = m;
      r[1] = l;
    }
#pragma unroll
    for (int e = 0; e < DS; ++e) r[2 + (e >> 3) * 64 + sl * 8 + (e & 7)] = o[e];
  }
  cbar();
  float* scr = rec_ptr<float>(c, kPOut) + (size_t)q.slot * NR * (D + 2);
  uint64_t* sm = rec_ptr<uint64_t>(c, kMirOut);  // the record's tagged pairs (read by a tagged combine), or null
  if (sm) sm += (size_t)q.slot * NR * (D + 2);
  for (int i = tid; i < NR * D; i += kConsumerThreads) {
    const int r = i / D, e = i - r * D;
    const int w0 = (r >> 2) * WPG, rs = r & 3;
    float M = -INFINITY;
    for (int w = w0; w < w0 + WPG; ++w) M = fmaxf(M, mrg[(w * 4 + rs) * (D + 2)]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = w0; w < w0 + WPG; ++w) {
        const float* rp = mrg + (w * 4 + rs) * (D + 2);
        const float f = exp2f(rp[0] - M);
        Ls = fmaf(rp[1], f, Ls);
        O = fmaf(rp[2 + e], f, O);
      }
    }
    scr[r * (D + 2) + 2 + e] = O;
    if (sm) st_relaxed_u64(sm + r * (D + 2) + 2 + e, ll_pack(O, c.p->tag));
    if (e == 0) {
      scr[r * (D + 2)] = M;
      scr[r * (D + 2) + 1] = Ls;
      if (sm) st_relaxed_v2u64(sm + r * (D + 2), ll_pack(M, c.p->tag), ll_pack(Ls, c.p->tag));
    }
  }
}

// Split-KV partial on tensor cores, for at most four query rows (token t,
// head h = row t * G + h).  The query tile (the three bf16 parts of each
// rotated, scaled query row: tile row 3 r + part) is staged once; per block
// of kKeyBlock cached keys the MMA warp computes S^T = K Q^T into a score
// buffer.  Warps 0-3 (softmax warps; one key per thread: tensor-memory lane
// = key) add the parts, take the block's row maxima, the new running maxima
// and the probabilities p = 2^(s - m) (a block-wise online softmax: the
// output sums of a block share one scale per row) and hand them, with the
// rescale factors, to warps 4-7 (P V warps), which accumulate P V on CUDA
// cores (warp w: keys w - 4, w, ...; lane: D / 32 dims) from the block's V
// rows while the softmax warps go on to the next block.  This step's keys
// (from qkv) are block 0 of that hand-off when the chunk holds some.  At
// the end the four P V warps' sums are added in warp order.
template <int DS, bool CH>
__device__ void tc_partial_body(Ctx& c, const mk_task_descriptor& d, const PartGeom& q) {
  constexpr int D = DS * 8;
  constexpr int DQ = D / 32;     // dims per lane in P V
  constexpr uint32_t NQ = 16;    // query tile rows
  const KParams& p = *c.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  TcCtl* ctl = c.ctl;
  const int G = q.G, NR = CH ? G * q.T : G;  // at most 4
  // shared scratch from its first 1024-byte boundary: the query tile
  // [D / 64][NQ][128 B] (4 KB), probabilities [2][kKeyBlock][4] (4 KB), qs
  // [4][D] (2 KB), nkv [2 T][D] bf16 (2 KB), block maxima and sums, rescale
  // factors, this step's key scores; at the end the P V warps' output sums
  // [4][4][D] (8 KB) over the tile
  const uint32_t s0 = smem_addr(c.scratch), sb = (s0 + 1023u) & ~1023u;
  uint8_t* base = reinterpret_cast<uint8_t*>(c.scratch) + (sb - s0);
  const uint32_t qt = sb;
  float* pb = reinterpret_cast<float*>(base + 4096);
  float* qs = reinterpret_cast<float*>(base + 8192);
  uint16_t* nkv = reinterpret_cast<uint16_t*>(base + 10240);
  float* red = reinterpret_cast<float*>(base + 12288);  // [2][32] maxima and sums, [2][4] factors, [32] new-key scores, [8] m, l
  float* osum = reinterpret_cast<float*>(base);
  if (tid == 0) {  // the MMA warp takes the task and waits for the query tile
    ctl->mb_task = c.task;
    ctl->mb_slot = c.rp.slot;
    ctl->mb_phase = c.rp.phase;
    ctl->mb_nblk = (uint32_t)q.nblk;
    ctl->mb_qt = qt;
    mbar_arrive(&ctl->task_go);
  }
  partial_stage<DS, CH>(c, q, qs, nkv);
  cbar();
  // query tile: dims (d2, d2 + 1) of row r, split into three bf16 parts
  // (each the rounding of what the previous leave), at tile rows 3 r + part
  for (int i = tid; i < NR * (D / 2); i += kConsumerThreads) {
    const int r = i / (D / 2), d2 = (i - r * (D / 2)) * 2;
    float v0 = qs[r * D + d2], v1 = qs[r * D + d2 + 1];
    const uint32_t kb = (uint32_t)d2 >> 6, kk = (uint32_t)d2 & 63u;
    const uint32_t ch = kk >> 3, cb = (kk & 7u) * 2u;
#pragma unroll
    for (int pt = 0; pt < 3; ++pt) {
      const __nv_bfloat162 a = __float22bfloat162_rn(make_float2(v0, v1));
      const uint32_t w = *reinterpret_cast<const uint32_t*>(&a);
      v0 -= bf_lo(w);
      v1 -= bf_hi(w);
      const uint32_t ra = qt + kb * (NQ * 128u) + (uint32_t)(3 * r + pt) * 128u;
      sts32(ra + ((ch ^ ((ra >> 7) & 7u)) << 4) + cb, w);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(&ctl->q_full);
  // hand-off blocks: this step's keys first (if any), then the cached blocks
  const int nb0 = q.has_new ? 1 : 0, nvb = nb0 + q.nblk;
  float o[4][DQ];  // P V warps: the output sums of rows 0-3 over this lane's dims
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int e = 0; e < DQ; ++e) o[r][e] = 0.f;
  if (warp < 4) {
    // ---- softmax warps
    float* ns = red + 72;  // [8 keys][4 rows] scores of this step's keys
    float m[4], l[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
    }
    if (q.has_new) {  // score (kk, r) by softmax warp (kk * NR + r) % 4
      for (int it = warp; it < q.nn * NR; it += 4) {
        const int kk = it / NR, r = it - kk * NR;
        float sc = 0.f;
#pragma unroll
        for (int e = 0; e < DQ; ++e)
          sc = fmaf(qs[r * D + lane * DQ + e], __uint_as_float((uint32_t)nkv[kk * D + lane * DQ + e] << 16), sc);
        sc = warp_sum(sc);
        const int tq = CH ? r / G : 0;  // row r sees this step's keys up to its own token
        if (lane == 0) ns[kk * 4 + r] = (q.nb0 + kk <= q.pos + tq) ? sc : -INFINITY;
      }
      named_bar_sync(2, 128);
    }
    for (int v = 0; v < nvb; ++v) {
      const int j = v & 1, b = v - nb0;
      float* P = pb + j * kKeyBlock * 4;
      float* rb = red + j * 32;  // [4 warps][4] maxima, [4 warps][4] sums
      const int key = warp * 32 + lane;
      float sc[4];
      if (b < 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) sc[r] = (key < q.nn && r < NR) ? ns[key * 4 + r] : -INFINITY;
      } else {
        const int nv = min(kKeyBlock, q.jst - (q.j0 + b * kKeyBlock));  // real keys in the block
        const int jb = b & 1;
        bar_wait(p, &ctl->s_full[jb], (c.tc_ph >> (3 + jb)) & 1u, c.task, false);  // every lane waits
        c.tc_ph ^= 1u << (3 + jb);
        if (b == 0) trace_mark(c, 0);
        tc_fence_after();
        float s16[16];
        tmem_ld16(c.taddr + ((uint32_t)(warp * 32) << 16) + c.pcol + (uint32_t)jb * NQ, s16);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (b + 2 < q.nblk) mbar_arrive(&ctl->s_empty[jb]);  // the MMA warp may refill the buffer
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
          sc[r] = (key < nv && r < NR) ? s16[3 * r] + s16[3 * r + 1] + s16[3 * r + 2] : -INFINITY;
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float mx = warp_max(sc[r]);
        if (lane == 0) rb[warp * 4 + r] = mx;
      }
      named_bar_sync(2, 128);
      float mn[4], pr[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float bm = fmaxf(fmaxf(rb[r], rb[4 + r]), fmaxf(rb[8 + r], rb[12 + r]));
        mn[r] = fmaxf(m[r], bm);
        pr[r] = sc[r] == -INFINITY ? 0.f : exp2f(sc[r] - mn[r]);
      }
      if (v >= 2) {  // the P V warps are done with buffer j (hand-off v - 2)
        bar_wait(p, &ctl->p_empty[j], (c.tc_ph >> (5 + j)) & 1u, c.task, false);  // every lane waits
        c.tc_ph ^= 1u << (5 + j);
      }
      *reinterpret_cast<float4*>(P + key * 4) = make_float4(pr[0], pr[1], pr[2], pr[3]);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float sm = warp_sum(pr[r]);
        if (lane == 0) rb[16 + warp * 4 + r] = sm;
      }
      named_bar_sync(2, 128);
      float* fac = red + 64 + j * 4;  // the rescale factors of hand-off v
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float al = mn[r] == -INFINITY ? 1.f : exp2f(m[r] - mn[r]);  // 0 while m is -inf and mn finite
        l[r] = fmaf(l[r], al, (rb[16 + r] + rb[20 + r]) + (rb[24 + r] + rb[28 + r]));
        m[r] = mn[r];
        if (tid == r) fac[r] = al;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[j]);  // release: the probabilities and factors
      if (b >= 0) {
        if (D == 128) c.rp.advance(c.nst);  // the K slot: the MMA warp hands it back
        // the V slot (or the block's slot at D = 64): the P V warps read it;
        // these warps count themselves in once it has been filled
        const uint32_t vslot = consume_begin(c);
        consume_end(c, vslot);
      }
    }
    trace_mark(c, 1);
#pragma unroll
    for (int r = 0; r < 4; ++r) {  // m and l of the rows, for the record
      if (tid == r) {
        red[104 + r] = m[r];
        red[108 + r] = l[r];
      }
    }
  } else {
    // ---- P V warps
    const int w4 = warp - 4;
    for (int v = 0; v < nvb; ++v) {
      const int j = v & 1, b = v - nb0;
      bar_wait(p, &ctl->p_full[j], (c.tc_ph >> (7 + j)) & 1u, c.task, false);  // every lane waits
      c.tc_ph ^= 1u << (7 + j);
      const float* fac = red + 64 + j * 4;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float al = fac[r];
#pragma unroll
        for (int e = 0; e < DQ; ++e) o[r][e] *= al;
      }
      int nv;
      uint32_t vb, vslot = 0;
      if (b < 0) {
        nv = q.nn;
        vb = smem_addr(nkv + q.T * D);  // this step's values
      } else {
        nv = min(kKeyBlock, q.jst - (q.j0 + b * kKeyBlock));
        if (D == 128) c.rp.advance(c.nst);  // the K slot: the MMA warp hands it back
        vslot = consume_begin(c);
        vb = smem_addr(c.ring + (size_t)vslot * kStageBytes) + (D == 128 ? 0u : kKeyBlock * 128u);
      }
      const uint32_t pa = smem_addr(pb + j * kKeyBlock * 4);
      for (int k = w4; k < nv; k += 4) {
        const uint4 pw = lds128(pa + (uint32_t)k * 16u);
        const float pk[4] = {__uint_as_float(pw.x), __uint_as_float(pw.y), __uint_as_float(pw.z),
                             __uint_as_float(pw.w)};
        float vv[DQ];
        if constexpr (DQ == 4) {
          const uint2 w = lds64(vb + (uint32_t)(k * D + lane * 4) * 2u);
          vv[0] = bf_lo(w.x); vv[1] = bf_hi(w.x); vv[2] = bf_lo(w.y); vv[3] = bf_hi(w.y);
        } else {
          const uint32_t w = lds32(vb + (uint32_t)(k * D + lane * 2) * 2u);
          vv[0] = bf_lo(w); vv[1] = bf_hi(w);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int e = 0; e < DQ; ++e) o[r][e] = fmaf(pk[r], vv[e], o[r][e]);
      }
      __syncwarp();
      if (lane == 0 && v + 2 < nvb) mbar_arrive(&ctl->p_empty[j]);  // the softmax warps may rewrite buffer j
      if (b >= 0) consume_end(c, vslot);
    }
  }
  cbar();  // every warp is done with the tile, the probabilities, qs and nkv; m and l are parked
  if (warp >= 4) {  // the P V warps' sums overlay the tile
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < DQ; ++e) osum[((warp - 4) * 4 + r) * D + lane * DQ + e] = o[r][e];
  }
  cbar();
  float* scr = rec_ptr<float>(c, kPOut) + (size_t)q.slot * NR * (D + 2);
  uint64_t* sm = rec_ptr<uint64_t>(c, kMirOut);  // the record's tagged pairs (read by a tagged combine), or null
  if (sm) sm += (size_t)q.slot * NR * (D + 2);
  for (int i = tid; i < NR * D; i += kConsumerThreads) {
    const int r = i / D, e = i - r * D;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) O += osum[(w * 4 + r) * D + e];
    scr[r * (D + 2) + 2 + e] = O;
    if (sm) st_relaxed_u64(sm + r * (D + 2) + 2 + e, ll_pack(O, c.p->tag));
    if (e == 0) {
      scr[r * (D + 2)] = red[104 + r];
      scr[r * (D + 2) + 1] = red[108 + r];
      if (sm) st_relaxed_v2u64(sm + r * (D + 2), ll_pack(red[104 + r], c.p->tag), ll_pack(red[108 + r], c.p->tag));
    }
  }
}

// The B <= 2 kernel has no tensor-core partials (its graphs carry no K-cache
// tensor maps): its decode chunks are short, and the code it would add to
// the consumer costs the hot GEMV loops more than it could save.
template <int BCLASS>
__device__ void partial_task(Ctx& c, const mk_task_descriptor& d) {
  PartGeom q;
  part_geom(c.state, d, q);
  if (q.bad) {
    if (threadIdx.x == 0) raise_error(*c.p, MK_DEV_CAPACITY, c.task);
    return;
  }
  if (BCLASS > 0 && tc_partial(d, c.rec->tm_rows, q.nblk)) {
    if constexpr (BCLASS > 0) {
      if (q.T == 1) {
        if (q.D == 128) tc_partial_body<16, false>(c, d, q);
        else tc_partial_body<8, false>(c, d, q);
      } else {
        if (q.D == 128) tc_partial_body<16, true>(c, d, q);
        else tc_partial_body<8, true>(c, d, q);
      }
    }
  } else if (q.T == 1) {
    if (q.D == 128) partial_body<16, false>(c, d, q);
    else partial_body<8, false>(c, d, q);
  } else {
    if (q.D == 128) partial_body<16, true>(c, d, q);
    else partial_body<8, true>(c, d, q);
  }
}

// Log-sum-exp merge of the P partials of one (sequence, kv head):
// out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k with M = max_k m_k;
// empty partials (m = -inf) add nothing.  Up to 32 partials, 8 / G warps
// serve each head: lane k reads partial k's (m, l) while every lane reads
// its output dims of all P partials at once (one L2 round trip), then the
// weights travel by shuffles.  More partials go through a running merge.
__device__ __forceinline__ void lse_fold(float& M, float& Ls, float& O0, float& O1, float m, float l, float o0,
                                         float o1) {
  if (m != -INFINITY) {
    const float Mn = fmaxf(M, m);
    const float a = exp2f(M - Mn), b = exp2f(m - Mn);
    Ls = fmaf(Ls, a, l * b);
    O0 = fmaf(O0, a, o0 * b);
    O1 = fmaf(O1, a, o1 * b);
    M = Mn;
  }
}

// Partials whose tagged records a decode combine loads at once (the 32
// partials of a full warp would take 128 registers of pairs).
constexpr int kCombGroup = 16;

__device__ void combine_task(Ctx& c, const mk_task_descriptor& d) {
  const KParams& p = *c.p;
  const int s = d.reserved[0], g = d.reserved[1], Hkv = d.reserved[2] & 0xFFFFu;
  const int T = (int)(d.reserved[2] >> 16) + 1;
  const int P = d.reserved[3], base = d.reserved[4];
  const int D = d.n, Hq = d.k, G = Hq / Hkv, NR = T * G;  // query rows (token t, head h) = t * G + h
  const int rec = NR * (D + 2);
  const float* scr = rec_ptr<const float>(c, kPIn0) + (size_t)base * rec;
  float* out = rec_ptr<float>(c, kPOut);
  uint64_t* om = rec_ptr<uint64_t>(c, kMirOut);
  const uint64_t* sm = rec_ptr<const uint64_t>(c, kMirX);  // the partials' tagged records (MEGA), or null
  if (P <= 32 && T == 1 && kConsumerWarps % G == 0) {
    // decode step: 8 / G warps per head, two output dims per lane; lane k
    // reads partial k's (m, l) while every lane reads its dims of all P
    // partials at once (one L2 round trip).  With tagged records this task
    // waited for no partial: while some lane holds a stale pair, the lowest
    // such lane polls it and the warp reloads what is stale.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wph = kConsumerWarps / G;
    const int h = warp / wph, dpw = D / wph;
    const int e = (warp % wph) * dpw + lane * 2;
    const bool mine = lane * 2 < dpw;
    if (sm) {
      // tagged records: (m, l) of partial `lane`, then the dims of the
      // partials in groups of kCombGroup (4 registers of pairs each in flight)
      const uint64_t* r = sm + (size_t)base * rec + h * (D + 2);
      ulonglong2 ml = lane < P ? ld_relaxed_v2u64(r + (size_t)lane * rec)
                               : make_ulonglong2(ll_pack(-INFINITY, p.tag), ll_pack(0.f, p.tag));
      float M = 0.f, L = 1.f, wk = 0.f, a0 = 0.f, a1 = 0.f;
      for (int k0 = 0; k0 < P; k0 += kCombGroup) {
        ulonglong2 qv[kCombGroup];
#pragma unroll
        for (int k = 0; k < kCombGroup; ++k)
          qv[k] = (k0 + k < P && mine) ? ld_relaxed_v2u64(r + (size_t)(k0 + k) * rec + 2 + e)
                                       : make_ulonglong2(ll_pack(0.f, p.tag), ll_pack(0.f, p.tag));
        for (;;) {  // while a lane holds stale pairs, the lowest such lane polls one
          uint32_t stale = (k0 == 0 && !(ll_ready(ml.x, p.tag) && ll_ready(ml.y, p.tag))) ? 1u << kCombGroup : 0u;
#pragma unroll
          for (int k = 0; k < kCombGroup; ++k)
            stale |= (ll_ready(qv[k].x, p.tag) && ll_ready(qv[k].y, p.tag)) ? 0u : 1u << k;
          const uint32_t want = __ballot_sync(0xffffffffu, stale != 0);
          if (!want) break;
          const int leader = __ffs(want) - 1;
          const int k = stale ? __ffs(stale) - 1 : 0;
          const uint64_t* pr = k == kCombGroup ? r + (size_t)lane * rec : r + (size_t)(k0 + k) * rec + 2 + e;
          // the stale half of the leader's pair of pairs
          bool second = ll_ready(ml.x, p.tag);
#pragma unroll
          for (int kk = 0; kk < kCombGroup; ++kk)  // no dynamic register indexing
            if (kk == k) second = ll_ready(qv[kk].x, p.tag);
          if (!ll_poll_warp(p, pr + (second ? 1 : 0), leader, c.task)) break;  // abort or timeout: carry on
          if (stale >> kCombGroup) ml = ld_relaxed_v2u64(r + (size_t)lane * rec);
#pragma unroll
          for (int k = 0; k < kCombGroup; ++k)
            if (stale & (1u << k)) qv[k] = ld_relaxed_v2u64(r + (size_t)(k0 + k) * rec + 2 + e);
        }
        if (k0 == 0) {
          const float mk = __uint_as_float((uint32_t)ml.x), lk = __uint_as_float((uint32_t)ml.y);
          M = warp_max(mk);
          wk = mk == -INFINITY ? 0.f : exp2f(mk - M);
          L = warp_sum(wk * lk);
        }
#pragma unroll
        for (int k = 0; k < kCombGroup; ++k) {
          const float w = __shfl_sync(0xffffffffu, wk, (k0 + k) & 31);
          a0 = fmaf(w, __uint_as_float((uint32_t)qv[k].x), a0);
          a1 = fmaf(w, __uint_as_float((uint32_t)qv[k].y), a1);
        }
      }
      if (mine) {
        const float inv = 1.f / L;
        const size_t o = (size_t)s * Hq * D + (size_t)(g * G + h) * D + e;
        *reinterpret_cast<float2*>(out + o) = make_float2(a0 * inv, a1 * inv);
        if (om) st_relaxed_v2u64(om + o, ll_pack(a0 * inv, p.tag), ll_pack(a1 * inv, p.tag));
      }
      return;
    }
    const float* r = scr + h * (D + 2);
    const float mk = lane < P ? __ldcg(r + (size_t)lane * rec) : -INFINITY;
    const float lk = lane < P ? __ldcg(r + (size_t)lane * rec + 1) : 0.f;
    float2 ov[32];
#pragma unroll
    for (int k = 0; k < 32; ++k)
      ov[k] = (k < P && mine) ? __ldcg(reinterpret_cast<const float2*>(r + (size_t)k * rec + 2 + e))
                              : make_float2(0.f, 0.f);
    const float M = warp_max(mk);
    const float wk = mk == -INFINITY ? 0.f : exp2f(mk - M);
    const float L = warp_sum(wk * lk);
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float w = __shfl_sync(0xffffffffu, wk, k);
      a0 = fmaf(w, ov[k].x, a0);
      a1 = fmaf(w, ov[k].y, a1);
    }
    if (mine) {
      const float inv = 1.f / L;
      const size_t o = (size_t)s * Hq * D + (size_t)(g * G + h) * D + e;
      *reinterpret_cast<float2*>(out + o) = make_float2(a0 * inv, a1 * inv);
      if (om) st_relaxed_v2u64(om + o, ll_pack(a0 * inv, p.tag), ll_pack(a1 * inv, p.tag));
    }
    return;
  }
  if (P <= 32) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // wpr warps share a row (its dims split between them) when the rows
    // divide the 8 warps, else each warp takes whole rows in turn
    const int wpr = (NR <= kConsumerWarps && kConsumerWarps % NR == 0) ? kConsumerWarps / NR : 1;
    const int dpw = D / wpr;
    for (int u = warp; u < NR * wpr; u += kConsumerWarps) {
      const int r = u / wpr, part = u - r * wpr;
      const int t = r / G, h = r - t * G;
      const float* rp = scr + r * (D + 2);
      // lane k reads partial k's (m, l) while every lane reads its first two
      // output dims of all P partials: one L2 round trip
      const float mk = lane < P ? __ldcg(rp + (size_t)lane * rec) : -INFINITY;
      const float lk = lane < P ? __ldcg(rp + (size_t)lane * rec + 1) : 0.f;
      const int e1 = (part + 1) * dpw;  // this warp's dims: [part * dpw, e1), two per lane
      float2 ov[32];
#pragma unroll
      for (int k = 0; k < 32; ++k)
        ov[k] = (k < P && part * dpw + lane * 2 < e1)
                    ? __ldcg(reinterpret_cast<const float2*>(rp + (size_t)k * rec + 2 + part * dpw + lane * 2))
                    : make_float2(0.f, 0.f);
      const float M = warp_max(mk);
      const float wk = mk == -INFINITY ? 0.f : exp2f(mk - M);
      const float L = warp_sum(wk * lk);
      const float inv = 1.f / L;
      const size_t ob = (size_t)(s * T + t) * Hq * D + (size_t)(g * G + h) * D;
      for (int e0 = part * dpw; e0 < e1; e0 += 64) {
        const int e = e0 + lane * 2;
        const bool mine = e < e1;
        if (e0 != part * dpw) {  // a whole row of D = 128 per warp: the second 64 dims
#pragma unroll
          for (int k = 0; k < 32; ++k)
            ov[k] = (k < P && mine) ? __ldcg(reinterpret_cast<const float2*>(rp + (size_t)k * rec + 2 + e))
                                    : make_float2(0.f, 0.f);
        }
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float w = __shfl_sync(0xffffffffu, wk, k);
          a0 = fmaf(w, ov[k].x, a0);
          a1 = fmaf(w, ov[k].y, a1);
        }
        if (mine) {
          *reinterpret_cast<float2*>(out + ob + e) = make_float2(a0 * inv, a1 * inv);
          if (om) st_relaxed_v2u64(om + ob + e, ll_pack(a0 * inv, p.tag), ll_pack(a1 * inv, p.tag));
        }
      }
    }
    return;
  }
  // each thread produces two adjacent outputs (e, e + 1) of one row
  for (int i = threadIdx.x; i < NR * D / 2; i += kConsumerThreads) {
    const int r = (2 * i) / D, e = (2 * i) % D;
    const int t = r / G, h = r - t * G;
    const float* rp = scr + r * (D + 2);
    float M = -INFINITY, Ls = 0.f, O0 = 0.f, O1 = 0.f;
    for (int k = 0; k < P; ++k) {
      const float* rr = rp + (size_t)k * rec;
      const float2 ov = __ldcg(reinterpret_cast<const float2*>(rr + 2 + e));
      lse_fold(M, Ls, O0, O1, __ldcg(rr), __ldcg(rr + 1), ov.x, ov.y);
    }
    const float inv = 1.f / Ls;
    const size_t o = (size_t)(s * T + t) * Hq * D + (size_t)(g * G + h) * D + e;
    *reinterpret_cast<float2*>(out + o) = make_float2(O0 * inv, O1 * inv);
    if (om) st_relaxed_v2u64(om + o, ll_pack(O0 * inv, p.tag), ll_pack(O1 * inv, p.tag));
  }
}

// Embedding gather of token t (the descriptor's step) of sequence s: token 0
// is the pending token in the state, later tokens of a chunk step come from
// the step's tokens buffer.
__device__ void embed_task(Ctx& c, const mk_task_descriptor& d) {
  const KParams& p = *c.p;
  const int s = d.reserved[0], V = d.reserved[1], H = d.n;
  const int T = (int)d.reserved[2] + 1, t = d.step, row = s * T + t;
  const int tok = t == 0 ? ld_relaxed(c.state + 2 * s) : rec_ptr<const int32_t>(c, kPIn1)[(size_t)s * T + t];
  if (tok < 0 || tok >= V || t >= T) {
    if (threadIdx.x == 0) raise_error(p, MK_DEV_BAD_INDEX, c.task);
    return;
  }
  const uint16_t* E = rec_ptr<const uint16_t>(c, kPIn0) + (size_t)tok * H;
  float* out = rec_ptr<float>(c, kPOut) + (size_t)row * H;
  uint64_t* om = rec_ptr<uint64_t>(c, kMirOut);
  for (int i = threadIdx.x * 8; i < H; i += kConsumerThreads * 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(E + i));
    float4 a = make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
    float4 b = make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w));
    *reinterpret_cast<float4*>(out + i) = a;
    *reinterpret_cast<float4*>(out + i + 4) = b;
    if (om) {
      uint64_t* m = om + (size_t)row * H + i;
      const uint32_t t = p.tag;
      st_relaxed_v2u64(m, ll_pack(a.x, t), ll_pack(a.y, t));
      st_relaxed_v2u64(m + 2, ll_pack(a.z, t), ll_pack(a.w, t));
      st_relaxed_v2u64(m + 4, ll_pack(b.x, t), ll_pack(b.y, t));
      st_relaxed_v2u64(m + 6, ll_pack(b.z, t), ll_pack(b.w, t));
    }
  }
}

// Standalone RMS norm of one sequence's row ("mega kernel initial", OpId
// table): y = x (+ residual with FUSED_RESIDUAL); out = y / sqrt(mean(y^2)
// + eps) * gamma.  A rare op: two plain passes over the row (the second
// reads it again from L2), kept small.
__device__ void rmsnorm_task(Ctx& c, const mk_task_descriptor& d) {
  const KParams& p = *c.p;
  const int s = (int)d.reserved[0], H = d.n, tid = threadIdx.x;
  const float* x = rec_ptr<const float>(c, kPIn0) + (size_t)s * H;
  const uint16_t* gamma = rec_ptr<const uint16_t>(c, kPIn1);
  const float* res = (d.flags & MK_F_ADD_RESIDUAL) ? rec_ptr<const float>(c, kPIn2) + (size_t)s * H : nullptr;
  float* out = rec_ptr<float>(c, kPOut) + (size_t)s * H;
  uint64_t* om = rec_ptr<uint64_t>(c, kMirOut);
  float* red = c.scratch;
  float ss = 0.f;
#pragma unroll 1
  for (int i = tid; i < H; i += kConsumerThreads) {
    const float y = __ldcg(x + i) + (res ? __ldcg(res + i) : 0.f);
    ss = fmaf(y, y, ss);
  }
  const float t = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = t;
  cbar();
  if (tid == 0) {
    float tot = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) tot += red[w];
    red[kConsumerWarps] = 1.0f / sqrtf(tot / (float)H + __uint_as_float(d.reserved[1]));
  }
  cbar();
  const float inv = red[kConsumerWarps];
#pragma unroll 1
  for (int i = tid; i < H; i += kConsumerThreads) {
    const float y = __ldcg(x + i) + (res ? __ldcg(res + i) : 0.f);
    const float o = y * inv * __uint_as_float((uint32_t)__ldg(gamma + i) << 16);
    out[i] = o;
    if (om) st_relaxed_u64(om + (size_t)s * H + i, ll_pack(o, p.tag));
  }
}

// The argmax of the sequence's last activation row over the lm_head tiles'
// (max, index) pairs; a chunk step of TQ tokens also records its input
// tokens 1 .. TQ-1 in the history, and the state advances by TQ.
__device__ void sample_task(Ctx& c, const mk_task_descriptor& d) {
  const KParams& p = *c.p;
  const int s = d.reserved[0], TQ = (int)d.reserved[1] + 1, M = d.m * TQ, T = d.k, cap = d.kv_len;
  const int col = s * TQ + TQ - 1;
  const mk_argmax_pair* pairs = rec_ptr<const mk_argmax_pair>(c, kPIn0);
  float bv = -FLT_MAX;
  int bi = INT_MAX;
  for (int t = threadIdx.x; t < T; t += kConsumerThreads) {
    const float2 pr = __ldcg(reinterpret_cast<const float2*>(pairs + (size_t)t * M + col));
    const int idx = __float_as_int(pr.y);
    if (pr.x > bv || (pr.x == bv && idx < bi)) {
      bv = pr.x;
      bi = idx;
    }
  }
  block_argmax(bv, bi, c.scratch);
  if (threadIdx.x == 0) {
    int32_t* state = c.state;
    int32_t* hist = rec_ptr<int32_t>(c, kPOut);
    const int pos = ld_relaxed(state + 2 * s + 1);
    if (pos < 0 || pos + TQ >= cap) {
      raise_error(p, MK_DEV_CAPACITY, c.task);
      return;
    }
    const int32_t* toks = rec_ptr<const int32_t>(c, kPIn1);
    for (int t = 1; t < TQ; ++t) hist[(size_t)s * cap + pos + t] = toks[(size_t)s * TQ + t];
    hist[(size_t)s * cap + pos + TQ] = bi;
    state[2 * s] = bi;
    state[2 * s + 1] = pos + TQ;
  }
}

// ------------------------------------------------------------------ consumer loop
// Wait (consumer warp 0) until every counter the task's plan names reaches
// epoch * count.  Lane i polls entry i with acquire loads; entries are
// usually none (tagged inputs), one (a whole-group counter or the task's
// own) or two, taken from the task record.  An abort is noticed while
// waiting; a task whose counters are already met just runs.
// Counters and targets are uint32 and wrap (a whole-group counter that
// gains a few thousand per step wraps after about a million steps), so the
// test is on the signed difference: at the start of step e a counter holds
// (e - 1) * count, never more than count < 2^31 below its target.
__device__ __forceinline__ bool counter_met(const uint32_t* ctr, uint32_t target) {
  return (int32_t)(ld_acquire(ctr) - target) >= 0;
}

__device__ bool wait_deps(const KParams& p, const TaskRec* r, int task) {
  const int lane = threadIdx.x & 31;
  const uint32_t w0 = r->w0, nw = r->nw;
  for (uint32_t base = 0; base < nw; base += 32) {
    const uint32_t i = base + lane;
    const bool mine = i < nw;
    const uint32_t* ctr = p.counters;
    uint32_t target = 0;
    if (mine) {
      const uint2 e = i < 4 ? r->wi[i] : __ldg(p.wait + w0 + i);
      ctr = p.counters + e.x;
      target = p.epoch * e.y;
    }
    bool done = !mine || counter_met(ctr, target);
    if (__all_sync(0xffffffffu, done)) continue;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      if (!done) done = counter_met(ctr, target);
      if (__all_sync(0xffffffffu, done)) break;
      if ((it & 63u) == 0) {
        if (aborted(p)) return false;
        if (globaltimer() - t0 > p.timeout_ns) {
          if (lane == 0) raise_error(p, MK_DEV_DEP_TIMEOUT, task);
          return false;
        }
      }
    }
  }
  return true;
}

// Grid barrier k of MK_MODE_LEVELS (consumer thread 0 of every CTA): one
// counter per level boundary, so a CTA that has run out of work can arrive
// at all remaining boundaries at once.
__device__ bool level_barrier(const KParams& p, int k) {
  red_release_add(p.level_bar + k, 1u);
  const uint32_t target = gridDim.x;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire(p.level_bar + k) >= target) return true;
    if ((it & 63u) == 0) {
      if (aborted(p)) return false;
      if (globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, MK_DEV_DEP_TIMEOUT, -1);
        return false;
      }
    }
  }
}

template <int BCLASS>
__device__ void consumer(const KParams& p, uint8_t* ring, uint64_t* full, uint64_t* empty, float* scratch,
                         volatile int* sflag, uint8_t* xbuf, TcCtl* ctl, uint32_t taddr, const TaskRec* recs,
                         uint64_t* rfull, uint64_t* rempty) {
  Ctx c{&p, ring, full, empty, scratch, RingPos{}, p.nstages, -1, {0, 0, 0}, 0u, xbuf, ctl, taddr, 0u,
        nullptr, static_cast<int32_t*>(p.bufs[MK_BUF_STATE]), tmem_part_col(BCLASS)};
  int cur_lvl = 0;
  const int tid = threadIdx.x;
  for (uint32_t k = 0;; ++k) {
    const uint32_t e = k & (kRecs - 1);
    const TaskRec* r = recs + e;
    c.mark[0] = c.mark[1] = c.mark[2] = 0;
    c.ring_waits = 0;
    uint64_t t_wait = 0, t_start = 0;
    if (tid < 32) {  // warp 0 takes the record, then waits (MEGA: all lanes; other modes: thread 0)
      int run = 1;   // 1: run the task, 0: stop (abort or timeout), 2: no more tasks
      // every lane acquires the record (no single-lane wait and warp barrier)
      if (!bar_wait(p, &rfull[e], (k / kRecs) & 1u, -1, true)) run = 0;
      run = __shfl_sync(0xffffffffu, run, 0);
      if (run && r->task < 0) run = 2;
      if (run == 1) {
        const int task = r->task;
        bool ok = true;
        if (p.trace) t_wait = globaltimer();
        if (p.mode == MK_MODE_MEGA) {
          ok = wait_deps(p, r, task);
        } else if (tid == 0 && p.mode == MK_MODE_LEVELS) {
          const int lvl = r->lvl;
          while (ok && cur_lvl < lvl) ok = level_barrier(p, ++cur_lvl);
          ok = ok && !aborted(p);
        } else if (p.mode == MK_MODE_PER_OP_PDL) {
          // the previous op's kernel has completed and its writes are
          // visible; only then may the next kernel launch (so its producer,
          // which starts before its own wait, never runs ahead of two ops)
          asm volatile("griddepcontrol.wait;" ::: "memory");
          if (tid == 0) {
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            ok = !aborted(p);
          }
        } else if (tid == 0) {
          ok = !aborted(p);
        }
        if (p.trace) t_start = globaltimer();
        if (!ok) run = 0;
      }
      if (tid == 0) *sflag = run;
    }
    cbar();
    const int run = *sflag;
    if (run == 0) return;
    if (run == 2) break;
    const mk_task_descriptor d = r->d;
    const int task = r->task;
    c.task = task;
    c.rec = r;
    switch (d.op_id) {
      case MK_OP_GEMV:
        if constexpr (BCLASS == 2) {
          if (d.config_id == 1 && r->tm_rows > 0) {
            tc_gemv_task(c, d);
            break;
          }
        }
        gemv_task<BCLASS>(c, d);
        break;
      case MK_OP_ATTENTION_APPEND: append_task(c, d); break;
      case MK_OP_ATTENTION_PARTIAL: partial_task<BCLASS>(c, d); break;
      case MK_OP_ATTENTION_COMBINE: combine_task(c, d); break;
      case MK_OP_MEMCPY: embed_task(c, d); break;
      case MK_OP_RMSNORM: rmsnorm_task(c, d); break;
      case MK_OP_SAMPLE: sample_task(c, d); break;
      case MK_OP_NOP: break;
      default:
        if (tid == 0) raise_error(p, MK_DEV_BAD_OP, task);
        break;
    }
    cbar();  // every output of the task is written
    if (p.trace && tid == 0) {
      // end stamp taken before the dependents are released, so a child's
      // start stamp is never earlier than its parents' end stamps
      uint64_t* tr = p.trace + (size_t)task * 8;
      tr[0] = ((uint64_t)blockIdx.x << 32) | smid();
      tr[1] = t_wait;
      tr[2] = t_start;
      tr[3] = globaltimer();
      tr[4] = c.mark[0];
      tr[5] = c.mark[1];
      tr[6] = c.mark[2];
      tr[7] = c.ring_waits;
    }
    if (tid < 32) {
      if (p.mode == MK_MODE_MEGA) {
        // release: one gpu-scope fence per signalling lane (covering, through
        // the barrier above, every consumer thread's output writes), then
        // relaxed adds that the dependents' acquire loads synchronise with
        const uint32_t s0 = r->s0, ns = r->ns;
        if ((uint32_t)tid < ns) fence_acq_rel_gpu();
        for (uint32_t i = tid; i < ns; i += 32) red_relaxed_add(p.counters + (i < 4 ? r->si[i] : __ldg(p.sig + s0 + i)), 1u);
      }
      __syncwarp();
      if (tid == 0) mbar_arrive(&rempty[e]);  // the record may be reused
    }
  }
  // LEVELS: arrive at the barriers of the remaining levels so no CTA waits on us
  if (p.mode == MK_MODE_LEVELS && tid == 0) {
    for (int k = cur_lvl + 1; k < p.num_levels; ++k) red_release_add(p.level_bar + k, 1u);
  }
}

// Shared memory: [activation staging (class-2 kernel)] [ring] [full, empty
// mbarriers] [control block] [task records] [record full, empty mbarriers]
// [scratch].
int smem_bytes_for(int nstages, int batch) {
  return (batch > 2 ? kXbufBytes : 0) + nstages * kStageBytes + 2 * nstages * 8 + kCtlBytes +
         kRecs * (kRecBytes + 16) + kScratchBytes;
}

template <int BCLASS>
__global__ void __launch_bounds__(kThreads, 1) mk_interpreter_kernel(const __grid_constant__ KParams p) {
  // 3 warpgroups: two consumer warpgroups and one producer warpgroup whose
  // first warp issues the copies.  Registers move from the producer group to
  // the consumers: 128 * kProducerRegs + 256 * kConsumerRegs equals
  // 384 * kLaunchRegs, the allocation the CTA is launched with (the host
  // refuses to launch if the compiled kernel's count differs).
  extern __shared__ __align__(1024) uint8_t smem[];
  const int nst = p.nstages;
  constexpr int xbytes = BCLASS == 2 ? kXbufBytes : 0;
  uint8_t* xbuf = smem;
  uint8_t* ring = smem + xbytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)nst * kStageBytes);
  uint64_t* empty = full + nst;
  TcCtl* ctl = reinterpret_cast<TcCtl*>(empty + nst);
  volatile int* sflag = &ctl->run;
  TaskRec* recs = reinterpret_cast<TaskRec*>(reinterpret_cast<uint8_t*>(ctl) + kCtlBytes);
  uint64_t* rfull = reinterpret_cast<uint64_t*>(recs + kRecs);
  uint64_t* rempty = rfull + kRecs;
  float* scratch = reinterpret_cast<float*>(rempty + kRecs);
  // the swizzled operand layouts assume 1024-byte aligned tiles
  const bool aligned = (smem_addr(smem) & 1023u) == 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(&ctl->mma_bar[0], 1);
    mbar_init(&ctl->mma_bar[1], 1);
    mbar_init(&ctl->x_full[0], kConsumerWarps);
    mbar_init(&ctl->x_full[1], kConsumerWarps);
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->acc_empty, 1);
    mbar_init(&ctl->task_go, 1);
    mbar_init(&ctl->s_full[0], 1);
    mbar_init(&ctl->s_full[1], 1);
    mbar_init(&ctl->s_empty[0], 4);  // the four softmax warps
    mbar_init(&ctl->s_empty[1], 4);
    mbar_init(&ctl->q_full, kConsumerWarps);
    mbar_init(&ctl->p_full[0], 4);   // the four softmax warps
    mbar_init(&ctl->p_full[1], 4);
    mbar_init(&ctl->p_empty[0], 4);  // the four P V warps
    mbar_init(&ctl->p_empty[1], 4);
    for (int i = 0; i < kRecs; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 2);  // the producer and consumer thread 0
    }
    fence_mbar_init();
    if (BCLASS > 0 && !aligned) raise_error(p, MK_DEV_BAD_OP, -1);  // the tensor-core operand tiles
  }
  constexpr uint32_t tcols = tmem_cols(BCLASS);
  if constexpr (tcols > 0) {
    if (threadIdx.x < 32) {  // one warp allocates the accumulator columns
      tmem_alloc(&ctl->tmem, tcols);
      tmem_relinquish();
    }
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (tcols > 0) tc_fence_after();
  const uint32_t taddr = tcols > 0 ? ctl->tmem : 0u;
  if (threadIdx.x >= kConsumerThreads) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    if (threadIdx.x < kConsumerThreads + 32) producer<BCLASS>(p, ring, full, empty, recs, rfull, rempty);
    else if (threadIdx.x < kConsumerThreads + 64) {
      if constexpr (tcols > 0) tc_mma_warp(p, ring, full, empty, ctl, smem_addr(xbuf), taddr, tmem_part_col(BCLASS));
    }
    else if (threadIdx.x < kConsumerThreads + 96)
      record_warp(p, recs, rfull, rempty);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
    if (BCLASS == 0 || aligned)
      consumer<BCLASS>(p, ring, full, empty, scratch, sflag, xbuf, ctl, taddr, recs, rfull, rempty);
    if constexpr (tcols > 0) {
      // every tensor-core operation has completed (the consumers waited for
      // each row group's last commit and each key block's scores): tell the
      // MMA warp to stop, free the columns
      named_bar_sync(1, kConsumerThreads);
      if (threadIdx.x == 0) {
        ctl->mb_task = -1;
        mbar_arrive(&ctl->task_go);
      }
      if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(taddr, tcols);
      }
    }
  }
}

}  // namespace mk

// Launch helpers used by the runtime (host side, same translation unit as the kernels).
namespace mk {

static const void* kernel_for(int batch) {
  return batch <= 2 ? (const void*)mk_interpreter_kernel<0> : (const void*)mk_interpreter_kernel<2>;
}

cudaError_t configure_interpreter(int batch, int nstages, int* num_regs) {
  const void* fn = kernel_for(batch);
  cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes_for(nstages, batch));
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, fn);
  if (e != cudaSuccess) return e;
  *num_regs = attr.numRegs;
  return cudaSuccess;
}

cudaError_t launch_interpreter(const KParams& p, int batch, int grid, bool cooperative, cudaStream_t stream) {
  const int smem = smem_bytes_for(p.nstages, batch);
  const void* fn = kernel_for(batch);
  void* args[] = {const_cast<KParams*>(&p)};
  if (cooperative)
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, (size_t)smem, stream);
  if (p.mode == MK_MODE_PER_OP_PDL) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
  }
  return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, (size_t)smem, stream);
}

cudaError_t max_coresident_ctas(int batch, int nstages, int* per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kernel_for(batch), kThreads,
                                                       smem_bytes_for(nstages, batch));
}

}  // namespace mk
