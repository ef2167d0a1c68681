// Host runtime of libmk: upload of the lowered graph, launches, status.
//
// Upload follows "mega kernel initial" (1y33.com, buffer-table and upload
// part): one contiguous device blob holding a 64-byte header, the task
// array and the edge array, copied with a single cudaMemcpy, plus the
// buffer pointer table.  Where the page keeps a pristine copy of the blob to
// restore between runs, this runtime keeps the descriptors immutable and
// makes dependency counters monotone: step e waits for counter >= e * deps,
// so nothing has to be restored between steps.
#include <cuda.h>  // CUtensorMap types; the encoder is fetched through the runtime
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "graph.h"
#include "kernel.h"

namespace mk {

cudaError_t configure_interpreter(int batch, int nstages, int* num_regs);
cudaError_t launch_interpreter(const KParams& p, int batch, int grid, bool cooperative, cudaStream_t stream);
cudaError_t max_coresident_ctas(int batch, int nstages, int* per_sm);

struct DeviceState {
  int device = -1;
  void* blob = nullptr;
  size_t blob_bytes = 0;
  mk_task_descriptor* tasks = nullptr;
  uint32_t* edges = nullptr;
  void** bufs = nullptr;
  uint32_t* counters = nullptr;
  uint32_t* wait_off = nullptr;
  uint2* wait = nullptr;
  uint32_t* sig_off = nullptr;
  uint32_t* sig = nullptr;
  size_t counter_words = 0;
  uint8_t* tmaps = nullptr;
  int32_t* tm_rows = nullptr;
  int tc_tiles = 0;  // GEMV tiles on the tensor-core path
  uint64_t** mirrors = nullptr;  // device table: per buffer, its tagged pairs or null
  uint32_t tag = 0;              // last step tag (never reset, so stale pairs never match)
  int32_t* queue_off = nullptr;
  int32_t* queue = nullptr;
  int32_t* level_off = nullptr;
  int32_t* level_tasks = nullptr;
  uint32_t* level_bar = nullptr;
  int32_t* status = nullptr;
  float* rope_cos = nullptr;
  float* rope_sin = nullptr;
  uint64_t* trace = nullptr;
  float* ksplit = nullptr;        // K-split partial-sum records
  uint32_t* karr_mega = nullptr;  // K-split arrivals in megakernel steps (monotone, like the counters)
  uint32_t* karr_step = nullptr;  // K-split arrivals in the other modes (cleared before each step)
  size_t krecords = 0;
  uint32_t epoch = 0;
  int nstages = kMaxStages;
  cudaGraphExec_t per_op_exec = nullptr;
  cudaGraph_t per_op_graph = nullptr;
};

}  // namespace mk

using namespace mk;

#define CUDA_TRY(call)                                                                       \
  do {                                                                                       \
    cudaError_t e__ = (call);                                                                \
    if (e__ != cudaSuccess)                                                                  \
      return fail(MK_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e__));         \
  } while (0)

int mk::query_sm_count(int* out) {
  int dev = 0, n = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
  *out = n;
  return MK_OK;
}

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

void free_device(DeviceState* d) {
  if (!d) return;
  if (d->per_op_exec) cudaGraphExecDestroy(d->per_op_exec);
  if (d->per_op_graph) cudaGraphDestroy(d->per_op_graph);
  if (d->blob) cudaFree(d->blob);
  delete d;
}

KParams base_params(const mk_graph* g) {
  const DeviceState* d = g->dev;
  KParams p{};
  p.tasks = d->tasks;
  p.edges = d->edges;
  p.bufs = d->bufs;
  p.counters = d->counters;
  p.wait_off = d->wait_off;
  p.wait = d->wait;
  p.sig_off = d->sig_off;
  p.sig = d->sig;
  p.tmaps = d->tmaps;
  p.tm_rows = d->tm_rows;
  p.mirrors = d->mirrors;
  p.tag = d->tag;
  p.num_bufs = (int32_t)g->bufs.size();
  p.queue_off = d->queue_off;
  p.queue = d->queue;
  p.level_off = d->level_off;
  p.level_tasks = d->level_tasks;
  p.level_bar = d->level_bar;
  p.status = d->status;
  p.rope_cos = d->rope_cos;
  p.rope_sin = d->rope_sin;
  p.trace = nullptr;
  p.timeout_ns = (uint64_t)g->timeout_us * 1000ull;
  p.epoch = d->epoch;
  p.mode = MK_MODE_MEGA;
  p.first_task = 0;
  p.num_levels = (int)g->level_off.size() - 1;
  p.nstages = d->nstages;
  p.rope_half = g->rope_D / 2;
  p.ksplit = d->ksplit;
  p.karr = d->karr_step;
  p.kmul = 1;
  return p;
}

// Clear the K-split arrival counters that a non-megakernel step counts in
// (their target is then S - 1 per block), on the step's stream.
cudaError_t clear_step_arrivals(const DeviceState* d, cudaStream_t stream) {
  if (!d->krecords) return cudaSuccess;
  return cudaMemsetAsync(d->karr_step, 0, d->krecords * 4, stream);
}

// Tensor maps of the weights that tensor-core GEMV tiles stream through the
// tensor-core path: a 2-D bf16 view [rows, K] with a box of 64 columns x RG
// rows in the 128-byte swizzle.  RG splits the op's tile width into row
// groups of at most 256 rows (128 per segment for SILU_MUL: gate and up
// share the 256 accumulator columns).  Ops with K not a multiple of 64 stay
// on the CUDA-core path (tm_rows 0).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int build_tensor_maps(const mk_graph* g, std::vector<uint8_t>& maps, std::vector<int32_t>& rows) {
  const size_t NB = g->bufs.size();
  maps.assign(NB * kTmapBytes, 0);
  rows.assign(NB, 0);
  EncodeTiledFn enc = nullptr;
  for (const OpRec& op : g->ops) {
    if (op.kind != K_MATMUL || op.B < kTcMinRows || op.k % 64 != 0) continue;
    const int seg = (op.flags & MK_F_SILU_MUL) ? 2 : 1;
    // the tile (or, K-split, the row block) width
    const int cw = ksplit_plan(op.n, op.k, op.flags, op.B, g->tiles_target, g->col_align).W;
    const int rgmax = seg == 2 ? 128 : 256;
    const int ng = (cw + rgmax - 1) / rgmax;
    const int rg = (cw + ng - 1) / ng;
    const int w = op.a[1];
    if (rows[w] != 0) {
      if (rows[w] != rg) return fail(MK_ERR_ARG, "mk_upload: weight buffer " + std::to_string(w) +
                                                   " used by tensor-core GEMVs with different tile widths");
      continue;
    }
    if (!enc) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return fail(MK_ERR_CUDA, "mk_upload: cuTensorMapEncodeTiled is not available");
      enc = reinterpret_cast<EncodeTiledFn>(fn);
    }
    const BufferRec& b = g->bufs[w];
    CUtensorMap m;
    const cuuint64_t gdim[2] = {(cuuint64_t)op.k, (cuuint64_t)b.rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)op.k * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)rg};
    const cuuint32_t estride[2] = {1u, 1u};
    const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b.ptr, gdim, gstride, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(MK_ERR_CUDA, "mk_upload: tensor map of buffer " + std::to_string(w) + " failed (" +
                                   std::to_string((int)r) + ")");
    static_assert(sizeof(CUtensorMap) == kTmapBytes, "tensor map size");
    std::memcpy(maps.data() + (size_t)w * kTmapBytes, &m, kTmapBytes);
    rows[w] = rg;
  }
  // K caches: a 2-D view [B * Hkv * capacity rows, D] with boxes of 64 dims
  // x kKeyBlockRows keys in the 128-byte swizzle, for the tensor-core
  // split-KV partials (their score MMAs read the key rows in that layout)
  for (const OpRec& op : g->ops) {
    // (the B <= 2 kernel runs its partials on CUDA cores)
    if (op.kind != K_ATTENTION || (op.D != 64 && op.D != 128) || g->rows() <= 2) continue;
    const int w = op.a[1];
    if (rows[w] != 0) continue;
    if (!enc) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return fail(MK_ERR_CUDA, "mk_upload: cuTensorMapEncodeTiled is not available");
      enc = reinterpret_cast<EncodeTiledFn>(fn);
    }
    const BufferRec& b = g->bufs[w];
    CUtensorMap m;
    const cuuint64_t gdim[2] = {(cuuint64_t)op.D, (cuuint64_t)b.rows * (cuuint64_t)op.cap};
    const cuuint64_t gstride[1] = {(cuuint64_t)op.D * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)kKeyBlockRows};
    const cuuint32_t estride[2] = {1u, 1u};
    const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b.ptr, gdim, gstride, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(MK_ERR_CUDA, "mk_upload: tensor map of K cache " + std::to_string(w) + " failed (" +
                                   std::to_string((int)r) + ")");
    std::memcpy(maps.data() + (size_t)w * kTmapBytes, &m, kTmapBytes);
    rows[w] = kKeyBlockRows;
  }
  return MK_OK;
}

int launch_per_op(mk_graph* g, cudaStream_t stream, uint64_t* trace, int mode = MK_MODE_PER_OP) {
  KParams p = base_params(g);
  p.mode = mode;
  p.trace = trace;
  CUDA_TRY(clear_step_arrivals(g->dev, stream));
  for (size_t i = 0; i + 1 < g->group_off.size(); ++i) {
    p.first_task = g->group_off[i];
    const int n = g->group_off[i + 1] - g->group_off[i];
    if (n <= 0) continue;
    CUDA_TRY(launch_interpreter(p, g->rows(), n, false, stream));
  }
  return MK_OK;
}

}  // namespace

extern "C" int mk_upload(mk_graph* g, void* stream_) {
  if (!g) return fail(MK_ERR_ARG, "mk_upload: null graph");
  if (!g->lowered) return fail(MK_ERR_STATE, "mk_upload: call mk_lower first");
  if (g->uploaded) return fail(MK_ERR_STATE, "mk_upload: already uploaded");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  auto* d = new (std::nothrow) DeviceState();
  if (!d) return fail(MK_ERR_NOMEM, "mk_upload: out of memory");
  int rc = MK_OK;
  do {
    if (cudaGetDevice(&d->device) != cudaSuccess) { rc = fail(MK_ERR_CUDA, "mk_upload: no device"); break; }
    // ring depth from the opt-in shared-memory limit, then co-residency check
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d->device);
    d->nstages = kMaxStages;
    while (d->nstages > 2 && smem_bytes_for(d->nstages, g->rows()) > optin) --d->nstages;
    int regs = 0;
    if (configure_interpreter(g->rows(), d->nstages, &regs) != cudaSuccess) {
      rc = fail(MK_ERR_CUDA, "mk_upload: cannot configure the interpreter kernel");
      break;
    }
    if (regs != kLaunchRegs) {
      // the producer/consumer register split assumes this launch allocation
      rc = fail(MK_ERR_CUDA, "mk_upload: interpreter kernel compiled with " + std::to_string(regs) +
                                 " registers per thread, expected " + std::to_string(kLaunchRegs));
      break;
    }
    int per_sm = 0, sms = 0;
    if (max_coresident_ctas(g->rows(), d->nstages, &per_sm) != cudaSuccess || per_sm < 1) {
      rc = fail(MK_ERR_CUDA, "mk_upload: the interpreter kernel cannot be resident");
      break;
    }
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d->device);
    if (g->num_ctas > per_sm * sms) {
      rc = fail(MK_ERR_LIMIT, "mk_upload: num_ctas " + std::to_string(g->num_ctas) + " exceeds co-resident CTAs " +
                                  std::to_string(per_sm * sms));
      break;
    }
    const size_t N = g->tasks.size(), E = g->edges.size(), NB = g->bufs.size();
    const int half = g->rope_D / 2, cap = g->rope_cap;
    std::vector<uint8_t> tmaps;
    std::vector<int32_t> tm_rows;
    if ((rc = build_tensor_maps(g, tmaps, tm_rows)) != MK_OK) break;
    // blob layout: header | tasks | edges | queue_off | queue | level_off | level_tasks | bufs | cos | sin |
    //              wait_off | wait | sig_off | sig, then (zeroed) counters | status | level_bar | trace
    size_t off = 0;
    auto take = [&](size_t bytes) {
      size_t o = off;
      off = align_up(off + bytes, 256);
      return o;
    };
    const size_t o_hdr = take(64), o_tasks = take(N * 64), o_edges = take(E * 4),
                 o_qoff = take(g->queue_off.size() * 4), o_q = take(g->queue.size() * 4),
                 o_loff = take(g->level_off.size() * 4), o_lt = take(g->level_tasks.size() * 4),
                 o_bufs = take(NB * 8), o_cos = take((size_t)cap * half * 4), o_sin = take((size_t)cap * half * 4),
                 o_woff = take(g->wait_off.size() * 4), o_wait = take(g->wait.size() * 4),
                 o_soff = take(g->sig_off.size() * 4), o_sig = take(g->sig.size() * 4),
                 o_tmap = take(tmaps.size()), o_tmr = take(tm_rows.size() * 4), o_mtab = take(NB * 8);
    const size_t static_bytes = off;
    std::vector<size_t> o_mir(NB, 0);  // tagged pairs of the buffers that carry them (zeroed)
    for (size_t b = 0; b < NB; ++b)
      if (b < g->ll_buf.size() && g->ll_buf[b]) o_mir[b] = take((size_t)g->bufs[b].rows * g->bufs[b].cols * 8);
    const size_t o_ctr = take((size_t)g->counter_words * 4), o_status = take(16), o_lbar = take(g->level_off.size() * 4),
                 o_trace = take(N * 64), o_kam = take((size_t)g->ksplit_records * 4),
                 o_kas = take((size_t)g->ksplit_records * 4),
                 o_ksp = take((size_t)g->ksplit_records * kKsplitRecFloats * 4);
    d->blob_bytes = off;
    if (cudaMalloc(&d->blob, d->blob_bytes) != cudaSuccess) {
      rc = fail(MK_ERR_NOMEM, "mk_upload: cudaMalloc of " + std::to_string(d->blob_bytes) + " bytes failed");
      break;
    }
    std::vector<uint8_t> img(static_bytes, 0);
    uint32_t hdr[16] = {0x31474B4Du /* "MKG1" */, MK_ABI_VERSION, (uint32_t)N, (uint32_t)E, (uint32_t)NB,
                        (uint32_t)g->num_ctas, (uint32_t)(g->level_off.size() - 1), 64u};
    std::memcpy(img.data() + o_hdr, hdr, 64);
    std::memcpy(img.data() + o_tasks, g->tasks.data(), N * 64);
    std::memcpy(img.data() + o_edges, g->edges.data(), E * 4);
    std::memcpy(img.data() + o_qoff, g->queue_off.data(), g->queue_off.size() * 4);
    std::memcpy(img.data() + o_q, g->queue.data(), g->queue.size() * 4);
    std::memcpy(img.data() + o_loff, g->level_off.data(), g->level_off.size() * 4);
    std::memcpy(img.data() + o_lt, g->level_tasks.data(), g->level_tasks.size() * 4);
    std::memcpy(img.data() + o_woff, g->wait_off.data(), g->wait_off.size() * 4);
    std::memcpy(img.data() + o_wait, g->wait.data(), g->wait.size() * 4);
    std::memcpy(img.data() + o_soff, g->sig_off.data(), g->sig_off.size() * 4);
    std::memcpy(img.data() + o_sig, g->sig.data(), g->sig.size() * 4);
    std::memcpy(img.data() + o_tmap, tmaps.data(), tmaps.size());
    std::memcpy(img.data() + o_tmr, tm_rows.data(), tm_rows.size() * 4);
    {
      std::vector<uint64_t*> mt(NB, nullptr);
      for (size_t b = 0; b < NB; ++b)
        if (o_mir[b]) mt[b] = reinterpret_cast<uint64_t*>(static_cast<char*>(d->blob) + o_mir[b]);
      std::memcpy(img.data() + o_mtab, mt.data(), NB * 8);
    }
    char* base = static_cast<char*>(d->blob);
    std::vector<void*> ptrs(NB);
    for (size_t i = 0; i < NB; ++i) ptrs[i] = g->bufs[i].ptr;
    ptrs[MK_BUF_ROPE_COS] = base + o_cos;
    ptrs[MK_BUF_ROPE_SIN] = base + o_sin;
    std::memcpy(img.data() + o_bufs, ptrs.data(), NB * 8);
    // RoPE tables: angle = pos * theta^(-2i/D), evaluated in double, stored as float
    {
      float* cs = reinterpret_cast<float*>(img.data() + o_cos);
      float* sn = reinterpret_cast<float*>(img.data() + o_sin);
      for (int i = 0; i < half; ++i) {
        const double inv = std::pow(g->rope_theta, -2.0 * i / (double)g->rope_D);
        for (int pos = 0; pos < cap; ++pos) {
          const double a = (double)pos * inv;
          cs[(size_t)pos * half + i] = (float)std::cos(a);
          sn[(size_t)pos * half + i] = (float)std::sin(a);
        }
      }
    }
    if (cudaMemcpy(d->blob, img.data(), static_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(base + static_bytes, 0, d->blob_bytes - static_bytes) != cudaSuccess) {
      rc = fail(MK_ERR_CUDA, "mk_upload: copy to device failed");
      break;
    }
    d->tasks = reinterpret_cast<mk_task_descriptor*>(base + o_tasks);
    d->edges = reinterpret_cast<uint32_t*>(base + o_edges);
    d->queue_off = reinterpret_cast<int32_t*>(base + o_qoff);
    d->queue = reinterpret_cast<int32_t*>(base + o_q);
    d->level_off = reinterpret_cast<int32_t*>(base + o_loff);
    d->level_tasks = reinterpret_cast<int32_t*>(base + o_lt);
    d->bufs = reinterpret_cast<void**>(base + o_bufs);
    d->rope_cos = reinterpret_cast<float*>(base + o_cos);
    d->rope_sin = reinterpret_cast<float*>(base + o_sin);
    d->counters = reinterpret_cast<uint32_t*>(base + o_ctr);
    d->counter_words = g->counter_words;
    d->wait_off = reinterpret_cast<uint32_t*>(base + o_woff);
    d->wait = reinterpret_cast<uint2*>(base + o_wait);
    d->sig_off = reinterpret_cast<uint32_t*>(base + o_soff);
    d->sig = reinterpret_cast<uint32_t*>(base + o_sig);
    d->tmaps = reinterpret_cast<uint8_t*>(base + o_tmap);
    d->tm_rows = reinterpret_cast<int32_t*>(base + o_tmr);
    d->mirrors = reinterpret_cast<uint64_t**>(base + o_mtab);
    for (const mk_task_descriptor& t : g->tasks)
      if (t.op_id == MK_OP_GEMV && t.config_id == 1 && g->rows() >= kTcMinRows && tm_rows[t.in_buf[1]] > 0) ++d->tc_tiles;
    d->status = reinterpret_cast<int32_t*>(base + o_status);
    d->level_bar = reinterpret_cast<uint32_t*>(base + o_lbar);
    d->trace = reinterpret_cast<uint64_t*>(base + o_trace);
    d->krecords = g->ksplit_records;
    d->karr_mega = reinterpret_cast<uint32_t*>(base + o_kam);
    d->karr_step = reinterpret_cast<uint32_t*>(base + o_kas);
    d->ksplit = reinterpret_cast<float*>(base + o_ksp);
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
      rc = fail(MK_ERR_CUDA, "mk_upload: stream synchronisation failed");
      break;
    }
  } while (0);
  if (rc != MK_OK) {
    free_device(d);
    return rc;
  }
  g->dev = d;
  g->uploaded = true;
  return MK_OK;
}

extern "C" int mk_decode_step_ex(mk_graph* g, void* stream_, int mode, uint32_t trace) {
  if (!g) return fail(MK_ERR_ARG, "mk_decode_step: null graph");
  if (!g->uploaded) return fail(MK_ERR_STATE, "mk_decode_step: call mk_upload first");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  DeviceState* d = g->dev;
  uint64_t* tr = trace ? d->trace : nullptr;
  switch (mode) {
    case MK_MODE_MEGA: {
      KParams p = base_params(g);
      p.epoch = d->epoch + 1;
      if (++d->tag == 0) d->tag = 1;  // 0 is the zeroed mirrors' tag: never a step's
      p.tag = d->tag;
      p.trace = tr;
      p.karr = d->karr_mega;
      p.kmul = p.epoch;
      CUDA_TRY(launch_interpreter(p, g->rows(), g->num_ctas, true, stream));
      d->epoch += 1;
      return MK_OK;
    }
    case MK_MODE_LEVELS: {
      KParams p = base_params(g);
      p.mode = MK_MODE_LEVELS;
      p.trace = tr;
      CUDA_TRY(cudaMemsetAsync(d->level_bar, 0, g->level_off.size() * 4, stream));
      CUDA_TRY(clear_step_arrivals(d, stream));
      CUDA_TRY(launch_interpreter(p, g->rows(), g->num_ctas, true, stream));
      return MK_OK;
    }
    case MK_MODE_PER_OP:
      return launch_per_op(g, stream, tr);
    case MK_MODE_PER_OP_PDL:
      return launch_per_op(g, stream, tr, MK_MODE_PER_OP_PDL);
    case MK_MODE_PER_OP_GRAPH: {
      if (trace) return fail(MK_ERR_ARG, "mk_decode_step_ex: tracing is not available in graph mode");
      if (!d->per_op_exec) {
        cudaStream_t cs;
        CUDA_TRY(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
        int rc = MK_OK;
        if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
          rc = fail(MK_ERR_CUDA, "mk_decode_step_ex: begin capture failed");
        } else {
          rc = launch_per_op(g, cs, nullptr);
          cudaGraph_t graph = nullptr;
          cudaError_t e = cudaStreamEndCapture(cs, &graph);
          if (rc == MK_OK && e != cudaSuccess) rc = fail(MK_ERR_CUDA, "mk_decode_step_ex: end capture failed");
          if (rc == MK_OK) {
            if (cudaGraphInstantiate(&d->per_op_exec, graph, 0) != cudaSuccess) {
              rc = fail(MK_ERR_CUDA, "mk_decode_step_ex: graph instantiation failed");
              cudaGraphDestroy(graph);
            } else {
              d->per_op_graph = graph;
            }
          } else if (graph) {
            cudaGraphDestroy(graph);
          }
        }
        cudaStreamDestroy(cs);
        if (rc != MK_OK) return rc;
      }
      CUDA_TRY(cudaGraphLaunch(d->per_op_exec, stream));
      return MK_OK;
    }
    default:
      return fail(MK_ERR_ARG, "mk_decode_step_ex: unknown mode " + std::to_string(mode));
  }
}

extern "C" int mk_decode_step(mk_graph* g, void* stream) { return mk_decode_step_ex(g, stream, MK_MODE_MEGA, 0); }

extern "C" int mk_decode_step_host(mk_graph* g, void* stream_, const int32_t* state_in, int32_t* tokens_out) {
  if (!g) return fail(MK_ERR_ARG, "mk_decode_step_host: null graph");
  if (!g->uploaded) return fail(MK_ERR_STATE, "mk_decode_step_host: call mk_upload first");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  void* state = g->bufs[MK_BUF_STATE].ptr;
  if (state_in) CUDA_TRY(cudaMemcpyAsync(state, state_in, (size_t)g->B * 8, cudaMemcpyHostToDevice, stream));
  int rc = mk_decode_step_ex(g, stream_, MK_MODE_MEGA, 0);
  if (rc != MK_OK) return rc;
  if (tokens_out)
    CUDA_TRY(cudaMemcpy2DAsync(tokens_out, 4, state, 8, 4, (size_t)g->B, cudaMemcpyDeviceToHost, stream));
  return MK_OK;
}

extern "C" int mk_status(mk_graph* g, void* stream_, int* dev_code, int32_t* task_id) {
  if (!g || !dev_code || !task_id) return fail(MK_ERR_ARG, "mk_status: null argument");
  if (!g->uploaded) return fail(MK_ERR_STATE, "mk_status: call mk_upload first");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  DeviceState* d = g->dev;
  CUDA_TRY(cudaStreamSynchronize(stream));
  int32_t st[4] = {0, 0, 0, 0};
  CUDA_TRY(cudaMemcpy(st, d->status, 16, cudaMemcpyDeviceToHost));
  *dev_code = st[kStatusCode];
  *task_id = st[kStatusCode] ? st[kStatusTask] : -1;
  if (st[kStatusCode] || st[kStatusAbort]) {
    // A failed step leaves counters part-way; start the epochs afresh.
    CUDA_TRY(cudaMemsetAsync(d->counters, 0, d->counter_words * 4, stream));
    if (d->krecords) CUDA_TRY(cudaMemsetAsync(d->karr_mega, 0, d->krecords * 4, stream));
    CUDA_TRY(cudaMemsetAsync(d->status, 0, 16, stream));
    CUDA_TRY(cudaStreamSynchronize(stream));
    d->epoch = 0;
  }
  return MK_OK;
}

extern "C" int mk_debug_set_epoch(mk_graph* g, void* stream_, uint32_t epoch, uint32_t tag) {
  if (!g) return fail(MK_ERR_ARG, "mk_debug_set_epoch: null graph");
  if (!g->uploaded) return fail(MK_ERR_STATE, "mk_debug_set_epoch: call mk_upload first");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  DeviceState* d = g->dev;
  // each counter gains, per step, one add per plan entry that names it
  std::vector<uint32_t> ctr(d->counter_words, 0u);
  for (uint32_t c : g->sig) {
    if (c >= d->counter_words) return fail(MK_ERR_ARG, "mk_debug_set_epoch: plan names a counter out of range");
    ctr[c] += 1u;
  }
  for (uint32_t& c : ctr) c *= epoch;  // modulo 2^32, as the device counters run
  // a K-split block's arrival counter gains S - 1 per megakernel step
  std::vector<uint32_t> karr(d->krecords, 0u);
  for (const mk_task_descriptor& t : g->tasks) {
    const uint32_t S = (uint32_t)t.kv_len >> 16, j = (uint32_t)t.kv_len & 0xFFFFu;
    if (t.op_id == MK_OP_GEMV && t.config_id == 1 && S >= 2 && j == S - 1 && t.reserved[4] < d->krecords)
      karr[t.reserved[4]] = epoch * (S - 1);
  }
  CUDA_TRY(cudaStreamSynchronize(stream));
  CUDA_TRY(cudaMemcpy(d->counters, ctr.data(), ctr.size() * 4, cudaMemcpyHostToDevice));
  if (d->krecords) CUDA_TRY(cudaMemcpy(d->karr_mega, karr.data(), karr.size() * 4, cudaMemcpyHostToDevice));
  d->epoch = epoch;
  d->tag = tag;
  return MK_OK;
}

extern "C" int mk_get_trace(mk_graph* g, const uint64_t** records, size_t* count) {
  if (!g || !records || !count) return fail(MK_ERR_ARG, "mk_get_trace: null argument");
  if (!g->uploaded) return fail(MK_ERR_STATE, "mk_get_trace: call mk_upload first");
  CUDA_TRY(cudaDeviceSynchronize());
  g->trace_host.resize(g->tasks.size() * 8);
  CUDA_TRY(cudaMemcpy(g->trace_host.data(), g->dev->trace, g->trace_host.size() * 8, cudaMemcpyDeviceToHost));
  *records = g->trace_host.data();
  *count = g->tasks.size();
  return MK_OK;
}

extern "C" int mk_kernel_info(const mk_graph* g, int* smem_bytes, int* threads, int* stages) {
  if (!g || !smem_bytes || !threads || !stages) return fail(MK_ERR_ARG, "mk_kernel_info: null argument");
  const int nst = g->dev ? g->dev->nstages : kMaxStages;
  *smem_bytes = smem_bytes_for(nst, g->rows());
  *threads = kThreads;
  *stages = nst;
  return MK_OK;
}

extern "C" int mk_gemv_tensor_core_tiles(const mk_graph* g, int* tiles) {
  if (!g || !tiles) return fail(MK_ERR_ARG, "mk_gemv_tensor_core_tiles: null argument");
  if (!g->uploaded) return fail(MK_ERR_STATE, "mk_gemv_tensor_core_tiles: call mk_upload first");
  *tiles = g->dev->tc_tiles;
  return MK_OK;
}

extern "C" void mk_destroy(mk_graph* g) {
  if (!g) return;
  free_device(g->dev);
  delete g;
}
