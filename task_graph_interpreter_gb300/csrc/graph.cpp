// Host side of libmk: graph building, lowering to task descriptors and the
// dependents edge array, per-CTA static queues and topological levels.
//
// Lowering follows "mega kernel initial" (1y33.com):
//  * lowering part: each op becomes one or more 64-byte descriptors; a matmul
//    fans out into one GEMV task per output-column tile (about one per SM;
//    3072 columns over 8 tiles -> 8 tasks of 384); attention becomes
//    ATTENTION_PARTIAL tasks per (sequence, KV-head group, KV chunk) plus a
//    combine; norm, residual and SiLU*mul are GEMV flags;
//  * every output remembers which task wrote which column range, and a
//    reader's parents are the writers of what it reads; parents are flipped
//    into dependents lists flattened into one edge array; tasks come out in
//    topological order (the edge-array part);
//  * levels: level = 1 + max parent level (the levels part), kept for the
//    level-synchronous ablation mode.
// In a KV cache block, columns [0, cap*D) stand for the rows of earlier steps
// and [cap*D, cap*D + D) for the row appended this step: APPEND writes only
// the latter and PARTIAL reads only the former (it takes the new key/value
// from qkv), so partials do not wait for the append.  COMBINE takes the
// appended row as an input, so the append completes before the attention
// output does and every reader of the decode state stays an ancestor of
// SAMPLE, which advances it.
#include <algorithm>
#include <map>
#include <cmath>
#include <cstring>
#include <limits>
#include <numeric>
#include <string>
#include <vector>

#include "graph.h"

namespace mk {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }
int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int tile_width(int n, int tiles_target, int col_align) {
  return (int)(cdiv(cdiv(n, tiles_target), col_align) * col_align);
}

int tile_count(int n, int tiles_target, int col_align) {
  return (int)cdiv(n, tile_width(n, tiles_target, col_align));
}

// Batch >= 8 GEMVs run on tensor cores, where every MMA instruction costs
// the same whatever its N (up to 256 weight rows): a tile must put as many
// rows as it can into each MMA.  When the per-SM tiles are narrow (seg *
// width < 128 rows, seg = 2 for SiLU*mul's stacked gate and up rows), the op
// is cut instead into row blocks of up to 256 / seg rows, each split into S
// consecutive K ranges (in 64-column blocks) so that blocks * S stays within
// tiles_target.  Split j of a block multiplies its K range only; the last
// split adds the others' partial sums, in order, and runs the epilogue.
// Ops with an argmax epilogue are never split.
KSplit ksplit_plan(int n, int k, uint32_t flags, int m, int tiles_target, int col_align) {
  KSplit r{tile_width(n, tiles_target, col_align), 1, 1};
  r.nb = (int)cdiv(n, r.W);
  const int seg = (flags & MK_F_SILU_MUL) ? 2 : 1;
  if (m < kTcMinRows || (flags & MK_F_ARGMAX_EPI) || seg * r.W >= 128 || k % 64) return r;
  const int nb = (int)cdiv((int64_t)seg * n, 256);
  const int W = (int)(cdiv(cdiv(n, nb), 8) * 8);
  const int S = std::max(1, std::min(k / 64, tiles_target / (int)cdiv(n, W)));
  if (S < 2) return r;
  r.W = W;
  r.nb = (int)cdiv(n, W);
  r.S = S;
  return r;
}

// Split-KV chunk count per sequence, fixed at lowering time.  chunk > 0:
// ceil(len0 / chunk).  chunk == 0: chunks of about
// E = max(128, ceil(Hkv * sum(len0) / num_ctas)) keys, so that the partials
// of a ragged batch carry similar bytes and number about one per SM.
std::vector<int> partials_per_sequence(const std::vector<int32_t>& len0, int Hkv, int chunk,
                                       int num_ctas) {
  std::vector<int> P(len0.size());
  if (chunk > 0) {
    for (size_t s = 0; s < len0.size(); ++s) P[s] = (int)std::max<int64_t>(1, cdiv(len0[s], chunk));
    return P;
  }
  // chunks of E keys: the smallest E >= max(128, Hkv * sum / num_ctas) whose
  // chunk count Hkv * sum_s max(1, ceil(len_s / E)) fits one wave of CTAs
  int64_t tot = 0, longest = 0;
  for (int32_t l : len0) {
    tot += l;
    longest = std::max<int64_t>(longest, l);
  }
  auto count = [&](int64_t E) {
    int64_t c = 0;
    for (int32_t l : len0) c += std::max<int64_t>(1, cdiv(l, E));
    return c * Hkv;
  };
  int64_t E = std::max<int64_t>(128, cdiv((int64_t)Hkv * tot, num_ctas));
  if (count(E) > num_ctas) {
    int64_t a = E, b = std::max(E, longest);
    while (b - a > 1) {
      const int64_t m = (a + b) / 2;
      if (count(m) <= num_ctas) b = m;
      else a = m;
    }
    E = b;
  }
  for (size_t s = 0; s < len0.size(); ++s) P[s] = (int)std::max<int64_t>(1, cdiv(len0[s], E));
  return P;
}

}  // namespace mk

using namespace mk;

extern "C" const char* mk_last_error(void) { return g_last_error.c_str(); }

extern "C" int mk_graph_create(const mk_config* cfg, mk_graph** out) {
  if (!cfg || !out) return fail(MK_ERR_ARG, "mk_graph_create: null argument");
  *out = nullptr;
  if (cfg->abi_version != MK_ABI_VERSION)
    return fail(MK_ERR_ABI, "mk_graph_create: abi_version " + std::to_string(cfg->abi_version) +
                                " != " + std::to_string(MK_ABI_VERSION));
  if (cfg->num_ctas < 0 || cfg->tiles_target < 0 || cfg->col_align < 0)
    return fail(MK_ERR_ARG, "mk_graph_create: negative size");
  int ctas = cfg->num_ctas;
  if (ctas == 0) {
    int rc = query_sm_count(&ctas);
    if (rc != MK_OK) return rc;
  }
  auto* g = new (std::nothrow) mk_graph();
  if (!g) return fail(MK_ERR_NOMEM, "mk_graph_create: out of memory");
  g->cfg = *cfg;
  g->num_ctas = ctas;
  g->tiles_target = cfg->tiles_target ? cfg->tiles_target : ctas;
  g->col_align = cfg->col_align ? cfg->col_align : 16;
  g->timeout_us = cfg->wait_timeout_us ? cfg->wait_timeout_us : 2000000u;
  g->bufs.resize(3);  // 0 state (set later), 1/2 RoPE tables (built at upload)
  *out = g;
  return MK_OK;
}

extern "C" int mk_set_state(mk_graph* g, void* state_dptr, int B) {
  if (!g) return fail(MK_ERR_ARG, "mk_set_state: null graph");
  if (g->lowered) return fail(MK_ERR_STATE, "mk_set_state: graph already lowered");
  if (g->state_set) return fail(MK_ERR_STATE, "mk_set_state: state already set");
  if (!state_dptr || B < 1 || B > 8) return fail(MK_ERR_ARG, "mk_set_state: need a pointer and 1 <= B <= 8");
  if (((uintptr_t)state_dptr) % 16) return fail(MK_ERR_ARG, "mk_set_state: pointer not 16-byte aligned");
  g->bufs[0] = BufferRec{state_dptr, MK_I32, B, 2};
  g->B = B;
  g->state_set = true;
  return MK_OK;
}

extern "C" int mk_add_buffer(mk_graph* g, void* dptr, int dtype, int64_t rows, int64_t cols,
                             uint16_t* out_idx) {
  if (!g || !out_idx) return fail(MK_ERR_ARG, "mk_add_buffer: null argument");
  if (g->lowered) return fail(MK_ERR_STATE, "mk_add_buffer: graph already lowered");
  if (!g->state_set) return fail(MK_ERR_STATE, "mk_add_buffer: call mk_set_state first");
  if (!dptr) return fail(MK_ERR_ARG, "mk_add_buffer: null device pointer");
  if (((uintptr_t)dptr) % 16) return fail(MK_ERR_ARG, "mk_add_buffer: pointer not 16-byte aligned");
  if (dtype < MK_BF16 || dtype > MK_PAIR) return fail(MK_ERR_ARG, "mk_add_buffer: bad dtype");
  if (rows <= 0 || cols <= 0) return fail(MK_ERR_ARG, "mk_add_buffer: rows and cols must be positive");
  if (g->bufs.size() >= 0xFFFF) return fail(MK_ERR_LIMIT, "mk_add_buffer: buffer table full (65535)");
  g->bufs.push_back(BufferRec{dptr, dtype, rows, cols});
  *out_idx = (uint16_t)(g->bufs.size() - 1);
  return MK_OK;
}

extern "C" int mk_set_chunk(mk_graph* g, int T, uint16_t tokens) {
  if (!g) return fail(MK_ERR_ARG, "mk_set_chunk: null graph");
  if (g->lowered) return fail(MK_ERR_STATE, "mk_set_chunk: graph already lowered");
  if (!g->state_set) return fail(MK_ERR_STATE, "mk_set_chunk: call mk_set_state first");
  if (!g->ops.empty() || g->T != 1) return fail(MK_ERR_STATE, "mk_set_chunk: must precede every op, once");
  if (T < 2 || g->B * T > 8) return fail(MK_ERR_ARG, "mk_set_chunk: need T >= 2 and B * T <= 8");
  if (tokens >= g->bufs.size() || tokens < 3 || g->bufs[tokens].dtype != MK_I32 || g->bufs[tokens].rows != g->B ||
      g->bufs[tokens].cols != T)
    return fail(MK_ERR_ARG, "mk_set_chunk: tokens must be a registered int32 [B, T] buffer");
  g->T = T;
  g->tokens = tokens;
  return MK_OK;
}

static int check_buf(const mk_graph* g, uint16_t idx, int dtype, int64_t rows, int64_t cols,
                     const char* what) {
  if (idx >= g->bufs.size() || idx < 3)
    return fail(MK_ERR_ARG, std::string(what) + ": bad buffer index " + std::to_string(idx));
  const BufferRec& b = g->bufs[idx];
  if (b.dtype != dtype)
    return fail(MK_ERR_ARG, std::string(what) + ": buffer " + std::to_string(idx) + " has wrong dtype");
  if ((rows >= 0 && b.rows != rows) || (cols >= 0 && b.cols != cols))
    return fail(MK_ERR_ARG, std::string(what) + ": buffer " + std::to_string(idx) + " is [" +
                                std::to_string(b.rows) + ", " + std::to_string(b.cols) + "], expected [" +
                                std::to_string(rows) + ", " + std::to_string(cols) + "]");
  return MK_OK;
}

#define CHECK(x)            \
  do {                      \
    int rc__ = (x);         \
    if (rc__) return rc__;  \
  } while (0)

static int add_common(mk_graph* g, const char* what) {
  if (!g) return fail(MK_ERR_ARG, std::string(what) + ": null graph");
  if (g->lowered) return fail(MK_ERR_STATE, std::string(what) + ": graph already lowered");
  if (!g->state_set) return fail(MK_ERR_STATE, std::string(what) + ": call mk_set_state first");
  return MK_OK;
}

extern "C" int mk_add_embed(mk_graph* g, uint16_t table, uint16_t out, int B, int H) {
  CHECK(add_common(g, "mk_add_embed"));
  if (B != g->B || H <= 0 || H % 8) return fail(MK_ERR_ARG, "mk_add_embed: B must equal the state's B, H a multiple of 8");
  CHECK(check_buf(g, table, MK_BF16, -1, H, "mk_add_embed table"));
  CHECK(check_buf(g, out, MK_F32, g->rows(), H, "mk_add_embed out"));
  OpRec op{K_EMBED};
  op.a[0] = table;
  op.a[1] = out;
  op.B = B;
  op.H = H;
  g->ops.push_back(op);
  return MK_OK;
}

extern "C" int mk_add_rmsnorm(mk_graph* g, uint16_t x, uint16_t gamma, uint16_t residual, uint16_t out, int B,
                              int H, float eps) {
  CHECK(add_common(g, "mk_add_rmsnorm"));
  if (B != g->B || H <= 0 || H % 8 || H > 16384)
    return fail(MK_ERR_ARG, "mk_add_rmsnorm: B must equal the state's B, H a multiple of 8 up to 16384");
  if (!std::isfinite(eps) || eps < 0.f) return fail(MK_ERR_ARG, "mk_add_rmsnorm: eps must be finite and >= 0");
  const int M = g->rows();
  CHECK(check_buf(g, x, MK_F32, M, H, "mk_add_rmsnorm x"));
  CHECK(check_buf(g, gamma, MK_BF16, 1, H, "mk_add_rmsnorm gamma"));
  CHECK(check_buf(g, out, MK_F32, M, H, "mk_add_rmsnorm out"));
  if (residual != MK_NO_BUF) CHECK(check_buf(g, residual, MK_F32, M, H, "mk_add_rmsnorm residual"));
  if (out == x || out == residual) return fail(MK_ERR_ARG, "mk_add_rmsnorm: out must not alias an input");
  OpRec op{K_RMSNORM};
  op.a[0] = x;
  op.a[1] = gamma;
  op.a[2] = out;
  op.a[3] = residual;
  op.B = B;
  op.H = H;
  op.eps = eps;
  op.flags = residual != MK_NO_BUF ? MK_F_ADD_RESIDUAL : 0u;
  g->ops.push_back(op);
  return MK_OK;
}

// Which ops read buffer b (any operand position).
static bool op_reads(const OpRec& op, uint16_t b) {
  switch (op.kind) {
    case K_EMBED: return op.a[0] == b;
    case K_MATMUL: return op.a[0] == b || op.a[1] == b || op.a[3] == b;
    case K_ATTENTION: return op.a[0] == b || op.a[1] == b || op.a[2] == b;
    case K_SAMPLE: return op.a[0] == b;
    case K_RMSNORM: return op.a[0] == b || op.a[1] == b || op.a[3] == b;
  }
  return false;
}

extern "C" int mk_fuse_rmsnorm(mk_graph* g, int* fused) {
  if (!g || !fused) return fail(MK_ERR_ARG, "mk_fuse_rmsnorm: null argument");
  if (g->lowered) return fail(MK_ERR_STATE, "mk_fuse_rmsnorm: graph already lowered");
  *fused = 0;
  std::vector<OpRec> kept;
  for (size_t i = 0; i < g->ops.size(); ++i) {
    const OpRec& nrm = g->ops[i];
    bool fuse = nrm.kind == K_RMSNORM && nrm.a[3] == MK_NO_BUF;
    int readers = 0;
    for (size_t j = 0; fuse && j < g->ops.size(); ++j) {
      if (j == i || !op_reads(g->ops[j], nrm.a[2])) continue;
      const OpRec& r = g->ops[j];
      // only as the x of a GEMV that has no aux operand, after the norm
      if (j < i || r.kind != K_MATMUL || r.a[0] != nrm.a[2] || r.a[1] == nrm.a[2] || r.a[3] != MK_NO_BUF ||
          (r.flags & (MK_F_RMS_NORM_INPUT | MK_F_ADD_RESIDUAL)))
        fuse = false;
      else
        ++readers;
    }
    if (!fuse || readers == 0) {
      kept.push_back(nrm);
      continue;
    }
    for (size_t j = i + 1; j < g->ops.size(); ++j) {
      OpRec& r = g->ops[j];
      if (r.kind == K_MATMUL && r.a[0] == nrm.a[2]) {
        r.a[0] = nrm.a[0];
        r.a[3] = nrm.a[1];
        r.flags |= MK_F_RMS_NORM_INPUT;
        r.eps = nrm.eps;
      }
    }
    ++*fused;
  }
  g->ops.swap(kept);
  return MK_OK;
}

extern "C" int mk_add_matmul(mk_graph* g, uint16_t x, uint16_t w, uint16_t out, uint16_t aux,
                             uint16_t pairs, uint32_t flags, int m, int n, int k, float eps) {
  CHECK(add_common(g, "mk_add_matmul"));
  if (flags & ~(MK_F_SILU_MUL | MK_F_ADD_RESIDUAL | MK_F_RMS_NORM_INPUT | MK_F_ARGMAX_EPI))
    return fail(MK_ERR_ARG, "mk_add_matmul: unknown flag bits");
  if ((flags & MK_F_RMS_NORM_INPUT) && (flags & MK_F_ADD_RESIDUAL))
    return fail(MK_ERR_ARG, "mk_add_matmul: RMS_NORM_INPUT and ADD_RESIDUAL share the aux slot");
  if (m < 1 || m > 8 || m != g->rows())
    return fail(MK_ERR_ARG, "mk_add_matmul: need 1 <= m <= 8 and m == B * T (the activation rows)");
  if (n < 1) return fail(MK_ERR_ARG, "mk_add_matmul: n must be positive");
  if (k < 256 || k % 256 || k > 65536) return fail(MK_ERR_ARG, "mk_add_matmul: k must be a multiple of 256 in [256, 65536]");
  if (!std::isfinite(eps) || eps < 0.f) return fail(MK_ERR_ARG, "mk_add_matmul: eps must be finite and >= 0");
  CHECK(check_buf(g, x, MK_F32, m, k, "mk_add_matmul x"));
  CHECK(check_buf(g, w, MK_BF16, (flags & MK_F_SILU_MUL) ? 2 * (int64_t)n : n, k, "mk_add_matmul W"));
  CHECK(check_buf(g, out, MK_F32, m, n, "mk_add_matmul out"));
  if (flags & MK_F_RMS_NORM_INPUT) {
    CHECK(check_buf(g, aux, MK_BF16, 1, k, "mk_add_matmul gamma"));
  } else if (flags & MK_F_ADD_RESIDUAL) {
    CHECK(check_buf(g, aux, MK_F32, m, n, "mk_add_matmul residual"));
    if (aux == out) return fail(MK_ERR_ARG, "mk_add_matmul: residual must not alias the output");
  } else if (aux != MK_NO_BUF) {
    return fail(MK_ERR_ARG, "mk_add_matmul: aux given without RMS_NORM_INPUT or ADD_RESIDUAL");
  }
  if (flags & MK_F_ARGMAX_EPI) {
    CHECK(check_buf(g, pairs, MK_PAIR, tile_count(n, g->tiles_target, g->col_align), m,
                    "mk_add_matmul pairs"));
    if (flags & MK_F_SILU_MUL) return fail(MK_ERR_ARG, "mk_add_matmul: ARGMAX_EPI with SILU_MUL is not supported");
  } else if (pairs != MK_NO_BUF) {
    return fail(MK_ERR_ARG, "mk_add_matmul: pairs given without ARGMAX_EPI");
  }
  if (x == out) return fail(MK_ERR_ARG, "mk_add_matmul: x must not alias the output");
  OpRec op{K_MATMUL};
  op.a[0] = x; op.a[1] = w; op.a[2] = out; op.a[3] = aux; op.a[4] = pairs;
  op.B = m; op.n = n; op.k = k; op.flags = flags; op.eps = eps;
  g->ops.push_back(op);
  if (m > g->max_m) g->max_m = m;
  return MK_OK;
}

extern "C" int mk_attention_scratch_rows(const mk_graph* g, int B, int Hkv, const int32_t* len0,
                                         int chunk, int64_t* rows) {
  if (!g || !len0 || !rows || B < 1 || Hkv < 1 || chunk < 0)
    return fail(MK_ERR_ARG, "mk_attention_scratch_rows: bad argument");
  std::vector<int32_t> l(len0, len0 + B);
  auto P = partials_per_sequence(l, Hkv, chunk, g->num_ctas);
  int64_t r = 0;
  for (int p : P) r += (int64_t)p * Hkv;
  *rows = r;
  return MK_OK;
}

extern "C" int mk_gemv_tiles(const mk_graph* g, int n, int32_t* tiles) {
  if (!g || !tiles || n < 1) return fail(MK_ERR_ARG, "mk_gemv_tiles: bad argument");
  *tiles = tile_count(n, g->tiles_target, g->col_align);
  return MK_OK;
}

extern "C" int mk_scratch_size(const mk_graph* g, uint16_t buf, size_t* bytes) {
  if (!g || !bytes) return fail(MK_ERR_ARG, "mk_scratch_size: null argument");
  size_t need = 0;
  bool used = false;
  for (const OpRec& op : g->ops) {
    if (op.kind == K_ATTENTION && op.a[4] == buf) {
      const auto P = partials_per_sequence(op.len0, op.Hkv, op.chunk, g->num_ctas);
      size_t rows = 0;
      for (int q : P) rows += (size_t)q * op.Hkv;
      need = std::max(need, rows * (size_t)g->T * (size_t)(op.Hq / op.Hkv) * (size_t)(op.D + 2) * 4);
      used = true;
    }
    if (op.kind == K_MATMUL && op.a[4] == buf && buf != MK_NO_BUF) {
      need = std::max(need, (size_t)tile_count(op.n, g->tiles_target, g->col_align) * (size_t)op.B * 8);
      used = true;
    }
  }
  if (!used) return fail(MK_ERR_ARG, "mk_scratch_size: buffer " + std::to_string(buf) +
                                         " is no op's attention scratch or argmax pairs");
  *bytes = need;
  return MK_OK;
}

extern "C" int mk_add_attention(mk_graph* g, uint16_t qkv, uint16_t kcache, uint16_t vcache,
                                uint16_t out, uint16_t scratch, int B, int Hq, int Hkv, int D,
                                int capacity, const int32_t* len0, int chunk, double rope_theta) {
  CHECK(add_common(g, "mk_add_attention"));
  if (B != g->B) return fail(MK_ERR_ARG, "mk_add_attention: B must equal the state's B");
  if (D != 64 && D != 128) return fail(MK_ERR_ARG, "mk_add_attention: D must be 64 or 128");
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq / Hkv > 4)
    return fail(MK_ERR_ARG, "mk_add_attention: need Hq a multiple of Hkv with Hq/Hkv <= 4");
  if (capacity < 2 || capacity > (1 << 24)) return fail(MK_ERR_ARG, "mk_add_attention: bad capacity");
  if (!len0) return fail(MK_ERR_ARG, "mk_add_attention: null len0");
  if (chunk < 0) return fail(MK_ERR_ARG, "mk_add_attention: negative chunk");
  if (!(rope_theta > 0.0) || !std::isfinite(rope_theta)) return fail(MK_ERR_ARG, "mk_add_attention: bad rope_theta");
  for (int s = 0; s < B; ++s)
    if (len0[s] < 0 || len0[s] >= capacity) return fail(MK_ERR_ARG, "mk_add_attention: len0 out of [0, capacity)");
  if (g->rope_D && (g->rope_D != D || g->rope_theta != rope_theta || g->rope_cap != capacity))
    return fail(MK_ERR_ARG, "mk_add_attention: every attention op must share D, rope_theta and capacity");
  const int G = Hq / Hkv, M = g->rows();
  if (G * g->T > 16) return fail(MK_ERR_ARG, "mk_add_attention: need (Hq / Hkv) * T <= 16");
  CHECK(check_buf(g, qkv, MK_F32, M, (int64_t)(Hq + 2 * Hkv) * D, "mk_add_attention qkv"));
  CHECK(check_buf(g, kcache, MK_BF16, (int64_t)B * Hkv, (int64_t)capacity * D, "mk_add_attention kcache"));
  CHECK(check_buf(g, vcache, MK_BF16, (int64_t)B * Hkv, (int64_t)capacity * D, "mk_add_attention vcache"));
  CHECK(check_buf(g, out, MK_F32, M, (int64_t)Hq * D, "mk_add_attention out"));
  {
    // a combine task stages 3 floats per (partial, head) in its shared scratch
    std::vector<int32_t> l(len0, len0 + B);
    for (int P : partials_per_sequence(l, Hkv, chunk, g->num_ctas))
      if ((int64_t)P * G > 2048)
        return fail(MK_ERR_LIMIT, "mk_add_attention: more than 2048 / (Hq/Hkv) chunks per sequence");
  }
  int64_t need = 0;
  CHECK(mk_attention_scratch_rows(g, B, Hkv, len0, chunk, &need));
  CHECK(check_buf(g, scratch, MK_F32, -1, (int64_t)g->T * G * (D + 2), "mk_add_attention scratch"));
  if (g->bufs[scratch].rows < need)
    return fail(MK_ERR_ARG, "mk_add_attention: scratch needs " + std::to_string(need) + " rows");
  if (kcache == vcache) return fail(MK_ERR_ARG, "mk_add_attention: kcache and vcache must differ");
  OpRec op{K_ATTENTION};
  op.a[0] = qkv; op.a[1] = kcache; op.a[2] = vcache; op.a[3] = out; op.a[4] = scratch;
  op.B = B; op.Hq = Hq; op.Hkv = Hkv; op.D = D; op.cap = capacity; op.chunk = chunk;
  op.len0.assign(len0, len0 + B);
  g->ops.push_back(op);
  g->rope_D = D;
  g->rope_theta = rope_theta;
  g->rope_cap = capacity;
  return MK_OK;
}

extern "C" int mk_add_sample(mk_graph* g, uint16_t pairs, uint16_t history, int B, int V, int capacity) {
  CHECK(add_common(g, "mk_add_sample"));
  if (B != g->B || V < 1 || capacity < 2) return fail(MK_ERR_ARG, "mk_add_sample: bad B, V or capacity");
  CHECK(check_buf(g, pairs, MK_PAIR, tile_count(V, g->tiles_target, g->col_align), g->rows(),
                  "mk_add_sample pairs"));
  CHECK(check_buf(g, history, MK_I32, B, capacity, "mk_add_sample history"));
  OpRec op{K_SAMPLE};
  op.a[0] = pairs; op.a[1] = history;
  op.B = B; op.V = V; op.cap = capacity;
  g->ops.push_back(op);
  return MK_OK;
}

// ------------------------------------------------------------------ lowering
namespace {

struct Rect {
  int buf;
  int64_t r0, r1, c0, c1;
};

struct Writer {
  int task;
  int64_t r0, r1, c0, c1;
};

struct Lowerer {
  mk_graph* g;
  std::vector<std::vector<Writer>> writes;  // per buffer (and the K-split scratch, last)
  std::vector<std::vector<int>> parents;
  std::vector<double> cost;                  // bytes-equivalent estimate per task

  explicit Lowerer(mk_graph* gr) : g(gr), writes(gr->bufs.size() + 1) {}

  std::vector<Writer>& at(int buf) { return buf == (int)kKsplitBuf ? writes.back() : writes[buf]; }

  int emit(const mk_task_descriptor& d, const std::vector<Rect>& reads, const std::vector<Rect>& wr,
           double c) {
    int t = (int)g->tasks.size();
    std::vector<int> ps;
    for (const Rect& r : reads)
      for (const Writer& w : at(r.buf))
        if (w.r0 < r.r1 && r.r0 < w.r1 && w.c0 < r.c1 && r.c0 < w.c1) ps.push_back(w.task);
    std::sort(ps.begin(), ps.end());
    ps.erase(std::unique(ps.begin(), ps.end()), ps.end());
    for (const Rect& r : wr) at(r.buf).push_back(Writer{t, r.r0, r.r1, r.c0, r.c1});
    g->tasks.push_back(d);
    parents.push_back(std::move(ps));
    cost.push_back(c);
    return t;
  }
};

mk_task_descriptor blank(uint16_t op) {
  mk_task_descriptor d;
  std::memset(&d, 0, sizeof(d));
  d.op_id = op;
  d.in_buf[0] = d.in_buf[1] = d.in_buf[2] = MK_NO_BUF;
  d.out_buf = MK_NO_BUF;
  return d;
}

uint32_t f32_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

constexpr double kTaskOverhead = 32768.0;  // fixed cost per task, in bytes of streaming
constexpr double kSyncLatency = 32768.0;   // cross-CTA dependency latency, same units

}  // namespace

extern "C" int mk_lower(mk_graph* g) {
  if (!g) return fail(MK_ERR_ARG, "mk_lower: null graph");
  if (g->lowered) return fail(MK_ERR_STATE, "mk_lower: already lowered");
  if (g->ops.empty()) return fail(MK_ERR_STATE, "mk_lower: no ops");
  Lowerer L(g);
  g->ksplit_records = 0;
  const int tt = g->tiles_target, al = g->col_align;
  const int T = g->T;  // tokens per sequence per step; activation row s * T + t
  g->group_off.clear();
  for (const OpRec& op : g->ops) {
    switch (op.kind) {
      case K_EMBED: {
        // one row gather per (sequence, token of the step): token 0 is the
        // pending token in the state, tokens 1.. come from the tokens buffer
        g->group_off.push_back((int)g->tasks.size());
        for (int s = 0; s < op.B; ++s)
          for (int t = 0; t < T; ++t) {
            mk_task_descriptor d = blank(MK_OP_MEMCPY);
            d.step = (uint16_t)t;
            d.in_buf[0] = op.a[0];
            if (T > 1) d.in_buf[1] = g->tokens;
            d.out_buf = op.a[1];
            d.m = op.B;
            d.n = op.H;
            d.reserved[0] = s;
            d.reserved[1] = (uint32_t)g->bufs[op.a[0]].rows;
            d.reserved[2] = (uint32_t)(T - 1);
            const int r = s * T + t;
            std::vector<Rect> rd;
            if (t == 0) rd.push_back({(int)MK_BUF_STATE, s, s + 1, 0, 2});
            else rd.push_back({(int)g->tokens, s, s + 1, t, t + 1});
            L.emit(d, rd, {{op.a[1], r, r + 1, 0, op.H}}, kTaskOverhead);
          }
        break;
      }
      case K_MATMUL: {
        g->group_off.push_back((int)g->tasks.size());
        const KSplit ks = ksplit_plan(op.n, op.k, op.flags, op.B, tt, al);
        if (ks.S > 1) {
          // split j of row block b: K columns [k0, k0 + kn); the last split
          // reads the others' partial sums (scratch records) and writes y
          const int KB = op.k / 64;
          const double rows = (op.flags & MK_F_SILU_MUL) ? 2.0 : 1.0;
          for (int c0 = 0; c0 < op.n; c0 += ks.W) {
            const int cn = std::min(ks.W, op.n - c0);
            const uint32_t rec0 = g->ksplit_records;
            for (int j = 0; j < ks.S; ++j) {
              const int k0 = (int)((int64_t)j * KB / ks.S) * 64, k1 = (int)((int64_t)(j + 1) * KB / ks.S) * 64;
              mk_task_descriptor d = blank(MK_OP_GEMV);
              d.config_id = 1;
              d.flags = (uint16_t)op.flags;
              d.in_buf[0] = op.a[0];
              d.in_buf[1] = op.a[1];
              d.in_buf[2] = op.a[3];
              d.out_buf = op.a[2];
              d.m = op.B;
              d.n = op.n;
              d.k = op.k;
              d.kv_len = j | (ks.S << 16);
              d.reserved[0] = c0;
              d.reserved[1] = cn;
              d.reserved[2] = (op.flags & MK_F_RMS_NORM_INPUT) ? f32_bits(op.eps) : 0u;
              d.reserved[3] = (uint32_t)k0 | ((uint32_t)(k1 - k0) << 16);
              d.reserved[4] = rec0 + (uint32_t)j;
              std::vector<Rect> rd{{op.a[0], 0, op.B, k0, k1}}, wr;
              if (j + 1 < ks.S) {
                wr.push_back({(int)kKsplitBuf, rec0 + j, rec0 + j + 1, 0, kKsplitRecFloats});
              } else {
                rd.push_back({(int)kKsplitBuf, rec0, rec0 + j, 0, kKsplitRecFloats});
                if (op.flags & MK_F_ADD_RESIDUAL) rd.push_back({op.a[3], 0, op.B, c0, c0 + cn});
                wr.push_back({op.a[2], 0, op.B, c0, c0 + cn});
              }
              L.emit(d, rd, wr, rows * cn * (k1 - k0) * 2.0 + kTaskOverhead);
            }
            g->ksplit_records += (uint32_t)ks.S;
          }
          break;
        }
        const int w = ks.W;
        int t = 0;
        for (int c0 = 0; c0 < op.n; c0 += w, ++t) {
          const int cn = std::min(w, op.n - c0);
          mk_task_descriptor d = blank(MK_OP_GEMV);
          d.config_id = op.B < kTcMinRows ? 0 : 1;
          d.flags = (uint16_t)op.flags;
          d.in_buf[0] = op.a[0];
          d.in_buf[1] = op.a[1];
          d.in_buf[2] = op.a[3];
          d.out_buf = op.a[2];
          d.m = op.B;
          d.n = op.n;
          d.k = op.k;
          d.reserved[0] = c0;
          d.reserved[1] = cn;
          d.reserved[2] = (op.flags & MK_F_RMS_NORM_INPUT) ? f32_bits(op.eps) : 0u;
          d.reserved[3] = (op.flags & MK_F_ARGMAX_EPI) ? op.a[4] : 0u;
          d.reserved[4] = (op.flags & MK_F_ARGMAX_EPI) ? (uint32_t)t : 0u;
          std::vector<Rect> rd{{op.a[0], 0, op.B, 0, op.k}};
          if (op.flags & MK_F_ADD_RESIDUAL) rd.push_back({op.a[3], 0, op.B, c0, c0 + cn});
          std::vector<Rect> wr{{op.a[2], 0, op.B, c0, c0 + cn}};
          if (op.flags & MK_F_ARGMAX_EPI) wr.push_back({op.a[4], t, t + 1, 0, op.B});
          double rows = (op.flags & MK_F_SILU_MUL) ? 2.0 * cn : cn;
          L.emit(d, rd, wr, rows * op.k * 2.0 + kTaskOverhead);
        }
        break;
      }
      case K_ATTENTION: {
        const int B = op.B, Hq = op.Hq, Hkv = op.Hkv, D = op.D, cap = op.cap, G = Hq / Hkv;
        const uint16_t cfg = D == 64 ? 0 : 1;
        const uint16_t qkv = op.a[0], kc = op.a[1], vc = op.a[2], out = op.a[3], scr = op.a[4];
        auto P = partials_per_sequence(op.len0, Hkv, op.chunk, g->num_ctas);
        std::vector<int> base(B * Hkv);
        int acc = 0;
        for (int s = 0; s < B; ++s) {
          for (int gg = 0; gg < Hkv; ++gg) base[s * Hkv + gg] = acc + gg * P[s];
          acc += Hkv * P[s];
        }
        auto common = [&](mk_task_descriptor& d) {
          d.config_id = cfg;
          d.m = B;
          d.n = D;
          d.k = Hq;
          d.kv_len = cap;
        };
        // Hkv in the low half of reserved[2], T - 1 in the high half
        const uint32_t hkvT = (uint32_t)Hkv | ((uint32_t)(T - 1) << 16);
        const int64_t cacheCols = (int64_t)cap * D;
        const int64_t RW = (int64_t)T * G * (D + 2);  // scratch record of one slot
        g->group_off.push_back((int)g->tasks.size());
        for (int s = 0; s < B; ++s)
          for (int gg = 0; gg < Hkv; ++gg)
            for (int t = 0; t < T; ++t) {
              // token t's row goes to position pos + t: columns
              // [cap*D + t*D, cap*D + (t+1)*D) of the (s, g) block stand for it
              mk_task_descriptor d = blank(MK_OP_ATTENTION_APPEND);
              common(d);
              d.step = (uint16_t)t;
              d.in_buf[0] = qkv; d.in_buf[1] = kc; d.in_buf[2] = vc;
              d.out_buf = kc;
              d.reserved[0] = s; d.reserved[1] = gg; d.reserved[2] = hkvT;
              const int64_t kcol = (int64_t)Hq * D + gg * D, vcol = (int64_t)(Hq + Hkv) * D + gg * D;
              const int64_t row = (int64_t)s * Hkv + gg, r = (int64_t)s * T + t;
              const int64_t a0 = cacheCols + (int64_t)t * D;
              L.emit(d,
                     {{qkv, r, r + 1, kcol, kcol + D}, {qkv, r, r + 1, vcol, vcol + D},
                      {(int)MK_BUF_STATE, s, s + 1, 0, 2}},
                     {{kc, row, row + 1, a0, a0 + D}, {vc, row, row + 1, a0, a0 + D}}, kTaskOverhead);
            }
        g->group_off.push_back((int)g->tasks.size());
        for (int s = 0; s < B; ++s)
          for (int gg = 0; gg < Hkv; ++gg) {
            const int64_t row = (int64_t)s * Hkv + gg;
            const double keys = std::ceil((op.len0[s] + 1.0) / P[s]);
            for (int c = 0; c < P[s]; ++c) {
              mk_task_descriptor d = blank(MK_OP_ATTENTION_PARTIAL);
              common(d);
              d.in_buf[0] = qkv; d.in_buf[1] = kc; d.in_buf[2] = vc;
              d.out_buf = scr;
              d.reserved[0] = s; d.reserved[1] = gg; d.reserved[2] = hkvT;
              d.reserved[3] = (uint32_t)c | ((uint32_t)P[s] << 16);
              d.reserved[4] = base[s * Hkv + gg];
              const int64_t slot = base[s * Hkv + gg] + c;
              const int64_t r0 = (int64_t)s * T, r1 = r0 + T;
              L.emit(d,
                     {{qkv, r0, r1, (int64_t)gg * G * D, (int64_t)(gg + 1) * G * D},
                      {qkv, r0, r1, (int64_t)Hq * D + gg * D, (int64_t)Hq * D + (gg + 1) * D},
                      {qkv, r0, r1, (int64_t)(Hq + Hkv) * D + gg * D, (int64_t)(Hq + Hkv) * D + (gg + 1) * D},
                      {kc, row, row + 1, 0, cacheCols}, {vc, row, row + 1, 0, cacheCols},
                      {(int)MK_BUF_STATE, s, s + 1, 0, 2}},
                     {{scr, slot, slot + 1, 0, RW}},
                     keys * D * 4.0 + kTaskOverhead);
            }
          }
        g->group_off.push_back((int)g->tasks.size());
        for (int s = 0; s < B; ++s)
          for (int gg = 0; gg < Hkv; ++gg) {
            mk_task_descriptor d = blank(MK_OP_ATTENTION_COMBINE);
            common(d);
            d.in_buf[0] = scr;
            d.in_buf[1] = kc;
            d.in_buf[2] = vc;
            d.out_buf = out;
            d.reserved[0] = s; d.reserved[1] = gg; d.reserved[2] = hkvT;
            d.reserved[3] = P[s];
            d.reserved[4] = base[s * Hkv + gg];
            const int64_t b0 = base[s * Hkv + gg];
            const int64_t row = (int64_t)s * Hkv + gg;
            const int64_t a1 = cacheCols + (int64_t)T * D;
            L.emit(d,
                   {{scr, b0, b0 + P[s], 0, RW}, {kc, row, row + 1, cacheCols, a1},
                    {vc, row, row + 1, cacheCols, a1}},
                   {{out, (int64_t)s * T, (int64_t)s * T + T, (int64_t)gg * G * D, (int64_t)(gg + 1) * G * D}},
                   kTaskOverhead);
          }
        break;
      }
      case K_RMSNORM: {
        g->group_off.push_back((int)g->tasks.size());
        for (int s = 0; s < op.B * T; ++s) {  // one task per activation row
          mk_task_descriptor d = blank(MK_OP_RMSNORM);
          d.flags = (uint16_t)op.flags;
          d.in_buf[0] = op.a[0];
          d.in_buf[1] = op.a[1];
          d.in_buf[2] = op.a[3];
          d.out_buf = op.a[2];
          d.m = op.B;
          d.n = op.H;
          d.reserved[0] = s;
          d.reserved[1] = f32_bits(op.eps);
          std::vector<Rect> rd{{op.a[0], s, s + 1, 0, op.H}};
          if (op.a[3] != MK_NO_BUF) rd.push_back({op.a[3], s, s + 1, 0, op.H});
          L.emit(d, rd, {{op.a[2], s, s + 1, 0, op.H}}, op.H * 4.0 + kTaskOverhead);
        }
        break;
      }
      case K_SAMPLE: {
        g->group_off.push_back((int)g->tasks.size());
        const int NT = tile_count(op.V, tt, al);
        for (int s = 0; s < op.B; ++s) {
          mk_task_descriptor d = blank(MK_OP_SAMPLE);
          d.in_buf[0] = op.a[0];
          d.out_buf = op.a[1];
          d.m = op.B;
          d.n = op.V;
          d.k = NT;
          d.kv_len = op.cap;
          d.reserved[0] = s;
          d.reserved[1] = (uint32_t)(T - 1);
          // the argmax of the sequence's last row; a chunk step also copies
          // its input tokens 1.. into the history
          const int lr = s * T + T - 1;
          std::vector<Rect> rd{{op.a[0], 0, NT, lr, lr + 1}, {(int)MK_BUF_STATE, s, s + 1, 0, 2}};
          if (T > 1) {
            d.in_buf[1] = g->tokens;
            rd.push_back({(int)g->tokens, s, s + 1, 0, T});
          }
          L.emit(d, rd, {{op.a[1], s, s + 1, 0, op.cap}, {(int)MK_BUF_STATE, s, s + 1, 0, 2}}, kTaskOverhead);
        }
        break;
      }
    }
  }
  const int N = (int)g->tasks.size();
  g->group_off.push_back(N);
  // drop empty groups (an op with no tasks cannot happen, but keep ranges tidy)
  g->group_off.erase(std::unique(g->group_off.begin(), g->group_off.end()), g->group_off.end());

  // parents -> dependents, flattened in task order (children ascending)
  std::vector<std::vector<int>> children(N);
  for (int t = 0; t < N; ++t)
    for (int p : L.parents[t]) children[p].push_back(t);
  g->edges.clear();
  uint32_t off = 0;
  for (int t = 0; t < N; ++t) {
    g->tasks[t].remaining_deps = (int32_t)L.parents[t].size();
    g->tasks[t].num_dependents = (int32_t)children[t].size();
    g->tasks[t].dependents_offset = off;
    for (int c : children[t]) g->edges.push_back((uint32_t)c);
    off += (uint32_t)children[t].size();
  }

  {
    // buffers written exactly once per step: by one op, whose tasks' write
    // rectangles tile the whole buffer without overlap
    const size_t NB = g->bufs.size();
    std::vector<int> group_of(N, 0);
    for (size_t k = 0; k + 1 < g->group_off.size(); ++k)
      for (int t = g->group_off[k]; t < g->group_off[k + 1]; ++t) group_of[t] = (int)k;
    std::vector<uint8_t> once(NB, 0);
    for (size_t b = 0; b < NB; ++b) {
      const std::vector<Writer>& ws = L.writes[b];
      if (ws.empty()) continue;
      bool ok = true;
      int64_t area = 0;
      for (size_t i = 0; i < ws.size() && ok; ++i) {
        const Writer& w = ws[i];
        ok = group_of[w.task] == group_of[ws[0].task] && w.r0 >= 0 && w.c0 >= 0 && w.r1 <= g->bufs[b].rows &&
             w.c1 <= g->bufs[b].cols;
        area += (w.r1 - w.r0) * (w.c1 - w.c0);
        for (size_t j = 0; j < i && ok; ++j)
          ok = !(ws[j].r0 < w.r1 && w.r0 < ws[j].r1 && ws[j].c0 < w.c1 && w.c0 < ws[j].c1);
      }
      once[b] = ok && area == g->bufs[b].rows * g->bufs[b].cols;
    }
    build_ll_plan(g, L.parents, once);
  }
  if (int rc = build_sync_plan(g)) return rc;

  // topological levels
  std::vector<int> level(N, 0);
  int nlev = 0;
  for (int t = 0; t < N; ++t) {
    for (int p : L.parents[t]) level[t] = std::max(level[t], level[p] + 1);
    nlev = std::max(nlev, level[t] + 1);
  }
  g->level_off.assign(nlev + 1, 0);
  for (int t = 0; t < N; ++t) g->level_off[level[t] + 1]++;
  for (int i = 0; i < nlev; ++i) g->level_off[i + 1] += g->level_off[i];
  g->level_tasks.assign(N, 0);
  {
    std::vector<int> fill(g->level_off.begin(), g->level_off.end() - 1);
    for (int t = 0; t < N; ++t) g->level_tasks[fill[level[t]]++] = t;
  }

  // Static per-CTA queues by list scheduling on an estimated timeline: each
  // task (in topological order) goes to the CTA that can finish it first;
  // ties go to the CTA that has been idle longest, then the lowest index.
  // Every queue is increasing in task index, so the lowest unfinished task is
  // always at the head of its queue and runnable: no deadlock while all CTAs
  // are co-resident.
  const int C = g->num_ctas;
  std::vector<double> freeAt(C, 0.0), finish(N, 0.0);
  std::vector<std::vector<int32_t>> q(C);
  for (int t = 0; t < N; ++t) {
    double ready = 0.0;
    for (int p : L.parents[t]) ready = std::max(ready, finish[p] + kSyncLatency);
    int best = 0;
    double bestFin = std::numeric_limits<double>::infinity(), bestFree = 0.0;
    for (int c = 0; c < C; ++c) {
      double fin = std::max(freeAt[c], ready) + L.cost[t];
      if (fin < bestFin || (fin == bestFin && freeAt[c] < bestFree)) {
        best = c;
        bestFin = fin;
        bestFree = freeAt[c];
      }
    }
    finish[t] = bestFin;
    freeAt[best] = bestFin;
    q[best].push_back(t);
  }
  g->queue_off.assign(C + 1, 0);
  g->queue.clear();
  for (int c = 0; c < C; ++c) {
    g->queue_off[c + 1] = g->queue_off[c] + (int32_t)q[c].size();
    g->queue.insert(g->queue.end(), q[c].begin(), q[c].end());
  }
  g->lowered = true;
  return MK_OK;
}

// Tagged hand-offs.  At one or two activation rows the activations a GEMV reads (its x, and
// its residual) and the qkv rows attention tasks read are also written
// by their producers as (step tag, value) pairs into a library-owned
// mirror.  Such a reader polls its inputs' tags instead of waiting on
// counters: the data and the news that it is ready
// arrive in one round trip, where a counter costs the producer's fence,
// the counter's round trip and then the data's.  A buffer qualifies when
// it is f32, written exactly once per step (once[b]) and only by GEMV,
// COMBINE, embedding MEMCPY or RMSNORM tasks (the bodies that write the
// pairs); a GEMV qualifies when its x and residual do and every one of its
// parents writes one of them (weights and gamma have no writers), a split-KV
// partial or a cache append when its qkv does and every parent writes qkv.
bool mk::combine_polls(const mk_task_descriptor& d) {
  const uint32_t Hkv = d.reserved[2] & 0xFFFFu, T = (d.reserved[2] >> 16) + 1u;
  return d.op_id == MK_OP_ATTENTION_COMBINE && T == 1u && d.reserved[3] <= 32u && Hkv > 0u && d.k % (int)Hkv == 0 &&
         8 % (d.k / (int)Hkv) == 0;
}

void mk::build_ll_plan(mk_graph* g, const std::vector<std::vector<int>>& parents,
                       const std::vector<uint8_t>& once) {
  const size_t NB = g->bufs.size(), N = g->tasks.size();
  g->ll_buf.assign(NB, 0);
  g->ll_task.assign(N, 0);
  if (g->rows() >= kTcMinRows) return;
  std::vector<uint8_t> read_as_input(NB, 0), bad_writer(NB, 0);
  for (const mk_task_descriptor& d : g->tasks) {
    if (d.op_id == MK_OP_GEMV) {
      read_as_input[d.in_buf[0]] = 1;
      if (d.flags & MK_F_ADD_RESIDUAL) read_as_input[d.in_buf[2]] = 1;
    }
    if (d.op_id == MK_OP_ATTENTION_PARTIAL || d.op_id == MK_OP_ATTENTION_APPEND) read_as_input[d.in_buf[0]] = 1;
    if (d.op_id == MK_OP_ATTENTION_COMBINE && d.in_buf[0] < NB) {
      // a combine polls its partials' records only on its decode path
      if (combine_polls(d)) read_as_input[d.in_buf[0]] = 1;
      else bad_writer[d.in_buf[0]] = 1;
    }
    if (d.out_buf >= NB) continue;
    const bool ok = d.op_id == MK_OP_GEMV || d.op_id == MK_OP_ATTENTION_COMBINE || d.op_id == MK_OP_MEMCPY ||
                    d.op_id == MK_OP_RMSNORM || d.op_id == MK_OP_ATTENTION_PARTIAL;
    if (!ok) bad_writer[d.out_buf] = 1;
  }
  for (size_t b = MK_BUF_ROPE_SIN + 1; b < NB; ++b)
    g->ll_buf[b] = read_as_input[b] && once[b] && !bad_writer[b] && g->bufs[b].dtype == MK_F32;
  for (size_t t = 0; t < N; ++t) {
    const mk_task_descriptor& d = g->tasks[t];
    if (d.op_id == MK_OP_ATTENTION_PARTIAL || d.op_id == MK_OP_ATTENTION_APPEND) {
      // the query and new key and value come from qkv; the cache rows a
      // partial reads and the decode state have no writer before them
      bool ok = g->ll_buf[d.in_buf[0]];
      for (int q : parents[t]) ok = ok && g->tasks[q].out_buf == d.in_buf[0];
      g->ll_task[t] = ok;
      continue;
    }
    if (d.op_id != MK_OP_GEMV) continue;
    const bool res = d.flags & MK_F_ADD_RESIDUAL;
    bool ok = g->ll_buf[d.in_buf[0]] && (!res || g->ll_buf[d.in_buf[2]]);
    for (int q : parents[t]) {
      const uint16_t o = g->tasks[q].out_buf;
      ok = ok && (o == d.in_buf[0] || (res && o == d.in_buf[2]));
    }
    g->ll_task[t] = ok;
  }
}

extern "C" int mk_get_ll_plan(const mk_graph* g, const uint8_t** task_ll, const uint8_t** buf_ll) {
  if (!g || !task_ll || !buf_ll) return fail(MK_ERR_ARG, "mk_get_ll_plan: null argument");
  if (!g->lowered) return fail(MK_ERR_STATE, "mk_get_ll_plan: not lowered");
  *task_ll = g->ll_task.data();
  *buf_ll = g->ll_buf.data();
  return MK_OK;
}

// Dependency-counter plan.  With one counter per task, a B = 1 GEMV tile
// whose ~150 children each need every tile of its op sends ~150 atomics,
// and one op hand-off puts ~150^2 atomics on a few cache lines of
// neighbouring counters.  Here a task whose parents include a whole launch
// group waits on that group's one counter (each group member adds 1 to it
// once).  The remaining parents signal one counter per distinct remaining
// set (the partials of one KV-head group share theirs), indexed by the
// first task with that set.  Group counters sit 128 bytes apart after the
// per-task counters.  The plan follows the descriptors' remaining_deps: the
// set counter is expected to reach remaining_deps minus the parents covered
// by group counters, so a descriptor patched to one dependency too many
// still times out.
int mk::build_sync_plan(mk_graph* g) {
  const int N = (int)g->tasks.size();
  const int NG = (int)g->group_off.size() - 1;
  std::vector<int> group_of(N, 0);
  for (int k = 0; k < NG; ++k)
    for (int t = g->group_off[k]; t < g->group_off[k + 1]; ++t) group_of[t] = k;
  std::vector<std::vector<int>> parents(N);
  for (int p = 0; p < N; ++p) {
    const mk_task_descriptor& d = g->tasks[p];
    if ((uint64_t)d.dependents_offset + (uint64_t)d.num_dependents > g->edges.size())
      return fail(MK_ERR_ARG, "sync plan: dependents range of task " + std::to_string(p) + " outside the edges");
    for (int i = 0; i < d.num_dependents; ++i) {
      const uint32_t c = g->edges[d.dependents_offset + i];
      if ((int)c <= p || (int)c >= N)
        return fail(MK_ERR_ARG, "sync plan: edge " + std::to_string(p) + "->" + std::to_string(c) +
                                    " does not point forward");
      parents[c].push_back(p);
    }
  }
  // The last split of a K-split row block waits for its sibling splits
  // inside its body (after its own partial product), through the block's
  // arrival counter in the K-split scratch: those parents leave the plan.
  // So do a combine's partials when their records carry tagged pairs: the
  // combine polls them (its cache appends stay in the plan).
  std::vector<int> deferred(N, 0);
  const bool ll_ready_plan = g->ll_buf.size() == g->bufs.size();
  for (int t = 0; t < N; ++t) {
    const mk_task_descriptor& d = g->tasks[t];
    if (ll_ready_plan && d.op_id == MK_OP_ATTENTION_COMBINE && d.in_buf[0] < g->bufs.size() && g->ll_buf[d.in_buf[0]]) {
      std::vector<int>& ps = parents[t];
      const size_t before = ps.size();
      ps.erase(std::remove_if(ps.begin(), ps.end(), [&](int q) { return g->tasks[q].out_buf == d.in_buf[0]; }),
               ps.end());
      deferred[t] = (int)(before - ps.size());
      continue;
    }
    const int S = (int)((uint32_t)d.kv_len >> 16), j = d.kv_len & 0xFFFF;
    if (d.op_id != MK_OP_GEMV || d.config_id != 1 || S < 2 || j != S - 1) continue;
    std::vector<int>& ps = parents[t];
    const size_t before = ps.size();
    ps.erase(std::remove_if(ps.begin(), ps.end(), [&](int q) { return q >= t - (S - 1) && q < t; }), ps.end());
    deferred[t] = (int)(before - ps.size());
  }
  const uint32_t npad = (uint32_t)((N + 31) / 32 * 32);
  auto group_size = [&](int k) { return g->group_off[k + 1] - g->group_off[k]; };
  auto group_counter = [&](int k) { return npad + 32u * (uint32_t)k; };
  std::vector<char> group_used(NG, 0);
  std::vector<std::vector<int>> whole(N);    // groups task t waits on as a whole
  std::vector<int> own(N, 0);                // count task t expects on its set counter
  std::vector<int> own_ctr(N, 0);            // that counter: the first task with the same set
  std::vector<std::vector<uint32_t>> own_sig(N);  // set counters parent p signals
  std::map<std::vector<int>, int> set_ctr;   // remaining-parent set -> its counter
  std::vector<int> cnt(NG, 0);
  const bool have_ll = g->ll_task.size() == (size_t)N;
  for (int t = 0; t < N; ++t) {
    if (have_ll && g->ll_task[t]) {
      // reads every parent's output as tagged pairs: no counter, except a
      // surplus in a patched descriptor (which then can never be met)
      own[t] = std::max(g->tasks[t].remaining_deps - deferred[t] - (int)parents[t].size(), 0);
      own_ctr[t] = t;
      continue;
    }
    for (int p : parents[t]) cnt[group_of[p]]++;
    int covered = 0;
    for (int p : parents[t]) {
      const int k = group_of[p];
      if (group_size(k) > 1 && cnt[k] == group_size(k)) {
        whole[t].push_back(k);
        group_used[k] = 1;
        covered += group_size(k);
        cnt[k] = -1;  // marks the group as waited on whole
      }
    }
    std::vector<int> rest;
    for (int p : parents[t])
      if (cnt[group_of[p]] != -1) rest.push_back(p);
    for (int p : parents[t]) cnt[group_of[p]] = 0;
    own[t] = std::max(g->tasks[t].remaining_deps - deferred[t] - covered, 0);
    own_ctr[t] = t;
    if (!rest.empty()) {  // tasks with the same remaining parents share one counter
      auto it = set_ctr.emplace(rest, t).first;
      own_ctr[t] = it->second;
      if (it->second == t)
        for (int p : rest) own_sig[p].push_back((uint32_t)t);
    }
  }
  g->wait_off.assign(N + 1, 0);
  g->wait.clear();
  g->sig_off.assign(N + 1, 0);
  g->sig.clear();
  for (int t = 0; t < N; ++t) {
    std::sort(whole[t].begin(), whole[t].end());
    for (int k : whole[t]) {
      g->wait.push_back(group_counter(k));
      g->wait.push_back((uint32_t)group_size(k));
    }
    if (own[t] > 0) {
      g->wait.push_back((uint32_t)own_ctr[t]);
      g->wait.push_back((uint32_t)own[t]);
    }
    g->wait_off[t + 1] = (uint32_t)(g->wait.size() / 2);
    if (group_used[group_of[t]]) g->sig.push_back(group_counter(group_of[t]));
    for (uint32_t c : own_sig[t]) g->sig.push_back(c);  // ascending: children come in order
    g->sig_off[t + 1] = (uint32_t)g->sig.size();
  }
  g->counter_words = npad + 32u * (uint32_t)NG;
  return MK_OK;
}

extern "C" int mk_get_sync_plan(const mk_graph* g, const uint32_t** wait_off, const uint32_t** wait,
                                const uint32_t** sig_off, const uint32_t** sig, uint32_t* counter_words) {
  if (!g || !wait_off || !wait || !sig_off || !sig || !counter_words)
    return fail(MK_ERR_ARG, "mk_get_sync_plan: null argument");
  if (!g->lowered) return fail(MK_ERR_STATE, "mk_get_sync_plan: not lowered");
  *wait_off = g->wait_off.data();
  *wait = g->wait.data();
  *sig_off = g->sig_off.data();
  *sig = g->sig.data();
  *counter_words = g->counter_words;
  return MK_OK;
}

extern "C" int mk_get_tasks(const mk_graph* g, const void** bytes, size_t* nbytes) {
  if (!g || !bytes || !nbytes) return fail(MK_ERR_ARG, "mk_get_tasks: null argument");
  if (!g->lowered) return fail(MK_ERR_STATE, "mk_get_tasks: not lowered");
  *bytes = g->tasks.data();
  *nbytes = g->tasks.size() * sizeof(mk_task_descriptor);
  return MK_OK;
}

extern "C" int mk_get_edges(const mk_graph* g, const uint32_t** edges, size_t* count) {
  if (!g || !edges || !count) return fail(MK_ERR_ARG, "mk_get_edges: null argument");
  if (!g->lowered) return fail(MK_ERR_STATE, "mk_get_edges: not lowered");
  *edges = g->edges.data();
  *count = g->edges.size();
  return MK_OK;
}

extern "C" int mk_debug_patch_task(mk_graph* g, int task, const mk_task_descriptor* d) {
  if (!g || !d) return fail(MK_ERR_ARG, "mk_debug_patch_task: null argument");
  if (!g->lowered || g->uploaded) return fail(MK_ERR_STATE, "mk_debug_patch_task: needs a lowered, not uploaded graph");
  if (task < 0 || task >= (int)g->tasks.size()) return fail(MK_ERR_ARG, "mk_debug_patch_task: bad task index");
  g->tasks[task] = *d;
  return build_sync_plan(g);
}

extern "C" int mk_get_queues(const mk_graph* g, const int32_t** offsets, const int32_t** tasks,
                             int* num_ctas) {
  if (!g || !offsets || !tasks || !num_ctas) return fail(MK_ERR_ARG, "mk_get_queues: null argument");
  if (!g->lowered) return fail(MK_ERR_STATE, "mk_get_queues: not lowered");
  *offsets = g->queue_off.data();
  *tasks = g->queue.data();
  *num_ctas = g->num_ctas;
  return MK_OK;
}

static_assert(sizeof(mk_task_descriptor) == 64, "ABI: descriptor must be 64 bytes");
static_assert(offsetof(mk_task_descriptor, remaining_deps) % 4 == 0, "remaining_deps must be 4-byte aligned");
static_assert(offsetof(mk_task_descriptor, in_buf) == 20, "ABI: in_buf at 20");
static_assert(offsetof(mk_task_descriptor, reserved) == 44, "ABI: reserved at 44");
