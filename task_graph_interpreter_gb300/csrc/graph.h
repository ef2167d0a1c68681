// Internal host-side state of an mk_graph (not part of the public ABI).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "mk.h"

namespace mk {

void set_error(const std::string& msg);
int fail(int code, const std::string& msg);

struct BufferRec {
  void* ptr = nullptr;
  int dtype = 0;
  int64_t rows = 0, cols = 0;
};

enum OpKind { K_EMBED, K_MATMUL, K_ATTENTION, K_SAMPLE, K_RMSNORM };

struct OpRec {
  OpKind kind;
  // embed: a0=table a1=out
  // matmul: a0=x a1=w a2=out a3=aux a4=pairs
  // attention: a0=qkv a1=k a2=v a3=out a4=scratch
  // sample: a0=pairs a1=history
  // rmsnorm: a0=x a1=gamma a2=out a3=residual
  uint16_t a[5] = {MK_NO_BUF, MK_NO_BUF, MK_NO_BUF, MK_NO_BUF, MK_NO_BUF};
  int B = 0, n = 0, k = 0, H = 0;
  int Hq = 0, Hkv = 0, D = 0, cap = 0, chunk = 0, V = 0;
  uint32_t flags = 0;
  float eps = 0.f;
  std::vector<int32_t> len0;
};

// Device-side resources owned by the library (runtime.cu).
struct DeviceState;

}  // namespace mk

struct mk_graph {
  mk_config cfg{};
  int num_ctas = 0, tiles_target = 0, col_align = 16;
  uint32_t timeout_us = 2000000;
  int B = 0;                       // sequences, from mk_set_state
  int T = 1;                       // tokens per sequence per step (mk_set_chunk)
  uint16_t tokens = MK_NO_BUF;     // int32 [B, T] input tokens of a chunk step (T > 1)
  bool state_set = false, lowered = false, uploaded = false;
  int rows() const { return B * T; }  // activation rows: row s * T + t
  std::vector<mk::BufferRec> bufs;  // index 0 state, 1/2 rope tables
  std::vector<mk::OpRec> ops;
  // rope parameters (shared by every attention op)
  double rope_theta = 0.0;
  int rope_D = 0, rope_cap = 0;
  // lowering output
  std::vector<mk_task_descriptor> tasks;
  std::vector<uint32_t> edges;
  std::vector<int32_t> queue_off, queue;       // per-CTA static queues
  std::vector<int32_t> level_off, level_tasks;  // topological levels
  std::vector<int32_t> group_off;               // per-op launch groups (task ranges)
  // dependency-counter plan (runtime only; descriptors and edges unchanged):
  // task t waits until counter[wait[i].first] >= epoch * wait[i].second for
  // every i in [wait_off[t], wait_off[t+1]), and when done adds 1 to
  // counter[sig[j]] for every j in [sig_off[t], sig_off[t+1]).
  std::vector<uint32_t> wait_off, wait, sig_off, sig;  // wait holds (counter, count) pairs
  uint32_t counter_words = 0;
  uint32_t ksplit_records = 0;     // K-split scratch records the lowering assigned
  // tagged hand-offs (one or two rows): buffers whose values are also written as
  // (step tag, value) pairs, and the GEMV, partial and append tasks that
  // read all their inputs from such pairs instead of waiting on counters
  std::vector<uint8_t> ll_buf, ll_task;
  // kernel geometry
  int max_m = 1;
  mk::DeviceState* dev = nullptr;
  std::vector<uint64_t> trace_host;
};

namespace mk {
// Row blocks and K splits of a GEMV op (ksplit_plan, graph.cpp): W rows per
// tile or block, nb blocks, S splits of K (1: not split).
struct KSplit {
  int W, nb, S;
};
KSplit ksplit_plan(int n, int k, uint32_t flags, int m, int tiles_target, int col_align);
// The library-owned scratch of the K-split partial sums, as a pseudo buffer
// index in dependency rectangles: one record of kKsplitRecFloats floats per
// split tile ([256 rows][8 batch] partial sums, then 8 partial sums of
// squares of x); the last split's record holds its block's arrival counter.
// Activation rows (B * T) from which GEMVs are dense contractions on the
// tensor cores (config_id 1, the batch-8 kernel; rows past B zero-padded)
constexpr int kTcMinRows = 3;
constexpr uint16_t kKsplitBuf = 0xFFFE;
constexpr int kKsplitRecFloats = 256 * 8 + 8;
int query_sm_count(int* out);  // runtime.cu
int tile_width(int n, int tiles_target, int col_align);
int tile_count(int n, int tiles_target, int col_align);
int build_sync_plan(mk_graph* g);  // graph.cpp; from the descriptors and edges
void build_ll_plan(mk_graph* g, const std::vector<std::vector<int>>& parents,
                   const std::vector<uint8_t>& once);  // graph.cpp; before build_sync_plan
// A COMBINE that polls its partials' tagged records when they have them:
// a decode step (T = 1) with at most 32 partials and G dividing 8 (graph.cpp)
bool combine_polls(const mk_task_descriptor& d);
std::vector<int> partials_per_sequence(const std::vector<int32_t>& len0, int Hkv, int chunk,
                                       int num_ctas);
}  // namespace mk
