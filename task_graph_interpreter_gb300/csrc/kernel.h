// Parameters and geometry shared by the persistent kernel and its host
// launcher (internal, not part of the public ABI).
#pragma once

#include <cstdint>

#include <vector_types.h>

#include "mk.h"

namespace mk {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 128;  // + one producer warpgroup
constexpr int kLaunchRegs = 168;    // registers per thread at launch (384 threads, 1 CTA/SM)
// The producer warpgroup runs the copy thread, the task-record warp and (in
// the class-2 kernel) the MMA warp.
constexpr int kProducerRegs = 56;   // after setmaxnreg.dec in the producer warpgroup
constexpr int kConsumerRegs = 224;  // after setmaxnreg.inc in the consumer warpgroups
static_assert(128 * kProducerRegs + 2 * 128 * kConsumerRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kStageBytes = 32768;               // one ring slot
constexpr int kStageElems = kStageBytes / 2;     // bf16 elements per slot
constexpr int kMaxStages = 5;                    // ring slots (a sixth only lengthened the HBM queues)
constexpr int kScratchBytes = 24576;             // per-task shared scratch
constexpr int kXbufBytes = 24576;                // class-2 kernel: two 12 KB activation staging tiles
constexpr int kTmemCols = 256;                   // class-2 kernel: GEMV accumulator columns
// Tensor memory per batch class: the class-2 kernel (three to eight
// activation rows) holds the GEMV accumulators (256 columns) and, after
// them, the split-KV partials' two 16-column score buffers; the class-0
// kernel (one or two rows) none: it runs no tensor-core work.
__host__ __device__ constexpr uint32_t tmem_cols(int bclass) { return bclass == 2 ? 512u : 0u; }
__host__ __device__ constexpr uint32_t tmem_part_col(int bclass) { return bclass == 2 ? 256u : 0u; }
constexpr int kTmapBytes = 128;                  // one CUtensorMap
constexpr int kKeyBlockRows = 128;               // keys per K box of the tensor-core split-KV partials
constexpr int kRecs = 8;                         // task-record FIFO entries (a power of two)
constexpr int kRecBytes = 256;                   // one task record
constexpr int kSlotFloats = 4096;                // GEMV per-warp partial slots
constexpr int kAccFloats = 1024;                 // GEMV per-row accumulators

// Status word layout (int32[4]): code, task, abort flag, spare.
constexpr int kStatusCode = 0, kStatusTask = 1, kStatusAbort = 2;

struct KParams {
  const mk_task_descriptor* tasks;
  const uint32_t* edges;
  void* const* bufs;          // buffer table (device pointers by index)
  uint32_t* counters;         // dependency counters (monotone): per task, then per launch group
  const uint32_t* wait_off;   // MEGA: task t waits on wait[wait_off[t] .. wait_off[t+1])
  const uint2* wait;          //   (counter index, count): counter >= epoch * count
  const uint32_t* sig_off;    // MEGA: task t then adds 1 to counters sig[sig_off[t] .. sig_off[t+1])
  const uint32_t* sig;
  const int32_t* queue_off;   // MEGA: per-CTA queue offsets
  const int32_t* queue;       // MEGA: task ids
  const int32_t* level_off;   // LEVELS: task range of each level
  const int32_t* level_tasks; // LEVELS: task ids grouped by level
  uint32_t* level_bar;        // LEVELS: one arrival counter per level boundary
  int32_t* status;            // int32[4]
  uint64_t* const* mirrors;   // MEGA, one or two rows: per buffer index, its (step tag, value) pairs or null
  uint32_t tag;               // MEGA: this step's tag (monotone across steps, never 0)
  const uint8_t* tmaps;       // CUtensorMap per buffer index (tensor-core weights), kTmapBytes each
  const int32_t* tm_rows;     // per buffer index: rows of its tensor map's box, 0 = no map
  const float* rope_cos;      // [cap, D/2]
  const float* rope_sin;
  uint64_t* trace;            // 8 x uint64 per task, or null
  uint64_t timeout_ns;
  uint32_t epoch;             // 1-based step counter (counter target = epoch * deps)
  int32_t mode;               // MK_MODE_MEGA / PER_OP / LEVELS
  int32_t first_task;         // PER_OP: first task of the launched group
  int32_t num_levels;         // LEVELS
  int32_t nstages;            // ring slots in use
  int32_t rope_half;          // D/2 of the tables
  int32_t num_bufs;           // entries of bufs / mirrors / tm_rows
  float* ksplit;              // K-split partial sums: kKsplitRecFloats floats per record
  uint32_t* karr;             // K-split arrival counters, one per record (the last split's is its block's)
  uint32_t kmul;              // a block's arrivals this step reach kmul * (S - 1)
};
constexpr int kKsplitRec = 256 * 8 + 8;  // floats per K-split record: [256 rows][8 batch] sums, 8 sums of squares

int smem_bytes_for(int nstages, int batch);

}  // namespace mk
