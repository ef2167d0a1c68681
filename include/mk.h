/*
 * mk.h -- C ABI of libmk, a decode "megakernel" that interprets a static task
 * DAG on one GB300 (sm_103a).
 *
 * Model.  A decode step of a Llama-style decoder is composed by calling ops
 * on a graph object ("mega kernel initial", 1y33.com: the graph-building
 * part, where a decoder layer is written as matmul / attention calls with
 * gamma=, residual= and silu_mul= keywords).  mk_lower() turns the ops into
 * 64-byte task descriptors in topological order plus a flat dependents edge
 * array (same page: the lowering part with its TaskDescriptor listing, and
 * the part on flipping parents into a dependents edge array).  mk_upload()
 * copies descriptors, edges and the buffer pointer table to the device
 * (same page: the buffer-table and upload part).  mk_decode_step() runs one
 * persistent kernel, one CTA per SM, that walks a static per-CTA queue of
 * tasks; each task waits only for its own producers, through counters in
 * global memory or, at one or two activation rows, by polling its inputs' (step tag, value)
 * pairs, with no grid-wide barrier ("Megakernels",
 * runhoid.com: the "Hoid's approach to megakernels" section and its Fig. 5,
 * the on-GPU interpreter in which a block waits only for its producers).
 *
 * Conventions.
 *  - Every function returns an int: MK_OK (0) or a negative MK_ERR_* code;
 *    mk_last_error() gives a message for the calling thread's last error.
 *  - A graph is not thread-safe; use one graph from one thread at a time.
 *  - `stream` is a cudaStream_t passed as void*.  Device work is enqueued
 *    asynchronously on it.  Only mk_upload (pageable copies) and mk_status
 *    synchronise the stream.
 *  - The CALLER owns every tensor registered with mk_add_buffer/mk_set_state
 *    (weights, KV caches, activations, scratch, state, history): it
 *    allocates them, keeps them alive while the graph exists and frees them
 *    after mk_destroy.  The LIBRARY owns what it allocates in mk_upload:
 *    the device blob (descriptors, edges, buffer table, per-CTA queues,
 *    dependency counters, tagged mirrors, status word, RoPE tables, trace
 *    ring).
 *  - Functions up to mk_get_queues need no GPU unless num_ctas is 0.
 *  - Sizes are elements unless stated; all device pointers must be 256-byte
 *    aligned (PyTorch allocations are).
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_ABI_VERSION 1u

/* ---- return codes ------------------------------------------------------ */
#define MK_OK 0
#define MK_ERR_ARG (-1)    /* bad index, dtype, shape or argument */
#define MK_ERR_STATE (-2)  /* call out of order (add after lower, step before upload) */
#define MK_ERR_LIMIT (-3)  /* more than 65535 buffers, or a size over a stated limit */
#define MK_ERR_ABI (-4)    /* mk_config.abi_version != MK_ABI_VERSION */
#define MK_ERR_CUDA (-5)   /* a CUDA runtime call failed (message has details) */
#define MK_ERR_NOMEM (-6)  /* host or device allocation failed */

/* ---- device status codes reported by mk_status ------------------------- */
#define MK_DEV_OK 0
#define MK_DEV_DEP_TIMEOUT (-10)   /* a dependency wait exceeded wait_timeout_us */
#define MK_DEV_BAD_OP (-11)        /* a descriptor had an unknown op_id */
#define MK_DEV_RING_TIMEOUT (-12)  /* a shared-memory pipeline wait timed out */
#define MK_DEV_CAPACITY (-13)      /* pos + 1 reached the KV / history capacity */
#define MK_DEV_ABORTED (-14)       /* stopped because another CTA failed */
#define MK_DEV_BAD_INDEX (-15)     /* a token id outside the embedding table */

/* ---- op ids: "mega kernel initial", the OpId table --------------------- */
#define MK_OP_NOP 0
#define MK_OP_MEMCPY 1            /* used as the embedding row gather */
#define MK_OP_GEMV 2
#define MK_OP_RMSNORM 3
#define MK_OP_ATTENTION 4
#define MK_OP_MLP 5
#define MK_OP_SAMPLE 6
#define MK_OP_ATTENTION_APPEND 7
#define MK_OP_ATTENTION_PARTIAL 8
#define MK_OP_ATTENTION_COMBINE 9

/* ---- epilogue flags: "mega kernel initial", the flags paragraph after
 *      the descriptor listing (bit0..bit2); bit3 is this library's ------- */
#define MK_F_SILU_MUL 1u
#define MK_F_ADD_RESIDUAL 2u
#define MK_F_RMS_NORM_INPUT 4u
#define MK_F_ARGMAX_EPI 8u        /* per-tile (max, index) pairs for SAMPLE */

/* ---- buffer dtypes ------------------------------------------------------ */
#define MK_BF16 1
#define MK_F32 2
#define MK_I32 3
#define MK_PAIR 4                  /* mk_argmax_pair, 8 bytes */

/* ---- execution modes for mk_decode_step_ex ------------------------------ */
#define MK_MODE_MEGA 0            /* persistent kernel, counters and tagged hand-offs */
#define MK_MODE_PER_OP 1          /* one kernel launch per op, one CTA per task */
#define MK_MODE_PER_OP_GRAPH 2    /* MK_MODE_PER_OP captured once into a CUDA graph */
#define MK_MODE_LEVELS 3          /* persistent kernel, barrier per topological level */
#define MK_MODE_PER_OP_PDL 4      /* MK_MODE_PER_OP with programmatic dependent launch: a kernel
                                     starts streaming its weights while the previous one runs */

#define MK_NO_BUF 0xFFFFu
#define MK_BUF_STATE 0u           /* int32 [B, 2]: (next token, its position) */
#define MK_BUF_ROPE_COS 1u        /* library-owned float [capacity, D/2] */
#define MK_BUF_ROPE_SIN 2u

/* The 64-byte task descriptor, field for field as "mega kernel initial"
 * gives it (the TaskDescriptor listing): standard layout, trivially
 * copyable, remaining_deps 4-byte aligned for atomics. */
typedef struct mk_task_descriptor {
  uint16_t op_id;              /*  0 */
  uint16_t config_id;          /*  2  GEMV: 0 if m < 3 else 1; attention: 0 if D=64, 1 if D=128 */
  uint16_t step;               /*  4  speculative draft step tag; always 0 */
  uint16_t flags;              /*  6  MK_F_* */
  int32_t remaining_deps;      /*  8  number of distinct parents */
  int32_t num_dependents;      /* 12  edges leaving the task */
  uint32_t dependents_offset;  /* 16  index into the edge array */
  uint16_t in_buf[3];          /* 20  buffer-table indices */
  uint16_t out_buf;            /* 26 */
  int32_t m;                   /* 28  batch */
  int32_t n;                   /* 32  GEMV: output columns; attention: D */
  int32_t k;                   /* 36  GEMV: inner dim; attention: Hq; SAMPLE: tile count */
  int32_t kv_len;              /* 40  attention / SAMPLE: cache capacity */
  uint32_t reserved[5];        /* 44  per-op scalars (see mk_lower) */
} mk_task_descriptor;

typedef struct mk_argmax_pair {
  float value;
  int32_t index;
} mk_argmax_pair;

typedef struct mk_graph mk_graph;

typedef struct mk_config {
  uint32_t abi_version;      /* must be MK_ABI_VERSION */
  int32_t num_ctas;          /* persistent CTAs; 0 = SM count of the current device */
  int32_t tiles_target;      /* GEMV tiles per op; 0 = num_ctas */
  int32_t col_align;         /* GEMV tile width alignment; 0 = 16 */
  uint32_t wait_timeout_us;  /* bound on every device wait; 0 = 2,000,000 */
} mk_config;

/* Create an empty graph: the object a decode step is composed on ("mega
 * kernel initial", 1y33.com, graph-building part: the decoder layer written
 * as ops called on a Graph object; abi_version is the check the same page
 * asks for when the descriptor layout on the two sides could drift: the
 * version is bumped and a mismatch fails loudly).  Errors:
 * MK_ERR_ABI on a version mismatch, MK_ERR_ARG on negative sizes,
 * MK_ERR_CUDA if num_ctas == 0 and no device can be queried.  Buffer
 * indices 1 and 2 are reserved for the RoPE tables; the caller frees the
 * graph with mk_destroy. */
int mk_graph_create(const mk_config* cfg, mk_graph** out);

/* Register the decode state as buffer 0: int32 [B, 2], row s = (token the
 * next step consumes, its position).  SAMPLE tasks overwrite it each step.
 * Must precede every other registration.  Errors: MK_ERR_ARG, MK_ERR_STATE. */
int mk_set_state(mk_graph* g, void* state_dptr, int B);

/* Append a caller-owned device tensor to the buffer table ("mega kernel
 * initial", buffer-table part: an append-only table of device pointers
 * indexed by uint16).  rows x cols in elements of dtype, row-major,
 * contiguous.  *out_idx receives the index.  Errors: MK_ERR_ARG (null
 * pointer, misalignment, bad dtype), MK_ERR_LIMIT (table full),
 * MK_ERR_STATE (after mk_lower). */
int mk_add_buffer(mk_graph* g, void* dptr, int dtype, int64_t rows, int64_t cols,
                  uint16_t* out_idx);

/* Make every step of this graph a chunk step of T >= 2 tokens per sequence
 * (a prefill chunk, or draft tokens to verify in speculative decoding):
 * token t of sequence s sits at position pos[s] + t and attends causally to
 * the cache and the chunk's earlier tokens.  Activations then have B * T
 * rows (row s * T + t) and every matmul has m = B * T (at most 8).  Token 0
 * is the pending token in the state; tokens 1..T-1 are read each step from
 * `tokens`, a registered int32 [B, T] buffer the caller fills (column 0 is
 * not read).  SAMPLE takes the argmax of each sequence's last row, writes
 * tokens 1..T-1 and the sampled token to history[s, pos+1 .. pos+T] and
 * advances the state by T.  Per-token tasks (the embedding gathers and the
 * cache appends) carry t in the descriptor's `step` field ("mega kernel
 * initial", 1y33.com, the TaskDescriptor listing: `step` is the tag of a
 * speculative draft step); attention descriptors carry T - 1 in the high
 * half of reserved[2].  Must follow mk_set_state and the registration of
 * `tokens`, and precede every op.  Errors: MK_ERR_ARG (T < 2, B * T > 8,
 * tokens not an int32 [B, T] buffer), MK_ERR_STATE (ops already added,
 * already set, or lowered). */
int mk_set_chunk(mk_graph* g, int T, uint16_t tokens);

/* Embedding row gather (a MEMCPY task per sequence, our reading: the OpId
 * table lists MEMCPY as a utility and no embedding op):
 * out[s, :] = float(table[state[s].token, :]).  table bf16 [V, H],
 * out f32 [B, H].  In a chunk step (mk_set_chunk) one task per (s, t):
 * out[s * T + t, :] = float(table[token t of s, :]), out f32 [B * T, H]. */
int mk_add_embed(mk_graph* g, uint16_t table, uint16_t out, int B, int H);

/* Standalone RMS norm, one RMSNORM task per activation row ("mega kernel
 * initial", OpId table: usually fused into a GEMV, rarely standalone):
 *   y = x (+ residual);  out[r, :] = y / sqrt(mean(y^2) + eps) * gamma.
 * B is the state's batch; x, residual, out f32 [B * T, H] (T = 1 unless
 * mk_set_chunk); gamma bf16 [1, H]; residual = MK_NO_BUF for
 * none (with one, the task carries FUSED_RESIDUAL, flag bit 1; our reading:
 * only the normalised sum is written).  H a multiple of 8, at most 16384.
 * Errors: MK_ERR_ARG, MK_ERR_STATE. */
int mk_add_rmsnorm(mk_graph* g, uint16_t x, uint16_t gamma, uint16_t residual, uint16_t out, int B,
                   int H, float eps);

/* Epilogue fusion pass, before mk_lower: every standalone RMS norm without a
 * residual whose output is read only as the x input of GEMV ops that have
 * no aux operand is folded into those GEMVs (they read the norm's input
 * with RMS_NORM_INPUT, its gain and its eps) and removed; the norm's output
 * buffer is then never written.  *fused receives the number of norms
 * removed.  Errors: MK_ERR_STATE (already lowered), MK_ERR_ARG. */
int mk_fuse_rmsnorm(mk_graph* g, int* fused);

/* y = epilogue(W x) fanned out into one GEMV task per output-column tile
 * ("mega kernel initial", lowering part: one task per column tile, roughly
 * one per SM; RMSNorm, residual and SiLU*mul as epilogue flags).
 *  x   f32 [m, k]                W bf16 [n, k], or [2n, k] = [gate; up] with SILU_MUL
 *  out f32 [m, n]                aux: gamma bf16 [1, k] (RMS_NORM_INPUT) or
 *                                     residual f32 [m, n] (ADD_RESIDUAL) or MK_NO_BUF
 *  pairs MK_PAIR [T, m] (tile-major; T = mk_gemv_tiles(n)) with ARGMAX_EPI, else MK_NO_BUF.
 *  RMS_NORM_INPUT: x_hat = x / sqrt(mean(x^2) + eps) * gamma.
 *  SILU_MUL: out = silu(W_gate x) * (W_up x).  ADD_RESIDUAL: out += residual.
 * Limits: m = B * T (the activation rows), 1 <= m <= 8; k a multiple of 256
 * and at most 65536.
 * Errors: MK_ERR_ARG (shape/dtype mismatch, both RMS_NORM_INPUT and
 * ADD_RESIDUAL, missing pairs), MK_ERR_STATE. */
int mk_add_matmul(mk_graph* g, uint16_t x, uint16_t w, uint16_t out, uint16_t aux,
                  uint16_t pairs, uint32_t flags, int m, int n, int k, float eps);

/* Attention for one decode token per sequence, lowered to ATTENTION_APPEND
 * per (sequence, KV head), ATTENTION_PARTIAL per (sequence, KV head, KV
 * chunk) and ATTENTION_COMBINE per (sequence, KV head): plain flash
 * decoding with a log-sum-exp merge ("mega kernel initial", lowering part
 * and the OpId table; the combine is per KV head, our reading).
 *  qkv  f32 [B, (Hq + 2 Hkv) D]: q heads, then k heads, then v heads.
 *  kcache / vcache bf16 [B * Hkv, capacity * D] (= [B, Hkv, capacity, D]).
 *  out  f32 [B, Hq D].     scratch f32 [mk_attention_scratch_rows, G (D + 2)].
 *  In a chunk step (mk_set_chunk) qkv and out have B * T rows, there is one
 *  APPEND per (sequence, KV head, token) storing token t's row at pos + t,
 *  each PARTIAL serves all T tokens (token t sees keys 0 .. pos + t), and
 *  the scratch has T G (D + 2) columns; (Hq / Hkv) T <= 16.
 *  len0[B]: cached keys per sequence when the graph is built (fixes the chunk
 *  count).  chunk: keys per chunk, 0 = automatic.  D in {64, 128}; Hq/Hkv <= 4;
 *  at most 2048 / (Hq/Hkv) chunks per sequence (MK_ERR_LIMIT beyond).
 * APPEND applies rotate-half RoPE (base rope_theta) to k at position pos and
 * stores bf16 k, v at row pos; PARTIAL applies RoPE to q and runs an online
 * softmax (scale 1/sqrt(D)) over its chunk of the pos + 1 keys. */
int mk_add_attention(mk_graph* g, uint16_t qkv, uint16_t kcache, uint16_t vcache,
                     uint16_t out, uint16_t scratch, int B, int Hq, int Hkv, int D,
                     int capacity, const int32_t* len0, int chunk, double rope_theta);

/* SAMPLE per sequence: token = argmax over the lm_head tiles' pairs (first
 * index on ties); history[s, pos + 1] = token; state[s] = (token, pos + 1).
 * pairs MK_PAIR [T, B] (tile-major), history int32 [B, capacity].  In a
 * chunk step of T tokens the pairs are [tiles, B * T] and the argmax is
 * taken over row s * T + T - 1; history[s, pos + 1 .. pos + T - 1] gets the
 * step's input tokens 1..T-1, history[s, pos + T] the sampled token, and
 * the state becomes (token, pos + T). */
int mk_add_sample(mk_graph* g, uint16_t pairs, uint16_t history, int B, int V, int capacity);

/* Rows the scratch buffer of mk_add_attention needs (its columns are
 * T * G * (D + 2) floats, T = 1 unless mk_set_chunk). */
int mk_attention_scratch_rows(const mk_graph* g, int B, int Hkv, const int32_t* len0,
                              int chunk, int64_t* rows);

/* Number of column tiles an n-column GEMV fans out into. */
int mk_gemv_tiles(const mk_graph* g, int n, int32_t* tiles);

/* Bytes the registered buffer `buf` needs as the scratch of the attention
 * ops or the argmax pairs of the matmul ops already added that name it (the
 * largest if several do); lets a caller check an allocation made from
 * mk_attention_scratch_rows / mk_gemv_tiles.  Errors: MK_ERR_ARG (null
 * argument, or no added op uses buf that way). */
int mk_scratch_size(const mk_graph* g, uint16_t buf, size_t* bytes);

/* Lower every op to descriptors and edges and build the per-CTA queues;
 * freezes the graph ("mega kernel initial", 1y33.com, lowering part: each op
 * becomes 64-byte TaskDescriptors, a matmul fans out into column tiles and
 * attention into split-KV partials and a combine; and the edge part: every
 * task's parents are found from the column ranges it reads, flipped into
 * dependents lists and flattened into one edge array in topological order).
 * Descriptor fields by op (unused in_buf = MK_NO_BUF, unused fields 0):
 *  RMSNORM  in={x,gamma,residual} out=out m=B n=H flags=FUSED_RESIDUAL (bit 1)
 *           with a residual; reserved={s, float bits of eps}
 *  GEMV     in={x,W,aux} out=y m=B n k; reserved={col_begin, col_count,
 *           float bits of eps (RMS_NORM_INPUT) or 0, pairs idx or 0,
 *           tile index (ARGMAX_EPI) or 0}.  config_id 1 (tensor cores, from
 *           three activation rows) with a K split: kv_len = j | S << 16
 *           (split j of S), reserved[3] = k_begin | k_count << 16,
 *           reserved[4] = the split's scratch record (the last split's
 *           record ends the block's S records)
 *  APPEND   in={qkv,K,V} out=K m=B n=D k=Hq kv_len=capacity reserved={s,g,Hkv,0,0}
 *  PARTIAL  in={qkv,K,V} out=scratch, same m/n/k/kv_len,
 *           reserved={s,g,Hkv, c | (P_s << 16), first slot of (s,g)}
 *  COMBINE  in={scratch,K,V} out=att, same m/n/k/kv_len, reserved={s,g,Hkv,P_s,first slot}
 *           (K and V order the append before the attention output)
 *  MEMCPY   in={table} out=h m=B n=H reserved={s, rows of the table}
 *  SAMPLE   in={pairs} out=history m=B n=V k=tiles kv_len=capacity reserved={s}
 * A chunk step of T tokens (mk_set_chunk) changes only: attention tasks
 * carry Hkv | (T-1) << 16 in reserved[2]; APPEND is one task per token t
 * with step = t; MEMCPY is one task per (s, t) with step = t, in_buf[1] =
 * tokens and reserved[2] = T-1; SAMPLE has in_buf[1] = tokens and
 * reserved[1] = T-1; RMSNORM is one task per activation row, reserved[0] =
 * the row.  With T = 1 every byte is as above.
 * Errors: MK_ERR_STATE (already lowered or no ops). */
int mk_lower(mk_graph* g);

/* Lowered descriptors (mk_task_descriptor[count]) and edges (uint32[count]);
 * the memory belongs to the graph and lives until mk_destroy. */
int mk_get_tasks(const mk_graph* g, const void** bytes, size_t* nbytes);
int mk_get_edges(const mk_graph* g, const uint32_t** edges, size_t* count);

/* Test hook for fault-detection tests: overwrite descriptor `task` of a
 * lowered, not yet uploaded graph (e.g. a dependency count one too high, or
 * an unknown op_id).  The device then reports MK_DEV_DEP_TIMEOUT or
 * MK_DEV_BAD_OP through mk_status instead of hanging or faulting.
 * Errors: MK_ERR_STATE (not lowered, or already uploaded), MK_ERR_ARG. */
int mk_debug_patch_task(mk_graph* g, int task, const mk_task_descriptor* d);

/* The dependency-counter plan the persistent kernel follows (a runtime
 * detail; descriptors and edges are not changed by it).  Task t waits until
 * counter[wait[2i]] >= epoch * wait[2i+1] for every i in
 * [wait_off[t], wait_off[t+1]) and, when done, adds 1 to counter[sig[j]]
 * for every j in [sig_off[t], sig_off[t+1]).  Parents that make up a whole
 * launch group (all GEMV tiles of one op, all partials of one attention op,
 * ...) are waited for through that group's one shared counter; the other
 * parents through one counter shared by every task with the same remaining
 * parents (its index is the first such task's); counter_words is the size
 * of the counter array.  Parents a task waits for in its body instead
 * (the sibling splits of a K-split block's last split; the partials whose
 * tagged records a decode COMBINE polls) leave its waits.  Arrays: wait_off
 * and sig_off uint32[N + 1], wait uint32[2 * wait_off[N]], sig
 * uint32[sig_off[N]]; they belong to the graph.  Errors: MK_ERR_STATE (not
 * lowered), MK_ERR_ARG. */
int mk_get_sync_plan(const mk_graph* g, const uint32_t** wait_off, const uint32_t** wait,
                     const uint32_t** sig_off, const uint32_t** sig, uint32_t* counter_words);

/* Tagged hand-offs (one or two activation rows, megakernel mode): task_ll[t] = 1 for the GEMV,
 * ATTENTION_PARTIAL and ATTENTION_APPEND tasks that read all their
 * activation inputs as (step tag, value) pairs and so wait on no counter;
 * buf_ll[b] = 1 for the buffers whose producers also write those pairs (into
 * library-owned mirrors: f32 buffers written once per step by one op's
 * GEMV, COMBINE, embedding or RMSNORM tasks, and the attention scratch
 * whose ATTENTION_PARTIAL records every reading COMBINE polls on its decode
 * path: T = 1, at most 32 partials, G dividing 8; such a combine waits
 * through counters for its appends only).  uint8 arrays of the task and
 * buffer counts, owned by the graph, fixed at lowering.  Errors: MK_ERR_ARG
 * (null argument), MK_ERR_STATE (not lowered). */
int mk_get_ll_plan(const mk_graph* g, const uint8_t** task_ll, const uint8_t** buf_ll);

/* Per-CTA task queues: offsets int32[num_ctas + 1] into tasks int32[]. */
int mk_get_queues(const mk_graph* g, const int32_t** offsets, const int32_t** tasks,
                  int* num_ctas);

/* Copy descriptors, edges, queues and the buffer pointer table to the
 * current device, build the RoPE tables (float64 on the host, stored as
 * float), and zero the dependency counters ("mega kernel initial",
 * 1y33.com, buffer-table and upload part: one contiguous blob of header,
 * tasks and edges copied to the device at once, with the table of buffer
 * pointers beside it).  The blob belongs to the library until mk_destroy.
 * Synchronises `stream`.  Errors: MK_ERR_STATE (not lowered), MK_ERR_CUDA,
 * MK_ERR_NOMEM. */
int mk_upload(mk_graph* g, void* stream);

/* Number of GEMV tiles of an uploaded graph that run on the tensor-core
 * path: tiles of ops with three to eight activation rows (config_id 1;
 * rows past B enter as zeros) whose K is a multiple of 64.
 * Their weights stream through TMA tensor copies (a tensor map per weight
 * buffer, built by mk_upload) and multiply on tcgen05 tensor cores with
 * f32 accumulators in tensor memory; the activations enter as three
 * bf16 parts (hi + mid + lo), which carry x to about f32 precision.
 * Other tiles run on CUDA cores.  Errors: MK_ERR_STATE (not uploaded),
 * MK_ERR_ARG. */
int mk_gemv_tensor_core_tiles(const mk_graph* g, int* tiles);

/* One decode step with the persistent kernel (MK_MODE_MEGA): one CTA per
 * SM walks its static queue, each task waits only for its own producers
 * and releases its dependents when done, with no grid-wide barrier
 * ("Megakernels", runhoid.com, "Hoid's approach to megakernels" and Fig. 5:
 * the on-GPU interpreter whose blocks wait only for their producers).
 * Enqueued on `stream`; the caller's registered tensors are read and
 * written in place (the state advances by one position per sequence).
 * Errors: MK_ERR_STATE (not uploaded), MK_ERR_CUDA (launch failed); device
 * failures are read with mk_status. */
int mk_decode_step(mk_graph* g, void* stream);

/* One decode step in `mode` (MK_MODE_*).  trace != 0 records, per task, the
 * CTA, SM and %globaltimer stamps (wait begin, start, end) readable with
 * mk_get_trace after the stream synchronises.  MK_MODE_PER_OP_GRAPH
 * captures the per-op launches into a CUDA graph on first use. */
int mk_decode_step_ex(mk_graph* g, void* stream, int mode, uint32_t trace);

/* One MK_MODE_MEGA step driven from host memory: copies state_in (int32
 * [B, 2], pinned host memory recommended; NULL = keep the device state)
 * to the state buffer, runs the step, and copies the sampled tokens
 * (int32 [B]) to tokens_out, all enqueued on `stream`; the caller
 * synchronises before reading tokens_out. */
int mk_decode_step_host(mk_graph* g, void* stream, const int32_t* state_in,
                        int32_t* tokens_out);

/* Synchronise `stream`, then read and clear the device status word:
 * *dev_code = MK_DEV_* and *task_id = the failing task (or -1). */
int mk_status(mk_graph* g, void* stream, int* dev_code, int32_t* task_id);

/* Trace records of the last traced step: uint64[count * 8] per task as
 * (cta << 32 | smid, t_wait_begin, t_start, t_end, mark0, mark1, mark2,
 * ring_waits), %globaltimer nanoseconds: the dependency wait began /
 * ended, the task's outputs were complete (before its dependents are
 * released), and marks inside the body (GEMV and PARTIAL: first ring slot
 * ready, all slots consumed, epilogue or merge done; 0 where unused);
 * ring_waits counts the task's ring slots whose copies had not landed when
 * the consumers reached them. */
int mk_get_trace(mk_graph* g, const uint64_t** records, size_t* count);

/* Test hook for the wrap-around of the dependency counters: put an uploaded
 * graph in the state it would have after `epoch` megakernel steps (every
 * counter at epoch times the adds it receives per step, modulo 2^32) with
 * `tag` as the last step tag; the next step is then step epoch + 1 with tag
 * tag + 1 (0 skipped).  Lets a test run steps across the point where
 * counters and their targets wrap.  Synchronises `stream`.  Errors:
 * MK_ERR_STATE (not uploaded), MK_ERR_CUDA. */
int mk_debug_set_epoch(mk_graph* g, void* stream, uint32_t epoch, uint32_t tag);

/* Bytes of shared memory the kernel uses per CTA and its thread count. */
int mk_kernel_info(const mk_graph* g, int* smem_bytes, int* threads, int* stages);

/* Decode attention that allocates nothing.  No counterpart in the paper:
 * this entry point exists for callers that cannot call cudaMalloc once they
 * run -- servers and plugins that give all of HBM to their own pool at start
 * up and forbid later device allocations, and latency-critical loops where
 * an allocation could synchronise the device.  It runs one step of the
 * attention op on device pointers the caller passes: the new k (rotate-half
 * RoPE, base rope_theta) and v rows of qkv f32 [B, (Hq + 2 Hkv) D] are
 * stored as bf16 at row pos[s] of kcache / vcache bf16 [B, Hkv, capacity, D],
 * and out f32 [B, Hq D] receives softmax(q K^T / sqrt(D)) V over keys
 * 0..pos[s], computed as split-KV partials (chunk count from len0 and chunk
 * as in mk_add_attention; chunk 0 uses the device's SM count) merged by a
 * log-sum-exp combine.  pos and len0 are host arrays [B].  Same limits as
 * mk_add_attention (B <= 8, D in {64, 128}, Hq/Hkv <= 4).
 * The partial scratch lives in a file-scope device array of
 * MK_NOALLOC_SCRATCH_FLOATS floats (4 MiB) that every GPU loading the
 * library holds until the process exits; a call needing more returns
 * MK_ERR_LIMIT.  No cudaMalloc, cudaFree or other allocation happens here.
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it for the life of the process; make that first
 * call before any stream capture, and do not call cudaDeviceReset after it.
 * All calls share the array: calls whose kernels overlap on the GPU race.
 * Enqueued on `stream`; errors: MK_ERR_ARG, MK_ERR_LIMIT, MK_ERR_CUDA (also
 * when an error from the caller's earlier work is pending: it is reported,
 * not cleared, and nothing is launched). */
#define MK_NOALLOC_SCRATCH_FLOATS (1 << 20)
int mk_attention_decode_noalloc(void* stream, const float* qkv, void* kcache, void* vcache, float* out,
                                int B, int Hq, int Hkv, int D, int capacity, const int32_t* pos,
                                const int32_t* len0, int chunk, double rope_theta);

/* Release everything the library allocated.  Safe on NULL. */
void mk_destroy(mk_graph* g);

/* Message for the calling thread's last error ("" if none). */
const char* mk_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MK_H */
