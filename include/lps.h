/*
 * lps.h -- C ABI of the layer-staged eager decode step on one GB300 (sm_103a).
 *
 * One eager decode step of a decoder-only transformer trunk whose layers are
 * split into N contiguous stages, all on one GPU (the repeated-device-id mode
 * of ninfer's pipeline-stages.md, "What it is and is not": `--devices 0,0`).
 * Each stage owns its layers' weights, KV cache and scratch and runs on its own
 * CUDA stream; the f32 hidden state [n_embd] is the only tensor that crosses a
 * stage boundary, through two persistent slots per boundary ordered by ev_tx /
 * ev_rx events (memra_engine::pp module docs, "M2 increment 1" and "Ownership
 * across a boundary"). Logits are read back eagerly or deferred on a dedicated
 * readback stream ("M2 increment 3", PendingLogits).
 *
 * Conventions for every call:
 *   - return 0 (LPS_OK) on success, a negative LPS_E* code on failure;
 *     last_error_string() then names the refusing call and the reason;
 *   - arguments are checked before any GPU work is enqueued; a refused call
 *     changes no state ("fail closed": memra_engine::pp, refuse_unsplit_if_remote);
 *   - pointers marked "host" are ordinary CPU memory owned by the caller and
 *     only read or written during the call; pointers marked "device" are
 *     device memory on the model's GPU;
 *   - a model is driven from one host thread at a time.
 */
#ifndef LPS_H
#define LPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes ------------------------------------------------------- */
#define LPS_OK 0
#define LPS_EINVAL (-1)    /* bad argument: cuts, shapes, token >= vocab, pos out of range, ... */
#define LPS_ENOMEM (-2)    /* a device or pinned-host allocation failed */
#define LPS_ECUDA (-3)     /* a CUDA call failed, or a kernel reported a device-side error;
                              the model is then unusable and must be destroyed */
#define LPS_ETIMEDOUT (-4) /* pending_wait ran out of time; the pending handle stays valid */
#define LPS_EBUSY (-5)     /* every deferred-readback slot is held by an unfreed pending handle */

/* ---- opaque handles ---------------------------------------------------- */
typedef struct lps_stage_plan lps_stage_plan;
typedef struct lps_model lps_model;
typedef struct lps_pending lps_pending;

/* ---- stage plan (host only, no GPU needed) ----------------------------- */

/* Build the stage fence of a trunk of n_layers layers from N-1 cuts
 * (memra_engine::pp, "Door": cuts strictly increasing, each in (0, n_layers);
 * pp_cuts: fence = [0, c1, .., cN-1, n_layers], stage s runs layers
 * [fence[s], fence[s+1])).
 *   cuts    host int[n_cuts], or NULL for the even split into n_cuts+1 stages,
 *           cut s = s * n_layers / (n_cuts + 1) (integer division);
 *   n_cuts  N-1 >= 0;
 *   out     receives a new plan, owned by the caller (stage_plan_destroy).
 * LPS_EINVAL if the cuts are not strictly increasing in (0, n_layers) or the
 * even split would leave a stage empty. */
int stage_plan_create(int n_layers, const int* cuts, int n_cuts, lps_stage_plan** out);

/* The same plan spelled as layer counts per stage (ninfer pipeline-stages.md,
 * "How it works": `--stage-layers 30,34`). counts: host int[n_stages], each >= 1.
 * LPS_EINVAL for NULL counts or out, n_stages < 1 or a count < 1. */
int stage_plan_from_counts(const int* counts, int n_stages, lps_stage_plan** out);

/* Free a plan (models bound from it keep their own copy). NULL is a no-op. */
void stage_plan_destroy(lps_stage_plan* plan);

/* Number of stages N (>= 1); LPS_EINVAL for NULL. */
int stage_plan_n_stages(const lps_stage_plan* plan);

/* Copy the fence (N+1 ints) into host fence[cap]; returns N+1, or LPS_EINVAL for
 * NULL arguments or cap < N+1. */
int stage_plan_fence(const lps_stage_plan* plan, int* fence, int cap);

/* The stage that owns layer il (memra_engine::pp, stage_of); LPS_EINVAL if il is out of range. */
int stage_of(const lps_stage_plan* plan, int il);

/* Memory-balancing cuts (ninfer pipeline-stages.md, "How it works":
 * solve_stage_plan -- the largest capacity every stage can hold, then the
 * least-full stage; when nothing fits, the layers dealt evenly). Stage s
 * holding layers [i, j) at a capacity of P units (a unit is one context
 * position of the per-stage KV cache) uses
 *     stage_fixed[s] + sum(layer_bytes[i..j)) + P * sum(layer_unit_bytes[i..j))
 * bytes and must stay within stage_free[s]. The cuts returned give the
 * largest P in [0, max_units] over all contiguous plans with every stage
 * non-empty; among those, the smallest fullest-stage fraction
 * max_s(used_s / stage_free[s]) (compared exactly); among those, the
 * lexicographically smallest cuts. Host only, exact (not a heuristic).
 *   layer_bytes, layer_unit_bytes  host uint64[n_layers]
 *   stage_free   host uint64[n_stages], each > 0 (stages sharing one device
 *                split its free bytes between them)
 *   stage_fixed  host uint64[n_stages] or NULL (zeros): bytes a stage needs
 *                beyond its layers (workspace; the embedding on stage 0, the
 *                final norm, LM head and logits on the last stage)
 *   cuts_out     host int[n_stages - 1], for stage_plan_create
 *   units_out    the capacity P, or -1 when no plan fits even at P = 0 (the
 *                cuts are then the even split of stage_plan_create)
 * LPS_EINVAL for NULL arguments, n_stages outside [1, n_layers], max_units < 0
 * or a stage with no free bytes. */
int stage_plan_solve(int n_layers, int n_stages, const uint64_t* layer_bytes, const uint64_t* layer_unit_bytes,
                     const uint64_t* stage_free, const uint64_t* stage_fixed, int64_t max_units, int* cuts_out,
                     int64_t* units_out);

/* ---- model description and weights ------------------------------------- */
#define LPS_WEIGHT_BF16 0          /* bf16 weights */
#define LPS_WEIGHT_INT8_ROWSCALE 1 /* int8 weights with one fp32 scale per output row: w = q * s_row */
#define LPS_KV_BF16 0              /* bf16 KV cache */

#define LPS_FLAG_SINGLE_STREAM 1u  /* test arm: every stage on one stream, each boundary two plain
                                      device-to-device copies (memra_engine::pp, pp2_streams_off) */
#define LPS_FLAG_KEEP_ATTN_OUT 2u  /* keep each layer's attention output of the latest step
                                      readable through model_attn_out (debug) */
#define LPS_FLAG_VERIFY 8u         /* speculative-verify rows (memra_engine::pp, spec_pp_on: the verify
                                      forward takes the stage split): the batch's B rows are B
                                      consecutive positions of ONE sequence -- pos[b] == pos[0] + b --
                                      with one KV cache; row b writes cache row pos[b] and attends
                                      [0, pos[b]], so it sees the rows before it in the same step,
                                      and the step returns the logits of every row. The cache calls
                                      (model_kv_export/import) take sequence 0 only. */
#define LPS_FLAG_PERSISTENT 16u     /* batch 1: run each stage's layers as ONE persistent kernel launch
                                      per stage and step (a cooperative grid, one CTA per SM, grid-wide
                                      barriers between the projection and attention phases, all stages
                                      on one stream) instead of the default chain of per-projection
                                      kernels. Same results within the oracle tolerance, the same bits
                                      in every stage plan; on the 8B bf16 step it measures slower than
                                      the default chain, so it is opt-in. Ignored (stats.persistent = 0)
                                      for batch > 1, verify rows, the single-stream arm and shapes
                                      the kernel does not take. */
#define LPS_FLAG_GRAPH 32u          /* every step replays as one CUDA graph (ninfer pipeline-stages.md,
                                      "StageLink": decode captures the whole pass into one graph):
                                      the step is captured from stage 0's stream, the other stages'
                                      streams fork from it and join back through the boundary
                                      events, and each step's capture updates the instantiated graph
                                      in place (positions, logits buffer and attention grid change)
                                      before it is launched. Same bits as the stream path. Graph
                                      steps run one after another (the next replay starts when the
                                      previous one has ended), so consecutive steps do not overlap
                                      as they do on the streams; the per-kernel timers do not time
                                      graph steps. Not with LPS_FLAG_PERSISTENT (LPS_EINVAL). */
#define LPS_FLAG_SERIAL_STEPS 4u   /* make stage 0 of step t+1 also wait for the last stage of step t.
                                      By default stages of consecutive steps overlap, bounded
                                      only by the slot events (tokens t+1.. keep running while
                                      token t drains: memra_engine::pp, "M2 increment 3"); the
                                      math is the same either way. */

typedef struct lps_model_desc {
  int n_layers;     /* trunk layers; must equal the plan's */
  int n_embd;       /* d; multiple of 8 (16 for int8) */
  int n_q_heads;    /* nq (the bound width, dummy heads included) */
  int n_kv_heads;   /* nkv; nq % nkv == 0; q head h reads kv head h / (nq / nkv) */
  int head_dim;     /* hd: 64 or 128 */
  int ffn;          /* SwiGLU hidden width; multiple of 8 (16 for int8) */
  int vocab;        /* V */
  int weight_dtype; /* LPS_WEIGHT_* */
  int kv_dtype;     /* LPS_KV_BF16 */
  int max_ctx;      /* cache rows per (layer, sequence, kv head) */
  int batch;        /* B independent sequences per step, 1..8 */
  int pending_depth;/* deferred-readback slots; 0 means 4 */
  float rope_theta; /* RoPE base (rotate-half pairs (i, i + hd/2), angle pos * theta^(-2i/hd)) */
  float rms_eps;    /* RMSNorm epsilon: xn = h * g / sqrt(mean(h^2) + eps) */
  uint32_t flags;   /* LPS_FLAG_* */
} lps_model_desc;

/* A host weight matrix [rows, cols], row-major (output row r, input column k).
 * w: bf16 bit patterns (uint16) or int8 values; scale: host float[rows] for
 * LPS_WEIGHT_INT8_ROWSCALE, else ignored. */
typedef struct lps_matrix {
  const void* w;
  const float* scale;
} lps_matrix;

typedef struct lps_layer_weights {
  const float* attn_norm; /* [n_embd] fp32 RMSNorm gain before attention */
  lps_matrix wq;          /* [nq*hd, n_embd], rows head-major (row = head*hd + i) */
  lps_matrix wk;          /* [nkv*hd, n_embd] */
  lps_matrix wv;          /* [nkv*hd, n_embd] */
  lps_matrix wo;          /* [n_embd, nq*hd] */
  const float* ffn_norm;  /* [n_embd] */
  lps_matrix w_gate;      /* [ffn, n_embd] */
  lps_matrix w_up;        /* [ffn, n_embd] */
  lps_matrix w_down;      /* [n_embd, ffn] */
} lps_layer_weights;

typedef struct lps_model_weights {
  lps_matrix embed;                /* [vocab, n_embd]: h = E[token] (stage 0 owns it) */
  const float* out_norm;           /* [n_embd] final RMSNorm gain (last stage) */
  lps_matrix lm_head;              /* [vocab, n_embd] untied head (last stage) */
  const lps_layer_weights* layers; /* [n_layers] */
} lps_model_weights;

/* The byte model stage_plan_solve takes, for a model bound with this
 * library: layer_bytes[l] = the weights of layer l (QKV, o, gate, up, down,
 * int8 row scales, both norms); layer_unit_bytes[l] = its KV cache per context
 * position (K and V rows of every sequence, bf16); first_stage_bytes = the
 * embedding; last_stage_bytes = the LM head, final norm and logits buffers;
 * every_stage_bytes = a stage's activations, attention partials (one per 64
 * positions, a bound), RoPE table and boundary slots at desc->max_ctx -- a
 * close estimate, not the exact allocation. Not counted: the chunked
 * prefill's workspace, allocated per stage at the first model_prefill call
 * (rows of 128 tokens: hidden, q and activation planes, the chunk
 * attention's partials over about 2 x SMs / n_kv_heads key chunks, the
 * GEMM's per-CTA partial tiles; about 120 MB per stage at the 8B shape on
 * 152 SMs); it depends on the device's SM count, which this host-only call
 * does not know. Host arrays of n_layers entries. LPS_EINVAL for NULL
 * arguments or a bad shape. */
int model_stage_bytes(const lps_model_desc* desc, uint64_t* layer_bytes, uint64_t* layer_unit_bytes,
                      uint64_t* first_stage_bytes, uint64_t* last_stage_bytes, uint64_t* every_stage_bytes);

/* Optional runtime hooks. alloc/free route every device allocation of the
 * model (weights, caches, scratch, slots) to the caller, e.g. PyTorch's
 * caching allocator; alloc must return 256-byte-aligned device memory or NULL.
 * streams, if not NULL, holds N+1 cudaStream_t handles: one per stage, then
 * the readback stream; the caller keeps them alive until model_destroy. */
typedef void* (*lps_alloc_fn)(void* ctx, size_t bytes);
typedef void (*lps_free_fn)(void* ctx, void* ptr);
typedef struct lps_runtime {
  int device;          /* CUDA device ordinal */
  lps_alloc_fn alloc;  /* NULL: cudaMalloc */
  lps_free_fn free;    /* required when alloc is set */
  void* alloc_ctx;
  void* const* streams;/* NULL: the model creates its own non-blocking streams */
} lps_runtime;

/* Upload a model onto one GPU, placed per stage: stage s holds the weights,
 * KV cache ([layers of s][B][nkv][max_ctx][hd] bf16) and scratch of its
 * layers; the embedding goes with stage 0, the final norm and LM head with
 * the last stage (memra_engine::pp, layer_engine and new_cache). The weights
 * are copied (the caller may free them on return); the load ends with one
 * synchronize per stage (memra_engine::pp, sync_stages_after_load).
 *   plan  a stage plan whose n_layers equals desc->n_layers (not retained);
 *   rt    optional runtime hooks, or NULL (device 0, cudaMalloc, own streams).
 * LPS_EINVAL for unsupported shapes, LPS_ENOMEM / LPS_ECUDA on device failure
 * (everything allocated so far is released). The descriptor, the weight
 * pointers and the runtime hooks are checked before the device is touched:
 * those refusals (LPS_EINVAL) come the same with or without a GPU; the
 * limits that depend on the device (shared memory per block, SM count for
 * batch > 1) are checked after. */
int model_bind(const lps_stage_plan* plan, const lps_model_desc* desc, const lps_model_weights* w,
               const lps_runtime* rt, lps_model** out);

/* Drain every stream and free the model; outstanding pending handles become
 * invalid (free them first). NULL is a no-op. */
void model_destroy(lps_model* m);

/* ---- the decode step --------------------------------------------------- */

/* One eager decode step for every sequence b: token tokens[b] at position
 * pos[b]. Writes KV row pos[b] of every layer, attends over rows [0, pos[b]],
 * and copies the logits to host logits[B][vocab] (fp32, caller-owned) before
 * returning. Requires 0 <= tokens[b] < vocab and 0 <= pos[b] <= filled[b]
 * (the rows written so far; rewinding is allowed, holes are not) and
 * pos[b] < max_ctx; afterwards filled[b] = pos[b] + 1. LPS_EINVAL when an
 * argument breaks these rules (nothing is enqueued); LPS_ECUDA when a CUDA
 * call fails or a kernel reports a device-side error (the model is then
 * unusable: every later step or prefill on it returns LPS_ECUDA). */
int decode_step(lps_model* m, const int32_t* tokens, const int32_t* pos, float* logits);

/* The same step, ending without the logits copy (memra_engine::pp,
 * decode_step_h_ppn_deferred): the logits stay on the device with a
 * completion event and *out receives a pending handle. Later steps may be
 * enqueued before it is waited. LPS_EBUSY if all pending_depth slots are held. */
int decode_step_deferred(lps_model* m, const int32_t* tokens, const int32_t* pos, lps_pending** out);

/* Wait for a deferred step and copy its logits to host logits[B][vocab]: the
 * readback stream waits the step's completion event, copies and synchronizes
 * (memra_engine::pp, PendingLogits::wait). timeout_ms < 0 waits without limit;
 * LPS_ETIMEDOUT leaves the handle valid. A handle may be waited more than once. */
int pending_wait(lps_pending* p, float* logits, int timeout_ms);

/* Release a pending handle, waited or not (dropping without waiting is safe);
 * its readback slot is free again. NULL is a no-op. */
void pending_free(lps_pending* p);

/* The step with device-resident input and output: tokens is a device int[B],
 * pos a host int[B] (the per-step position snapshot), logits a device
 * float[B][vocab]. Returns once the step is enqueued; the logits are ready
 * when model_synchronize returns or after work ordered on the stream that
 * model_stream(m, N-1) returns. The same refusals as decode_step, except that
 * the token ids, being on the device, are not range-checked here: each must be
 * in [0, vocab). */
int decode_step_device(lps_model* m, const int32_t* tokens, const int32_t* pos, float* logits);

/* ---- chunked prefill through the stages -------------------------------- */

/* Prefill (memra_engine::pp, prime_pp_on / prime_pipe_on; ninfer
 * pipeline-stages.md, "Prefill micro-chunk overlap"): run the n prompt tokens
 * tokens[0..n) (host int32) of sequence b at positions pos0 .. pos0 + n - 1
 * through the stages, in chunks of `chunk` tokens (0 = 128, the maximum). Each
 * chunk's projections run as tcgen05 tensor-core GEMMs over its token rows,
 * its attention is causal inside the chunk over the cache rows [0, pos], and
 * the chunk's f32 hidden rows [chunk][n_embd] cross each stage boundary
 * through two slots ordered by events, so stage s works on chunk c while
 * stage s + 1 works on chunk c - 1. Writes the KV rows pos0 .. pos0 + n - 1
 * of every layer; afterwards filled[b] = max(filled[b], pos0 + n), and decode
 * continues at pos0 + n. logits (host float[vocab], may be NULL) receives the
 * last prompt token's logits. Returns once the prefill has completed.
 * Requires a batch-1 model (the row-major weight layout; bf16 weights, or int8
 * ones widened to bf16 in shared memory with the row scale on the result),
 * 0 <= pos0 <= filled[b], pos0 + n <= max_ctx and 0 <= tokens[i] < vocab;
 * else LPS_EINVAL. The first call allocates the prefill buffers (through the
 * model's allocator; LPS_ENOMEM on failure). Results match the oracle within
 * the decode tolerance and are the same bits for every stage plan. */
int model_prefill(lps_model* m, int b, const int32_t* tokens, int n, int pos0, int chunk, float* logits);

/* Block until every stream of the model is idle; reports device-side errors. */
int model_synchronize(lps_model* m);

/* Test hook: the SM cycles that every bounded device-side wait of this model's
 * kernels (a copy into a shared-memory ring, a ring slot's release) may take
 * before the kernel gives up, records an error and returns; 0 restores the
 * default of about two seconds. A kernel that gives up still waits, with its
 * own fixed bound, for the copies it has issued before it ends, and the next
 * readback or model_synchronize returns LPS_ECUDA with a message naming the
 * kernel that failed first; the model is then unusable. Synchronizes the model
 * first. LPS_EINVAL for cycles < 0. */
int model_set_wait_limit(lps_model* m, long long cycles);

/* Switch step overlap off (serial = 1: stage 0 of a step waits for the last
 * stage of the previous step, as LPS_FLAG_SERIAL_STEPS does at bind time) or
 * back on (serial = 0). Synchronizes the model first; results are unchanged
 * (each stage's kernels run in the same order either way). Used to time a
 * kernel family without other stages' kernels running beside it. */
int model_set_serial_steps(lps_model* m, int serial);

/* The cudaStream_t of stage s (0..N-1) or of the readback stream (s = N), into
 * *stream. LPS_EINVAL for NULL arguments or s outside 0..N. */
int model_stream(const lps_model* m, int s, void** stream);

/* ---- errors, counters, test hooks ---------------------------------------- */

/* Thread-local message of the last failure on this thread ("" if none). */
const char* last_error_string(void);

typedef struct lps_stats {
  uint64_t steps;              /* decode steps enqueued (all entry points) */
  uint64_t deferred_steps;     /* of which deferred */
  uint64_t stage_walks;        /* per-stage layer walks enqueued (N per step) */
  uint64_t boundary_crossings; /* hidden-state hand-overs across a cut (N-1 per step) */
  uint64_t pending_drains;     /* completed pending_wait readbacks */
  uint64_t kernel_launches;    /* this library's kernel launches */
  int n_stages;
  int fence[17];               /* the first min(N, 16)+1 entries of the fence */
  int persistent;              /* 1: steps run on the persistent stage kernel (LPS_FLAG_PERSISTENT),
                                  0: the chained per-projection kernels (the default) */
} lps_stats;

/* Copy the counters into *out (host). LPS_EINVAL for NULL arguments. */
int model_stats(const lps_model* m, lps_stats* out);

/* Copy the cache rows of (layer, sequence b) out of or into the device:
 * host buffer [2][nkv][max_ctx][hd] bf16 (K then V), bytes must equal
 * 4 * nkv * max_ctx * hd. Import also sets filled[b] = filled (0..max_ctx).
 * Both synchronize the owning stage's stream. With LPS_FLAG_VERIFY only b = 0
 * exists. LPS_EINVAL for a NULL model or buffer, a layer or sequence out of
 * range, another byte count, or (import) filled outside 0..max_ctx. */
int model_kv_export(const lps_model* m, int layer, int b, void* host, size_t bytes);
int model_kv_import(lps_model* m, int layer, int b, const void* host, size_t bytes, int filled);

/* Attention output of (layer, sequence b) in the latest step, host float[nq*hd];
 * synchronizes the layer's stage. LPS_EINVAL for bad arguments or a model bound
 * without LPS_FLAG_KEEP_ATTN_OUT. */
int model_attn_out(const lps_model* m, int layer, int b, float* host);

/* Per-kernel timing with CUDA events on the launching stream, for the kernel
 * family `kind` (LPS_KERNEL_QKV .. LPS_KERNEL_STAGE). Enabling starts a new
 * measurement; reading synchronizes and returns the summed device time and
 * launch count. A model on the persistent stage kernel launches only
 * LPS_KERNEL_STAGE; the per-projection families apply to the chained kernels.
 * LPS_EINVAL for a NULL model or output, or a kind above LPS_KERNEL_STAGE (the
 * kinds after it name launches in the trace only). */
#define LPS_KERNEL_QKV 0
#define LPS_KERNEL_ATTN 1
#define LPS_KERNEL_OPROJ 2
#define LPS_KERNEL_GATEUP 3
#define LPS_KERNEL_DOWN 4
#define LPS_KERNEL_HEAD 5
#define LPS_KERNEL_EMBED 6
#define LPS_KERNEL_STAGE 7  /* the persistent stage kernel (batch 1): one launch per stage and step */
#define LPS_KERNEL_MERGE 8  /* trace only: the persistent kernel's merge of the attention chunks */
#define LPS_KERNEL_PF_SPLIT 9   /* trace only: prefill, activation split (with the RMSNorm) */
#define LPS_KERNEL_PF_GEMM 10   /* trace only: prefill, a tcgen05 projection GEMM */
#define LPS_KERNEL_PF_ATTN 11   /* trace only: prefill, the chunk attention */
#define LPS_KERNEL_PF_MERGE 12  /* trace only: prefill, the merge of the chunk attention's key chunks */
int model_time_kernel(lps_model* m, int kind, int enable);
int model_kernel_time(lps_model* m, int kind, double* total_ms, uint64_t* launches);

/* ---- launch trace --------------------------------------------------------- */

/* One launch of a decode step or a prefill chunk: its kernel family, where it
 * ran, and the device clock (%globaltimer, ns) of its earliest CTA start and
 * latest warp end, so that overlapping launches (stages, programmatic
 * dependent launch, consecutive steps or chunks) show as they ran. */
typedef struct {
  int32_t kind;      /* LPS_KERNEL_* */
  int32_t stage;
  int32_t layer;     /* -1 for the embedding and the LM head */
  int32_t step;      /* the model's step counter when the launch was enqueued; for a
                        prefill launch (the LPS_KERNEL_PF_* kinds, and the embedding
                        and LM head of a prefill) the model's prefill chunk counter */
  uint64_t start_ns;
  uint64_t end_ns;   /* 0 if the launch has not finished or left early */
} lps_trace_record;

/* Record every launch of the following steps, up to `capacity` records (a
 * device buffer of 16 bytes per record, from the model's allocator; launches
 * past it are counted as dropped). Each kernel then does one extra atomic per
 * CTA as it starts and one per warp as it ends; results are unchanged. LPS_EINVAL for capacity < 1. */
int model_trace_enable(lps_model* m, int capacity);
/* Synchronize, copy up to max_records records (launch order) into out, return
 * their count and the dropped count, and start a new recording. LPS_EINVAL for
 * NULL arguments or when tracing is not enabled. */
int model_trace_read(lps_model* m, lps_trace_record* out, int max_records, int* n_records, uint64_t* dropped);
/* Stop recording and release the buffer (LPS_OK when tracing is already off). */
int model_trace_disable(lps_model* m);

/* ---- allocation-free attention ------------------------------------------ */

/* The staged runtime on the pages has no counterpart to this entry point. It
 * serves callers that may not allocate device memory once they run -- a
 * serving loop with a hard latency budget (allocation can synchronize the
 * device), or a program whose GPU memory is handed out once by its own pool.
 * It runs the same split-K GQA
 * decode attention as the decode step, without a model: its scratch (partial
 * results and chunk counters) is one file-scope device array of
 * LPS_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * exit. It calls no allocator.
 *   q        device float [batch][n_q_heads * head_dim]
 *   k_cache  device bf16 [batch][n_kv_heads][max_ctx][head_dim] (one layer),
 *   v_cache  same layout; 16-byte aligned; rows [0, pos[b]] are read
 *   out      device float [batch][n_q_heads * head_dim], written
 *   pos      host int[batch], 0 <= pos[b] < max_ctx
 *   stream   cudaStream_t to run on (NULL: the default stream)
 * Runs on the calling thread's current device and returns once enqueued.
 * The first call on a device looks up the array's address there. All calls
 * share the array (it keeps the last call's contents; the counters are
 * cleared by each call): calls that overlap on the GPU race, so keep them in
 * order on one stream. LPS_EINVAL for unsupported shapes, for
 * batch * n_kv_heads * max_ctx >= 2^31 (cache rows are addressed with 32-bit
 * coordinates), or when the call would need more scratch than the array holds
 * (message from attention_decode_noalloc_error()); LPS_ECUDA if a CUDA call
 * fails. A device-side wait that gives up (a copy that never lands) is not
 * seen by this call, which only enqueues: it sets a status word in the array,
 * and attention_decode_noalloc_status() reports it. */
#define LPS_NOALLOC_SCRATCH_BYTES (8u << 20)
int attention_decode_noalloc(const float* q, const void* k_cache, const void* v_cache, float* out, int batch,
                             int n_q_heads, int n_kv_heads, int head_dim, int max_ctx, const int32_t* pos,
                             void* stream);
const char* attention_decode_noalloc_error(void);

/* Synchronize `stream` (cudaStream_t, NULL: the default stream) and read the
 * status word that attention_decode_noalloc's kernel sets on the current
 * device when one of its bounded waits gives up. LPS_OK: no call since the
 * last check failed on the device. LPS_ECUDA: at least one call's `out` is
 * invalid (message from attention_decode_noalloc_error(), naming the kernel);
 * the word is then cleared. The word is shared by all calls on the device,
 * like the rest of the array. Allocates nothing. */
int attention_decode_noalloc_status(void* stream);

/* The scratch bytes attention_decode_noalloc needs for these shapes on the
 * current device (the call is refused when they exceed
 * LPS_NOALLOC_SCRATCH_BYTES), or -1 for unsupported shapes or without a
 * device. Launches nothing. */
long long attention_decode_noalloc_scratch_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim, int max_pos);

#ifdef __cplusplus
}
#endif

#endif /* LPS_H */
