// Kernel parameter blocks and host-side launchers of the decode-step kernels.
// Shapes are validated by the runtime before any launcher is called.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>

namespace lps {

constexpr int kMaxBatch = 8;
constexpr int kMaxDevices = 64;

// A device-side status (two words: error kinds OR-ed, the first report whole;
// see ptx.cuh) as a message naming the kernel that reported first.
std::string describe_status(int kinds, int first);

// The opt-in dynamic shared memory of a kernel belongs to each device's
// context: set it on the current device unless `done` (the launcher's own
// per-device record) shows at least `bytes` there already. Thread-safe.
template <class Kern>
cudaError_t set_smem_attr(Kern kern, int bytes, std::atomic<int>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) {
    int cur = done[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !done[dev].compare_exchange_weak(cur, bytes, std::memory_order_release)) {
    }
  }
  return e;
}

// ---- weight-streaming GEMV (batch 1) --------------------------------------
// y = W x over a row-major weight matrix whose rows are grouped into "units"
// of unit_rows consecutive rows (1, or 2 for a RoPE pair / a gate-up pair).
// Rows are packed at bind time so that every unit, and every CTA's range of
// units, is one contiguous byte range streamed by 1D bulk copies.
enum GemvEpilogue : int {
  kEpiQkv = 0,     // unit = (row i, row i + hd/2) of one head: RoPE, q out, K/V cache append
  kEpiResidual = 1,// unit = 1 row: h_out[r] = h_in[r] + y
  kEpiSwiglu = 2,  // unit = (gate_i, up_i): a[i] = silu(gate) * up
  kEpiStore = 3,   // unit = 1 row: out[r] = y (logits)
};

struct GemvParams {
  const void* w;        // packed weights [rows][K] (bf16 or int8)
  const float* wscale;  // int8: per packed row scale; else nullptr
  int rows, K;
  int unit_rows, units;
  int units_per_buf, nbuf;
  // input vector: either x (used as is) or rmsnorm(h) * gain
  const float* x;
  const float* h;
  const float* gain;
  float eps;
  // epilogue
  float* out;           // q [nq*hd] | a [ffn] | logits [rows]
  const float* h_in;    // residual input (may alias h_out)
  float* h_out;
  __nv_bfloat16* kc;    // K cache of this layer and sequence: [nkv][max_ctx][hd]
  __nv_bfloat16* vc;
  const float2* rope;   // (cos, sin) [hd/2] at this step's position
  int nq, nkv, hd, max_ctx, pos;
  int nwarps;           // consumer warps (set from the plan at launch)
  long long wait_limit; // cycles a buffer wait may take before it reports an error (<= 0: default)
  int* status;          // int[2]: error kinds, first error (see ptx.cuh)
  unsigned long long* trace;  // launch trace record, or nullptr
};

struct GemvPlan {
  int grid, smem, units_per_buf, nbuf, nwarps;
};
GemvPlan gemv_plan(int rows, int K, int unit_rows, bool int8, int num_sms, int max_smem);
bool gemv_supported(int K, int unit_rows, bool int8, int max_smem);
cudaError_t launch_gemv(const GemvParams& p, int epi, bool norm, bool int8, const GemvPlan& plan,
                        cudaStream_t s, bool pdl);

// ---- skinny GEMM, batch 2..8, on tensor cores --------------------------------
// Same epilogues as the GEMV, for all sequences of the batch at once; weights
// in the tiled layout of skinny_offset().
struct SkinnyParams {
  const void* w;           // tiled packed weights
  const float* wscale;     // int8: per packed row scale
  int rows, K, KC, KP, units, kw, rc, pu, batch;  // KP: K padded to whole k-chunks; see SkinnyPlan
  const float* x;          // [B][K]: the input, or h for the fused RMSNorm
  const float* gain;
  float eps;
  float* out;              // q [B][nq*hd] | a [B][ffn] | logits [B][rows] | h_out
  size_t out_stride;       // per sequence, in floats (also of h_in / h_out)
  const float* h_in;
  float* h_out;
  __nv_bfloat16* kc;       // layer cache [B][nkv][max_ctx][hd]
  __nv_bfloat16* vc;
  size_t kv_stride;        // per sequence, in elements
  const float2* rope;      // the whole (cos, sin) table [max_ctx][hd/2]
  int nq, nkv, hd, max_ctx;
  int pos[kMaxBatch];
  long long wait_limit;    // cycles a stage wait may take before it reports an error (<= 0: default)
  int* status;
  unsigned long long* trace;  // launch trace record, or nullptr
};
struct SkinnyPlan {
  int grid, smem, kc, units;
  int kw;          // k-groups: warp groups that each own every kw-th k-chunk (1, 2, 4 or 8)
  int pu;          // units per pass: a CTA's units are taken pu at a time, each pass over all of K
  int rc;          // k-chunks of a k-group's tiles in flight (its ring holds rc * pu tiles)
  int upw;         // units per warp in a pass (1, 2, 4 or 8)
  int kp;          // K padded to a whole number of k-chunks (zero columns)
  int rows_p;      // rows padded to whole 16-row units (zero rows)
};
SkinnyPlan skinny_plan(int rows, int K, bool int8, int batch, int num_sms, int max_smem);
// Complete a plan whose grid, units, kc, kw, pu and rc are set; false if it does not fit.
bool skinny_plan_finish(SkinnyPlan& g, int K, bool int8, int batch, int max_smem);
bool skinny_supported(int rows, int K, bool int8, int batch, int num_sms, int max_smem);
__host__ __device__ size_t skinny_offset(int r, int k, int kp, int kc, int units, int grid, int eb);
cudaError_t launch_skinny(const SkinnyParams& p, int epi, bool norm, bool int8, const SkinnyPlan& plan,
                          cudaStream_t s, bool pdl);
// Rearrange a row-major [rows][K] matrix (elements of eb bytes) into the tiled
// layout of `plan` for a [rows_p][kp] zero-padded matrix (dst must be zeroed first).
cudaError_t launch_retile(const void* src, void* dst, int rows, int K, const SkinnyPlan& plan, int eb, cudaStream_t s);

// ---- split-K GQA decode attention -----------------------------------------
struct AttnParams {
  CUtensorMap tmap_k;          // this layer's K cache as a 2D bf16 tensor [B*nkv*max_ctx rows][hd],
  CUtensorMap tmap_v;          // boxes of 64 elements x sub-tile rows, 128-byte swizzle
  const float* q;              // [B][nq*hd]
  const __nv_bfloat16* kc;     // layer base: [B][nkv][max_ctx][hd]
  const __nv_bfloat16* vc;
  float* out;                  // [B][nq*hd]
  float* part;                 // scratch [B][nq][max_chunks][hd + 4]: acc, m, l, pad
  int* counter;                // scratch [B][nkv], zero between launches
  int nq, nkv, hd, max_ctx, max_chunks;
  int chunk;                   // positions per CTA (multiple of the sub-tile)
  int pos[kMaxBatch];
  float scale;                 // 1/sqrt(hd)
  int early_dependents;        // 1: let the next kernel launch once every CTA has started
                               // (pays when it is the batch-1 GEMV), 0: once every CTA ends
  long long wait_limit;        // cycles a sub-tile wait may take before it reports an error (<= 0: default)
  int* status;
  unsigned long long* trace;  // launch trace record, or nullptr
};
int attn_sub_tile(int hd);
// Positions per attention CTA at max_pos (a function of the shapes, the
// position and the SM count only, so every stage plan gets the same bits).
int attn_chunk(int hd, int nkv, int batch, int max_pos, int num_sms);
int attn_max_chunks(int hd, int nkv, int batch, int max_ctx, int num_sms);
cudaError_t launch_attention(const AttnParams& p, int batch, int max_pos, cudaStream_t s, bool pdl);

// ---- prefill chunk: GEMM on tcgen05 tensor cores ---------------------------------
// Y[j][r] = sum_k W[r][k] X[j][k] for the ntok token rows of one prefill chunk
// (token j at position pos0 + j of sequence seq), W the packed bf16 weights
// [R][K] row-major, X two bf16 planes (hi rows [0, NP), lo rows [NP, 2 NP)).
// Epilogues: kEpiQkv (RoPE, q [ntok][nq*hd] and the K/V cache rows),
// kEpiResidual (h[j][r] += y), kEpiSwiglu (a = silu(gate) * up written as the
// down projection's two bf16 planes xo [2][NP][ldx]).
struct TcGemmParams {
  CUtensorMap tmap_w;          // W [R][K]: bf16 (box 64 x 128, 128-byte swizzle) or int8 (box 64 x 128, unswizzled)
  const float* wscale;         // int8: per packed row scale; else nullptr
  int int8;                    // 1: int8 weights, widened to bf16 in shared memory
  CUtensorMap tmap_x;          // X [2*NP][K] bf16: box 64 x NP, 128-byte swizzle
  int R, K, NP, ntok, epi;
  int stages, tmem_cols;       // set from the plan at launch
  int pos0, seq;
  float* q;
  __nv_bfloat16* kc;           // layer cache base [seqs][nkv][max_ctx][hd]
  __nv_bfloat16* vc;
  int nq, nkv, hd, max_ctx;
  const float2* rope;          // [max_ctx][hd/2]
  float* h;                    // residual rows [ntok][ldh]
  int ldh;
  __nv_bfloat16* xo;           // swiglu output planes [2][NP][ldx]
  int ldx;
  float* part;                 // scratch [grid][2][NP][128]
  int* counter;                // scratch [tiles], zero between launches
  long long wait_limit;
  int* status;
  unsigned long long* trace;
};
struct TcGemmPlan {
  int grid, smem, stages, tmem_cols;
  bool ok;
};
constexpr int kTcMaxTokens = 128;  // token rows of one prefill chunk (NP <= 128)
TcGemmPlan tc_gemm_plan(int NP, bool int8, int num_sms, int max_smem);
int tc_gemm_tiles(int R);
cudaError_t launch_tc_gemm(const TcGemmParams& p, const TcGemmPlan& plan, cudaStream_t s, bool pdl);
// 2D bf16 tensor map over a row-major [rows][cols] matrix with boxes of 64
// columns x box_rows rows and the 128-byte swizzle.
bool make_bf16_map(CUtensorMap* map, const void* base, unsigned long long cols, unsigned long long rows, int box_rows);
// The same for a row-major int8 matrix, boxes of 64 columns (bytes) x box_rows
// rows without a swizzle.
bool make_i8_map(CUtensorMap* map, const void* base, unsigned long long cols, unsigned long long rows, int box_rows);

// ---- prefill chunk: activation planes and chunk attention ------------------------
// Rows j < ntok of src [ntok][lds] (RMS-normalised with gain when gain != null)
// as two bf16 planes x [2][NP][K]: x[j] = bf16(v), x[NP + j] = bf16(v - bf16(v));
// rows [ntok, NP) of both planes are zeroed.
struct PrepParams {
  const float* src;
  int lds, K, NP, ntok;
  const float* gain;
  float eps;
  __nv_bfloat16* x;
  unsigned long long* trace;
};
cudaError_t launch_prep(const PrepParams& p, cudaStream_t s, bool pdl);

// Causal attention of ntok consecutive tokens (positions pos0 ..) of sequence
// seq over its cache rows, split by key chunks, then merged into the o-proj
// activation planes xo [2][NP][nq*hd].
struct ChunkAttnParams {
  CUtensorMap tmap_k;          // the layer's cache maps (box 64 x sub-tile rows, 128-byte swizzle)
  CUtensorMap tmap_v;
  const float* q;              // [ntok][nq*hd]
  float* part;                 // [ntok][nq][max_chunks][hd + 4]: o, m, l
  float* out;                  // when set: the merged o as fp32 [ntok][nq*hd] instead of the planes
  __nv_bfloat16* xo;
  int nq, nkv, hd, max_ctx, max_chunks;
  int chunk, nchunks, qblock;  // keys per CTA, CTAs per (block, kv head), tokens per block: chunk_attn_split
  int seq, pos0, ntok, NP;
  float scale;
  long long wait_limit;
  int* status;
  unsigned long long* trace;        // attention launch record, or nullptr
  unsigned long long* trace_merge;  // merge launch record, or nullptr
};
int chunk_attn_sub_tile(int hd);
int chunk_attn_max_chunks(int nkv, int num_sms);
void chunk_attn_split(int hd, int nq, int nkv, int ntok, int pos0, int num_sms, int* nchunks, int* chunk,
                      int* qblock);
cudaError_t launch_chunk_attn(const ChunkAttnParams& p, cudaStream_t s, bool pdl);

// ---- persistent stage kernel (batch 1) -----------------------------------------
// One launch runs every layer of a stage (and the embedding on stage 0, the
// final norm + LM head on the last stage) for one decode step; see stage.cu.
struct StageLayer {            // one layer's device pointers, in a device table
  CUtensorMap tmap_k;          // the layer's K cache as a 2D bf16 tensor [nkv*max_ctx rows][hd]
  CUtensorMap tmap_v;
  const void* w_qkv;           // packed as for the GEMV (RoPE pairs adjacent)
  const float* s_qkv;
  const void* w_o;
  const float* s_o;
  const void* w_gu;            // (gate_i, up_i) row pairs
  const float* s_gu;
  const void* w_d;
  const float* s_d;
  const float* attn_norm;
  const float* ffn_norm;
  __nv_bfloat16* kc;           // [nkv][max_ctx][hd]
  __nv_bfloat16* vc;
  float* o_out;                // attention output [nq*hd] (the layer's own with LPS_FLAG_KEEP_ATTN_OUT)
};

struct StageParams {
  const StageLayer* layers;    // device table [n_layers] of this stage
  int n_layers;
  int d, nq, nkv, hd, ffn, vocab, max_ctx;
  float eps, scale;
  int pos, tok;                // the step's position; the token when tok_dev is null
  const int* tok_dev;
  const void* embed;           // stage 0: the embedding table, else nullptr
  const float* embed_s;
  const void* head;            // last stage: the LM head, else nullptr
  const float* head_s;
  const float* out_norm;
  float* logits;               // [vocab]
  const float* h_in;           // the boundary slot a later stage reads, or nullptr (stage 0)
  float* h;                    // this stage's residual stream [d]
  float* h_out;                // where the last layer's down projection writes (next slot, or h)
  float* q;                    // [nq*hd]
  float* a;                    // [ffn]
  float* part;                 // attention chunk partials [nq][nch_max][hd + 4]
  const float2* rope;          // (cos, sin) table [max_ctx][hd/2]
  int nch, chunk;              // attention chunks per kv head at this position, positions per chunk
  int nch_max, nw, depth, xs_bytes, seg_cap;  // set from the plan at launch
  unsigned long long* bar;     // this stage's grid-barrier counter (monotonic)
  unsigned long long bar_base; // its value when this launch starts
  long long wait_limit;        // cycles a wait may take before it reports an error (<= 0: default)
  int* status;
  unsigned long long* trace;   // [n_phases][2] trace words of this launch, or nullptr
};

struct StageKernelPlan {
  bool ok;                     // the shapes fit the kernel
  int grid, nw, depth, smem, xs_bytes, seg_cap, nch_max;
};
StageKernelPlan stage_kernel_plan(int d, int nq, int nkv, int hd, int ffn, int vocab, bool int8, int num_sms,
                                  int max_smem);
void stage_attn_chunks(const StageKernelPlan& g, int hd, int nkv, int pos, int* nch, int* chunk);
int stage_sub_tile(int hd);  // positions per K/V sub-tile of the stage kernel (its tensor maps' box rows)
int stage_barriers(const StageParams& p);
cudaError_t launch_stage(const StageParams& p, bool int8, const StageKernelPlan& plan, cudaStream_t s, bool pdl);

// ---- embedding -------------------------------------------------------------
struct EmbedParams {
  const void* table;     // [vocab][d] bf16 or int8
  const float* scale;    // int8 row scales
  const int* tok_dev;    // device tokens, or nullptr to use tok[]
  int tok[kMaxBatch];
  int d, vocab, batch;
  float* h;              // [B][d]
  int* status;
  unsigned long long* trace;  // launch trace record, or nullptr
};
cudaError_t launch_embed(const EmbedParams& p, bool int8, cudaStream_t s, bool pdl);

}  // namespace lps
