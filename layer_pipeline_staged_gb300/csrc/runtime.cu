// Host runtime behind the C ABI of include/lps.h: stage plans, per-stage
// placement and upload, the step schedule across per-stage streams with
// double-buffered boundary slots ordered by ev_tx / ev_rx events, eager and
// deferred logits readback, counters and test hooks.
//
// Structure follows the pages' N-stage runtime (memra_engine::pp): per-stage
// execution homes (StageRt: stream + stage-owned weights, cache and scratch),
// N-1 boundaries with two persistent slots each and their own step counter,
// the fence of pp_cuts, the load barrier of sync_stages_after_load and the
// PendingLogits readback on a dedicated stream. Differences from the pages'
// design: one device and one context; every buffer is allocated at bind
// (nothing is allocated per step); the hand-over is fused into the kernels
// (the last layer of stage s writes its residual output straight into the
// boundary slot and stage s+1's first layer reads it from there); and all
// shared mutable state of a step is per stage, so stages of consecutive
// steps can overlap on one device.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "kernels.h"
#include "lps.h"

namespace lps {
bool attn_supported(int hd, int group);
}  // namespace lps

using namespace lps;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fn, const std::string& why) {
  g_err = std::string(fn) + ": " + why;
  return code;
}

int cuda_fail(const char* fn, const char* what, cudaError_t e) {
  return fail(LPS_ECUDA, fn, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CK(expr, what)                                   \
  do {                                                   \
    cudaError_t e_ = (expr);                             \
    if (e_ != cudaSuccess) return cuda_fail(FN, what, e_); \
  } while (0)

}  // namespace

namespace lps {
// The thread's last error, for host code in other files (the stage solver).
int host_fail(int code, const char* fn, const std::string& why) { return fail(code, fn, why); }

std::string describe_status(int kinds, int first) {
  static const char* const kKernels[] = {"unknown kernel",
                                         "RMSNorm + QKV + RoPE + KV append",
                                         "o-proj / down projection + residual",
                                         "RMSNorm + gate/up + SwiGLU",
                                         "final RMSNorm + LM head",
                                         "split-K attention",
                                         "split-K attention (merge of the chunks)",
                                         "embedding",
                                         "persistent stage kernel",
                                         "prefill GEMM (tcgen05)",
                                         "prefill chunk attention",
                                         "prefill RMSNorm / activation split"};
  const int kid = (first >> 8) & 0xf;
  std::string what;
  const int k = first & 0xff ? first & 0xff : kinds;
  if (k & 1) what += "a copy wait timed out; ";
  if (k & 2) what += "a buffer-release wait timed out; ";
  if (k & 4) what += "draining in-flight copies timed out; ";
  if (k & 8) what += "a kernel argument was out of range; ";
  if (k & 16) what += "a grid-wide barrier wait timed out; ";
  if (what.empty()) what = "unknown error; ";
  std::string name = kKernels[kid < 12 ? kid : 0];
  if (first & 0x1000) name += " (batch > 1 tensor-core GEMM)";
  char buf[96];
  std::snprintf(buf, sizeof buf, "(status 0x%x, first report 0x%x, detail %d)", kinds, first,
                static_cast<int>(static_cast<unsigned>(first) >> 13));
  return "device-side error in " + name + ": " + what + buf;
}
}  // namespace lps

// ---------------------------------------------------------------------------
// stage plan
// ---------------------------------------------------------------------------

struct lps_stage_plan {
  int n_layers;
  std::vector<int> fence;  // N+1 entries
};

extern "C" int stage_plan_create(int n_layers, const int* cuts, int n_cuts, lps_stage_plan** out) {
  static const char* FN = "stage_plan_create";
  if (!out) return fail(LPS_EINVAL, FN, "out is NULL");
  *out = nullptr;
  if (n_layers < 1) return fail(LPS_EINVAL, FN, "n_layers must be >= 1");
  if (n_cuts < 0 || n_cuts >= n_layers) return fail(LPS_EINVAL, FN, "need 0 <= n_cuts < n_layers");
  const int N = n_cuts + 1;
  std::vector<int> fence(N + 1);
  fence[0] = 0;
  fence[N] = n_layers;
  for (int s = 1; s < N; ++s) fence[s] = cuts ? cuts[s - 1] : static_cast<int>(static_cast<long long>(s) * n_layers / N);
  for (int s = 0; s < N; ++s)
    if (fence[s + 1] <= fence[s])
      return fail(LPS_EINVAL, FN, "cuts must be strictly increasing and inside (0, n_layers)");
  *out = new lps_stage_plan{n_layers, fence};
  return LPS_OK;
}

extern "C" int stage_plan_from_counts(const int* counts, int n_stages, lps_stage_plan** out) {
  static const char* FN = "stage_plan_from_counts";
  if (!out) return fail(LPS_EINVAL, FN, "out is NULL");
  *out = nullptr;
  if (!counts || n_stages < 1) return fail(LPS_EINVAL, FN, "need counts and n_stages >= 1");
  std::vector<int> fence(n_stages + 1, 0);
  for (int s = 0; s < n_stages; ++s) {
    if (counts[s] < 1) return fail(LPS_EINVAL, FN, "every stage needs at least one layer");
    fence[s + 1] = fence[s] + counts[s];
  }
  *out = new lps_stage_plan{fence[n_stages], fence};
  return LPS_OK;
}

extern "C" void stage_plan_destroy(lps_stage_plan* p) { delete p; }

extern "C" int stage_plan_n_stages(const lps_stage_plan* p) {
  if (!p) return fail(LPS_EINVAL, "stage_plan_n_stages", "plan is NULL");
  return static_cast<int>(p->fence.size()) - 1;
}

extern "C" int stage_plan_fence(const lps_stage_plan* p, int* fence, int cap) {
  static const char* FN = "stage_plan_fence";
  if (!p || !fence) return fail(LPS_EINVAL, FN, "NULL argument");
  const int n = static_cast<int>(p->fence.size());
  if (cap < n) return fail(LPS_EINVAL, FN, "cap smaller than N+1");
  std::memcpy(fence, p->fence.data(), sizeof(int) * n);
  return n;
}

extern "C" int stage_of(const lps_stage_plan* p, int il) {
  static const char* FN = "stage_of";
  if (!p) return fail(LPS_EINVAL, FN, "plan is NULL");
  if (il < 0 || il >= p->n_layers) return fail(LPS_EINVAL, FN, "layer out of range");
  const int N = static_cast<int>(p->fence.size()) - 1;
  for (int s = 0; s < N; ++s)
    if (il < p->fence[s + 1]) return s;
  return N - 1;
}

// ---------------------------------------------------------------------------
// model
// ---------------------------------------------------------------------------

namespace {

struct LayerDev {
  void* w_qkv = nullptr;  // packed RoPE pairs: rows (head h, i) and (h, i + hd/2) adjacent
  float* s_qkv = nullptr;
  void* w_o = nullptr;
  float* s_o = nullptr;
  void* w_gu = nullptr;   // packed (gate_i, up_i) row pairs
  float* s_gu = nullptr;
  void* w_d = nullptr;
  float* s_d = nullptr;
  float* attn_norm = nullptr;
  float* ffn_norm = nullptr;
  __nv_bfloat16* kc = nullptr;  // [B][nkv][max_ctx][hd]
  __nv_bfloat16* vc = nullptr;
  float* o_keep = nullptr;      // [B][nq*hd] with LPS_FLAG_KEEP_ATTN_OUT
  CUtensorMap tmap_k{}, tmap_v{};  // the caches as 2D TMA tensors (attention sub-tile boxes)
  // the weights in the row-major layout as 2D TMA tensors (64 x 128 boxes;
  // bf16 with the 128-byte swizzle, int8 unswizzled) for the prefill's GEMMs
  CUtensorMap tm_qkv{}, tm_o{}, tm_gu{}, tm_d{};
};

struct StageDev {
  int l0 = 0, l1 = 0;
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  std::vector<LayerDev> layers;
  float* h = nullptr;      // [B][d] this stage's residual stream
  float* q = nullptr;      // [B][nq*hd]
  float* o = nullptr;      // [B][nq*hd]
  float* a = nullptr;      // [B][ffn]
  float* part = nullptr;   // attention partials
  int* counter = nullptr;  // attention chunk counters [B][nkv]
  float2* rope = nullptr;  // [max_ctx][hd/2] (cos, sin)
  void* embed = nullptr;   // stage 0
  float* embed_s = nullptr;
  void* head = nullptr;    // last stage
  float* head_s = nullptr;
  float* out_norm = nullptr;
  GemvPlan plan_qkv{}, plan_o{}, plan_gu{}, plan_d{}, plan_head{};
  SkinnyPlan sk_qkv{}, sk_o{}, sk_gu{}, sk_d{}, sk_head{};  // batch > 1
  StageLayer* ltab = nullptr;          // persistent kernel: device table of this stage's layers
  unsigned long long* bar = nullptr;   // persistent kernel: grid-barrier counter
  uint64_t bar_count = 0;              // grid barriers completed by earlier launches
};

struct Boundary {
  float* slot[2] = {nullptr, nullptr};  // [B][d] f32
  cudaEvent_t ev_tx[2] = {nullptr, nullptr};
  cudaEvent_t ev_rx[2] = {nullptr, nullptr};
  uint64_t steps = 0;
};

// Prefill buffers of one stage, allocated at the first model_prefill call
// (NP = the chunk's token rows padded to 16; C <= kTcMaxTokens).
struct PrefillStage {
  float* h = nullptr;               // [C][E] the chunk's residual rows
  float* q = nullptr;               // [C][nq*hd]
  __nv_bfloat16* x = nullptr;       // [2][NP][E] planes of the normalised input (QKV, gate/up)
  __nv_bfloat16* xo = nullptr;      // [2][NP][nq*hd] planes of the attention output (o-proj)
  __nv_bfloat16* xd = nullptr;      // [2][NP][ffn] planes of the SwiGLU output (down)
  float* apart = nullptr;           // chunk-attention partials [C][nq][max_chunks][hd + 4]
  float* gpart = nullptr;           // GEMM partials [grid][2][NP][128]
  int* gcnt = nullptr;              // GEMM tile counters (zero between launches)
  int32_t* tok = nullptr;           // stage 0: the prompt's token ids [max_ctx]
  CUtensorMap map_x{}, map_xo{}, map_xd{};
};
struct PrefillState {
  bool ready = false;
  int C = 0, NP = 0, max_chunks = 0;
  TcGemmPlan plan{};
  std::vector<PrefillStage> st;
  std::vector<Boundary> bd;         // [N-1] boundary slots [C][E], ev_tx / ev_rx per chunk parity
  uint64_t chunks = 0;              // chunks enqueued (their parity picks the slot)
};

struct PendingSlot {
  float* logits_dev = nullptr;
  float* host = nullptr;  // pinned [B][V]
  int* status_host = nullptr;
  cudaEvent_t ev_done = nullptr;
  bool held = false;
  bool drained = false;
  uint64_t step = 0;
};

struct KTimer {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev;
  size_t used = 0;
  double total_ms = 0;
  uint64_t launches = 0;
};

}  // namespace

struct lps_model {
  lps_model_desc d{};
  int N = 0;
  std::vector<int> fence;
  int device = 0;
  int num_sms = 0;
  bool int8 = false;
  bool single = false;
  bool skinny = false;  // batch > 1: tensor-core skinny GEMMs on the tiled weight layout
  bool verify = false;  // LPS_FLAG_VERIFY: the batch rows are consecutive positions of one sequence
  bool persist = false; // batch 1: one persistent stage kernel per stage and step, all on one stream
  bool graph = false;   // LPS_FLAG_GRAPH: every step replays as one CUDA graph
  bool capturing = false;  // a step is being captured: no cross-step waits, no timers
  cudaGraphExec_t gexec = nullptr;
  std::vector<cudaEvent_t> gjoin;  // per stage: its stream's work so far, for the graph's fork and join
  cudaEvent_t gdone = nullptr;     // the graph launch, for the stage streams' later work
  uint64_t graph_instantiations = 0;
  StageKernelPlan skp{};
  lps_alloc_fn alloc = nullptr;
  lps_free_fn free_fn = nullptr;
  void* alloc_ctx = nullptr;
  std::vector<void*> dev_allocs;
  std::vector<void*> host_allocs;
  std::vector<StageDev> st;
  std::vector<Boundary> bd;
  cudaStream_t rb = nullptr;
  bool own_rb = false;
  bool overlap = true;            // off with LPS_FLAG_SERIAL_STEPS
  cudaEvent_t ev_step = nullptr;  // recorded by the last stage after each step
  int* status_dev = nullptr;
  int* status_host = nullptr;
  std::vector<int> filled;
  std::vector<PendingSlot> pend;
  float* eager_logits_dev = nullptr;
  float* eager_host = nullptr;
  uint64_t step_count = 0;
  lps_stats stats{};
  bool failed = false;
  bool alloc_failed = false;  // a device allocation failed (bind gives up; see dev_alloc)
  long long wait_limit = 0;  // device-side wait limit in cycles (0: the kernels' default)
  int attn_max_chunks = 0;
  KTimer timers[LPS_KERNEL_STAGE + 1];
  PrefillState pf;
  // launch trace: device records [cap][2] (zeroed), host metadata per record
  unsigned long long* trace_dev = nullptr;
  int trace_cap = 0, trace_n = 0;
  uint64_t trace_dropped = 0;
  std::vector<lps_trace_record> trace_meta;

  cudaStream_t stream(int s) const { return (single || persist) ? st[0].stream : st[s].stream; }
};

struct lps_pending {
  lps_model* m;
  int slot;
  uint64_t step;
};

namespace {

// After one allocation has failed, the allocations that follow return nullptr
// without asking the allocator again (a failed bind stops allocating at once).
void* dev_alloc(lps_model* m, size_t bytes) {
  if (m->alloc_failed) return nullptr;
  if (bytes == 0) bytes = 256;
  void* p = nullptr;
  if (m->alloc) {
    p = m->alloc(m->alloc_ctx, bytes);
  } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    p = nullptr;
  }
  if (p)
    m->dev_allocs.push_back(p);
  else
    m->alloc_failed = true;
  return p;
}

void dev_free(lps_model* m, void* p) {
  for (size_t i = 0; i < m->dev_allocs.size(); ++i)
    if (m->dev_allocs[i] == p) {
      m->dev_allocs.erase(m->dev_allocs.begin() + static_cast<long>(i));
      if (m->free_fn)
        m->free_fn(m->alloc_ctx, p);
      else
        cudaFree(p);
      return;
    }
}

void* host_alloc(lps_model* m, size_t bytes) {
  void* p = nullptr;
  if (cudaHostAlloc(&p, bytes ? bytes : 16, cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  m->host_allocs.push_back(p);
  return p;
}

void release(lps_model* m) {
  cudaSetDevice(m->device);
  for (auto& s : m->st)
    if (s.stream) cudaStreamSynchronize(s.stream);
  if (m->rb) cudaStreamSynchronize(m->rb);
  for (auto& b : m->bd)
    for (int i = 0; i < 2; ++i) {
      if (b.ev_tx[i]) cudaEventDestroy(b.ev_tx[i]);
      if (b.ev_rx[i]) cudaEventDestroy(b.ev_rx[i]);
    }
  for (auto& b : m->pf.bd)
    for (int i = 0; i < 2; ++i) {
      if (b.ev_tx[i]) cudaEventDestroy(b.ev_tx[i]);
      if (b.ev_rx[i]) cudaEventDestroy(b.ev_rx[i]);
    }
  for (auto& p : m->pend)
    if (p.ev_done) cudaEventDestroy(p.ev_done);
  if (m->ev_step) cudaEventDestroy(m->ev_step);
  for (cudaEvent_t e : m->gjoin)
    if (e) cudaEventDestroy(e);
  if (m->gdone) cudaEventDestroy(m->gdone);
  if (m->gexec) cudaGraphExecDestroy(m->gexec);
  for (auto& t : m->timers)
    for (auto& e : t.ev) {
      cudaEventDestroy(e.first);
      cudaEventDestroy(e.second);
    }
  for (void* p : m->dev_allocs) {
    if (m->free_fn)
      m->free_fn(m->alloc_ctx, p);
    else
      cudaFree(p);
  }
  for (void* p : m->host_allocs) cudaFreeHost(p);
  for (auto& s : m->st)
    if (s.own_stream && s.stream) cudaStreamDestroy(s.stream);
  if (m->own_rb && m->rb) cudaStreamDestroy(m->rb);
  cudaGetLastError();
}

// Double-buffered pinned staging for host -> device uploads on one stream.
struct Uploader {
  static constexpr size_t kCap = 64ull << 20;
  void* buf[2] = {nullptr, nullptr};
  cudaEvent_t ev[2] = {nullptr, nullptr};
  int cur = 0;
  size_t fill = 0;
  char* dst = nullptr;  // device address of buf[cur]'s first byte
  cudaStream_t s = nullptr;
  cudaError_t err = cudaSuccess;

  bool init() {
    for (int i = 0; i < 2; ++i) {
      if (cudaHostAlloc(&buf[i], kCap, cudaHostAllocDefault) != cudaSuccess) return false;
      if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) return false;
    }
    return true;
  }
  ~Uploader() {
    for (int i = 0; i < 2; ++i) {
      if (ev[i]) {
        cudaEventSynchronize(ev[i]);
        cudaEventDestroy(ev[i]);
      }
      if (buf[i]) cudaFreeHost(buf[i]);
    }
  }
  void flush() {
    if (fill && err == cudaSuccess) {
      err = cudaMemcpyAsync(dst, buf[cur], fill, cudaMemcpyHostToDevice, s);
      if (err == cudaSuccess) err = cudaEventRecord(ev[cur], s);
      cur ^= 1;
      if (err == cudaSuccess) err = cudaEventSynchronize(ev[cur]);
    }
    fill = 0;
    dst = nullptr;
  }
  // Copy `bytes` from host `src` to device `d`, through staging. Consecutive
  // puts are merged into one copy only when `same_alloc` says that d continues
  // the previous put inside the same device allocation (two allocations can be
  // adjacent in the address space, and one copy must not span both).
  void put(void* d, const void* src, size_t bytes, bool same_alloc = false) {
    const char* sp = static_cast<const char*>(src);
    char* dp = static_cast<char*>(d);
    if (!same_alloc) flush();
    while (bytes) {
      if (dst && (dst + fill != dp || fill == kCap)) flush();
      if (!dst) dst = dp;
      const size_t n = std::min(bytes, kCap - fill);
      std::memcpy(static_cast<char*>(buf[cur]) + fill, sp, n);
      fill += n;
      sp += n;
      dp += n;
      bytes -= n;
    }
  }
};

size_t elem_bytes(const lps_model* m) { return m->int8 ? 1 : 2; }

// Upload a packed [rows, K] matrix: device row r is host row row_ptr(r) (with
// scale row_scale(r) for int8). Batch 1 keeps it row-major; batch > 1 stores the
// tiled layout of the skinny GEMM (uploaded row-major into `temp`, then
// rearranged on the device).
template <class RowPtr, class RowScale>
bool place_matrix(lps_model* m, Uploader& up, int rows, int K, RowPtr row_ptr, RowScale row_scale, void** w_dev,
                  float** s_dev, const SkinnyPlan* sk, void* temp, std::string* why) {
  const size_t rb = static_cast<size_t>(K) * elem_bytes(m);
  const size_t bytes = m->skinny ? static_cast<size_t>(sk->rows_p) * sk->kp * elem_bytes(m) : rb * rows;
  *w_dev = dev_alloc(m, bytes);
  if (!*w_dev) {
    *why = "device allocation of " + std::to_string(bytes) + " bytes failed";
    return false;
  }
  char* dst = static_cast<char*>(m->skinny ? temp : *w_dev);
  for (int r = 0; r < rows; ++r) up.put(dst + rb * r, row_ptr(r), rb, r > 0);
  if (m->skinny) {
    up.flush();
    cudaError_t e = up.err;
    if (e == cudaSuccess) e = cudaMemsetAsync(*w_dev, 0, bytes, up.s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(up.s);
    if (e == cudaSuccess)
      e = launch_retile(temp, *w_dev, rows, K, *sk, static_cast<int>(elem_bytes(m)), up.s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(up.s);
    if (e != cudaSuccess) {
      *why = std::string("retiling: ") + cudaGetErrorString(e);
      return false;
    }
  }
  if (m->int8) {
    *s_dev = static_cast<float*>(dev_alloc(m, sizeof(float) * rows));
    if (!*s_dev) {
      *why = "device allocation of row scales failed";
      return false;
    }
    std::vector<float> sc(rows);
    for (int r = 0; r < rows; ++r) sc[r] = row_scale(r);
    up.put(*s_dev, sc.data(), sizeof(float) * rows);
    up.flush();
  }
  if (up.err != cudaSuccess) *why = std::string("host-to-device copy: ") + cudaGetErrorString(up.err);
  return up.err == cudaSuccess;
}

bool check_matrix(bool int8, const lps_matrix& x) { return x.w && (!int8 || x.scale); }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda
// link), looked up once per process (a function-local static: models bound on
// several threads at once initialise it once).
PFN_cuTensorMapEncodeTiled_v12000 lookup_tensor_map_encoder() {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  cudaGetLastError();
  return nullptr;
}
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = lookup_tensor_map_encoder();
  return fn;
}

// A cache [rows][hd] bf16 as a 2D tensor read in boxes of 64 elements x box_rows
// rows with the 128-byte swizzle; rows past the end read as zeros.
bool make_kv_map(CUtensorMap* map, void* base, int hd, unsigned long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(hd), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(hd) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace lps {
// A row-major [rows][cols] bf16 matrix as a 2D tensor read in boxes of 64
// columns x box_rows rows with the 128-byte swizzle; reads past either edge
// give zeros.
bool make_bf16_map(CUtensorMap* map, const void* base, unsigned long long cols, unsigned long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_i8_map(CUtensorMap* map, const void* base, unsigned long long cols, unsigned long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace lps

namespace {

// The trace record of the next launch (two zeroed 64-bit words), or nullptr;
// `step` is the decode step (or, for prefill launches, the chunk) it belongs to.
unsigned long long* trace_slot_at(lps_model* m, int kind, int stage, int layer, int64_t step) {
  if (!m->trace_dev) return nullptr;
  if (m->trace_n >= m->trace_cap) {
    ++m->trace_dropped;
    return nullptr;
  }
  lps_trace_record r{};
  r.kind = kind;
  r.stage = stage;
  r.layer = layer;
  r.step = static_cast<int32_t>(step);
  m->trace_meta.push_back(r);
  return m->trace_dev + 2 * static_cast<size_t>(m->trace_n++);
}

unsigned long long* trace_slot(lps_model* m, int kind, int stage, int layer) {
  return trace_slot_at(m, kind, stage, layer, static_cast<int64_t>(m->step_count));
}

// n consecutive trace records (the phases of one persistent launch), or
// nullptr (all n counted as dropped) when they do not all fit.
unsigned long long* trace_block(lps_model* m, int n) {
  if (!m->trace_dev) return nullptr;
  if (m->trace_n + n > m->trace_cap) {
    m->trace_dropped += n;
    return nullptr;
  }
  unsigned long long* p = m->trace_dev + 2 * static_cast<size_t>(m->trace_n);
  m->trace_n += n;
  return p;
}

int timer_begin(lps_model* m, int kind, cudaStream_t s, cudaEvent_t* stop) {
  *stop = nullptr;
  KTimer& t = m->timers[kind];
  if (!t.on || m->capturing) return 0;
  if (t.used == t.ev.size()) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return -1;
    t.ev.emplace_back(a, b);
  }
  cudaEventRecord(t.ev[t.used].first, s);
  *stop = t.ev[t.used].second;
  ++t.used;
  return 0;
}

void timer_end(lps_model* m, int kind, cudaStream_t s, cudaEvent_t stop) {
  if (stop) {
    cudaEventRecord(stop, s);
    ++m->timers[kind].launches;
  }
}

}  // namespace

extern "C" int model_bind(const lps_stage_plan* plan, const lps_model_desc* desc, const lps_model_weights* w,
                          const lps_runtime* rt, lps_model** out) {
  static const char* FN = "model_bind";
  if (!out) return fail(LPS_EINVAL, FN, "out is NULL");
  *out = nullptr;
  if (!plan || !desc || !w) return fail(LPS_EINVAL, FN, "plan, desc and weights are required");
  const lps_model_desc& d = *desc;
  if (d.n_layers != plan->n_layers) return fail(LPS_EINVAL, FN, "desc->n_layers differs from the plan's");
  if (d.weight_dtype != LPS_WEIGHT_BF16 && d.weight_dtype != LPS_WEIGHT_INT8_ROWSCALE)
    return fail(LPS_EINVAL, FN, "unsupported weight_dtype");
  if (d.kv_dtype != LPS_KV_BF16) return fail(LPS_EINVAL, FN, "unsupported kv_dtype");
  if (d.n_embd < 1 || d.n_q_heads < 1 || d.n_kv_heads < 1 || d.ffn < 1 || d.vocab < 1 || d.max_ctx < 1)
    return fail(LPS_EINVAL, FN, "shape fields must be positive");
  if (d.batch < 1 || d.batch > kMaxBatch) return fail(LPS_EINVAL, FN, "batch must be in 1..8");
  if ((d.flags & LPS_FLAG_GRAPH) && (d.flags & LPS_FLAG_PERSISTENT))
    return fail(LPS_EINVAL, FN, "LPS_FLAG_GRAPH replays the chained kernels; it does not combine with LPS_FLAG_PERSISTENT");
  if (d.n_q_heads % d.n_kv_heads) return fail(LPS_EINVAL, FN, "n_q_heads must be a multiple of n_kv_heads");
  if (!attn_supported(d.head_dim, d.n_q_heads / d.n_kv_heads))
    return fail(LPS_EINVAL, FN, "head_dim must be 64 or 128 and n_q_heads/n_kv_heads in {1,2,4,8}");
  if (d.n_embd % 4) return fail(LPS_EINVAL, FN, "n_embd must be a multiple of 4");
  if (!(d.rms_eps > 0.f) || !(d.rope_theta > 0.f)) return fail(LPS_EINVAL, FN, "rms_eps and rope_theta must be > 0");
  // the attention addresses a layer's cache rows with 32-bit TMA coordinates
  if (static_cast<long long>(d.batch) * d.n_kv_heads * d.max_ctx > 0x7fffffffll)
    return fail(LPS_EINVAL, FN, "batch * n_kv_heads * max_ctx must stay below 2^31 cache rows per layer");
  if (!w->layers || !w->out_norm || !w->embed.w || !w->lm_head.w) return fail(LPS_EINVAL, FN, "missing weights");
  const bool int8 = d.weight_dtype == LPS_WEIGHT_INT8_ROWSCALE;
  for (int l = 0; l < d.n_layers; ++l) {
    const lps_layer_weights& L = w->layers[l];
    if (!L.attn_norm || !L.ffn_norm || !check_matrix(int8, L.wq) || !check_matrix(int8, L.wk) ||
        !check_matrix(int8, L.wv) || !check_matrix(int8, L.wo) || !check_matrix(int8, L.w_gate) ||
        !check_matrix(int8, L.w_up) || !check_matrix(int8, L.w_down))
      return fail(LPS_EINVAL, FN, "layer " + std::to_string(l) + " has a missing tensor or scale");
  }
  if (!check_matrix(int8, w->embed) || !check_matrix(int8, w->lm_head))
    return fail(LPS_EINVAL, FN, "embed or lm_head is missing its row scales");
  if (rt && rt->alloc && !rt->free) return fail(LPS_EINVAL, FN, "rt->free is required with rt->alloc");
  // (every check above reads the arguments only; the ones below ask the device)
  const int qw = d.n_q_heads * d.head_dim;
  const int dev = rt ? rt->device : 0;
  int max_smem = 0;
  if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(LPS_ECUDA, FN, "cannot query device " + std::to_string(dev));
  }
  if (!gemv_supported(d.n_embd, 2, int8, max_smem) || !gemv_supported(qw, 1, int8, max_smem) ||
      !gemv_supported(d.ffn, 1, int8, max_smem))
    return fail(LPS_EINVAL, FN, "n_embd, n_q_heads*head_dim and ffn need whole 16-byte weight rows, and two "
                                "rows (row pairs) plus the fp32 input vector must fit in shared memory");
  if (d.batch > 1) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return fail(LPS_ECUDA, FN, "cannot query device " + std::to_string(dev));
    }
    const int rows_qkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
    if (!skinny_supported(rows_qkv, d.n_embd, int8, d.batch, sms, max_smem) ||
        !skinny_supported(d.n_embd, qw, int8, d.batch, sms, max_smem) ||
        !skinny_supported(2 * d.ffn, d.n_embd, int8, d.batch, sms, max_smem) ||
        !skinny_supported(d.n_embd, d.ffn, int8, d.batch, sms, max_smem) ||
        !skinny_supported(d.vocab, d.n_embd, int8, d.batch, sms, max_smem))
      return fail(LPS_EINVAL, FN, "batch > 1 needs every projection's columns in multiples of 16, rows even and "
                                  "at most 64 16-row units (1024 rows) per SM");
  }

  lps_model* m = new lps_model();
  m->d = d;
  m->int8 = int8;
  m->single = (d.flags & LPS_FLAG_SINGLE_STREAM) != 0;
  m->overlap = (d.flags & LPS_FLAG_SERIAL_STEPS) == 0;
  m->fence = plan->fence;
  m->N = static_cast<int>(plan->fence.size()) - 1;
  m->device = rt ? rt->device : 0;
  if (rt) {
    m->alloc = rt->alloc;
    m->free_fn = rt->free;
    m->alloc_ctx = rt->alloc_ctx;
  }

  auto bail = [&](int code, const std::string& why) {
    release(m);
    delete m;
    return fail(code, FN, why);
  };
  cudaError_t e = cudaSetDevice(m->device);
  if (e != cudaSuccess) return bail(LPS_ECUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(e));
  if (cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess)
    return bail(LPS_ECUDA, "cudaDeviceGetAttribute failed");
  m->skinny = d.batch > 1;

  const int N = m->N, B = d.batch, hd = d.head_dim, nq = d.n_q_heads, nkv = d.n_kv_heads, E = d.n_embd;
  const int half = hd / 2;
  m->st.resize(N);
  m->bd.resize(N > 1 ? N - 1 : 0);
  // streams
  for (int s = 0; s < N; ++s) {
    StageDev& S = m->st[s];
    S.l0 = m->fence[s];
    S.l1 = m->fence[s + 1];
    if (rt && rt->streams) {
      S.stream = static_cast<cudaStream_t>(rt->streams[s]);
    } else {
      if (cudaStreamCreateWithFlags(&S.stream, cudaStreamNonBlocking) != cudaSuccess)
        return bail(LPS_ECUDA, "cudaStreamCreate failed");
      S.own_stream = true;
    }
  }
  if (rt && rt->streams) {
    m->rb = static_cast<cudaStream_t>(rt->streams[N]);
  } else {
    if (cudaStreamCreateWithFlags(&m->rb, cudaStreamNonBlocking) != cudaSuccess)
      return bail(LPS_ECUDA, "cudaStreamCreate failed");
    m->own_rb = true;
  }

  // chunking of the attention partials, sized for the longest context (the
  // verify arm runs the causal chunk attention instead)
  m->verify = (d.flags & LPS_FLAG_VERIFY) != 0;
  m->attn_max_chunks = attn_max_chunks(hd, nkv, m->verify ? 1 : B, d.max_ctx, m->num_sms);
  // batch 1, on request: the persistent stage kernel where its shapes fit
  m->skp = stage_kernel_plan(E, nq, nkv, hd, d.ffn, d.vocab, int8, m->num_sms, max_smem);
  m->persist = B == 1 && !m->verify && !m->single && (d.flags & LPS_FLAG_PERSISTENT) && m->skp.ok;
  m->graph = (d.flags & LPS_FLAG_GRAPH) != 0;

  // rope table (cos, sin) of angle pos * theta^(-2i/hd), computed in double
  std::vector<float2> rope(static_cast<size_t>(d.max_ctx) * half);
  for (int p = 0; p < d.max_ctx; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang = static_cast<double>(p) * std::pow(static_cast<double>(d.rope_theta), -2.0 * i / hd);
      rope[static_cast<size_t>(p) * half + i] = make_float2(static_cast<float>(std::cos(ang)),
                                                            static_cast<float>(std::sin(ang)));
    }

  m->status_dev = static_cast<int*>(dev_alloc(m, 2 * sizeof(int)));
  m->status_host = static_cast<int*>(host_alloc(m, 2 * sizeof(int)));
  if (!m->status_dev || !m->status_host) return bail(LPS_ENOMEM, "status word allocation failed");
  if (cudaMemset(m->status_dev, 0, 2 * sizeof(int)) != cudaSuccess) return bail(LPS_ECUDA, "cudaMemset failed");

  const int seqs = m->verify ? 1 : B;  // sequences with a cache of their own
  const size_t kv_elems = static_cast<size_t>(seqs) * nkv * d.max_ctx * hd;
  std::string why;
  // batch > 1: a row-major staging buffer on the device for retiling (the largest matrix)
  void* temp = nullptr;
  if (m->skinny) {
    size_t biggest = 0;
    const size_t sizes[5] = {static_cast<size_t>((nq + 2 * nkv) * hd) * E, static_cast<size_t>(E) * qw,
                             static_cast<size_t>(2 * d.ffn) * E, static_cast<size_t>(E) * d.ffn,
                             static_cast<size_t>(d.vocab) * E};
    for (size_t z : sizes) biggest = z > biggest ? z : biggest;
    temp = dev_alloc(m, biggest * elem_bytes(m));
    if (!temp) return bail(LPS_ENOMEM, "retiling buffer allocation failed");
  }
  for (int s = 0; s < N; ++s) {
    StageDev& S = m->st[s];
    Uploader up;
    up.s = S.stream;
    if (!up.init()) return bail(LPS_ENOMEM, "pinned staging allocation failed");
    // scratch
    S.h = static_cast<float*>(dev_alloc(m, sizeof(float) * B * E));
    S.q = static_cast<float*>(dev_alloc(m, sizeof(float) * B * qw));
    S.o = static_cast<float*>(dev_alloc(m, sizeof(float) * B * qw));
    S.a = static_cast<float*>(dev_alloc(m, sizeof(float) * B * d.ffn));
    const size_t part_chunks = m->persist  ? static_cast<size_t>(m->skp.nch_max)
                               : m->verify ? static_cast<size_t>(chunk_attn_max_chunks(nkv, m->num_sms))
                                           : static_cast<size_t>(m->attn_max_chunks);
    S.part = static_cast<float*>(dev_alloc(m, sizeof(float) * B * nq * part_chunks * (hd + 4)));
    S.counter = static_cast<int*>(dev_alloc(m, sizeof(int) * B * nkv));
    S.rope = static_cast<float2*>(dev_alloc(m, sizeof(float2) * rope.size()));
    if (!S.h || !S.q || !S.o || !S.a || !S.part || !S.counter || !S.rope)
      return bail(LPS_ENOMEM, "stage " + std::to_string(s) + " scratch allocation failed");
    if (cudaMemsetAsync(S.counter, 0, sizeof(int) * B * nkv, S.stream) != cudaSuccess ||
        cudaMemsetAsync(S.h, 0, sizeof(float) * B * E, S.stream) != cudaSuccess)
      return bail(LPS_ECUDA, "cudaMemsetAsync failed");
    up.put(S.rope, rope.data(), sizeof(float2) * rope.size());

    // kernel plans (grid and ring sizing) of this stage's GEMVs
    const int rows_qkv = (nq + 2 * nkv) * hd;
    // When three or more stages overlap (own streams, steps not serialized),
    // the layer's smaller projections (QKV, o-proj, down) take half the SMs and
    // leave the rest to the other stages' kernels; the gate/up projection and
    // the LM head keep every SM. The GEMV's sums do not depend on its grid, so
    // the bits do not change. Measured on the 8B bf16 step (4 stages, context
    // 8192): 2.872 ms with every projection on all 152 SMs, 2.726 with these on
    // 76 (114: 2.752; 57: 2.776; gate/up on fewer SMs as well: slower); with 2
    // stages (8B int8) 2% slower, so not there. Graph steps replay one after
    // another (no other step's stages run beside them): full grids there.
    const int shared_sms = (N >= 3 && !m->single && m->overlap && !m->graph) ? m->num_sms / 2 : m->num_sms;
    S.plan_qkv = gemv_plan(rows_qkv, E, 2, int8, shared_sms, max_smem);
    S.plan_o = gemv_plan(E, qw, 1, int8, shared_sms, max_smem);
    S.plan_gu = gemv_plan(2 * d.ffn, E, 2, int8, m->num_sms, max_smem);
    S.plan_d = gemv_plan(E, d.ffn, 1, int8, shared_sms, max_smem);
    S.plan_head = gemv_plan(d.vocab, E, 1, int8, m->num_sms, max_smem);
    S.sk_qkv = skinny_plan(rows_qkv, E, int8, B, m->num_sms, max_smem);
    S.sk_o = skinny_plan(E, qw, int8, B, m->num_sms, max_smem);
    S.sk_gu = skinny_plan(2 * d.ffn, E, int8, B, m->num_sms, max_smem);
    S.sk_d = skinny_plan(E, d.ffn, int8, B, m->num_sms, max_smem);
    S.sk_head = skinny_plan(d.vocab, E, int8, B, m->num_sms, max_smem);

    // layers owned by this stage
    S.layers.resize(S.l1 - S.l0);
    const size_t rbE = static_cast<size_t>(E) * elem_bytes(m);
    for (int l = S.l0; l < S.l1; ++l) {
      LayerDev& D = S.layers[l - S.l0];
      const lps_layer_weights& L = w->layers[l];
      // W_qkv packed into RoPE pairs: packed unit u = (head hh, i) holds rows
      // (hh*hd + i, hh*hd + i + hd/2) of [W_q; W_k; W_v]
      auto qkv_src = [&](int r, const lps_matrix** mat) {
        const int u = r >> 1, hh = u / half, i = u % half;
        const int src = hh * hd + i + ((r & 1) ? half : 0);  // row of the concatenation
        if (src < qw) {
          *mat = &L.wq;
          return src;
        }
        if (src < qw + nkv * hd) {
          *mat = &L.wk;
          return src - qw;
        }
        *mat = &L.wv;
        return src - qw - nkv * hd;
      };
      if (!place_matrix(
              m, up, rows_qkv, E,
              [&](int r) {
                const lps_matrix* mat;
                const int row = qkv_src(r, &mat);
                return static_cast<const char*>(mat->w) + rbE * row;
              },
              [&](int r) {
                const lps_matrix* mat;
                const int row = qkv_src(r, &mat);
                return mat->scale[row];
              },
              &D.w_qkv, &D.s_qkv, &S.sk_qkv, temp, &why))
        return bail(LPS_ENOMEM, "W_qkv upload: " + why);
      const size_t rbQ = static_cast<size_t>(qw) * elem_bytes(m);
      if (!place_matrix(
              m, up, E, qw, [&](int r) { return static_cast<const char*>(L.wo.w) + rbQ * r; },
              [&](int r) { return L.wo.scale[r]; }, &D.w_o, &D.s_o, &S.sk_o, temp, &why))
        return bail(LPS_ENOMEM, "W_o upload: " + why);
      // gate/up packed as row pairs (gate_i, up_i)
      if (!place_matrix(
              m, up, 2 * d.ffn, E,
              [&](int r) { return static_cast<const char*>(((r & 1) ? L.w_up : L.w_gate).w) + rbE * (r >> 1); },
              [&](int r) { return ((r & 1) ? L.w_up : L.w_gate).scale[r >> 1]; }, &D.w_gu, &D.s_gu, &S.sk_gu, temp,
              &why))
        return bail(LPS_ENOMEM, "W_gate/W_up upload: " + why);
      const size_t rbF = static_cast<size_t>(d.ffn) * elem_bytes(m);
      if (!place_matrix(
              m, up, E, d.ffn, [&](int r) { return static_cast<const char*>(L.w_down.w) + rbF * r; },
              [&](int r) { return L.w_down.scale[r]; }, &D.w_d, &D.s_d, &S.sk_d, temp, &why))
        return bail(LPS_ENOMEM, "W_down upload: " + why);
      // the row-major weights as TMA tensors for the prefill's tensor-core GEMMs
      if (!m->skinny) {
        auto mk = int8 ? make_i8_map : make_bf16_map;
        if (!(mk(&D.tm_qkv, D.w_qkv, E, rows_qkv, 128) && mk(&D.tm_o, D.w_o, qw, E, 128) &&
              mk(&D.tm_gu, D.w_gu, E, 2 * d.ffn, 128) && mk(&D.tm_d, D.w_d, d.ffn, E, 128)))
          return bail(LPS_ECUDA, "cuTensorMapEncodeTiled failed for a weight matrix");
      }
      D.attn_norm = static_cast<float*>(dev_alloc(m, sizeof(float) * E));
      D.ffn_norm = static_cast<float*>(dev_alloc(m, sizeof(float) * E));
      D.kc = static_cast<__nv_bfloat16*>(dev_alloc(m, kv_elems * 2));
      D.vc = static_cast<__nv_bfloat16*>(dev_alloc(m, kv_elems * 2));
      if (!D.attn_norm || !D.ffn_norm || !D.kc || !D.vc) return bail(LPS_ENOMEM, "KV cache allocation failed");
      if (!make_kv_map(&D.tmap_k, D.kc, hd, static_cast<unsigned long long>(seqs) * nkv * d.max_ctx, attn_sub_tile(hd)) ||
          !make_kv_map(&D.tmap_v, D.vc, hd, static_cast<unsigned long long>(seqs) * nkv * d.max_ctx, attn_sub_tile(hd)))
        return bail(LPS_ECUDA, "cuTensorMapEncodeTiled failed for the KV cache");
      up.put(D.attn_norm, L.attn_norm, sizeof(float) * E);
      up.put(D.ffn_norm, L.ffn_norm, sizeof(float) * E);
      if (cudaMemsetAsync(D.kc, 0, kv_elems * 2, S.stream) != cudaSuccess ||
          cudaMemsetAsync(D.vc, 0, kv_elems * 2, S.stream) != cudaSuccess)
        return bail(LPS_ECUDA, "cudaMemsetAsync failed");
      if (d.flags & LPS_FLAG_KEEP_ATTN_OUT) {
        D.o_keep = static_cast<float*>(dev_alloc(m, sizeof(float) * B * qw));
        if (!D.o_keep) return bail(LPS_ENOMEM, "attention-output allocation failed");
      }
    }
    if (s == 0) {  // the embedding is gathered row by row, so it stays row-major
      const bool was = m->skinny;
      m->skinny = false;
      const bool ok = place_matrix(
          m, up, d.vocab, E, [&](int r) { return static_cast<const char*>(w->embed.w) + rbE * r; },
          [&](int r) { return w->embed.scale[r]; }, &S.embed, &S.embed_s, nullptr, nullptr, &why);
      m->skinny = was;
      if (!ok) return bail(LPS_ENOMEM, "embedding upload: " + why);
    }
    if (s == N - 1) {
      if (!place_matrix(
              m, up, d.vocab, E, [&](int r) { return static_cast<const char*>(w->lm_head.w) + rbE * r; },
              [&](int r) { return w->lm_head.scale[r]; }, &S.head, &S.head_s, &S.sk_head, temp, &why))
        return bail(LPS_ENOMEM, "LM head upload: " + why);
      S.out_norm = static_cast<float*>(dev_alloc(m, sizeof(float) * E));
      if (!S.out_norm) return bail(LPS_ENOMEM, "allocation failed");
      up.put(S.out_norm, w->out_norm, sizeof(float) * E);
    }
    if (m->persist) {
      // the persistent kernel's table of this stage's layers, and its barrier counter
      std::vector<StageLayer> tab(S.layers.size());
      for (size_t i = 0; i < S.layers.size(); ++i) {
        const LayerDev& D = S.layers[i];
        StageLayer& T = tab[i];
        // the stage kernel's K/V sub-tiles are shorter than the chained attention's
        const unsigned long long kv_rows = static_cast<unsigned long long>(seqs) * nkv * d.max_ctx;
        if (!make_kv_map(&T.tmap_k, D.kc, hd, kv_rows, stage_sub_tile(hd)) ||
            !make_kv_map(&T.tmap_v, D.vc, hd, kv_rows, stage_sub_tile(hd)))
          return bail(LPS_ECUDA, "cuTensorMapEncodeTiled failed for the KV cache");
        T.w_qkv = D.w_qkv;
        T.s_qkv = D.s_qkv;
        T.w_o = D.w_o;
        T.s_o = D.s_o;
        T.w_gu = D.w_gu;
        T.s_gu = D.s_gu;
        T.w_d = D.w_d;
        T.s_d = D.s_d;
        T.attn_norm = D.attn_norm;
        T.ffn_norm = D.ffn_norm;
        T.kc = D.kc;
        T.vc = D.vc;
        T.o_out = D.o_keep ? D.o_keep : S.o;
      }
      S.ltab = static_cast<StageLayer*>(dev_alloc(m, sizeof(StageLayer) * tab.size()));
      S.bar = static_cast<unsigned long long*>(dev_alloc(m, sizeof(unsigned long long)));
      if (!S.ltab || !S.bar) return bail(LPS_ENOMEM, "stage table allocation failed");
      up.put(S.ltab, tab.data(), sizeof(StageLayer) * tab.size());
      if (cudaMemsetAsync(S.bar, 0, sizeof(unsigned long long), S.stream) != cudaSuccess)
        return bail(LPS_ECUDA, "cudaMemsetAsync failed");
    }
    up.flush();
    if (up.err != cudaSuccess) return bail(LPS_ECUDA, std::string("upload: ") + cudaGetErrorString(up.err));
    // load barrier: one synchronize per stage (memra_engine::pp, sync_stages_after_load)
    e = cudaStreamSynchronize(S.stream);
    if (e != cudaSuccess) return bail(LPS_ECUDA, std::string("load barrier: ") + cudaGetErrorString(e));
  }

  if (temp) dev_free(m, temp);

  // boundaries: two persistent slots each, owned by the receiving stage
  for (int b = 0; b + 1 < N; ++b) {
    Boundary& Bd = m->bd[b];
    for (int i = 0; i < 2; ++i) {
      Bd.slot[i] = static_cast<float*>(dev_alloc(m, sizeof(float) * B * E));
      if (!Bd.slot[i]) return bail(LPS_ENOMEM, "boundary slot allocation failed");
      if (cudaMemset(Bd.slot[i], 0, sizeof(float) * B * E) != cudaSuccess ||
          cudaEventCreateWithFlags(&Bd.ev_tx[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&Bd.ev_rx[i], cudaEventDisableTiming) != cudaSuccess)
        return bail(LPS_ECUDA, "boundary setup failed");
    }
  }

  if (cudaEventCreateWithFlags(&m->ev_step, cudaEventDisableTiming) != cudaSuccess)
    return bail(LPS_ECUDA, "cudaEventCreate failed");
  if (m->graph) {
    m->gjoin.assign(N, nullptr);
    for (auto& e : m->gjoin)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
        return bail(LPS_ECUDA, "cudaEventCreate failed");
    if (cudaEventCreateWithFlags(&m->gdone, cudaEventDisableTiming) != cudaSuccess)
      return bail(LPS_ECUDA, "cudaEventCreate failed");
  }

  // logits: one eager buffer and the deferred-readback ring
  const size_t logits_bytes = sizeof(float) * B * static_cast<size_t>(d.vocab);
  m->eager_logits_dev = static_cast<float*>(dev_alloc(m, logits_bytes));
  m->eager_host = static_cast<float*>(host_alloc(m, logits_bytes));
  if (!m->eager_logits_dev || !m->eager_host) return bail(LPS_ENOMEM, "logits allocation failed");
  const int depth = d.pending_depth > 0 ? d.pending_depth : 4;
  m->pend.resize(depth);
  for (auto& p : m->pend) {
    p.logits_dev = static_cast<float*>(dev_alloc(m, logits_bytes));
    p.host = static_cast<float*>(host_alloc(m, logits_bytes));
    p.status_host = static_cast<int*>(host_alloc(m, 2 * sizeof(int)));
    if (!p.logits_dev || !p.host || !p.status_host) return bail(LPS_ENOMEM, "pending slot allocation failed");
    if (cudaEventCreateWithFlags(&p.ev_done, cudaEventDisableTiming) != cudaSuccess)
      return bail(LPS_ECUDA, "cudaEventCreate failed");
  }
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return bail(LPS_ECUDA, std::string("bind: ") + cudaGetErrorString(e));
  m->filled.assign(seqs, 0);
  m->stats.n_stages = N;
  m->stats.persistent = m->persist ? 1 : 0;
  for (int i = 0; i <= N && i < 17; ++i) m->stats.fence[i] = m->fence[i];
  *out = m;
  return LPS_OK;
}

extern "C" void model_destroy(lps_model* m) {
  if (!m) return;
  release(m);
  delete m;
}

// ---------------------------------------------------------------------------
// the step
// ---------------------------------------------------------------------------

namespace {

int check_step(lps_model* m, const int32_t* tokens, const int32_t* pos, bool tokens_on_host, const char* FN) {
  if (!m) return fail(LPS_EINVAL, FN, "model is NULL");
  if (m->failed) return fail(LPS_ECUDA, FN, "model is in a failed state after an earlier device error");
  if (!tokens || !pos) return fail(LPS_EINVAL, FN, "tokens and pos are required");
  for (int b = 0; b < m->d.batch; ++b) {
    if (tokens_on_host && (tokens[b] < 0 || tokens[b] >= m->d.vocab))
      return fail(LPS_EINVAL, FN, "token " + std::to_string(b) + " out of [0, vocab)");
    if (pos[b] < 0 || pos[b] >= m->d.max_ctx)
      return fail(LPS_EINVAL, FN, "pos " + std::to_string(b) + " out of [0, max_ctx)");
    if (m->verify) {
      // the rows are consecutive positions of the one sequence
      if (pos[b] != pos[0] + b) return fail(LPS_EINVAL, FN, "verify rows need pos[b] == pos[0] + b");
    } else if (pos[b] > m->filled[b]) {
      return fail(LPS_EINVAL, FN, "pos " + std::to_string(b) + " skips unwritten cache rows (pos > filled)");
    }
  }
  if (m->verify && pos[0] > m->filled[0])
    return fail(LPS_EINVAL, FN, "pos 0 skips unwritten cache rows (pos > filled)");
  return LPS_OK;
}

SkinnyParams skinny_params(const lps_model* m, const void* w, const float* wscale, int rows, int K,
                           const int32_t* pos) {
  SkinnyParams p{};
  p.w = w;
  p.wscale = wscale;
  p.rows = rows;
  p.K = K;
  p.batch = m->d.batch;
  p.eps = m->d.rms_eps;
  p.nq = m->d.n_q_heads;
  p.nkv = m->d.n_kv_heads;
  p.hd = m->d.head_dim;
  p.max_ctx = m->d.max_ctx;
  // verify rows all write the one sequence's cache (row pos[b] each)
  p.kv_stride = m->verify ? 0 : static_cast<size_t>(m->d.n_kv_heads) * m->d.max_ctx * m->d.head_dim;
  for (int b = 0; b < m->d.batch; ++b) p.pos[b] = pos[b];
  p.status = m->status_dev;
  p.wait_limit = m->wait_limit;
  return p;
}

// One step on the persistent stage kernel: one launch per stage, in stage
// order on one stream, chained by programmatic dependent launch; stage s
// writes its last layer's output into boundary slot [s][step parity] and
// stage s + 1 reads it from there.
int enqueue_persistent(lps_model* m, const int32_t* tok_host, const int32_t* tok_dev, const int32_t* pos,
                       float* logits_dev, const char* FN) {
  const lps_model_desc& d = m->d;
  const int N = m->N;
  const int par = static_cast<int>(m->step_count & 1);
  const cudaStream_t cs = m->st[0].stream;
  int nch = 1, chunk = 1;
  stage_attn_chunks(m->skp, d.head_dim, d.n_kv_heads, pos[0], &nch, &chunk);
  static const int32_t kPhaseKind[] = {LPS_KERNEL_QKV, LPS_KERNEL_ATTN, LPS_KERNEL_MERGE,
                                       LPS_KERNEL_OPROJ, LPS_KERNEL_GATEUP, LPS_KERNEL_DOWN};
  for (int s = 0; s < N; ++s) {
    StageDev& S = m->st[s];
    StageParams p{};
    p.layers = S.ltab;
    p.n_layers = S.l1 - S.l0;
    p.d = d.n_embd;
    p.nq = d.n_q_heads;
    p.nkv = d.n_kv_heads;
    p.hd = d.head_dim;
    p.ffn = d.ffn;
    p.vocab = d.vocab;
    p.max_ctx = d.max_ctx;
    p.eps = d.rms_eps;
    p.scale = 1.0f / std::sqrt(static_cast<float>(d.head_dim));
    p.pos = pos[0];
    p.tok = tok_host ? tok_host[0] : 0;
    p.tok_dev = tok_dev;
    if (s == 0) {
      p.embed = S.embed;
      p.embed_s = S.embed_s;
    }
    if (s == N - 1) {
      p.head = S.head;
      p.head_s = S.head_s;
      p.out_norm = S.out_norm;
      p.logits = logits_dev;
    }
    p.h_in = s > 0 ? m->bd[s - 1].slot[par] : nullptr;
    p.h = S.h;
    p.h_out = s + 1 < N ? m->bd[s].slot[par] : S.h;
    p.q = S.q;
    p.a = S.a;
    p.part = S.part;
    p.rope = S.rope;
    p.nch = nch;
    p.chunk = chunk;
    p.bar = S.bar;
    p.bar_base = S.bar_count * static_cast<unsigned long long>(m->skp.grid);
    p.wait_limit = m->wait_limit;
    p.status = m->status_dev;
    const int nb = stage_barriers(p);
    const int nph = nb + 1;
    p.trace = trace_block(m, nph);
    if (p.trace) {
      // metadata of the phases, in the kernel's order
      auto rec = [&](int kind, int layer) {
        lps_trace_record r{};
        r.kind = kind;
        r.stage = s;
        r.layer = layer;
        r.step = static_cast<int32_t>(m->step_count);
        m->trace_meta.push_back(r);
      };
      if (s == 0) rec(LPS_KERNEL_EMBED, -1);
      for (int l = S.l0; l < S.l1; ++l)
        for (int k : kPhaseKind) rec(k, l);
      if (s == N - 1) rec(LPS_KERNEL_HEAD, -1);
    }
    cudaEvent_t stop;
    if (timer_begin(m, LPS_KERNEL_STAGE, cs, &stop)) return fail(LPS_ECUDA, FN, "timer event");
    const cudaError_t e = launch_stage(p, m->int8, m->skp, cs, true);
    if (e != cudaSuccess) {
      m->failed = true;
      return cuda_fail(FN, "stage kernel launch", e);
    }
    timer_end(m, LPS_KERNEL_STAGE, cs, stop);
    S.bar_count += static_cast<uint64_t>(nb);
    if (s + 1 < N) {
      ++m->bd[s].steps;
      ++m->stats.boundary_crossings;
    }
    ++m->stats.stage_walks;
  }
  m->filled[0] = pos[0] + 1;
  ++m->step_count;
  ++m->stats.steps;
  m->stats.kernel_launches += static_cast<uint64_t>(N);
  return LPS_OK;
}

// Enqueue one step's kernels on the stage streams; the last stage writes logits_dev [B][V].
int enqueue_step_streams(lps_model* m, const int32_t* tok_host, const int32_t* tok_dev, const int32_t* pos,
                         float* logits_dev, const char* FN) {
  const lps_model_desc& d = m->d;
  const int N = m->N, B = d.batch, E = d.n_embd, hd = d.head_dim, nq = d.n_q_heads, nkv = d.n_kv_heads;
  const int qw = nq * hd, half = hd / 2;
  const int par = static_cast<int>(m->step_count & 1);
  int max_pos = 0;
  for (int b = 0; b < B; ++b) max_pos = pos[b] > max_pos ? pos[b] : max_pos;
  const int chunk = attn_chunk(hd, nkv, B, max_pos, m->num_sms);
  // Programmatic dependent launch chains the kernels inside a stage walk; the
  // first kernel of each walk follows cross-stream event waits and is launched
  // with full stream ordering instead.
  bool pdl = false;
  uint64_t launches = 0;
  cudaEvent_t stop;
  int s_trace = 0, layer_trace = -1;  // stage and layer of the next launch, for the trace

#define LAUNCH(kind, stream, params, call)                                  \
  do {                                                                      \
    (params).trace = trace_slot(m, kind, s_trace, layer_trace);             \
    if (timer_begin(m, kind, stream, &stop)) return fail(LPS_ECUDA, FN, "timer event"); \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) {                                                \
      m->failed = true;                                                     \
      return cuda_fail(FN, "kernel launch", e_);                            \
    }                                                                       \
    timer_end(m, kind, stream, stop);                                       \
    ++launches;                                                             \
    pdl = true;                                                             \
  } while (0)

  for (int s = 0; s < N; ++s) {
    StageDev& S = m->st[s];
    const cudaStream_t cs = m->stream(s);
    pdl = false;
    s_trace = s;
    layer_trace = -1;
    if (!m->single) {
      if (s > 0) CK(cudaStreamWaitEvent(cs, m->bd[s - 1].ev_tx[par], 0), "wait ev_tx");
      // (a captured step replays only after the previous graph launch has
      // completed, so it waits for no earlier step)
      if (s + 1 < N && !m->capturing) CK(cudaStreamWaitEvent(cs, m->bd[s].ev_rx[par], 0), "wait ev_rx");
      if (s == 0 && N > 1 && !m->overlap && !m->capturing)
        CK(cudaStreamWaitEvent(cs, m->ev_step, 0), "wait previous step");
    } else if (s > 0) {
      CK(cudaMemcpyAsync(S.h, m->bd[s - 1].slot[par], sizeof(float) * B * E, cudaMemcpyDeviceToDevice, cs),
         "boundary copy");
    }
    const float* h_first = (s == 0 || m->single) ? S.h : m->bd[s - 1].slot[par];
    if (s == 0) {
      EmbedParams ep{};
      ep.table = S.embed;
      ep.scale = S.embed_s;
      ep.tok_dev = tok_dev;
      for (int b = 0; b < B; ++b) ep.tok[b] = tok_host ? tok_host[b] : 0;
      ep.d = E;
      ep.vocab = d.vocab;
      ep.batch = B;
      ep.h = S.h;
      ep.status = m->status_dev;
      LAUNCH(LPS_KERNEL_EMBED, cs, ep, launch_embed(ep, m->int8, cs, pdl));
    }
    for (int l = S.l0; l < S.l1; ++l) {
      const LayerDev& L = S.layers[l - S.l0];
      const bool first = (l == S.l0), last = (l == S.l1 - 1);
      layer_trace = l;
      const float* hin = first ? h_first : S.h;
      float* o_buf = L.o_keep ? L.o_keep : S.o;
      // RMSNorm -> QKV -> RoPE -> q and KV-cache row pos (per sequence)
      if (m->skinny) {
        SkinnyParams p = skinny_params(m, L.w_qkv, L.s_qkv, (nq + 2 * nkv) * hd, E, pos);
        p.x = hin;
        p.gain = L.attn_norm;
        p.out = S.q;
        p.out_stride = qw;
        p.kc = L.kc;
        p.vc = L.vc;
        p.rope = S.rope;
        LAUNCH(LPS_KERNEL_QKV, cs, p, launch_skinny(p, kEpiQkv, true, m->int8, S.sk_qkv, cs, pdl));
      }
      for (int b = 0; b < (m->skinny ? 0 : B); ++b) {
        GemvParams p{};
        p.w = L.w_qkv;
        p.wscale = L.s_qkv;
        p.rows = (nq + 2 * nkv) * hd;
        p.K = E;
        p.unit_rows = 2;
        p.units = p.rows / 2;
        p.units_per_buf = S.plan_qkv.units_per_buf;
        p.nbuf = S.plan_qkv.nbuf;
        p.h = hin + static_cast<size_t>(b) * E;
        p.gain = L.attn_norm;
        p.eps = d.rms_eps;
        p.out = S.q + static_cast<size_t>(b) * qw;
        const size_t seq = m->verify ? 0 : static_cast<size_t>(b);
        p.kc = L.kc + seq * nkv * d.max_ctx * hd;
        p.vc = L.vc + seq * nkv * d.max_ctx * hd;
        p.rope = S.rope + static_cast<size_t>(pos[b]) * half;
        p.nq = nq;
        p.nkv = nkv;
        p.hd = hd;
        p.max_ctx = d.max_ctx;
        p.pos = pos[b];
        p.status = m->status_dev;
        p.wait_limit = m->wait_limit;
        LAUNCH(LPS_KERNEL_QKV, cs, p, launch_gemv(p, kEpiQkv, true, m->int8, S.plan_qkv, cs, pdl));
      }
      // split-K attention over [0, pos]
      {
        AttnParams ap{};
        ap.tmap_k = L.tmap_k;
        ap.tmap_v = L.tmap_v;
        ap.q = S.q;
        ap.kc = L.kc;
        ap.vc = L.vc;
        ap.out = o_buf;
        ap.part = S.part;
        ap.counter = S.counter;
        ap.nq = nq;
        ap.nkv = nkv;
        ap.hd = hd;
        ap.max_ctx = d.max_ctx;
        ap.max_chunks = m->attn_max_chunks;
        ap.chunk = chunk;
        for (int b = 0; b < B; ++b) ap.pos[b] = pos[b];
        ap.scale = 1.0f / std::sqrt(static_cast<float>(hd));
        ap.early_dependents = m->skinny ? 0 : 1;  // the GEMV o-proj follows
        ap.status = m->status_dev;
        ap.wait_limit = m->wait_limit;
        if (!m->verify) {
          LAUNCH(LPS_KERNEL_ATTN, cs, ap, launch_attention(ap, B, max_pos, cs, pdl));
        } else {
          // verify rows share the one cache: row b (position pos[0] + b) attends
          // [0, pos[0] + b], rows pos[0].. written by this step's QKV: one
          // causal chunk-attention launch (and its merge) for all rows
          ChunkAttnParams cp{};
          cp.tmap_k = L.tmap_k;
          cp.tmap_v = L.tmap_v;
          cp.q = S.q;
          cp.part = S.part;
          cp.out = o_buf;
          cp.nq = nq;
          cp.nkv = nkv;
          cp.hd = hd;
          cp.max_ctx = d.max_ctx;
          cp.max_chunks = chunk_attn_max_chunks(nkv, m->num_sms);
          chunk_attn_split(hd, nq, nkv, B, pos[0], m->num_sms, &cp.nchunks, &cp.chunk, &cp.qblock);
          cp.seq = 0;
          cp.pos0 = pos[0];
          cp.ntok = B;
          cp.NP = B;
          cp.scale = ap.scale;
          cp.wait_limit = m->wait_limit;
          cp.status = m->status_dev;
          cp.trace_merge = nullptr;
          LAUNCH(LPS_KERNEL_ATTN, cs, cp, launch_chunk_attn(cp, cs, pdl));
          ++launches;  // the merge
        }
      }
      // o-proj + residual (the first layer of a later stage reads the boundary slot)
      if (m->skinny) {
        SkinnyParams p = skinny_params(m, L.w_o, L.s_o, E, qw, pos);
        p.x = o_buf;
        p.h_in = hin;
        p.h_out = S.h;
        p.out_stride = E;
        LAUNCH(LPS_KERNEL_OPROJ, cs, p, launch_skinny(p, kEpiResidual, false, m->int8, S.sk_o, cs, pdl));
      }
      for (int b = 0; b < (m->skinny ? 0 : B); ++b) {
        GemvParams p{};
        p.w = L.w_o;
        p.wscale = L.s_o;
        p.rows = E;
        p.K = qw;
        p.unit_rows = 1;
        p.units = E;
        p.units_per_buf = S.plan_o.units_per_buf;
        p.nbuf = S.plan_o.nbuf;
        p.x = o_buf + static_cast<size_t>(b) * qw;
        p.h_in = hin + static_cast<size_t>(b) * E;
        p.h_out = S.h + static_cast<size_t>(b) * E;
        p.status = m->status_dev;
        p.wait_limit = m->wait_limit;
        LAUNCH(LPS_KERNEL_OPROJ, cs, p, launch_gemv(p, kEpiResidual, false, m->int8, S.plan_o, cs, pdl));
      }
      if (first && s > 0 && !m->single && !m->capturing)
        CK(cudaEventRecord(m->bd[s - 1].ev_rx[par], cs), "record ev_rx");
      // RMSNorm -> gate/up -> SwiGLU
      if (m->skinny) {
        SkinnyParams p = skinny_params(m, L.w_gu, L.s_gu, 2 * d.ffn, E, pos);
        p.x = S.h;
        p.gain = L.ffn_norm;
        p.out = S.a;
        p.out_stride = d.ffn;
        LAUNCH(LPS_KERNEL_GATEUP, cs, p, launch_skinny(p, kEpiSwiglu, true, m->int8, S.sk_gu, cs, pdl));
      }
      for (int b = 0; b < (m->skinny ? 0 : B); ++b) {
        GemvParams p{};
        p.w = L.w_gu;
        p.wscale = L.s_gu;
        p.rows = 2 * d.ffn;
        p.K = E;
        p.unit_rows = 2;
        p.units = d.ffn;
        p.units_per_buf = S.plan_gu.units_per_buf;
        p.nbuf = S.plan_gu.nbuf;
        p.h = S.h + static_cast<size_t>(b) * E;
        p.gain = L.ffn_norm;
        p.eps = d.rms_eps;
        p.out = S.a + static_cast<size_t>(b) * d.ffn;
        p.status = m->status_dev;
        p.wait_limit = m->wait_limit;
        LAUNCH(LPS_KERNEL_GATEUP, cs, p, launch_gemv(p, kEpiSwiglu, true, m->int8, S.plan_gu, cs, pdl));
      }
      // down + residual (the last layer of an earlier stage writes the boundary slot)
      float* h_out = (last && s + 1 < N && !m->single) ? m->bd[s].slot[par] : S.h;
      if (m->skinny) {
        SkinnyParams p = skinny_params(m, L.w_d, L.s_d, E, d.ffn, pos);
        p.x = S.a;
        p.h_in = S.h;
        p.h_out = h_out;
        p.out_stride = E;
        LAUNCH(LPS_KERNEL_DOWN, cs, p, launch_skinny(p, kEpiResidual, false, m->int8, S.sk_d, cs, pdl));
      }
      for (int b = 0; b < (m->skinny ? 0 : B); ++b) {
        GemvParams p{};
        p.w = L.w_d;
        p.wscale = L.s_d;
        p.rows = E;
        p.K = d.ffn;
        p.unit_rows = 1;
        p.units = E;
        p.units_per_buf = S.plan_d.units_per_buf;
        p.nbuf = S.plan_d.nbuf;
        p.x = S.a + static_cast<size_t>(b) * d.ffn;
        p.h_in = S.h + static_cast<size_t>(b) * E;
        p.h_out = h_out + static_cast<size_t>(b) * E;
        p.status = m->status_dev;
        p.wait_limit = m->wait_limit;
        LAUNCH(LPS_KERNEL_DOWN, cs, p, launch_gemv(p, kEpiResidual, false, m->int8, S.plan_d, cs, pdl));
      }
    }
    if (s + 1 < N) {
      if (m->single)
        CK(cudaMemcpyAsync(m->bd[s].slot[par], S.h, sizeof(float) * B * E, cudaMemcpyDeviceToDevice, cs),
           "boundary copy");
      else
        CK(cudaEventRecord(m->bd[s].ev_tx[par], cs), "record ev_tx");
      ++m->bd[s].steps;
      ++m->stats.boundary_crossings;
    }
    ++m->stats.stage_walks;
  }
  // the last stage: final RMSNorm -> LM head
  {
    StageDev& S = m->st[N - 1];
    const cudaStream_t cs = m->stream(N - 1);
    s_trace = N - 1;
    layer_trace = -1;
    if (m->skinny) {
      SkinnyParams p = skinny_params(m, S.head, S.head_s, d.vocab, E, pos);
      p.x = S.h;
      p.gain = S.out_norm;
      p.out = logits_dev;
      p.out_stride = d.vocab;
      LAUNCH(LPS_KERNEL_HEAD, cs, p, launch_skinny(p, kEpiStore, true, m->int8, S.sk_head, cs, pdl));
    }
    for (int b = 0; b < (m->skinny ? 0 : B); ++b) {
      GemvParams p{};
      p.w = S.head;
      p.wscale = S.head_s;
      p.rows = d.vocab;
      p.K = E;
      p.unit_rows = 1;
      p.units = d.vocab;
      p.units_per_buf = S.plan_head.units_per_buf;
      p.nbuf = S.plan_head.nbuf;
      p.h = S.h + static_cast<size_t>(b) * E;
      p.gain = S.out_norm;
      p.eps = d.rms_eps;
      p.out = logits_dev + static_cast<size_t>(b) * d.vocab;
      p.status = m->status_dev;
      p.wait_limit = m->wait_limit;
      LAUNCH(LPS_KERNEL_HEAD, cs, p, launch_gemv(p, kEpiStore, true, m->int8, S.plan_head, cs, pdl));
    }
    if (N > 1 && !m->single && !m->overlap && !m->capturing) CK(cudaEventRecord(m->ev_step, cs), "record step event");
  }
#undef LAUNCH
  if (m->verify)
    m->filled[0] = pos[B - 1] + 1;
  else
    for (int b = 0; b < B; ++b) m->filled[b] = pos[b] + 1;
  ++m->step_count;
  ++m->stats.steps;
  m->stats.kernel_launches += launches;
  return LPS_OK;
}

// ---- prefill -------------------------------------------------------------------

// The prefill buffers, boundary slots and tensor maps, at the first prefill call.
int prefill_init(lps_model* m, const char* FN) {
  PrefillState& P = m->pf;
  if (P.ready) return LPS_OK;
  // an earlier call that failed part way: release what it made (once the
  // clears it enqueued have run) before starting again
  if (!P.st.empty() || !P.bd.empty())
    for (int s = 0; s < m->N; ++s) CK(cudaStreamSynchronize(m->stream(s)), "stage stream");
  for (auto& b : P.bd)
    for (int i = 0; i < 2; ++i) {
      if (b.ev_tx[i]) cudaEventDestroy(b.ev_tx[i]);
      if (b.ev_rx[i]) cudaEventDestroy(b.ev_rx[i]);
      dev_free(m, b.slot[i]);
    }
  P.bd.clear();
  for (auto& F : P.st)
    for (void* p : {static_cast<void*>(F.h), static_cast<void*>(F.q), static_cast<void*>(F.x),
                    static_cast<void*>(F.xo), static_cast<void*>(F.xd), static_cast<void*>(F.apart),
                    static_cast<void*>(F.gpart), static_cast<void*>(F.gcnt), static_cast<void*>(F.tok)})
      dev_free(m, p);
  P.st.clear();
  const lps_model_desc& d = m->d;
  const int N = m->N, E = d.n_embd, nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim, ffn = d.ffn;
  const int qw = nq * hd, rows_qkv = (nq + 2 * nkv) * hd;
  int max_smem = 0;
  CK(cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, m->device), "device attribute");
  const int C = kTcMaxTokens, NP = kTcMaxTokens;
  P.plan = tc_gemm_plan(NP, m->int8, m->num_sms, max_smem);
  if (!P.plan.ok) return fail(LPS_EINVAL, FN, "the prefill GEMM does not fit this device");
  P.C = C;
  P.NP = NP;
  P.max_chunks = chunk_attn_max_chunks(nkv, m->num_sms);
  const int max_tiles = tc_gemm_tiles(std::max(std::max(rows_qkv, E), 2 * ffn));
  P.st.assign(N, PrefillStage{});
  for (int s = 0; s < N; ++s) {
    StageDev& S = m->st[s];
    PrefillStage& F = P.st[s];
    F.h = static_cast<float*>(dev_alloc(m, sizeof(float) * C * E));
    F.q = static_cast<float*>(dev_alloc(m, sizeof(float) * C * qw));
    F.x = static_cast<__nv_bfloat16*>(dev_alloc(m, sizeof(__nv_bfloat16) * 2 * NP * E));
    F.xo = static_cast<__nv_bfloat16*>(dev_alloc(m, sizeof(__nv_bfloat16) * 2 * NP * qw));
    F.xd = static_cast<__nv_bfloat16*>(dev_alloc(m, sizeof(__nv_bfloat16) * 2 * NP * ffn));
    F.apart = static_cast<float*>(dev_alloc(m, sizeof(float) * C * nq * static_cast<size_t>(P.max_chunks) * (hd + 4)));
    F.gpart = static_cast<float*>(dev_alloc(m, sizeof(float) * P.plan.grid * 2 * NP * 128));
    F.gcnt = static_cast<int*>(dev_alloc(m, sizeof(int) * max_tiles));
    if (s == 0) F.tok = static_cast<int32_t*>(dev_alloc(m, sizeof(int32_t) * d.max_ctx));
    if (!F.h || !F.q || !F.x || !F.xo || !F.xd || !F.apart || !F.gpart || !F.gcnt || (s == 0 && !F.tok))
      return fail(LPS_ENOMEM, FN, "prefill buffer allocation failed");
    CK(cudaMemsetAsync(F.gcnt, 0, sizeof(int) * max_tiles, S.stream), "cudaMemsetAsync");
    CK(cudaMemsetAsync(F.x, 0, sizeof(__nv_bfloat16) * 2 * NP * E, S.stream), "cudaMemsetAsync");
    CK(cudaMemsetAsync(F.xo, 0, sizeof(__nv_bfloat16) * 2 * NP * qw, S.stream), "cudaMemsetAsync");
    CK(cudaMemsetAsync(F.xd, 0, sizeof(__nv_bfloat16) * 2 * NP * ffn, S.stream), "cudaMemsetAsync");
    bool ok = make_bf16_map(&F.map_x, F.x, E, 2 * NP, NP) && make_bf16_map(&F.map_xo, F.xo, qw, 2 * NP, NP) &&
              make_bf16_map(&F.map_xd, F.xd, ffn, 2 * NP, NP);
    if (!ok) return fail(LPS_ECUDA, FN, "cuTensorMapEncodeTiled failed for a prefill operand");
  }
  P.bd.assign(N > 1 ? N - 1 : 0, Boundary{});
  for (auto& b : P.bd)
    for (int i = 0; i < 2; ++i) {
      b.slot[i] = static_cast<float*>(dev_alloc(m, sizeof(float) * C * E));
      if (!b.slot[i]) return fail(LPS_ENOMEM, FN, "prefill boundary allocation failed");
      CK(cudaEventCreateWithFlags(&b.ev_tx[i], cudaEventDisableTiming), "cudaEventCreate");
      CK(cudaEventCreateWithFlags(&b.ev_rx[i], cudaEventDisableTiming), "cudaEventCreate");
    }
  P.ready = true;
  return LPS_OK;
}

// Enqueue one chunk: ntok prompt tokens (ids at tok[tok_off..]) of sequence
// seq at positions pos0 .. pos0 + ntok - 1, through every stage. Stage s waits
// for stage s - 1's slot of this chunk's parity (ev_tx) and for stage s + 1 to
// have read its own slot of the same parity two chunks ago (ev_rx), so stage s
// works on chunk c while stage s + 1 works on chunk c - 1. With want_logits
// the last stage writes the logits of the chunk's last token.
int enqueue_prefill_chunk(lps_model* m, int seq, int pos0, int ntok, int tok_off, bool want_logits, const char* FN) {
  PrefillState& P = m->pf;
  const lps_model_desc& d = m->d;
  const int N = m->N, E = d.n_embd, nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim, ffn = d.ffn;
  const int qw = nq * hd, NP = P.NP;
  const int par = static_cast<int>(P.chunks & 1);
  const int64_t chunk_no = static_cast<int64_t>(P.chunks);
  auto tr = [&](int kind, int stage, int layer) { return trace_slot_at(m, kind, stage, layer, chunk_no); };
  int nchunks = 1, achunk = 1, qblock = 16;
  chunk_attn_split(hd, nq, nkv, ntok, pos0, m->num_sms, &nchunks, &achunk, &qblock);
  uint64_t launches = 0;
  bool pdl = false;
#define PF_LAUNCH(call)                                 \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) {                            \
      m->failed = true;                                 \
      return cuda_fail(FN, "prefill kernel launch", e_); \
    }                                                   \
    ++launches;                                         \
    pdl = true;                                         \
  } while (0)
  for (int s = 0; s < N; ++s) {
    StageDev& S = m->st[s];
    PrefillStage& F = P.st[s];
    const cudaStream_t cs = m->stream(s);
    pdl = false;
    if (s > 0) CK(cudaStreamWaitEvent(cs, P.bd[s - 1].ev_tx[par], 0), "wait prefill ev_tx");
    if (s + 1 < N) CK(cudaStreamWaitEvent(cs, P.bd[s].ev_rx[par], 0), "wait prefill ev_rx");
    if (s == 0) {
      EmbedParams ep{};
      ep.table = S.embed;
      ep.scale = S.embed_s;
      ep.tok_dev = F.tok + tok_off;
      ep.d = E;
      ep.vocab = d.vocab;
      ep.batch = ntok;
      ep.h = F.h;
      ep.status = m->status_dev;
      ep.trace = tr(LPS_KERNEL_EMBED, s, -1);
      PF_LAUNCH(launch_embed(ep, m->int8, cs, pdl));
    } else {
      CK(cudaMemcpyAsync(F.h, P.bd[s - 1].slot[par], sizeof(float) * ntok * E, cudaMemcpyDeviceToDevice, cs),
         "prefill boundary copy");
      CK(cudaEventRecord(P.bd[s - 1].ev_rx[par], cs), "record prefill ev_rx");
      pdl = false;
    }
    TcGemmParams g{};
    g.NP = NP;
    g.ntok = ntok;
    g.pos0 = pos0;
    g.seq = seq;
    g.nq = nq;
    g.nkv = nkv;
    g.hd = hd;
    g.max_ctx = d.max_ctx;
    g.rope = S.rope;
    g.h = F.h;
    g.ldh = E;
    g.part = F.gpart;
    g.counter = F.gcnt;
    g.wait_limit = m->wait_limit;
    g.status = m->status_dev;
    g.int8 = m->int8 ? 1 : 0;
    PrepParams pp{};
    pp.src = F.h;
    pp.lds = E;
    pp.K = E;
    pp.NP = NP;
    pp.ntok = ntok;
    pp.eps = d.rms_eps;
    pp.x = F.x;
    for (int l = S.l0; l < S.l1; ++l) {
      const int i = l - S.l0;
      const LayerDev& L = S.layers[i];
      // RMSNorm -> QKV -> RoPE -> q and the chunk's cache rows
      pp.gain = L.attn_norm;
      pp.trace = tr(LPS_KERNEL_PF_SPLIT, s, l);
      PF_LAUNCH(launch_prep(pp, cs, pdl));
      TcGemmParams gq = g;
      gq.tmap_w = L.tm_qkv;
      gq.wscale = L.s_qkv;
      gq.tmap_x = F.map_x;
      gq.R = (nq + 2 * nkv) * hd;
      gq.K = E;
      gq.epi = kEpiQkv;
      gq.q = F.q;
      gq.kc = L.kc;
      gq.vc = L.vc;
      gq.trace = tr(LPS_KERNEL_PF_GEMM, s, l);
      PF_LAUNCH(launch_tc_gemm(gq, P.plan, cs, pdl));
      // causal attention of the chunk, merged into the o-proj input planes
      ChunkAttnParams ap{};
      ap.tmap_k = L.tmap_k;
      ap.tmap_v = L.tmap_v;
      ap.q = F.q;
      ap.part = F.apart;
      ap.xo = F.xo;
      ap.nq = nq;
      ap.nkv = nkv;
      ap.hd = hd;
      ap.max_ctx = d.max_ctx;
      ap.max_chunks = P.max_chunks;
      ap.chunk = achunk;
      ap.nchunks = nchunks;
      ap.qblock = qblock;
      ap.seq = seq;
      ap.pos0 = pos0;
      ap.ntok = ntok;
      ap.NP = NP;
      ap.scale = 1.0f / std::sqrt(static_cast<float>(hd));
      ap.wait_limit = m->wait_limit;
      ap.status = m->status_dev;
      ap.trace = tr(LPS_KERNEL_PF_ATTN, s, l);
      ap.trace_merge = tr(LPS_KERNEL_PF_MERGE, s, l);
      PF_LAUNCH(launch_chunk_attn(ap, cs, pdl));
      ++launches;  // the merge
      // o-proj + residual
      TcGemmParams go = g;
      go.tmap_w = L.tm_o;
      go.wscale = L.s_o;
      go.tmap_x = F.map_xo;
      go.R = E;
      go.K = qw;
      go.epi = kEpiResidual;
      go.trace = tr(LPS_KERNEL_PF_GEMM, s, l);
      PF_LAUNCH(launch_tc_gemm(go, P.plan, cs, pdl));
      // RMSNorm -> gate/up -> SwiGLU (into the down projection's input planes)
      pp.gain = L.ffn_norm;
      pp.trace = tr(LPS_KERNEL_PF_SPLIT, s, l);
      PF_LAUNCH(launch_prep(pp, cs, pdl));
      TcGemmParams gg = g;
      gg.tmap_w = L.tm_gu;
      gg.wscale = L.s_gu;
      gg.tmap_x = F.map_x;
      gg.R = 2 * ffn;
      gg.K = E;
      gg.epi = kEpiSwiglu;
      gg.xo = F.xd;
      gg.ldx = ffn;
      gg.trace = tr(LPS_KERNEL_PF_GEMM, s, l);
      PF_LAUNCH(launch_tc_gemm(gg, P.plan, cs, pdl));
      // down + residual
      TcGemmParams gd = g;
      gd.tmap_w = L.tm_d;
      gd.wscale = L.s_d;
      gd.tmap_x = F.map_xd;
      gd.R = E;
      gd.K = ffn;
      gd.epi = kEpiResidual;
      gd.trace = tr(LPS_KERNEL_PF_GEMM, s, l);
      PF_LAUNCH(launch_tc_gemm(gd, P.plan, cs, pdl));
    }
    if (s + 1 < N) {
      CK(cudaMemcpyAsync(P.bd[s].slot[par], F.h, sizeof(float) * ntok * E, cudaMemcpyDeviceToDevice, cs),
         "prefill boundary copy");
      CK(cudaEventRecord(P.bd[s].ev_tx[par], cs), "record prefill ev_tx");
      ++m->stats.boundary_crossings;
    }
    ++m->stats.stage_walks;
  }
  if (want_logits) {
    // the last token's final RMSNorm -> LM head, on the batch-1 GEMV
    StageDev& S = m->st[N - 1];
    const cudaStream_t cs = m->stream(N - 1);
    GemvParams p{};
    p.w = S.head;
    p.wscale = S.head_s;
    p.rows = d.vocab;
    p.K = E;
    p.unit_rows = 1;
    p.units = d.vocab;
    p.units_per_buf = S.plan_head.units_per_buf;
    p.nbuf = S.plan_head.nbuf;
    p.h = P.st[N - 1].h + static_cast<size_t>(ntok - 1) * E;
    p.gain = S.out_norm;
    p.eps = d.rms_eps;
    p.out = m->eager_logits_dev;
    p.status = m->status_dev;
    p.wait_limit = m->wait_limit;
    p.trace = tr(LPS_KERNEL_HEAD, N - 1, -1);
    PF_LAUNCH(launch_gemv(p, kEpiStore, true, m->int8, S.plan_head, cs, pdl));
  }
#undef PF_LAUNCH
  ++P.chunks;
  m->stats.kernel_launches += launches;
  return LPS_OK;
}

// One step as a CUDA graph (the pages' decode captures the whole pass into one
// graph: ninfer pipeline-stages.md, "StageLink"). The step is captured from
// stage 0's stream -- the other stages' streams join through the ev_tx events
// and are joined back at the end -- and the captured graph updates the
// instantiated one in place (cudaGraphExecUpdate: the positions, the logits
// buffer and the attention's grid change from step to step; a fresh
// instantiation when the topology changes), which is then launched on stage
// 0's stream. Every replay runs after the previous one, so the captured step
// drops the waits on earlier steps' events: graph steps do not overlap one
// another, only the stages inside a step do.
int enqueue_step_graph(lps_model* m, const int32_t* tok_host, const int32_t* tok_dev, const int32_t* pos,
                       float* logits_dev, const char* FN) {
  const int N = m->N;
  const cudaStream_t s0 = m->stream(0);
  // the replay follows everything already enqueued on any stage's stream
  for (int s = 1; s < N; ++s) {
    if (m->stream(s) == s0) continue;
    CK(cudaEventRecord(m->gjoin[s], m->stream(s)), "record join event");
    CK(cudaStreamWaitEvent(s0, m->gjoin[s], 0), "wait join event");
  }
  CK(cudaStreamBeginCapture(s0, cudaStreamCaptureModeRelaxed), "cudaStreamBeginCapture");
  m->capturing = true;
  int rc = enqueue_step_streams(m, tok_host, tok_dev, pos, logits_dev, FN);
  cudaError_t e = cudaSuccess;
  for (int s = 1; s < N && rc == LPS_OK && e == cudaSuccess; ++s) {
    if (m->stream(s) == s0) continue;
    e = cudaEventRecord(m->gjoin[s], m->stream(s));
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s0, m->gjoin[s], 0);
  }
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(s0, &g);
  m->capturing = false;
  if (rc != LPS_OK || e != cudaSuccess || ec != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    m->failed = true;
    if (rc != LPS_OK) return rc;
    return cuda_fail(FN, "step capture", e != cudaSuccess ? e : ec);
  }
  if (m->gexec) {
    cudaGraphExecUpdateResultInfo info;
    if (cudaGraphExecUpdate(m->gexec, g, &info) != cudaSuccess) {
      cudaGetLastError();
      cudaGraphExecDestroy(m->gexec);
      m->gexec = nullptr;
    }
  }
  if (!m->gexec) {
    e = cudaGraphInstantiate(&m->gexec, g, 0);
    if (e != cudaSuccess) {
      cudaGraphDestroy(g);
      m->gexec = nullptr;
      m->failed = true;
      return cuda_fail(FN, "graph instantiation", e);
    }
    ++m->graph_instantiations;
  }
  cudaGraphDestroy(g);
  e = cudaGraphLaunch(m->gexec, s0);
  if (e != cudaSuccess) {
    m->failed = true;
    return cuda_fail(FN, "graph launch", e);
  }
  // whatever follows on a stage's stream (readback, events, prefill) follows the replay
  CK(cudaEventRecord(m->gdone, s0), "record graph event");
  for (int s = 1; s < N; ++s)
    if (m->stream(s) != s0) CK(cudaStreamWaitEvent(m->stream(s), m->gdone, 0), "wait graph event");
  return LPS_OK;
}

// Enqueue one step; the last stage writes logits_dev [B][V].
int enqueue_step(lps_model* m, const int32_t* tok_host, const int32_t* tok_dev, const int32_t* pos, float* logits_dev,
                 const char* FN) {
  if (m->persist) return enqueue_persistent(m, tok_host, tok_dev, pos, logits_dev, FN);
  if (m->graph) return enqueue_step_graph(m, tok_host, tok_dev, pos, logits_dev, FN);
  return enqueue_step_streams(m, tok_host, tok_dev, pos, logits_dev, FN);
}

int read_status(lps_model* m, const int* status, const char* FN) {
  if (status[0] != 0 || status[1] != 0) {
    m->failed = true;
    return fail(LPS_ECUDA, FN, lps::describe_status(status[0], status[1]));
  }
  return LPS_OK;
}

}  // namespace

extern "C" int decode_step(lps_model* m, const int32_t* tokens, const int32_t* pos, float* logits) {
  static const char* FN = "decode_step";
  int rc = check_step(m, tokens, pos, true, FN);
  if (rc) return rc;
  if (!logits) return fail(LPS_EINVAL, FN, "logits is NULL");
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  rc = enqueue_step(m, tokens, nullptr, pos, m->eager_logits_dev, FN);
  if (rc) return rc;
  const cudaStream_t last = m->stream(m->N - 1);
  const size_t bytes = sizeof(float) * m->d.batch * static_cast<size_t>(m->d.vocab);
  CK(cudaMemcpyAsync(m->eager_host, m->eager_logits_dev, bytes, cudaMemcpyDeviceToHost, last), "logits copy");
  CK(cudaMemcpyAsync(m->status_host, m->status_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost, last), "status copy");
  // the last stage's wait chain orders every earlier stage, so this drains the step
  cudaError_t e = cudaStreamSynchronize(last);
  if (e != cudaSuccess) {
    m->failed = true;
    return cuda_fail(FN, "step", e);
  }
  rc = read_status(m, m->status_host, FN);
  if (rc) return rc;
  std::memcpy(logits, m->eager_host, bytes);
  return LPS_OK;
}

extern "C" int decode_step_deferred(lps_model* m, const int32_t* tokens, const int32_t* pos, lps_pending** out) {
  static const char* FN = "decode_step_deferred";
  if (!out) return fail(LPS_EINVAL, FN, "out is NULL");
  *out = nullptr;
  int rc = check_step(m, tokens, pos, true, FN);
  if (rc) return rc;
  int slot = -1;
  for (size_t i = 0; i < m->pend.size(); ++i)
    if (!m->pend[i].held) {
      slot = static_cast<int>(i);
      break;
    }
  if (slot < 0) return fail(LPS_EBUSY, FN, "every deferred-readback slot is held; wait and free a pending handle");
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  PendingSlot& P = m->pend[slot];
  rc = enqueue_step(m, tokens, nullptr, pos, P.logits_dev, FN);
  if (rc) return rc;
  CK(cudaEventRecord(P.ev_done, m->stream(m->N - 1)), "record completion event");
  P.held = true;
  P.drained = false;
  P.step = m->step_count - 1;
  ++m->stats.deferred_steps;
  *out = new lps_pending{m, slot, P.step};
  return LPS_OK;
}

extern "C" int pending_wait(lps_pending* p, float* logits, int timeout_ms) {
  static const char* FN = "pending_wait";
  if (!p || !logits) return fail(LPS_EINVAL, FN, "pending and logits are required");
  lps_model* m = p->m;
  PendingSlot& P = m->pend[p->slot];
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  const size_t bytes = sizeof(float) * m->d.batch * static_cast<size_t>(m->d.vocab);
  if (!P.drained) {
    if (timeout_ms >= 0) {
      const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
      for (;;) {
        const cudaError_t q = cudaEventQuery(P.ev_done);
        if (q == cudaSuccess) break;
        if (q != cudaErrorNotReady) {
          m->failed = true;
          return cuda_fail(FN, "completion event", q);
        }
        if (std::chrono::steady_clock::now() >= deadline)
          return fail(LPS_ETIMEDOUT, FN, "the step has not completed yet");
        std::this_thread::sleep_for(std::chrono::microseconds(20));
      }
    }
    // the dedicated readback stream waits the completion event, copies, syncs
    CK(cudaStreamWaitEvent(m->rb, P.ev_done, 0), "readback wait");
    CK(cudaMemcpyAsync(P.host, P.logits_dev, bytes, cudaMemcpyDeviceToHost, m->rb), "logits copy");
    CK(cudaMemcpyAsync(P.status_host, m->status_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost, m->rb), "status copy");
    const cudaError_t e = cudaStreamSynchronize(m->rb);
    if (e != cudaSuccess) {
      m->failed = true;
      return cuda_fail(FN, "readback", e);
    }
    P.drained = true;
    ++m->stats.pending_drains;
  }
  const int rc = read_status(m, P.status_host, FN);
  if (rc) return rc;
  std::memcpy(logits, P.host, bytes);
  return LPS_OK;
}

extern "C" void pending_free(lps_pending* p) {
  if (!p) return;
  p->m->pend[p->slot].held = false;
  delete p;
}

extern "C" int decode_step_device(lps_model* m, const int32_t* tokens, const int32_t* pos, float* logits) {
  static const char* FN = "decode_step_device";
  int rc = check_step(m, tokens, pos, false, FN);
  if (rc) return rc;
  if (!logits) return fail(LPS_EINVAL, FN, "logits is NULL");
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  return enqueue_step(m, nullptr, tokens, pos, logits, FN);
}

extern "C" int model_prefill(lps_model* m, int b, const int32_t* tokens, int n, int pos0, int chunk,
                             float* logits) {
  static const char* FN = "model_prefill";
  if (!m) return fail(LPS_EINVAL, FN, "model is NULL");
  if (m->failed) return fail(LPS_ECUDA, FN, "model is in a failed state after an earlier device error");
  const lps_model_desc& d = m->d;
  if (m->skinny || m->verify)
    return fail(LPS_EINVAL, FN, "prefill needs the row-major weight layout of a batch-1 model (not batch > 1, "
                                "not verify rows)");
  if (!tokens || n < 1) return fail(LPS_EINVAL, FN, "tokens is NULL or n < 1");
  if (b < 0 || b >= static_cast<int>(m->filled.size())) return fail(LPS_EINVAL, FN, "sequence out of range");
  if (pos0 < 0 || pos0 > m->filled[b]) return fail(LPS_EINVAL, FN, "pos0 skips unwritten cache rows (pos0 > filled)");
  if (static_cast<long long>(pos0) + n > d.max_ctx) return fail(LPS_EINVAL, FN, "pos0 + n exceeds max_ctx");
  if (chunk < 0 || chunk > kTcMaxTokens) return fail(LPS_EINVAL, FN, "chunk out of [0, 128]");
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= d.vocab)
      return fail(LPS_EINVAL, FN, "token " + std::to_string(i) + " out of [0, vocab)");
  const int C = chunk ? chunk : kTcMaxTokens;
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  int rc = prefill_init(m, FN);
  if (rc) return rc;
  const cudaStream_t first = m->stream(0), last = m->stream(m->N - 1);
  CK(cudaMemcpyAsync(m->pf.st[0].tok, tokens, sizeof(int32_t) * n, cudaMemcpyHostToDevice, first), "token upload");
  for (int c0 = 0; c0 < n; c0 += C) {
    const int ntok = n - c0 < C ? n - c0 : C;
    rc = enqueue_prefill_chunk(m, b, pos0 + c0, ntok, c0, logits && c0 + ntok == n, FN);
    if (rc) return rc;
  }
  if (pos0 + n > m->filled[b]) m->filled[b] = pos0 + n;
  const size_t bytes = sizeof(float) * static_cast<size_t>(d.vocab);
  if (logits) CK(cudaMemcpyAsync(m->eager_host, m->eager_logits_dev, bytes, cudaMemcpyDeviceToHost, last), "logits copy");
  CK(cudaMemcpyAsync(m->status_host, m->status_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost, last), "status copy");
  // every stage's last chunk is ordered before the last stage's, so this drains the prefill
  cudaError_t e = cudaStreamSynchronize(last);
  if (e != cudaSuccess) {
    m->failed = true;
    return cuda_fail(FN, "prefill", e);
  }
  rc = read_status(m, m->status_host, FN);
  if (rc) return rc;
  if (logits) std::memcpy(logits, m->eager_host, bytes);
  return LPS_OK;
}

extern "C" int model_synchronize(lps_model* m) {
  static const char* FN = "model_synchronize";
  if (!m) return fail(LPS_EINVAL, FN, "model is NULL");
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  for (int s = 0; s < m->N; ++s) {
    const cudaError_t e = cudaStreamSynchronize(m->st[s].stream);
    if (e != cudaSuccess) {
      m->failed = true;
      return cuda_fail(FN, "stage stream", e);
    }
  }
  CK(cudaStreamSynchronize(m->rb), "readback stream");
  CK(cudaMemcpy(m->status_host, m->status_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost), "status copy");
  return read_status(m, m->status_host, FN);
}

extern "C" int model_stream(const lps_model* m, int s, void** stream) {
  static const char* FN = "model_stream";
  if (!m || !stream || s < 0 || s > m->N) return fail(LPS_EINVAL, FN, "bad argument");
  *stream = s == m->N ? m->rb : m->stream(s);
  return LPS_OK;
}

// ---------------------------------------------------------------------------
// errors, counters, test hooks
// ---------------------------------------------------------------------------

extern "C" const char* last_error_string(void) { return g_err.c_str(); }

extern "C" int model_stats(const lps_model* m, lps_stats* out) {
  if (!m || !out) return fail(LPS_EINVAL, "model_stats", "NULL argument");
  *out = m->stats;
  return LPS_OK;
}

namespace {
int kv_locate(const lps_model* m, int layer, int b, size_t bytes, const LayerDev** L, cudaStream_t* stream,
              const char* FN) {
  if (!m || layer < 0 || layer >= m->d.n_layers || b < 0 || b >= (m->verify ? 1 : m->d.batch))
    return fail(LPS_EINVAL, FN, "bad model, layer or sequence");
  const size_t want = 4ull * m->d.n_kv_heads * m->d.max_ctx * m->d.head_dim;
  if (bytes != want) return fail(LPS_EINVAL, FN, "bytes must be 4 * nkv * max_ctx * hd");
  int s = 0;
  while (layer >= m->fence[s + 1]) ++s;
  *L = &m->st[s].layers[layer - m->fence[s]];
  *stream = m->stream(s);
  return LPS_OK;
}
}  // namespace

extern "C" int model_kv_export(const lps_model* m, int layer, int b, void* host, size_t bytes) {
  static const char* FN = "model_kv_export";
  const LayerDev* L;
  cudaStream_t s;
  int rc = kv_locate(m, layer, b, bytes, &L, &s, FN);
  if (rc) return rc;
  if (!host) return fail(LPS_EINVAL, FN, "host is NULL");
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  const size_t half = bytes / 2, off = static_cast<size_t>(b) * m->d.n_kv_heads * m->d.max_ctx * m->d.head_dim;
  CK(cudaStreamSynchronize(s), "stage stream");
  CK(cudaMemcpy(host, L->kc + off, half, cudaMemcpyDeviceToHost), "K copy");
  CK(cudaMemcpy(static_cast<char*>(host) + half, L->vc + off, half, cudaMemcpyDeviceToHost), "V copy");
  return LPS_OK;
}

extern "C" int model_kv_import(lps_model* m, int layer, int b, const void* host, size_t bytes, int filled) {
  static const char* FN = "model_kv_import";
  const LayerDev* L;
  cudaStream_t s;
  int rc = kv_locate(m, layer, b, bytes, &L, &s, FN);
  if (rc) return rc;
  if (!host || filled < 0 || filled > m->d.max_ctx) return fail(LPS_EINVAL, FN, "bad host buffer or filled");
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  const size_t half = bytes / 2, off = static_cast<size_t>(b) * m->d.n_kv_heads * m->d.max_ctx * m->d.head_dim;
  CK(cudaStreamSynchronize(s), "stage stream");
  CK(cudaMemcpy(L->kc + off, host, half, cudaMemcpyHostToDevice), "K copy");
  CK(cudaMemcpy(L->vc + off, static_cast<const char*>(host) + half, half, cudaMemcpyHostToDevice), "V copy");
  m->filled[b] = filled;
  return LPS_OK;
}

extern "C" int model_attn_out(const lps_model* m, int layer, int b, float* host) {
  static const char* FN = "model_attn_out";
  if (!m || !host || layer < 0 || layer >= m->d.n_layers || b < 0 || b >= m->d.batch)
    return fail(LPS_EINVAL, FN, "bad argument");
  if (!(m->d.flags & LPS_FLAG_KEEP_ATTN_OUT)) return fail(LPS_EINVAL, FN, "bind with LPS_FLAG_KEEP_ATTN_OUT");
  int s = 0;
  while (layer >= m->fence[s + 1]) ++s;
  const LayerDev& L = m->st[s].layers[layer - m->fence[s]];
  const size_t qw = static_cast<size_t>(m->d.n_q_heads) * m->d.head_dim;
  CK(cudaSetDevice(m->device), "cudaSetDevice");
  CK(cudaStreamSynchronize(m->stream(s)), "stage stream");
  CK(cudaMemcpy(host, L.o_keep + b * qw, qw * sizeof(float), cudaMemcpyDeviceToHost), "copy");
  return LPS_OK;
}

extern "C" int model_set_wait_limit(lps_model* m, long long cycles) {
  static const char* FN = "model_set_wait_limit";
  if (!m || cycles < 0) return fail(LPS_EINVAL, FN, "model and cycles >= 0 are required");
  const int rc = model_synchronize(m);
  if (rc) return rc;
  m->wait_limit = cycles;
  return LPS_OK;
}

extern "C" int model_set_serial_steps(lps_model* m, int serial) {
  if (!m) return fail(LPS_EINVAL, "model_set_serial_steps", "model is NULL");
  const int rc = model_synchronize(m);
  if (rc) return rc;
  m->overlap = serial == 0;
  return LPS_OK;
}

extern "C" int model_trace_enable(lps_model* m, int capacity) {
  static const char* FN = "model_trace_enable";
  if (!m || capacity < 1) return fail(LPS_EINVAL, FN, "model and capacity >= 1 are required");
  int rc = model_trace_disable(m);
  if (rc) return rc;
  const size_t bytes = 16 * static_cast<size_t>(capacity);
  m->alloc_failed = false;
  m->trace_dev = static_cast<unsigned long long*>(dev_alloc(m, bytes));
  if (!m->trace_dev) return fail(LPS_ENOMEM, FN, "trace buffer allocation failed");
  CK(cudaMemset(m->trace_dev, 0, bytes), "cudaMemset");
  m->trace_cap = capacity;
  m->trace_n = 0;
  m->trace_dropped = 0;
  m->trace_meta.clear();
  return LPS_OK;
}

extern "C" int model_trace_read(lps_model* m, lps_trace_record* out, int max_records, int* n_records,
                                uint64_t* dropped) {
  static const char* FN = "model_trace_read";
  if (!m || !n_records || (max_records > 0 && !out)) return fail(LPS_EINVAL, FN, "bad argument");
  if (!m->trace_dev) return fail(LPS_EINVAL, FN, "tracing is not enabled");
  int rc = model_synchronize(m);
  if (rc) return rc;
  const int n = m->trace_n < max_records ? m->trace_n : (max_records > 0 ? max_records : 0);
  std::vector<unsigned long long> words(2 * static_cast<size_t>(m->trace_n));
  if (m->trace_n)
    CK(cudaMemcpy(words.data(), m->trace_dev, 16 * static_cast<size_t>(m->trace_n), cudaMemcpyDeviceToHost),
       "cudaMemcpy");
  for (int i = 0; i < n; ++i) {
    out[i] = m->trace_meta[i];
    out[i].start_ns = words[2 * i] ? ~words[2 * i] : 0;
    out[i].end_ns = words[2 * i + 1];
  }
  *n_records = n;
  if (dropped) *dropped = m->trace_dropped;
  CK(cudaMemset(m->trace_dev, 0, 16 * static_cast<size_t>(m->trace_cap)), "cudaMemset");
  m->trace_n = 0;
  m->trace_dropped = 0;
  m->trace_meta.clear();
  return LPS_OK;
}

extern "C" int model_trace_disable(lps_model* m) {
  if (!m) return fail(LPS_EINVAL, "model_trace_disable", "model is NULL");
  if (!m->trace_dev) return LPS_OK;
  int rc = model_synchronize(m);
  if (rc) return rc;
  dev_free(m, m->trace_dev);
  m->trace_dev = nullptr;
  m->trace_cap = m->trace_n = 0;
  m->trace_meta.clear();
  return LPS_OK;
}

extern "C" int model_time_kernel(lps_model* m, int kind, int enable) {
  if (!m || kind < 0 || kind > LPS_KERNEL_STAGE) return fail(LPS_EINVAL, "model_time_kernel", "bad argument");
  KTimer& t = m->timers[kind];
  t.on = enable != 0;
  t.used = 0;
  t.total_ms = 0;
  t.launches = 0;
  return LPS_OK;
}

extern "C" int model_kernel_time(lps_model* m, int kind, double* total_ms, uint64_t* launches) {
  static const char* FN = "model_kernel_time";
  if (!m || kind < 0 || kind > LPS_KERNEL_STAGE || !total_ms || !launches) return fail(LPS_EINVAL, FN, "bad argument");
  int rc = model_synchronize(m);
  if (rc) return rc;
  KTimer& t = m->timers[kind];
  for (size_t i = 0; i < t.used; ++i) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, t.ev[i].first, t.ev[i].second), "cudaEventElapsedTime");
    t.total_ms += ms;
  }
  t.used = 0;
  *total_ms = t.total_ms;
  *launches = t.launches;
  return LPS_OK;
}
