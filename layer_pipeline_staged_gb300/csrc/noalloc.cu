// attention_decode_noalloc: the split-K decode attention for callers that may
// not allocate device memory.
//
// Who needs it: code whose device memory is fixed before it starts work and
// that must not allocate afterwards -- e.g. a serving loop with a hard latency
// budget (cudaMalloc can synchronize the device and stall every stream), or a
// host program whose GPU memory is handed out once by its own pool and where a
// later allocation may simply fail. The regular decode path keeps its
// attention scratch inside the model (allocated at bind time); this entry
// point needs no model at all, so its scratch -- the per-chunk partial
// results and the chunk counters -- lives in one file-scope device array
// instead.
//
// The array (kScratchBytes) is part of the library's device image: every GPU
// that loads the library holds it until the process exits. Its device address
// is looked up once per device, on the first call made with that device
// current. All calls share the array and it keeps the last call's contents;
// the counters that must start at zero are cleared at the start of every call
// (on the caller's stream). Two calls whose work overlaps on the GPU -- on
// different streams, or on different host threads -- race on the array and
// give wrong results; order them on one stream.
//
// The array's first 256 bytes hold a status (two ints) that the kernel sets
// when one of its bounded waits gives up, in which case that call's output is
// invalid. The status is sticky across calls: attention_decode_noalloc_status
// reads it (after synchronizing the caller's stream) and clears it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <string>

#include "kernels.h"
#include "lps.h"

namespace lps {
int attn_chunk(int hd, int nkv, int batch, int max_pos, int num_sms);
int attn_sub_tile(int hd);
bool attn_supported(int hd, int group);
}  // namespace lps

namespace {

constexpr size_t kScratchBytes = LPS_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[lps::kMaxDevices] = {};
int g_num_sms[lps::kMaxDevices] = {};

thread_local std::string g_err;

int fail(int code, const std::string& why) {
  g_err = "attention_decode_noalloc: " + why;
  return code;
}

// Scratch layout: the status (two ints) in a 256-byte block, the chunk
// counters [B][nkv] (rounded up to 256 bytes), then the partials
// [B][nq][nchunks][hd + 4] floats.
constexpr size_t kStatusBytes = 256;

// The array's device address on device `dev` (which must be current).
cudaError_t scratch_on(int dev, void** addr, int* num_sms) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    g_num_sms[dev] = sms;
  }
  *addr = g_scratch_addr[dev];
  *num_sms = g_num_sms[dev];
  return cudaSuccess;
}

// The driver's tensor-map encoder, looked up once per process (a function-local
// static, so concurrent first calls initialise it once).
PFN_cuTensorMapEncodeTiled_v12000 lookup_encoder() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool encode_cache(CUtensorMap* map, const void* base, int hd, unsigned long long rows, int box_rows) {
  static const PFN_cuTensorMapEncodeTiled_v12000 enc = lookup_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(hd), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(hd) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" const char* attention_decode_noalloc_error(void) { return g_err.c_str(); }

namespace {
// Scratch of one call: the status block and the counters (each rounded up to 256 bytes), then the partials.
void scratch_need(int batch, int n_q_heads, int n_kv_heads, int head_dim, int nchunks, size_t* counter_bytes,
                  size_t* part_bytes) {
  *counter_bytes = kStatusBytes + (static_cast<size_t>(batch) * n_kv_heads * sizeof(int) + 255) / 256 * 256;
  *part_bytes = static_cast<size_t>(batch) * n_q_heads * nchunks * (head_dim + 4) * sizeof(float);
}
}  // namespace

extern "C" long long attention_decode_noalloc_scratch_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                                            int max_pos) {
  using namespace lps;
  if (batch < 1 || batch > kMaxBatch || n_kv_heads < 1 || n_q_heads % n_kv_heads ||
      !attn_supported(head_dim, n_q_heads / n_kv_heads) || max_pos < 0)
    return -1;
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  const int chunk = attn_chunk(head_dim, n_kv_heads, batch, max_pos, num_sms);
  size_t counter_bytes = 0, part_bytes = 0;
  scratch_need(batch, n_q_heads, n_kv_heads, head_dim, (max_pos + 1 + chunk - 1) / chunk, &counter_bytes, &part_bytes);
  return static_cast<long long>(counter_bytes + part_bytes);
}

extern "C" int attention_decode_noalloc(const float* q, const void* k_cache, const void* v_cache, float* out,
                                        int batch, int n_q_heads, int n_kv_heads, int head_dim, int max_ctx,
                                        const int32_t* pos, void* stream) {
  using namespace lps;
  if (!q || !k_cache || !v_cache || !out || !pos) return fail(LPS_EINVAL, "q, caches, out and pos are required");
  if (batch < 1 || batch > kMaxBatch) return fail(LPS_EINVAL, "batch must be in 1..8");
  if (n_kv_heads < 1 || n_q_heads % n_kv_heads || !attn_supported(head_dim, n_q_heads / n_kv_heads))
    return fail(LPS_EINVAL, "head_dim must be 64 or 128 and n_q_heads / n_kv_heads in {1, 2, 4, 8}");
  if (max_ctx < 1) return fail(LPS_EINVAL, "max_ctx must be positive");
  int max_pos = 0;
  for (int b = 0; b < batch; ++b) {
    if (pos[b] < 0 || pos[b] >= max_ctx) return fail(LPS_EINVAL, "pos out of [0, max_ctx)");
    max_pos = pos[b] > max_pos ? pos[b] : max_pos;
  }
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return fail(LPS_EINVAL, "caches must be 16-byte aligned");
  // the kernel addresses cache rows with 32-bit TMA coordinates
  if (static_cast<long long>(batch) * n_kv_heads * max_ctx > 0x7fffffffll)
    return fail(LPS_EINVAL, "batch * n_kv_heads * max_ctx must stay below 2^31 cache rows");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= lps::kMaxDevices) return fail(LPS_ECUDA, "no usable current device");
  void* base = nullptr;
  int num_sms = 0;
  e = scratch_on(dev, &base, &num_sms);
  if (e != cudaSuccess) return fail(LPS_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));

  const int chunk = attn_chunk(head_dim, n_kv_heads, batch, max_pos, num_sms);
  const int nchunks = (max_pos + 1 + chunk - 1) / chunk;
  size_t counter_bytes = 0, part_bytes = 0;
  scratch_need(batch, n_q_heads, n_kv_heads, head_dim, nchunks, &counter_bytes, &part_bytes);
  if (counter_bytes + part_bytes > kScratchBytes)
    return fail(LPS_EINVAL, "needs " + std::to_string(counter_bytes + part_bytes) + " bytes of scratch, more than the " +
                                std::to_string(kScratchBytes) + " this entry point holds; use fewer sequences or "
                                "positions, or the regular decode path");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(static_cast<unsigned char*>(base) + kStatusBytes, 0, counter_bytes - kStatusBytes, s);
  if (e != cudaSuccess) return fail(LPS_ECUDA, std::string("clearing the counters: ") + cudaGetErrorString(e));

  AttnParams p{};
  const unsigned long long rows = static_cast<unsigned long long>(batch) * n_kv_heads * max_ctx;
  if (!encode_cache(&p.tmap_k, k_cache, head_dim, rows, attn_sub_tile(head_dim)) ||
      !encode_cache(&p.tmap_v, v_cache, head_dim, rows, attn_sub_tile(head_dim)))
    return fail(LPS_ECUDA, "cuTensorMapEncodeTiled failed for a cache");
  p.q = q;
  p.kc = static_cast<const __nv_bfloat16*>(k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(v_cache);
  p.out = out;
  p.counter = reinterpret_cast<int*>(static_cast<unsigned char*>(base) + kStatusBytes);
  p.part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + counter_bytes);
  p.nq = n_q_heads;
  p.nkv = n_kv_heads;
  p.hd = head_dim;
  p.max_ctx = max_ctx;
  p.max_chunks = nchunks;
  p.chunk = chunk;
  for (int b = 0; b < batch; ++b) p.pos[b] = pos[b];
  p.scale = 1.0f / std::sqrt(static_cast<float>(head_dim));
  p.status = static_cast<int*>(base);  // sticky until attention_decode_noalloc_status reads it
  e = launch_attention(p, batch, max_pos, s, false);
  if (e != cudaSuccess) return fail(LPS_ECUDA, std::string("launch: ") + cudaGetErrorString(e));
  return LPS_OK;
}

extern "C" int attention_decode_noalloc_status(void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= lps::kMaxDevices) return fail(LPS_ECUDA, "no usable current device");
  void* base = nullptr;
  int num_sms = 0;
  e = scratch_on(dev, &base, &num_sms);
  if (e != cudaSuccess) return fail(LPS_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
  e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(LPS_ECUDA, std::string("stream: ") + cudaGetErrorString(e));
  int st[2] = {0, 0};
  e = cudaMemcpy(st, base, sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(LPS_ECUDA, std::string("reading the status: ") + cudaGetErrorString(e));
  if (st[0] == 0 && st[1] == 0) return LPS_OK;
  e = cudaMemset(base, 0, sizeof st);
  if (e != cudaSuccess) return fail(LPS_ECUDA, std::string("clearing the status: ") + cudaGetErrorString(e));
  return fail(LPS_ECUDA, "an earlier call's output is invalid: " + lps::describe_status(st[0], st[1]));
}
