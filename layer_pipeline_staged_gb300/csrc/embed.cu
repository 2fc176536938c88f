// Stage 0's embedding lookup: h[b] = E[token_b] as fp32 (bf16 exact, or
// int8 * row scale), for every sequence of the batch.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

template <bool INT8>
__global__ void __launch_bounds__(256) embed_kernel(const __grid_constant__ EmbedParams p) {
  trace_start(p.trace);
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const int tok = p.tok_dev ? p.tok_dev[b] : p.tok[b];
  pdl_wait();  // the previous step may still be reading h
  if (tok < 0 || tok >= p.vocab) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report_error(p.status, kErrBadArg | (kKidEmbed << 8));
    return;
  }
  float* h = p.h + static_cast<size_t>(b) * p.d;
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) * 4; i < p.d; i += gridDim.x * blockDim.x * 4) {
    float4 v;
    if (INT8) {
      const int8_t* row = static_cast<const int8_t*>(p.table) + static_cast<size_t>(tok) * p.d;
      const float s = p.scale[tok];
      const char4 q = *reinterpret_cast<const char4*>(row + i);
      v = make_float4(q.x * s, q.y * s, q.z * s, q.w * s);
    } else {
      const uint16_t* row = static_cast<const uint16_t*>(p.table) + static_cast<size_t>(tok) * p.d;
      const uint2 w = *reinterpret_cast<const uint2*>(row + i);
      v = make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
    }
    *reinterpret_cast<float4*>(h + i) = v;
  }
  trace_end(p.trace);
}

}  // namespace

cudaError_t launch_embed(const EmbedParams& p, bool int8, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.d + 1023) / 1024, p.batch);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int8 ? cudaLaunchKernelEx(&cfg, embed_kernel<true>, p) : cudaLaunchKernelEx(&cfg, embed_kernel<false>, p);
}

}  // namespace lps
