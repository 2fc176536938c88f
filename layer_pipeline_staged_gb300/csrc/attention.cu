// Split-K GQA decode attention over a stage-owned contiguous bf16 KV cache
// (flash-decoding): the positions [0, pos] of each (sequence, kv head) are cut
// into equal chunks; one CTA per chunk computes, for every q head of the
// group, a partial (running max m, running sum l, unnormalised output acc)
// with an online softmax over sub-tiles streamed by 1D bulk copies; the last
// CTA of the group to finish combines the partials in chunk order.
//
// The q heads of one group share the group's K/V rows, so every cached byte is
// read once per step (q head h reads kv head h / (nq / nkv): "TP3 support via
// zero-padded dummy heads", Implementation status item 2). Sub-tiles that lie
// strictly before the current position are prefetched before the
// programmatic-dependent-launch wait (earlier steps wrote them); the sub-tile
// holding row pos is loaded after it (the QKV kernel just wrote that row).
// The combine order is fixed, and the chunk length depends only on pos, so the
// result is the same bits for every stage plan and stream schedule.
#include "kernels.h"
#include "ptx.cuh"

namespace lps {
namespace {

constexpr int kThreads = 128;
constexpr int kRing = 3;

template <int HD>
struct AttnShape {
  static constexpr int TS = 8192 / HD;          // positions per sub-tile (16 KB of K, 16 KB of V)
  static constexpr int NPART = HD / 64;         // 64-element parts of a row in the score phase
  static constexpr int NG = kThreads / (HD / 2);// position groups in the PV phase
  static constexpr int TILE = TS * HD;          // bf16 elements per K (or V) sub-tile
};

template <int HD, int G>
struct AttnSmem {
  using S = AttnShape<HD>;
  __nv_bfloat16 k[kRing][S::TILE];
  __nv_bfloat16 v[kRing][S::TILE];
  float q[G][S::NPART][8][12];      // q chunks of 8 floats, padded to 12 against bank conflicts
  float s[S::NPART][G][S::TS];      // partial scores per row part
  float p[S::TS][G];                // softmax numerators of the sub-tile
  float red[S::NG][G][HD];          // cross-group reduction of the PV accumulators
  float m[G], l[G], alpha[G];
  uint64_t full[kRing];
  int last;
};

template <int HD, int G>
__global__ void __launch_bounds__(kThreads, 2) attn_kernel(const __grid_constant__ AttnParams p) {
  using S = AttnShape<HD>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  AttnSmem<HD, G>& sm = *reinterpret_cast<AttnSmem<HD, G>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int pos = p.pos[b];
  const int n_total = pos + 1;
  const int t_begin = c * p.chunk;
  if (t_begin >= n_total) return;  // beyond this sequence's positions (uniform per CTA)
  const int t_end = min(t_begin + p.chunk, n_total);
  const int nsub = (t_end - t_begin + S::TS - 1) / S::TS;
  const int nchunks = (n_total + p.chunk - 1) / p.chunk;
  const size_t kv_off = static_cast<size_t>(b * p.nkv + g) * p.max_ctx * HD;
  const __nv_bfloat16* kbase = p.kc + kv_off;
  const __nv_bfloat16* vbase = p.vc + kv_off;

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) mbar_init(&sm.full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint64_t pol = 0;
  auto issue = [&](int j) {
    const int slot = j % kRing;
    const int t0 = t_begin + j * S::TS;
    const int rows = min(S::TS, t_end - t0);
    const uint32_t bytes = static_cast<uint32_t>(rows) * HD * 2;
    mbar_arrive_expect_tx(&sm.full[slot], 2 * bytes);
    bulk_g2s(sm.k[slot], kbase + static_cast<size_t>(t0) * HD, bytes, &sm.full[slot], pol);
    bulk_g2s(sm.v[slot], vbase + static_cast<size_t>(t0) * HD, bytes, &sm.full[slot], pol);
  };
  const int first = min(kRing, nsub);
  int issued = 0;
  if (tid == 0) {
    pol = l2_evict_first();
    // sub-tiles whose rows all lie before pos were written by earlier steps
    while (issued < first && t_begin + (issued + 1) * S::TS <= pos) issue(issued++);
  }
  pdl_wait();
  if (tid == 0)
    while (issued < first) issue(issued++);

  // q of the group's heads, in padded 8-float chunks
  for (int i = tid; i < G * HD; i += kThreads) {
    const int hh = i / HD, e = i - hh * HD;
    const int part = e / 64, ch = (e % 64) / 8, k = e % 8;
    sm.q[hh][part][ch][k] = p.q[static_cast<size_t>(b) * p.nq * HD + (g * G + hh) * HD + e];
  }
  if (tid < G) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
  }
  float a0[G], a1[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) a0[hh] = a1[hh] = 0.f;
  __syncthreads();

  for (int j = 0; j < nsub; ++j) {
    const int slot = j % kRing;
    const bool got = mbar_wait(&sm.full[slot], (j / kRing) & 1);
    if (__syncthreads_or(!got)) {
      if (tid == 0) {
        report_error(p.status, kErrWaitFull);
        for (int k = j + 1; k < min(nsub, j + kRing); ++k)
          if (!mbar_wait(&sm.full[k % kRing], (k / kRing) & 1)) {
            report_error(p.status, kErrDrain);
            break;
          }
      }
      return;
    }
    const int rows = min(S::TS, t_end - (t_begin + j * S::TS));

    // scores: thread = (position pp, row part); chunks visited in a rotated
    // order so the 8 lanes of a shared-memory phase hit distinct banks
    {
      const int pp = tid % S::TS, part = tid / S::TS;
      float sc[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) sc[hh] = 0.f;
      if (pp < rows) {
        const uint8_t* krow = reinterpret_cast<const uint8_t*>(sm.k[slot]) + pp * HD * 2 + part * 128;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int ch = (jj + pp) & 7;
          const uint4 kw = *reinterpret_cast<const uint4*>(krow + ch * 16);
          const float k8[8] = {bf16lo(kw.x), bf16hi(kw.x), bf16lo(kw.y), bf16hi(kw.y),
                               bf16lo(kw.z), bf16hi(kw.z), bf16lo(kw.w), bf16hi(kw.w)};
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const float4 qa = *reinterpret_cast<const float4*>(&sm.q[hh][part][ch][0]);
            const float4 qb = *reinterpret_cast<const float4*>(&sm.q[hh][part][ch][4]);
            float acc = sc[hh];
            acc = fmaf(k8[0], qa.x, acc); acc = fmaf(k8[1], qa.y, acc);
            acc = fmaf(k8[2], qa.z, acc); acc = fmaf(k8[3], qa.w, acc);
            acc = fmaf(k8[4], qb.x, acc); acc = fmaf(k8[5], qb.y, acc);
            acc = fmaf(k8[6], qb.z, acc); acc = fmaf(k8[7], qb.w, acc);
            sc[hh] = acc;
          }
        }
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) sm.s[part][hh][pp] = sc[hh];
    }
    __syncthreads();

    // online softmax update, one warp per head
    for (int hh = warp; hh < G; hh += kThreads / 32) {
      float sv[S::TS / 32];
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < S::TS / 32; ++k) {
        const int pp = lane + 32 * k;
        float s = -INFINITY;
        if (pp < rows) {
          float t = sm.s[0][hh][pp];
#pragma unroll
          for (int part = 1; part < S::NPART; ++part) t += sm.s[part][hh][pp];
          s = t * p.scale;
        }
        sv[k] = s;
        mx = fmaxf(mx, s);
      }
      mx = warp_max(mx);
      const float m_old = sm.m[hh];
      const float m_new = fmaxf(m_old, mx);
      float ls = 0.f;
#pragma unroll
      for (int k = 0; k < S::TS / 32; ++k) {
        const int pp = lane + 32 * k;
        const float e = (pp < rows) ? expf(sv[k] - m_new) : 0.f;
        sm.p[pp][hh] = e;
        ls += e;
      }
      ls = warp_sum(ls);
      if (lane == 0) {
        const float alpha = expf(m_old - m_new);
        sm.alpha[hh] = alpha;
        sm.m[hh] = m_new;
        sm.l[hh] = sm.l[hh] * alpha + ls;
      }
    }
    __syncthreads();

    // acc = acc * alpha + sum_p P[p] * V[p]: thread = (dim pair, position group)
    {
      const int i2 = tid % (HD / 2), pg = tid / (HD / 2);
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float al = sm.alpha[hh];
        a0[hh] *= al;
        a1[hh] *= al;
      }
      const uint32_t* vt = reinterpret_cast<const uint32_t*>(sm.v[slot]);
      for (int pp = pg; pp < rows; pp += S::NG) {
        const uint32_t vw = vt[pp * (HD / 2) + i2];
        const float v0 = bf16lo(vw), v1 = bf16hi(vw);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float pr = sm.p[pp][hh];
          a0[hh] = fmaf(pr, v0, a0[hh]);
          a1[hh] = fmaf(pr, v1, a1[hh]);
        }
      }
    }
    __syncthreads();  // sub-tile `slot` fully consumed
    if (tid == 0 && j + kRing < nsub) issue(j + kRing);
  }

  // reduce the position groups in order and write this chunk's partial
  {
    const int i2 = tid % (HD / 2), pg = tid / (HD / 2);
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      sm.red[pg][hh][2 * i2] = a0[hh];
      sm.red[pg][hh][2 * i2 + 1] = a1[hh];
    }
  }
  __syncthreads();
  const int stride = HD + 2;
  for (int o = tid; o < G * HD; o += kThreads) {
    const int hh = o / HD, i = o - hh * HD;
    float acc = sm.red[0][hh][i];
#pragma unroll
    for (int pg = 1; pg < S::NG; ++pg) acc += sm.red[pg][hh][i];
    float* dst = p.part + ((static_cast<size_t>(b) * p.nq + g * G + hh) * p.max_chunks + c) * stride;
    dst[i] = acc;
    if (i == 0) {
      dst[HD] = sm.m[hh];
      dst[HD + 1] = sm.l[hh];
    }
  }

  // the last CTA of (b, g) combines every chunk's partial, in chunk order
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&p.counter[b * p.nkv + g], 1);
    sm.last = (prev == nchunks - 1);
  }
  __syncthreads();
  if (sm.last) {
    __threadfence();
    for (int o = tid; o < G * HD; o += kThreads) {
      const int hh = o / HD, i = o - hh * HD;
      const float* base = p.part + (static_cast<size_t>(b) * p.nq + g * G + hh) * p.max_chunks * stride;
      float M = -INFINITY;
      for (int cc = 0; cc < nchunks; ++cc) M = fmaxf(M, __ldcg(base + cc * stride + HD));
      float L = 0.f, O = 0.f;
      for (int cc = 0; cc < nchunks; ++cc) {
        const float w = expf(__ldcg(base + cc * stride + HD) - M);
        L = fmaf(__ldcg(base + cc * stride + HD + 1), w, L);
        O = fmaf(__ldcg(base + cc * stride + i), w, O);
      }
      p.out[static_cast<size_t>(b) * p.nq * HD + (g * G + hh) * HD + i] = O / L;
    }
    if (tid == 0) p.counter[b * p.nkv + g] = 0;
  }
  pdl_launch_dependents();
}

template <int HD, int G>
cudaError_t launch_hg(const AttnParams& p, int batch, int max_pos, cudaStream_t s, bool pdl) {
  auto kern = attn_kernel<HD, G>;
  const int smem = static_cast<int>(sizeof(AttnSmem<HD, G>));
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((max_pos + 1 + p.chunk - 1) / p.chunk, p.nkv, batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int HD>
cudaError_t launch_h(const AttnParams& p, int batch, int max_pos, cudaStream_t s, bool pdl) {
  switch (p.nq / p.nkv) {
    case 1: return launch_hg<HD, 1>(p, batch, max_pos, s, pdl);
    case 2: return launch_hg<HD, 2>(p, batch, max_pos, s, pdl);
    case 4: return launch_hg<HD, 4>(p, batch, max_pos, s, pdl);
    case 8: return launch_hg<HD, 8>(p, batch, max_pos, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int attn_sub_tile(int hd) { return 8192 / hd; }

// Positions per CTA: a whole number of sub-tiles, sized so the grid holds
// about two CTAs per SM (one resident wave).
int attn_chunk(int hd, int nkv, int batch, int max_pos, int num_sms) {
  const int ts = attn_sub_tile(hd);
  const int nsub = (max_pos + 1 + ts - 1) / ts;
  int per_group = (2 * num_sms) / (nkv * batch);
  per_group = per_group < 1 ? 1 : per_group;
  const int subs = (nsub + per_group - 1) / per_group;
  return subs * ts;
}

int attn_max_chunks(int hd, int nkv, int batch, int max_ctx, int num_sms) {
  int worst = 1;
  // the chunk count is (pos + 1) / chunk(pos), rounded up; take its maximum over pos
  const int ts = attn_sub_tile(hd);
  for (int n = 1; n <= max_ctx; n += (n < ts ? 1 : ts)) {
    const int ch = attn_chunk(hd, nkv, batch, n - 1, num_sms);
    const int k = (n + ch - 1) / ch;
    worst = k > worst ? k : worst;
  }
  const int ch = attn_chunk(hd, nkv, batch, max_ctx - 1, num_sms);
  const int k = (max_ctx + ch - 1) / ch;
  return k > worst ? k : worst;
}

bool attn_supported(int hd, int group) {
  return (hd == 64 || hd == 128) && (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_attention(const AttnParams& p, int batch, int max_pos, cudaStream_t s, bool pdl) {
  if (p.hd == 64) return launch_h<64>(p, batch, max_pos, s, pdl);
  if (p.hd == 128) return launch_h<128>(p, batch, max_pos, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace lps
