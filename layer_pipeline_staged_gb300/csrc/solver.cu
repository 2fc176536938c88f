// Memory-balancing stage plan (host only): which contiguous layers each stage
// owns so that the context every stage can hold is as large as possible, and
// among those plans the one whose fullest stage is least full (ninfer
// pipeline-stages.md, "How it works": solve_stage_plan, "maximum page groups
// every stage can hold, then least-full stage", checked against a brute-force
// partition oracle; when nothing fits it deals the layers evenly).
//
// Cost model. Stage s, holding layers [i, j), at capacity P units (a unit is
// one context position of the per-stage cache) uses
//     U_s(P) = fixed[s] + sum_{l in [i,j)} bytes[l] + P * sum_{l in [i,j)} unit[l]
// and fits when U_s(P) <= free[s]. A plan's capacity is the largest P in
// [0, max_units] at which every stage fits (-1 if none does at P = 0).
//
// Algorithm (exact):
//   1. the best capacity P* by bisection on P (feasibility is monotone in P),
//      each P checked by reachability over (stage, layers held so far);
//   2. at P*, a dynamic program over (stage, first layer) for the smallest
//      fullest-stage fraction max_s U_s(P*) / free[s], with fractions compared
//      exactly (128-bit cross products);
//   3. among optimal plans the lexicographically smallest cuts.
#include <algorithm>
#include <cstdint>
#include <string>
#include <vector>

#include "lps.h"

namespace lps {
int host_fail(int code, const char* fn, const std::string& why);
}  // namespace lps

namespace {

using u128 = unsigned __int128;

struct Instance {
  int L, N;
  const uint64_t* bytes;
  const uint64_t* unit;
  const uint64_t* free_b;
  std::vector<uint64_t> fixed;
  std::vector<u128> pre_b, pre_u;  // prefix sums over layers
};

// U_s(P) for stage s holding layers [i, j), exact in 128 bits (saturated when
// P times the unit bytes could not fit in 128 bits: such a stage never fits).
u128 usage(const Instance& in, int s, int i, int j, int64_t P) {
  const u128 w = in.pre_b[j] - in.pre_b[i];
  const u128 k = in.pre_u[j] - in.pre_u[i];
  if (P > 0 && (k >> 64) != 0) return ~static_cast<u128>(0);
  return static_cast<u128>(in.fixed[s]) + w + static_cast<u128>(P) * k;  // < 2^64 L + 2^127
}

bool fits(const Instance& in, int s, int i, int j, int64_t P) { return usage(in, s, i, j, P) <= in.free_b[s]; }

// Whether some plan fits at capacity P: reach[j] after stage s says whether
// stages 0..s can hold exactly layers [0, j). (A greedy "fill each stage
// as far as it goes" is not enough: taking a small layer early can leave a
// small later stage a layer it cannot hold.)
bool feasible(const Instance& in, int64_t P) {
  std::vector<char> reach(in.L + 1, 0), next(in.L + 1, 0);
  reach[0] = 1;
  for (int s = 0; s < in.N; ++s) {
    std::fill(next.begin(), next.end(), 0);
    const int rest = in.N - 1 - s;  // stages after s, one layer each at least
    for (int i = s; i <= in.L - 1 - rest; ++i) {
      if (!reach[i]) continue;
      for (int j = i + 1; j <= in.L - rest; ++j) {
        if (!fits(in, s, i, j, P)) break;  // longer stages only use more
        next[j] = 1;
      }
    }
    reach.swap(next);
  }
  return reach[in.L] != 0;
}

// a/b < c/d for b, d > 0. The numerators compared are usages of stages that
// fit, so a, c <= free[s] < 2^64, and the products stay below 2^128.
bool frac_less(u128 a, uint64_t b, u128 c, uint64_t d) { return a * d < c * b; }

}  // namespace

namespace lps {

// Parameters are checked by the caller (stage_plan_solve below).
int solve_plan(int L, int N, const uint64_t* bytes, const uint64_t* unit, const uint64_t* free_b,
               const uint64_t* fixed, int64_t max_units, std::vector<int>& fence, int64_t& units) {
  Instance in{L, N, bytes, unit, free_b, std::vector<uint64_t>(N, 0), std::vector<u128>(L + 1, 0),
              std::vector<u128>(L + 1, 0)};
  for (int s = 0; s < N; ++s) in.fixed[s] = fixed ? fixed[s] : 0;
  for (int l = 0; l < L; ++l) {
    in.pre_b[l + 1] = in.pre_b[l] + bytes[l];
    in.pre_u[l + 1] = in.pre_u[l] + unit[l];
  }
  fence.assign(N + 1, 0);
  if (!feasible(in, 0)) {
    // nothing fits: the even split, capacity -1
    for (int s = 0; s <= N; ++s) fence[s] = static_cast<int>(static_cast<long long>(s) * L / N);
    units = -1;
    return LPS_OK;
  }
  int64_t lo = 0, hi = max_units;  // feasible(lo) holds
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo + 1) / 2;
    if (feasible(in, mid))
      lo = mid;
    else
      hi = mid - 1;
  }
  const int64_t P = lo;
  units = P;

  // best[s][i]: the smallest fullest-stage fraction of stages s..N-1 holding
  // layers [i, L), as (numerator, denominator); invalid when den == 0.
  struct Frac {
    u128 num;
    uint64_t den;
  };
  std::vector<std::vector<Frac>> best(N + 1, std::vector<Frac>(L + 1, Frac{0, 0}));
  best[N][L] = Frac{0, 1};
  auto worse = [](const Frac& a, const Frac& b) { return frac_less(b.num, b.den, a.num, a.den); };  // a > b
  for (int s = N - 1; s >= 0; --s) {
    const int rest = N - 1 - s;  // stages after s, one layer each at least
    for (int i = s; i <= L - 1 - rest; ++i) {
      Frac cur{0, 0};
      for (int j = i + 1; j <= L - rest; ++j) {
        const Frac& tail = best[s + 1][j];
        if (tail.den == 0) continue;
        if (!fits(in, s, i, j, P)) break;  // longer stages only use more
        const Frac mine{usage(in, s, i, j, P), free_b[s]};
        const Frac m = worse(mine, tail) ? mine : tail;
        if (cur.den == 0 || frac_less(m.num, m.den, cur.num, cur.den)) cur = m;
      }
      best[s][i] = cur;
    }
  }
  // walk from the left taking the smallest end that keeps the optimum
  const Frac opt = best[0][0];
  int i = 0;
  fence[0] = 0;
  for (int s = 0; s < N; ++s) {
    const int rest = N - 1 - s;
    int chosen = -1;
    for (int j = i + 1; j <= L - rest; ++j) {
      const Frac& tail = best[s + 1][j];
      if (tail.den == 0 || !fits(in, s, i, j, P)) continue;
      const Frac mine{usage(in, s, i, j, P), free_b[s]};
      // max(mine, tail) <= opt
      if (!worse(mine, opt) && !worse(tail, opt)) {
        chosen = j;
        break;
      }
    }
    if (chosen < 0) return host_fail(LPS_EINVAL, "stage_plan_solve", "internal: no plan at the solved capacity");
    fence[s + 1] = chosen;
    i = chosen;
  }
  return LPS_OK;
}

}  // namespace lps

extern "C" int stage_plan_solve(int n_layers, int n_stages, const uint64_t* layer_bytes,
                                const uint64_t* layer_unit_bytes, const uint64_t* stage_free,
                                const uint64_t* stage_fixed, int64_t max_units, int* cuts_out, int64_t* units_out) {
  static const char* FN = "stage_plan_solve";
  if (!layer_bytes || !layer_unit_bytes || !stage_free || !units_out || (n_stages > 1 && !cuts_out))
    return lps::host_fail(LPS_EINVAL, FN, "NULL argument");
  if (n_layers < 1 || n_stages < 1 || n_stages > n_layers)
    return lps::host_fail(LPS_EINVAL, FN, "need 1 <= n_stages <= n_layers");
  if (max_units < 0) return lps::host_fail(LPS_EINVAL, FN, "max_units must be >= 0");
  for (int s = 0; s < n_stages; ++s)
    if (stage_free[s] == 0) return lps::host_fail(LPS_EINVAL, FN, "every stage needs free bytes > 0");
  std::vector<int> fence;
  int64_t units = -1;
  const int rc = lps::solve_plan(n_layers, n_stages, layer_bytes, layer_unit_bytes, stage_free, stage_fixed,
                                 max_units, fence, units);
  if (rc != LPS_OK) return rc;
  for (int s = 1; s < n_stages; ++s) cuts_out[s - 1] = fence[s];
  *units_out = units;
  return LPS_OK;
}

extern "C" int model_stage_bytes(const lps_model_desc* d, uint64_t* layer_bytes, uint64_t* layer_unit_bytes,
                                 uint64_t* first_stage_bytes, uint64_t* last_stage_bytes,
                                 uint64_t* every_stage_bytes) {
  static const char* FN = "model_stage_bytes";
  if (!d || !layer_bytes || !layer_unit_bytes || !first_stage_bytes || !last_stage_bytes || !every_stage_bytes)
    return lps::host_fail(LPS_EINVAL, FN, "NULL argument");
  if (d->n_layers < 1 || d->n_embd < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 || d->head_dim < 2 ||
      d->ffn < 1 || d->vocab < 1 || d->batch < 1 || d->max_ctx < 1)
    return lps::host_fail(LPS_EINVAL, FN, "bad model shape");
  const bool int8 = d->weight_dtype == LPS_WEIGHT_INT8_ROWSCALE;
  const uint64_t eb = int8 ? 1 : 2;
  const uint64_t E = d->n_embd, qw = static_cast<uint64_t>(d->n_q_heads) * d->head_dim,
                 kw = static_cast<uint64_t>(d->n_kv_heads) * d->head_dim, F = d->ffn, V = d->vocab,
                 B = d->batch;
  // weights of one layer: QKV, o, gate/up, down (+ one fp32 scale per row), two norms
  const uint64_t rows = (qw + 2 * kw) + E + 2 * F + E;
  const uint64_t w = ((qw + 2 * kw) * E + E * qw + 2 * F * E + E * F) * eb + (int8 ? rows * 4 : 0) + 2 * E * 4;
  // cache of one layer per context position: K and V rows of every sequence, bf16
  const uint64_t kv = B * kw * 2 * 2;
  for (int l = 0; l < d->n_layers; ++l) {
    layer_bytes[l] = w;
    layer_unit_bytes[l] = kv;
  }
  const uint64_t table = V * E * eb + (int8 ? V * 4 : 0);
  *first_stage_bytes = table;                                              // embedding
  const uint64_t depth = d->pending_depth > 0 ? d->pending_depth : 4;
  *last_stage_bytes = table + E * 4 + (depth + 1) * B * V * 4;             // LM head, final norm, logits
  // activations, attention partials (a rough bound: one partial per 64
  // positions), the RoPE table and two boundary slots
  const uint64_t parts = B * static_cast<uint64_t>(d->n_q_heads) * ((d->max_ctx + 63) / 64) * (d->head_dim + 4) * 4;
  *every_stage_bytes = B * (E + 2 * qw + F) * 4 + parts + static_cast<uint64_t>(d->max_ctx) * d->head_dim * 4 +
                       2 * B * E * 4;
  return LPS_OK;
}
