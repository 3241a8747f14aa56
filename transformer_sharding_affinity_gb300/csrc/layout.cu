// layout.cu -- host-only helpers of the C ABI (include/affinity.h) that turn
// per-layer affinity matrices into a layout score: unit-mass normalisation,
// the group gain, the scoring of every balanced KV-group partition, the
// per-layer best head map and the total co-located affinity J
// ("Affinity-Aware Sharding for Delayed Tensor Parallelism", §3 "Objective",
// equation (6), and "Optimiser"), plus the token-weighted merge of S matrices
// calibrated on disjoint token shards.  Nothing here touches a GPU.
#include "affinity.h"

#include <cmath>
#include <cstddef>
#include <vector>

namespace {

constexpr int kMaxGroups = 16;

// G! / ((G/L)!)^L evaluated as a product of binomials in double precision.
double balanced_count(int G, int L) {
  const int cap = G / L;
  double total = 1.0, rem = G;
  for (int l = 0; l < L; ++l) {
    double b = 1.0;
    for (int i = 0; i < cap; ++i) b = b * (rem - i) / (i + 1);
    total *= b;
    rem -= cap;
  }
  return total;
}

bool partition_args_ok(int32_t G, int32_t L) { return G >= 1 && L >= 1 && G <= kMaxGroups && L <= G && G % L == 0; }

// Visit every balanced map h (G/L groups per device) in lexicographic order of
// (h(0), ..., h(G-1)): a depth-first walk that tries devices in increasing order.
template <class Visit>
int64_t for_each_partition(int G, int L, Visit&& visit) {
  const int cap = G / L;
  int h[kMaxGroups], used[kMaxGroups] = {0};
  for (int i = 0; i < G; ++i) h[i] = -1;
  int64_t n = 0;
  int g = 0;
  while (g >= 0) {
    if (g == G) {
      visit(n, h);
      ++n;
      --g;
      continue;
    }
    if (h[g] >= 0) used[h[g]]--;
    int l = h[g] + 1;
    while (l < L && used[l] >= cap) ++l;
    if (l < L) {
      h[g] = l;
      used[l]++;
      ++g;
      if (g < G) h[g] = -1;
    } else {
      h[g] = -1;
      --g;
    }
  }
  return n;
}

bool map_ok(const int32_t* m, int64_t n, int32_t L) {
  for (int64_t i = 0; i < n; ++i)
    if (m[i] < 0 || m[i] >= L) return false;
  return true;
}

void gain(const double* Su, const int32_t* nu, const double* Sd, const int32_t* nu_prev, int32_t G, int64_t I,
          int32_t L, double* C) {
  for (int64_t i = 0; i < (int64_t)G * L; ++i) C[i] = 0.0;
  for (int g = 0; g < G; ++g)
    for (int64_t k = 0; k < I; ++k) C[(size_t)g * L + nu[k]] += Su[(size_t)g * I + k];
  if (Sd)
    for (int64_t k = 0; k < I; ++k)
      for (int g = 0; g < G; ++g) C[(size_t)g * L + nu_prev[k]] += Sd[(size_t)k * G + g];
}

}  // namespace

extern "C" {

aff_status affinity_score_partitions(const double* C, int32_t G, int32_t L, double* scores, int64_t* count,
                                     int64_t* best_index, int32_t* best_assign) {
  if (!C || !count || !best_index || !partition_args_ok(G, L)) return AFF_ERR_INVALID_ARG;
  if (balanced_count(G, L) > 1e8) return AFF_ERR_UNSUPPORTED_SHAPE;
  int64_t best = -1;
  double best_score = 0.0;
  const int64_t n = for_each_partition(G, L, [&](int64_t idx, const int* h) {
    double sc = 0.0;
    for (int i = 0; i < G; ++i) sc += C[(size_t)i * L + h[i]];
    if (scores) scores[idx] = sc;
    if (best < 0 || sc > best_score) {
      best = idx;
      best_score = sc;
      if (best_assign)
        for (int i = 0; i < G; ++i) best_assign[i] = h[i];
    }
  });
  *count = n;
  *best_index = best;
  return AFF_OK;
}

aff_status affinity_group_gain(const double* Shat_up_i, const int32_t* nu_i, const double* Shat_down_prev,
                               const int32_t* nu_prev, int32_t G, int64_t I, int32_t L, double* C) {
  if (!Shat_up_i || !nu_i || !C || G < 1 || I < 1 || L < 1) return AFF_ERR_INVALID_ARG;
  if ((Shat_down_prev == nullptr) != (nu_prev == nullptr)) return AFF_ERR_INVALID_ARG;
  if (!map_ok(nu_i, I, L) || (nu_prev && !map_ok(nu_prev, I, L))) return AFF_ERR_INVALID_ARG;
  gain(Shat_up_i, nu_i, Shat_down_prev, nu_prev, G, I, L, C);
  return AFF_OK;
}

aff_status affinity_objective(const double* Shat_up, const double* Shat_down, const int32_t* h, const int32_t* nu,
                              int32_t N, int32_t G, int64_t I, double* J) {
  if (!Shat_up || !h || !nu || !J || N < 1 || G < 1 || I < 1) return AFF_ERR_INVALID_ARG;
  if (N > 1 && !Shat_down) return AFF_ERR_INVALID_ARG;
  double s = 0.0;
  for (int i = 0; i < N; ++i) {
    const double* S = Shat_up + (size_t)i * G * I;
    const int32_t* hi = h + (size_t)i * G;
    const int32_t* ni = nu + (size_t)i * I;
    for (int g = 0; g < G; ++g)
      for (int64_t k = 0; k < I; ++k)
        if (hi[g] == ni[k]) s += S[(size_t)g * I + k];
  }
  for (int i = 0; i + 1 < N; ++i) {
    const double* S = Shat_down + (size_t)i * I * G;
    const int32_t* ni = nu + (size_t)i * I;
    const int32_t* hn = h + (size_t)(i + 1) * G;
    for (int64_t k = 0; k < I; ++k)
      for (int g = 0; g < G; ++g)
        if (ni[k] == hn[g]) s += S[(size_t)k * G + g];
  }
  *J = s;
  return AFF_OK;
}

aff_status affinity_unit_mass(const float* S, int64_t n, double* out) {
  if (!S || !out || n < 1) return AFF_ERR_INVALID_ARG;
  double total = 0.0;
  for (int64_t i = 0; i < n; ++i) total += (double)S[i];
  if (!(total > 0.0) || !std::isfinite(total)) return AFF_ERR_INVALID_ARG;
  const double inv = 1.0 / total;
  for (int64_t i = 0; i < n; ++i) out[i] = (double)S[i] * inv;
  return AFF_OK;
}

aff_status affinity_best_heads(const double* Shat_up, const double* Shat_down, const int32_t* nu, int32_t N,
                               int32_t G, int64_t I, int32_t L, int32_t* h_out, double* J_out) {
  if (!Shat_up || !nu || !h_out || N < 1 || I < 1 || !partition_args_ok(G, L)) return AFF_ERR_INVALID_ARG;
  if (N > 1 && !Shat_down) return AFF_ERR_INVALID_ARG;
  if (!map_ok(nu, (int64_t)N * I, L)) return AFF_ERR_INVALID_ARG;
  if (balanced_count(G, L) > 1e8) return AFF_ERR_UNSUPPORTED_SHAPE;
  // With every nu_i fixed, h_i enters J only through layer i's up term and
  // layer i-1's down term, so choosing each h_i by its own gain maximises J.
  std::vector<double> C((size_t)G * L);
  for (int i = 0; i < N; ++i) {
    const double* Sd = i > 0 ? Shat_down + (size_t)(i - 1) * I * G : nullptr;
    const int32_t* np = i > 0 ? nu + (size_t)(i - 1) * I : nullptr;
    gain(Shat_up + (size_t)i * G * I, nu + (size_t)i * I, Sd, np, G, I, L, C.data());
    int64_t count = 0, best = 0;
    const aff_status st = affinity_score_partitions(C.data(), G, L, nullptr, &count, &best, h_out + (size_t)i * G);
    if (st != AFF_OK) return st;
  }
  if (J_out) return affinity_objective(Shat_up, Shat_down, h_out, nu, N, G, I, J_out);
  return AFF_OK;
}

aff_status affinity_combine_shards(const float* const* S_shards, const int64_t* T_shards, int32_t n_shards,
                                   int64_t n, float* out) {
  if (!S_shards || !T_shards || !out || n_shards < 1 || n < 0) return AFF_ERR_INVALID_ARG;
  double T_total = 0.0;
  for (int r = 0; r < n_shards; ++r) {
    if (T_shards[r] < 0) return AFF_ERR_INVALID_ARG;
    if (T_shards[r] > 0 && !S_shards[r]) return AFF_ERR_INVALID_ARG;
    T_total += (double)T_shards[r];
  }
  if (!(T_total > 0.0)) return AFF_ERR_INVALID_ARG;
  for (int64_t j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int r = 0; r < n_shards; ++r)  // fixed shard order: the merge is deterministic
      if (T_shards[r] > 0) acc += (double)T_shards[r] * (double)S_shards[r][j];
    out[j] = (float)(acc / T_total);
  }
  return AFF_OK;
}

}  // extern "C"
