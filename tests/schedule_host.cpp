// Host-side check of the attention kernels' work decomposition (tva_common.cuh), built
// with a plain C++ compiler: the header is included unmodified, with single-thread
// stand-ins for the few device built-ins its staging helpers name.
//
// For each problem (one sequence or a ragged batch; stream-K ranges, ranges aligned to
// row groups, and teams sharing K/V tiles), every worker's range is walked segment by
// segment, exactly as the partials kernels do, and the walk must:
//   - cover every (row group, key tile) unit of every sequence exactly once;
//   - keep each segment inside one row group (and inside the worker's range);
//   - give each (worker, segment) pair its own partial slot, below U + B * Hkv * MP_max
//     (the workspace the host reserves).
// Prints "ok <problems>" or the first violation, and exits non-zero on a violation.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <set>
#include <vector>

#include <cuda_runtime.h>

static uint3 threadIdx = {0, 0, 0};
static dim3 blockDim(1, 1, 1);
template <typename T>
static inline T __ldg(const T* p) { return *p; }
static inline void __syncthreads() {}
static inline int atomicCAS(int* a, int cmp, int v) {
  const int old = *a;
  if (old == cmp) *a = v;
  return old;
}
static inline float __uint_as_float(unsigned u) {
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

#include "tva_internal.h"

namespace {

int g_problems = 0;

bool fail(const char* what, int u, long long x) {
  std::printf("FAIL problem %d: %s (worker %d, value %lld)\n", g_problems, what, u, x);
  return false;
}

// prefix lengths and tree sizes per sequence; null cu arrays for one sequence when `single`
bool check(const std::vector<int>& P, const std::vector<int>& m, int Hkv, int G, int W, int U, int mode,
           bool single) {
  ++g_problems;
  const int B = (int)P.size();
  const int npt = 128 / G;                  // nodes per M-tile
  int max_prefix = 0, max_nodes = 1;
  for (int b = 0; b < B; ++b) {
    max_prefix = P[b] > max_prefix ? P[b] : max_prefix;
    max_nodes = m[b] > max_nodes ? m[b] : max_nodes;
  }
  std::vector<int32_t> cu_p(B + 1, 0), cu_n(B + 1, 0);
  for (int b = 0; b < B; ++b) {
    cu_p[b + 1] = cu_p[b] + P[b];
    cu_n[b + 1] = cu_n[b] + m[b];
  }
  tva::Problem pr{};
  pr.cu_prefix = single ? nullptr : cu_p.data();
  pr.cu_nodes = single ? nullptr : cu_n.data();
  pr.single_prefix = P[0];
  pr.single_nodes = m[0];
  pr.B = B;
  pr.Hkv = Hkv;
  pr.G = G;
  pr.Hq = Hkv * G;
  pr.d = 128;
  pr.RG = W * npt * G;
  pr.U = U;
  pr.max_prefix = max_prefix;
  pr.max_nodes = max_nodes;
  pr.kv_capacity = cu_p[B];
  pr.node_capacity = cu_n[B];
  const int mp_max = (max_nodes + W * npt - 1) / (W * npt);
  pr.share = mode == 2 ? mp_max : 0;
  pr.align = mode == 1 ? U / Hkv : 0;
  const bool shared = pr.share != 0;
  const long long slots = (long long)U + (long long)B * Hkv * mp_max;

  // every unit, by (global row group, tile)
  std::vector<std::vector<int>> hits;
  long long T = 0;
  for (int b = 0; b < B; ++b) {
    const int MP = (m[b] * G + pr.RG - 1) / pr.RG, tiles = (P[b] + 127) / 128 + 1;
    for (int q = 0; q < Hkv * MP; ++q) hits.emplace_back(tiles, 0);
    T += (long long)Hkv * MP * tiles;
  }
  if (!shared && mode == 0 && tva::total_units(pr) != T) return fail("total_units", -1, tva::total_units(pr));
  std::set<long long> used;
  for (int u = 0; u < U; ++u) {
    long long t0 = 0, t1 = 0;
    tva::worker_range(pr, u, t0, t1, shared);
    long long t = t0;
    tva::Segment S;
    int guard = 0;
    while (tva::next_segment(pr, u, t, t1, S, shared)) {
      if (++guard > 1 << 20) return fail("walk does not end", u, t);
      const tva::Loc& L = S.L;
      if (S.n <= 0) return fail("empty segment", u, S.n);
      if (L.q < 0 || L.q >= (int)hits.size()) return fail("row group out of range", u, L.q);
      if (S.tile0 < 0 || S.tile0 + S.n > L.tiles) return fail("segment leaves its row group", u, S.tile0);
      if ((int)hits[L.q].size() != L.tiles) return fail("row group's tile count", u, L.tiles);
      for (int i = 0; i < S.n; ++i) ++hits[L.q][S.tile0 + i];
      const long long slot = tva::partial_slot(pr, u, L, shared);
      if (slot < 0 || slot >= slots) return fail("partial slot outside the workspace", u, slot);
      if (!used.insert(slot).second) return fail("partial slot used twice", u, slot);
    }
    if (t < t1) return fail("walk stopped early", u, t);
  }
  for (size_t q = 0; q < hits.size(); ++q)
    for (size_t i = 0; i < hits[q].size(); ++i)
      if (hits[q][i] != 1) return fail("unit not covered exactly once", -1, (long long)q * 100000 + (long long)i);
  return true;
}

}  // namespace

int main() {
  bool ok = true;
  const int sms = 152;
  // one sequence: the attention workloads (64k prefix / 64-node tree; 128k / 128 nodes at
  // G = 8; 16k chain; 32k beam tree of 68 nodes), with every mode whose precondition holds
  struct One { int P, m, Hkv, G; };
  const One ones[] = {{65536, 64, 8, 4}, {131072, 128, 8, 8}, {16384, 8, 8, 4}, {32768, 68, 8, 4},
                      {0, 5, 2, 4},      {1500, 40, 8, 4},    {900, 128, 8, 8}, {300, 1, 1, 4},
                      {129, 127, 4, 3},  {127, 33, 8, 16},    {4096, 100, 2, 2}};
  for (const One& o : ones) {
    for (int W = 1; W <= 2; ++W) {
      const int npt = 128 / o.G;
      const int mp_max = (o.m + W * npt - 1) / (W * npt);
      for (int U : {sms, sms / 2, 7, 1, 300}) {
        for (bool single : {true, false}) {
          ok = ok && check({o.P}, {o.m}, o.Hkv, o.G, W, U, 0, single);
          if (mp_max == 1 && U % o.Hkv == 0) ok = ok && check({o.P}, {o.m}, o.Hkv, o.G, W, U, 1, single);
          if (mp_max >= 2 && U >= mp_max) ok = ok && check({o.P}, {o.m}, o.Hkv, o.G, W, U, 2, single);
        }
      }
    }
  }
  // ragged batches (stream-K): prefixes 4k-32k with 32-node trees, empty prefixes and
  // trees, and uneven tree sizes
  std::srand(7);
  for (int rep = 0; rep < 40; ++rep) {
    const int B = 1 + std::rand() % 9;
    std::vector<int> P(B), m(B);
    for (int b = 0; b < B; ++b) {
      P[b] = rep % 3 == 0 ? 4096 + std::rand() % 28673 : std::rand() % 2000;
      m[b] = rep % 5 == 0 ? 32 : std::rand() % 129;
    }
    const int G = (rep % 4 == 0) ? 8 : 4;
    for (int W = 1; W <= 2; ++W)
      for (int U : {sms, 19, 1}) ok = ok && check(P, m, 8, G, W, U, 0, false);
  }
  if (ok) std::printf("ok %d\n", g_problems);
  return ok ? 0 : 1;
}
