// k_gdn.cu - tree verification for Gated DeltaNet layers ("DFlash-TfM", Method 3,
// rollback-free tree verification for GDN).
//
// A GDN layer updates its state by S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} +
// beta_t k_t v_t^T; a tree node's output o_i = S_i^T q_i is the recurrence run along its
// root-to-node path from the committed state S_0.  With gamma_i the product of alpha
// over that path, writing w_j for gamma_j times the j-th delta-rule update vector turns
// the whole tree into one unit-lower-triangular system over the topologically ordered
// nodes (the page's "(I + X) U = beta V"):
//     w_i + sum_{j proper ancestor of i} beta_i (gamma_i / gamma_j) (k_i . k_j) w_j
//         = beta_i (v_i - gamma_i S_0^T k_i),
//     o_i = gamma_i S_0^T q_i + sum_{j ancestor-or-self of i} (gamma_i / gamma_j) (k_j . q_i) w_j,
// and the state itself is never updated here (the commit waits for the accepted branch).
// The ratios gamma_i / gamma_j are products of alpha walked up from i to j (no division).
//
// One CTA (1024 threads) per (sequence, head), fp32 throughout:
//   1. parents -> depth, per-node offsets into compact ancestor lists (thread 0; m <= 128);
//      K staged in shared memory with padded rows;
//   2. interaction values over ancestor pairs only: X (k.k) and Y (q.k), one pair per thread;
//   3. K S_0 and Q S_0 for the thread's (rows, column) with S_0 read column-wise (coalesced);
//      the right-hand side goes to shared memory, gamma_i Q S_0 stays in registers;
//   4. forward substitution one depth level at a time (nodes of a level are independent);
//   5. the output sum over each node's ancestors-or-self.
#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

constexpr int kThreadsGdn = 1024;
constexpr int kMaxPairs = kMaxNodes * (kMaxNodes + 1) / 2;   // a chain of kMaxNodes

template <int D>
struct GdnSmem {
  static constexpr int kKPitch = D + 1;                 // padded rows: distinct rows, distinct banks
  static constexpr int kK = 0;                          // float [m][D+1]
  static constexpr int kW = kK + kMaxNodes * kKPitch;   // float [m][D]
  static constexpr int kX = kW + kMaxNodes * D;         // float [kMaxPairs] (proper-ancestor pairs)
  static constexpr int kY = kX + kMaxPairs;             // float [kMaxPairs] (ancestor-or-self pairs)
  static constexpr int kFloats = kY + kMaxPairs;
  static constexpr int kInts = 4 * kMaxNodes + 2 * (kMaxNodes + 2);   // par, dep, off, lvl, lvl0, fill
  static constexpr size_t kBytes = (size_t)kFloats * 4 + (size_t)kInts * 4 + (size_t)kMaxNodes * 4;
};

template <int D>
__global__ void __launch_bounds__(kThreadsGdn, 1) gdn_tree_kernel(GdnArgs a) {
  using SM = GdnSmem<D>;
  extern __shared__ float gsm[];
  float* sK = gsm + SM::kK;
  float* sW = gsm + SM::kW;
  float* sX = gsm + SM::kX;
  float* sY = gsm + SM::kY;
  int* s_par = reinterpret_cast<int*>(gsm + SM::kFloats);
  int* s_dep = s_par + kMaxNodes;      // depth, root = 1
  int* s_off = s_dep + kMaxNodes;      // first entry of node i's ancestor-or-self list
  int* s_lvl = s_off + kMaxNodes;      // nodes sorted by depth
  int* s_lvl0 = s_lvl + kMaxNodes;     // first index in s_lvl of each depth d (d <= m + 1)
  int* s_fill = s_lvl0 + kMaxNodes + 2;
  float* s_gam = reinterpret_cast<float*>(s_fill + kMaxNodes + 2);   // gamma_i
  __shared__ int s_ok, s_maxdep, s_pairs;

  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int n0 = __ldg(a.cu_nodes + b);
  const int m = __ldg(a.cu_nodes + b + 1) - n0;
  if (!(n0 >= 0 && m >= 0 && m <= a.max_nodes && (long long)n0 + m <= a.node_capacity)) {
    if (threadIdx.x == 0) set_status(a.status, kStatusInvalidArg);
    return;
  }
  if (m == 0) return;
  const int tid = threadIdx.x;
  const size_t hs = (size_t)a.H * D;   // stride between nodes in q / k / v / o

  // ---- 1. tree bookkeeping and K
  for (int i = tid; i < m; i += kThreadsGdn) s_par[i] = __ldg(a.parent + n0 + i);
  for (int e = tid; e < m * D; e += kThreadsGdn) {
    const int i = e / D, r = e % D;
    sK[i * SM::kKPitch + r] = __ldg(a.k + (size_t)(n0 + i) * hs + (size_t)h * D + r);
  }
  __syncthreads();
  if (tid == 0) {
    int ok = 1, off = 0, maxdep = 0;
    for (int i = 0; i < m; ++i) {
      const int p = s_par[i];
      if (p < -1 || p >= i) { ok = 0; break; }
      s_dep[i] = p < 0 ? 1 : s_dep[p] + 1;
      s_off[i] = off;
      off += s_dep[i];
      maxdep = max(maxdep, s_dep[i]);
      const float al = __ldg(a.alpha + (size_t)(n0 + i) * a.H + h);
      s_gam[i] = p < 0 ? al : al * s_gam[p];
    }
    if (ok) {   // counting sort by depth (depths 1..maxdep <= m <= kMaxNodes)
      for (int d = 0; d <= maxdep + 1; ++d) s_lvl0[d] = 0;
      for (int i = 0; i < m; ++i) s_lvl0[s_dep[i]]++;
      int run = 0;
      for (int d = 0; d <= maxdep; ++d) { const int c = s_lvl0[d]; s_lvl0[d] = run; run += c; }
      s_lvl0[maxdep + 1] = run;
      for (int d = 0; d <= maxdep; ++d) s_fill[d] = s_lvl0[d];
      for (int i = 0; i < m; ++i) s_lvl[s_fill[s_dep[i]]++] = i;
    }
    s_ok = ok;
    s_maxdep = maxdep;
    s_pairs = off;
  }
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) set_status(a.status, kStatusBadTree);
    return;
  }
  const int pairs = s_pairs;

  // ---- 2. interaction values over ancestor pairs: pair index -> (node i, a-th entry of
  // its ancestor-or-self list, walked up from i: a = 0 is i itself)
  for (int pi = tid; pi < pairs; pi += kThreadsGdn) {
    int lo = 0, hi = m - 1;          // node i: largest i with s_off[i] <= pi
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= pi) lo = mid; else hi = mid - 1;
    }
    const int i = lo, aidx = pi - s_off[i];
    int j = i;
    float ratio = 1.f;               // gamma_i / gamma_j
    for (int t = 0; t < aidx; ++t) {
      ratio *= __ldg(a.alpha + (size_t)(n0 + j) * a.H + h);
      j = s_par[j];
    }
    const float* kj = sK + j * SM::kKPitch;
    const float* ki = sK + i * SM::kKPitch;
    const float* qi = a.q + (size_t)(n0 + i) * hs + (size_t)h * D;
    float kk = 0.f, qk = 0.f;
#pragma unroll 8
    for (int r = 0; r < D; ++r) {
      kk = fmaf(ki[r], kj[r], kk);
      qk = fmaf(__ldg(qi + r), kj[r], qk);
    }
    const float beta_i = __ldg(a.beta + (size_t)(n0 + i) * a.H + h);
    sX[pi] = aidx > 0 ? beta_i * ratio * kk : 0.f;
    sY[pi] = ratio * qk;
  }

  // ---- 3. K S_0 and Q S_0: thread -> column c, rows g, g + G, g + 2G, ...
  constexpr int G = kThreadsGdn / D;          // row groups
  constexpr int RPT = kMaxNodes / G;          // rows per thread (at most)
  const int c = tid % D, g = tid / D;
  float ks[RPT], qs[RPT];
#pragma unroll
  for (int t = 0; t < RPT; ++t) { ks[t] = 0.f; qs[t] = 0.f; }
  const float* S0 = a.S0 + ((size_t)b * a.H + h) * D * D;
  for (int r = 0; r < D; ++r) {
    const float s = __ldg(S0 + (size_t)r * D + c);
#pragma unroll
    for (int t = 0; t < RPT; ++t) {
      const int i = g + t * G;
      if (i < m) {
        ks[t] = fmaf(sK[i * SM::kKPitch + r], s, ks[t]);
        qs[t] = fmaf(__ldg(a.q + (size_t)(n0 + i) * hs + (size_t)h * D + r), s, qs[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < RPT; ++t) {
    const int i = g + t * G;
    if (i < m) {
      const size_t row = (size_t)(n0 + i) * hs + (size_t)h * D + c;
      const float bt = __ldg(a.beta + (size_t)(n0 + i) * a.H + h);
      sW[i * D + c] = bt * (__ldg(a.v + row) - s_gam[i] * ks[t]);   // right-hand side
      qs[t] *= s_gam[i];
    }
  }
  __syncthreads();

  // ---- 4. forward substitution, one depth level at a time
  const int maxdep = s_maxdep;
  for (int d = 2; d <= maxdep; ++d) {
    const int l0 = s_lvl0[d], l1 = s_lvl0[d + 1];
    for (int e = tid; e < (l1 - l0) * D; e += kThreadsGdn) {
      const int i = s_lvl[l0 + e / D], cc = e % D;
      float acc = sW[i * D + cc];
      int j = s_par[i];
      for (int t = 1; t < s_dep[i]; ++t) {      // proper ancestors, nearest first
        acc = fmaf(-sX[s_off[i] + t], sW[j * D + cc], acc);
        j = s_par[j];
      }
      sW[i * D + cc] = acc;
    }
    __syncthreads();
  }

  // ---- 5. outputs
#pragma unroll
  for (int t = 0; t < RPT; ++t) {
    const int i = g + t * G;
    if (i < m) {
      float acc = qs[t];
      int j = i;
      for (int aa = 0; aa < s_dep[i]; ++aa) {   // ancestors-or-self, self first
        acc = fmaf(sY[s_off[i] + aa], sW[j * D + c], acc);
        j = s_par[j];
      }
      a.o[(size_t)(n0 + i) * hs + (size_t)h * D + c] = acc;
    }
  }
}

template <int D>
cudaError_t launch_gdn_typed(const GdnArgs& a, cudaStream_t s) {
  constexpr size_t smem = GdnSmem<D>::kBytes;
  cudaError_t e = check_cuda(cudaFuncSetAttribute(gdn_tree_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)smem),
                             "cudaFuncSetAttribute(gdn_tree_kernel)");
  if (e != cudaSuccess) return e;
  return check_cuda(launch_pdl(gdn_tree_kernel<D>, dim3((unsigned)(a.B * a.H)), dim3(kThreadsGdn), smem, s, a),
                    "launch gdn_tree_kernel");
}

}  // namespace

cudaError_t launch_gdn(const GdnArgs& a, cudaStream_t s) {
  return a.d == 64 ? launch_gdn_typed<64>(a, s) : launch_gdn_typed<128>(a, s);
}

}  // namespace tva
