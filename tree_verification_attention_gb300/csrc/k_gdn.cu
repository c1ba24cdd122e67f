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
// D / 32 CTAs (1024 threads) per (sequence, head), each owning 32 columns of the output.
// q, k, v and the output are fp32 or bf16 (T); beta, alpha and the state are fp32, and all
// arithmetic is fp32 (bf16 inputs are widened as they are staged; the output is rounded to
// T once):
//   1. K, Q (16-byte loads, all issued before the first store) and this CTA's columns of
//      S_0 staged in shared memory; parents -> depth and path product (a thread per node),
//      list offsets (a scan) and the depth-level order;
//   2. interaction values over ancestor pairs only: X (k.k) and Y (q.k), one pair per
//      thread, which also records the pair's ancestor id (the lists that steps 4 and 5 walk);
//   3. K S_0 and Q S_0: a warp takes 4 nodes (K and Q rows) x 16 columns, its lanes split
//      the sum over the D rows of S_0 eight ways (k = 8 kk + lane % 8), so that each 16-byte
//      load of S_0 brings distinct data to every lane, and a reduce-scatter of shuffles
//      leaves each lane 4 finished sums; the right-hand side goes to shared memory over Q,
//      gamma_i Q S_0 over K;
//   4. forward substitution one depth level at a time (nodes of a level are independent);
//   5. the output sum over each node's ancestors-or-self.
#include <cuda_bf16.h>

#include <type_traits>

#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

// four consecutive elements (16-byte aligned for float, 8-byte for bf16)
__device__ __forceinline__ float4 gdn_load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 gdn_load4(const __nv_bfloat16* p) {
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
}
__device__ __forceinline__ void gdn_store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void gdn_store4(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  *reinterpret_cast<uint2*>(p) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

constexpr int kThreadsGdn = 1024;
constexpr int kMaxPairs = kMaxNodes * (kMaxNodes + 1) / 2;   // a chain of kMaxNodes

constexpr int kCols = 32;   // output columns (of d_v) per CTA

template <int D>
struct GdnSmem {
  static constexpr int kKPitch = D + 1;                 // padded rows: distinct rows, distinct banks
  static constexpr int kQPitch = D + 4;                 // padded, 16-byte aligned rows (Q, then W)
  static constexpr int kSPitch = kCols + 4;             // 16-byte rows; the k-split reads hit 8 bank groups
  static constexpr int kWPitch = kCols + 4;
  static constexpr int kK = 0;                          // float [m][D+1]
  static constexpr int kQ = kK + ((kMaxNodes * kKPitch + 3) & ~3);   // float [m][D+4], later W [m][kCols+4]
  static constexpr int kS = kQ + kMaxNodes * kQPitch;   // float [D][kCols+4]: this CTA's columns of S_0
  static constexpr int kX = kS + D * kSPitch;           // float [kMaxPairs] (proper-ancestor pairs)
  static constexpr int kY = kX + kMaxPairs;             // float [kMaxPairs] (ancestor-or-self pairs)
  static constexpr int kFloats = kY + kMaxPairs;
  static constexpr int kInts = 4 * kMaxNodes + 2 * (kMaxNodes + 2);   // par, dep, off, lvl, lvl0, fill
  // + gamma, alpha, beta (float [m]) and the pairs' ancestor ids (uint8 [kMaxPairs])
  static constexpr size_t kBytes =
      (size_t)kFloats * 4 + (size_t)kInts * 4 + (size_t)kMaxNodes * 4 * 3 + (size_t)kMaxPairs;
};

template <int D, typename T>
__global__ void __launch_bounds__(kThreadsGdn, 1) gdn_tree_kernel(GdnArgs a) {
  using SM = GdnSmem<D>;
  constexpr int CS = D / kCols;                // CTAs per (sequence, head)
  extern __shared__ float gsm[];
  float* sK = gsm + SM::kK;
  float* sQ = gsm + SM::kQ;
  float* sW = gsm + SM::kQ;                    // over Q once Q is no longer read
  float* sG = gsm + SM::kK;                    // gamma_i Q S_0 [m][kCols+4], over K after step 3
  float* sS = gsm + SM::kS;
  float* sX = gsm + SM::kX;
  float* sY = gsm + SM::kY;
  int* s_par = reinterpret_cast<int*>(gsm + SM::kFloats);
  int* s_dep = s_par + kMaxNodes;      // depth, root = 1
  int* s_off = s_dep + kMaxNodes;      // first entry of node i's ancestor-or-self list
  int* s_lvl = s_off + kMaxNodes;      // nodes sorted by depth
  int* s_lvl0 = s_lvl + kMaxNodes;     // first index in s_lvl of each depth d (d <= m + 1)
  int* s_fill = s_lvl0 + kMaxNodes + 2;
  float* s_gam = reinterpret_cast<float*>(s_fill + kMaxNodes + 2);   // gamma_i
  float* s_alpha = s_gam + kMaxNodes;
  float* s_beta = s_alpha + kMaxNodes;
  uint8_t* s_anc = reinterpret_cast<uint8_t*>(s_beta + kMaxNodes);   // node id of each list entry
  __shared__ int s_maxdep, s_pairs;

  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int cs = blockIdx.x % CS;
  const int bh = blockIdx.x / CS;
  const int b = bh / a.H, h = bh % a.H;
  const int n0 = __ldg(a.cu_nodes + b);
  const int m = __ldg(a.cu_nodes + b + 1) - n0;
  if (!(n0 >= 0 && m >= 0 && m <= a.max_nodes && (long long)n0 + m <= a.node_capacity)) {
    if (threadIdx.x == 0 && cs == 0) set_status(a.status, kStatusInvalidArg);
    return;
  }
  if (m == 0) return;
  const int tid = threadIdx.x;
  const size_t hs = (size_t)a.H * D;   // stride between nodes in q / k / v / o
  const int c0 = cs * kCols;           // this CTA's first column of d_v
  // v is read after the contractions: its rows start towards L2 now
  if (tid < m) ptx::prefetch_l2(static_cast<const T*>(a.v) + (size_t)(n0 + tid) * hs + (size_t)h * D + c0);

  // ---- 1. K, Q, this CTA's columns of S_0 and the tree's scalars; then the bookkeeping
  for (int i = tid; i < m; i += kThreadsGdn) {
    s_par[i] = __ldg(a.parent + n0 + i);
    s_alpha[i] = __ldg(a.alpha + (size_t)(n0 + i) * a.H + h);
    s_beta[i] = __ldg(a.beta + (size_t)(n0 + i) * a.H + h);
  }
  {
    constexpr int D4 = D / 4;
    constexpr int kStage = (kMaxNodes * D4 + kThreadsGdn - 1) / kThreadsGdn;
    constexpr int kS0 = (D * (kCols / 4) + kThreadsGdn - 1) / kThreadsGdn;
    const float* S0 = a.S0 + ((size_t)b * a.H + h) * D * D + c0;
    float4 kv[kStage], qv[kStage], sv[kS0];
#pragma unroll
    for (int t = 0; t < kStage; ++t) {   // every load issued before the first store
      const int e = tid + t * kThreadsGdn;
      if (e < m * D4) {
        const size_t src = (size_t)(n0 + e / D4) * hs + (size_t)h * D + 4 * (e % D4);
        kv[t] = gdn_load4(static_cast<const T*>(a.k) + src);
        qv[t] = gdn_load4(static_cast<const T*>(a.q) + src);
      }
    }
#pragma unroll
    for (int t = 0; t < kS0; ++t) {
      const int e = tid + t * kThreadsGdn;
      if (e < D * (kCols / 4))
        sv[t] = __ldg(reinterpret_cast<const float4*>(S0 + (size_t)(e / (kCols / 4)) * D) + e % (kCols / 4));
    }
#pragma unroll
    for (int t = 0; t < kStage; ++t) {
      const int e = tid + t * kThreadsGdn;
      if (e < m * D4) {
        const int i = e / D4, r = 4 * (e % D4);
        float* kd = sK + i * SM::kKPitch + r;
        kd[0] = kv[t].x; kd[1] = kv[t].y; kd[2] = kv[t].z; kd[3] = kv[t].w;
        *reinterpret_cast<float4*>(sQ + i * SM::kQPitch + r) = qv[t];
      }
    }
#pragma unroll
    for (int t = 0; t < kS0; ++t) {
      const int e = tid + t * kThreadsGdn;
      if (e < D * (kCols / 4))
        *reinterpret_cast<float4*>(sS + (e / (kCols / 4)) * SM::kSPitch + 4 * (e % (kCols / 4))) = sv[t];
    }
  }
  if (tid == 0) s_maxdep = 0;
  for (int d = tid; d < kMaxNodes + 2; d += kThreadsGdn) s_lvl0[d] = 0;
  __syncthreads();
  // depth and gamma: one thread per node walks its own path (bounded: a parent id
  // outside [-1, j) ends the walk; such a tree is rejected below)
  bool ok = true;
  if (tid < m) {
    const int p0 = s_par[tid];
    ok = p0 >= -1 && p0 < tid;
    int j = tid, dep = 0;
    float g = 1.f;
    while (j >= 0 && dep < m) {
      const int pj = s_par[j];
      if (pj < -1 || pj >= j) break;
      g *= s_alpha[j];
      ++dep;
      j = pj;
    }
    s_dep[tid] = dep;
    s_gam[tid] = g;
    atomicMax(&s_maxdep, dep);
    atomicAdd(&s_lvl0[dep], 1);
  }
  if (!__syncthreads_and(ok)) {
    if (tid == 0 && cs == 0) set_status(a.status, kStatusBadTree);
    return;
  }
  // offsets of the ancestor-or-self lists: exclusive scan of the depths (m <= 128, four warps)
  if (tid < kMaxNodes) {
    const int lane = tid & 31, w = tid >> 5;
    const int x = tid < m ? s_dep[tid] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_fill[w] = incl;   // warp totals (s_fill is reused below)
    __syncwarp();
    s_off[tid] = incl - x;              // within the warp; warp offsets added next
  }
  __syncthreads();
  if (tid < kMaxNodes) {
    int wo = 0;
    for (int w = 0; w < (tid >> 5); ++w) wo += s_fill[w];
    s_off[tid] += wo;
    if (tid == m - 1) s_pairs = s_off[tid] + s_dep[tid];
  }
  __syncthreads();
  // level order: counts are in s_lvl0; their exclusive prefix (depths 0..maxdep+1), then
  // each node takes a slot of its level
  if (tid == 0) {
    int run = 0;
    for (int d = 0; d <= s_maxdep + 1; ++d) { const int c = s_lvl0[d]; s_lvl0[d] = run; s_fill[d] = run; run += c; }
  }
  __syncthreads();
  if (tid < m) s_lvl[atomicAdd(&s_fill[s_dep[tid]], 1)] = tid;
  __syncthreads();
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
      ratio *= s_alpha[j];
      j = s_par[j];
    }
    const float* kj = sK + j * SM::kKPitch;
    const float* ki = sK + i * SM::kKPitch;
    const float* qi = sQ + i * SM::kQPitch;
    float kk = 0.f, qk = 0.f;
#pragma unroll 8
    for (int r = 0; r < D; ++r) {
      kk = fmaf(ki[r], kj[r], kk);
      qk = fmaf(qi[r], kj[r], qk);
    }
    sX[pi] = aidx > 0 ? s_beta[i] * ratio * kk : 0.f;
    sY[pi] = ratio * qk;
    s_anc[pi] = (uint8_t)j;
  }

  // ---- 3. K S_0 and Q S_0 on this CTA's columns.  Warp w takes the column half w % 2
  // (16 columns) and the nodes w / 2 + 16 t (t < 4) of each 64-node chunk; lane = kg + 8 cg
  // takes columns 4 cg .. 4 cg + 3 of the half and the rows k = 8 kk + kg of S_0, so its 32
  // partial sums (node slot t, K or Q, 4 columns: index 8 t + 4 kq + c) are reduced over
  // the eight kg lanes by a reduce-scatter that leaves lane kg the sums 4 kg .. 4 kg + 3:
  // node slot kg / 2, K (kg even) or Q (kg odd).
  const int lane = tid & 31, warp = tid >> 5;
  const int kg = lane & 7, cl = 16 * (warp & 1) + 4 * (lane >> 3), rset = warp >> 1;
  const int kq = kg & 1;
  float4 mine[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll
  for (int chunk = 0; chunk < 2; ++chunk) {
    const int base = 64 * chunk;
    if (base >= m) break;   // uniform over the CTA
    float acc[32];
#pragma unroll
    for (int x = 0; x < 32; ++x) acc[x] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < D / 8; ++kk) {
      const int k = 8 * kk + kg;
      const float4 sv = *reinterpret_cast<const float4*>(sS + k * SM::kSPitch + cl);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int i = base + rset + 16 * t;
        if (i < m) {   // uniform over the warp
          const float kv = sK[i * SM::kKPitch + k], qv = sQ[i * SM::kQPitch + k];
          float* ak = acc + 8 * t;
          ak[0] = fmaf(kv, sv.x, ak[0]); ak[1] = fmaf(kv, sv.y, ak[1]);
          ak[2] = fmaf(kv, sv.z, ak[2]); ak[3] = fmaf(kv, sv.w, ak[3]);
          ak[4] = fmaf(qv, sv.x, ak[4]); ak[5] = fmaf(qv, sv.y, ak[5]);
          ak[6] = fmaf(qv, sv.z, ak[6]); ak[7] = fmaf(qv, sv.w, ak[7]);
        }
      }
    }
    // reduce-scatter over kg (lane bits 2, 1, 0 of kg select index bits 4, 3, 2)
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const bool up = (kg & 4) != 0;
      const float give = up ? acc[x] : acc[16 + x], keep = up ? acc[16 + x] : acc[x];
      acc[x] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
    }
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const bool up = (kg & 2) != 0;
      const float give = up ? acc[x] : acc[8 + x], keep = up ? acc[8 + x] : acc[x];
      acc[x] = keep + __shfl_xor_sync(0xffffffffu, give, 2);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const bool up = (kg & 1) != 0;
      const float give = up ? acc[x] : acc[4 + x], keep = up ? acc[4 + x] : acc[x];
      acc[x] = keep + __shfl_xor_sync(0xffffffffu, give, 1);
    }
    mine[chunk] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
  __syncthreads();   // every read of Q is done: the buffer now takes the right-hand side
#pragma unroll
  for (int chunk = 0; chunk < 2; ++chunk) {
    const int i = 64 * chunk + rset + 16 * (kg >> 1);
    if (i < m) {
      const float gm = s_gam[i];
      const float4 x = mine[chunk];
      if (kq == 0) {   // K S_0: the right-hand side beta_i (v_i - gamma_i S_0^T k_i)
        const float4 vv = gdn_load4(static_cast<const T*>(a.v) + (size_t)(n0 + i) * hs + (size_t)h * D + c0 + cl);
        const float bt = s_beta[i];
        *reinterpret_cast<float4*>(sW + i * SM::kWPitch + cl) =
            make_float4(bt * (vv.x - gm * x.x), bt * (vv.y - gm * x.y), bt * (vv.z - gm * x.z), bt * (vv.w - gm * x.w));
      } else {         // Q S_0: gamma_i S_0^T q_i, parked over K (read by nobody after step 3)
        *reinterpret_cast<float4*>(sG + i * SM::kWPitch + cl) = make_float4(gm * x.x, gm * x.y, gm * x.z, gm * x.w);
      }
    }
  }
  __syncthreads();

  // ---- 4. forward substitution, one depth level at a time
  const int maxdep = s_maxdep;
  for (int d = 2; d <= maxdep; ++d) {
    const int l0 = s_lvl0[d], l1 = s_lvl0[d + 1];
    for (int e = tid; e < (l1 - l0) * kCols; e += kThreadsGdn) {
      const int i = s_lvl[l0 + e / kCols], cc = e % kCols;
      const int off = s_off[i], dep = s_dep[i];
      float acc = sW[i * SM::kWPitch + cc];
      for (int t = 1; t < dep; ++t)      // proper ancestors, nearest first
        acc = fmaf(-sX[off + t], sW[s_anc[off + t] * SM::kWPitch + cc], acc);
      sW[i * SM::kWPitch + cc] = acc;
    }
    __syncthreads();
  }

  // ---- 5. outputs: thread -> node tid / 8, columns 4 (tid % 8) .. + 3
  for (int e = tid; e < m * (kCols / 4); e += kThreadsGdn) {
    const int i = e / (kCols / 4), c = 4 * (e % (kCols / 4));
    float4 acc = *reinterpret_cast<const float4*>(sG + i * SM::kWPitch + c);
    const int off = s_off[i], dep = s_dep[i];
    for (int aa = 0; aa < dep; ++aa) {   // ancestors-or-self, self first
      const float y = sY[off + aa];
      const float4 w = *reinterpret_cast<const float4*>(sW + s_anc[off + aa] * SM::kWPitch + c);
      acc.x = fmaf(y, w.x, acc.x); acc.y = fmaf(y, w.y, acc.y);
      acc.z = fmaf(y, w.z, acc.z); acc.w = fmaf(y, w.w, acc.w);
    }
    gdn_store4(static_cast<T*>(a.o) + (size_t)(n0 + i) * hs + (size_t)h * D + c0 + c, acc);
  }
}

template <int D, typename T>
cudaError_t launch_gdn_typed(const GdnArgs& a, cudaStream_t s) {
  constexpr size_t smem = GdnSmem<D>::kBytes;
  cudaError_t e = check_cuda(cudaFuncSetAttribute(gdn_tree_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)smem),
                             "cudaFuncSetAttribute(gdn_tree_kernel)");
  if (e != cudaSuccess) return e;
  return check_cuda(launch_pdl(gdn_tree_kernel<D, T>, dim3((unsigned)(a.B * a.H * (D / kCols))), dim3(kThreadsGdn),
                               smem, s, a),
                    "launch gdn_tree_kernel");
}

}  // namespace

cudaError_t launch_gdn(const GdnArgs& a, cudaStream_t s) {
  if (a.bf16) return a.d == 64 ? launch_gdn_typed<64, __nv_bfloat16>(a, s) : launch_gdn_typed<128, __nv_bfloat16>(a, s);
  return a.d == 64 ? launch_gdn_typed<64, float>(a, s) : launch_gdn_typed<128, float>(a, s);
}

}  // namespace tva
