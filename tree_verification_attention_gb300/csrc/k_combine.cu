// k_combine.cu - merge of the attention partials (LongSpec, "Fast Tree Attention",
// Aggregation, and the appendix "Correctness of attention aggregation").
//
// For a query row with partials (O_s, LSE_s), s = 1..S, over disjoint key ranges
// covering the prefix and the tree:
//     LSE = log sum_s exp(LSE_s),     out = sum_s O_s * exp(LSE_s - LSE).
// The page writes the two-part case (cache, specs); the proof only uses that the
// softmax numerator and denominator are sums over the key groups, so it holds for
// any number of groups.  Partials are kept in base 2 (log2-sum-exp2 of base-2
// logits); the natural-log LSE is produced here.  The maximum is subtracted before
// exponentiating (the stable form of the same expression).
//
// One warp per (node, query head) row; each lane owns d/32 consecutive columns, so a
// partial row is one coalesced 16-byte (d=128) or 8-byte (d=64) load per lane.
#include "tva_internal.h"

namespace tva {
namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  constexpr int V = D / 32;
  const Problem& pr = a.pr;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= (long long)pr.node_capacity * pr.Hq) return;
  const int n = (int)(row / pr.Hq);
  const int h = (int)(row % pr.Hq);
  RowLoc R;
  if (!locate_row(pr, n, h, R)) return;
  const long long c = chunk_units(pr, R.T);
  const int u0 = (int)(R.start / c);
  const int u1 = (int)((R.start + R.tiles - 1) / c);

  float M = -INFINITY;
  for (int u = u0; u <= u1; ++u)
    M = fmaxf(M, __ldg(a.lse_part + (size_t)(u + R.q) * pr.RG + R.r));

  float den = 0.f;
  float acc[V];
#pragma unroll
  for (int k = 0; k < V; ++k) acc[k] = 0.f;
#pragma unroll 4
  for (int u = u0; u <= u1; ++u) {
    const size_t prow = (size_t)(u + R.q) * pr.RG + R.r;
    const float w = exp2f(__ldg(a.lse_part + prow) - M);
    den += w;
    const float* op = a.o_part + prow * D + lane * V;
    if constexpr (V == 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(op));
      acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
    } else {
      const float2 v = __ldg(reinterpret_cast<const float2*>(op));
      acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
    }
  }
  const float inv = 1.f / den;
  const size_t orow = ((size_t)n * pr.Hq + h) * D + lane * V;
  if constexpr (sizeof(T) == 4) {
    float* out = static_cast<float*>(a.out) + orow;
#pragma unroll
    for (int k = 0; k < V; ++k) out[k] = acc[k] * inv;
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + orow;
#pragma unroll
    for (int k = 0; k < V; k += 2)
      *reinterpret_cast<__nv_bfloat162*>(out + k) = __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
  }
  if (lane == 0) a.lse[(size_t)n * pr.Hq + h] = (M + log2f(den)) * 0.69314718055994530942f;
}

template <typename T, int D>
cudaError_t launch_typed(const CombineArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.pr.node_capacity * a.pr.Hq;
  const long long blocks = (rows + 7) / 8;
  if (blocks <= 0) return cudaSuccess;
  combine_kernel<T, D><<<(unsigned)blocks, 256, 0, s>>>(a);
  return check_cuda(cudaGetLastError(), "launch combine_kernel");
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 1) return a.pr.d == 64 ? launch_typed<float, 64>(a, s) : launch_typed<float, 128>(a, s);
  return a.pr.d == 64 ? launch_typed<__nv_bfloat16, 64>(a, s) : launch_typed<__nv_bfloat16, 128>(a, s);
}

}  // namespace tva
