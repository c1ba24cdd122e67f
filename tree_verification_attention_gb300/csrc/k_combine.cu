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
// partial row is one coalesced 16-byte (d=128) or 8-byte (d=64) load per lane.  The
// kernel is bound by the latency of those loads, so a warp issues up to 16 of them
// before consuming any.  It is launched as a programmatic dependent of the partials
// kernel: its blocks become resident early and wait for the partials to be complete.
#include <type_traits>

#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

constexpr int kBatch = 16;  // partial rows in flight per warp
constexpr int kCuCap = 2048;  // ints of shared memory for the staged cu_* arrays

template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  constexpr int V = D / 32;
  using Vec = typename std::conditional<V == 4, float4, float2>::type;
  ptx::pdl_wait();  // partials (and every earlier write) are visible after this
  ptx::pdl_launch_dependents();
  __shared__ int cu_buf[kCuCap];
  Problem pr = a.pr;
  stage_cu(pr, cu_buf, kCuCap);
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

  // Lane k (mod 32) holds the LSE of partial u0 + k.  The first kBatch partial rows
  // of O are requested together with the LSEs (they do not depend on the maximum), so
  // a row with up to kBatch partials costs one round of loads.
  const int np = u1 - u0 + 1;
  if ((long long)u1 + R.q >= a.slots) {  // cannot happen for a consistent layout
    if (lane == 0) set_status(a.status, kStatusInvalidArg);
    return;
  }
  const float* lrow = a.lse_part + (size_t)(u0 + R.q) * pr.RG + R.r;
  const float* obase = a.o_part + ((size_t)(u0 + R.q) * pr.RG + R.r) * D + lane * V;
  const size_t ostride = (size_t)pr.RG * D;
  auto load_o = [&](int k) -> float4 {
    const float* op = obase + (size_t)k * ostride;
    if constexpr (V == 4) {
      return __ldg(reinterpret_cast<const float4*>(op));
    } else {
      const float2 t = __ldg(reinterpret_cast<const float2*>(op));
      return make_float4(t.x, t.y, 0.f, 0.f);
    }
  };
  float lk = lane < np ? __ldg(lrow + (size_t)lane * pr.RG) : -INFINITY;
  float4 v[kBatch];
  const int cnt0 = min(kBatch, np);
#pragma unroll
  for (int j = 0; j < kBatch; ++j) v[j] = j < cnt0 ? load_o(j) : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = lk;
  for (int k = lane + 32; k < np; k += 32) M = fmaxf(M, __ldg(lrow + (size_t)k * pr.RG));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float den = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < np; k0 += 32) {
    if (k0 > 0) lk = k0 + lane < np ? __ldg(lrow + (size_t)(k0 + lane) * pr.RG) : -INFINITY;
    const float wk = k0 + lane < np ? exp2f(lk - M) : 0.f;
    den += wk;
    for (int j0 = 0; j0 < 32 && k0 + j0 < np; j0 += kBatch) {
      const int cnt = min(kBatch, np - k0 - j0);
      if (k0 + j0 > 0) {
#pragma unroll
        for (int j = 0; j < kBatch; ++j) v[j] = j < cnt ? load_o(k0 + j0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float wj = __shfl_sync(0xffffffffu, wk, j0 + j);
        if (j < cnt) {
          acc[0] = fmaf(wj, v[j].x, acc[0]);
          acc[1] = fmaf(wj, v[j].y, acc[1]);
          acc[2] = fmaf(wj, v[j].z, acc[2]);
          acc[3] = fmaf(wj, v[j].w, acc[3]);
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
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
  return check_cuda(launch_pdl(combine_kernel<T, D>, dim3((unsigned)blocks), dim3(256), 0, s, a),
                    "launch combine_kernel");
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 1) return a.pr.d == 64 ? launch_typed<float, 64>(a, s) : launch_typed<float, 128>(a, s);
  return a.pr.d == 64 ? launch_typed<__nv_bfloat16, 64>(a, s) : launch_typed<__nv_bfloat16, 128>(a, s);
}

}  // namespace tva
