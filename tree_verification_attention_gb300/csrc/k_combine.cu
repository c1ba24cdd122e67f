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
// A (node, query head) row is handled by a group of LPR lanes of one warp (LPR = 32,
// 16 or 8, so a warp holds 32 / LPR rows); each lane owns D / LPR consecutive columns,
// read as 16-byte loads.  The kernel is bound by load latency, so a group issues the
// loads of up to NB partial rows (and their LSEs) in one round; LPR and NB are picked
// per launch from the expected number of partials per row, so that the rows of a launch
// fit in one wave of resident warps.  It is launched as a programmatic dependent of the
// partials kernel: the sequence walk that locates a row reads only the caller's cu_*
// arrays and runs before the wait for the partials.
#include <type_traits>

#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

constexpr int kCuCap = 2048;      // ints of shared memory for the staged cu_* arrays
constexpr int kWarpsPerBlock = 2;

template <typename T, int D, int LPR, int NB>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) combine_kernel(CombineArgs a) {
  constexpr int V = D / LPR;  // columns per lane
  constexpr int V4 = V / 4;   // 16-byte loads per lane per partial row
  static_assert(V % 4 == 0, "at least four columns per lane");
  static_assert(NB <= LPR, "a round's weights come from one group of lanes");
  constexpr int RPW = 32 / LPR;  // rows per warp
  __shared__ int cu_buf[kCuCap];
  Problem pr = a.pr;
  stage_cu(pr, cu_buf, kCuCap);  // block-wide; reads caller inputs only
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;               // lane within the row's group
  const int base = lane - sub;              // first lane of the group
  const long long row =
      ((long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * RPW + lane / LPR;
  RowLoc R;
  bool valid = row < (long long)pr.node_capacity * pr.Hq;
  const int n = valid ? (int)(row / pr.Hq) : 0;
  const int h = valid ? (int)(row % pr.Hq) : 0;
  if (valid) valid = locate_row(pr, n, h, R);
  int u0 = 0, np = 0;
  if (valid) {
    const long long c = chunk_units(pr, R.T);
    u0 = (int)(R.start / c);
    np = (int)((R.start + R.tiles - 1) / c) - u0 + 1;
    if ((long long)u0 + np - 1 + R.q >= a.slots) {  // cannot happen for a consistent layout
      if (sub == 0) set_status(a.status, kStatusInvalidArg);
      valid = false;
      np = 0;
    }
  }

  ptx::pdl_wait();  // the partials (and every earlier write) are visible after this
  ptx::pdl_launch_dependents();

  const float* lrow = valid ? a.lse_part + (size_t)(u0 + R.q) * pr.RG + R.r : a.lse_part;
  const float* obase = valid ? a.o_part + ((size_t)(u0 + R.q) * pr.RG + R.r) * D + sub * V : a.o_part;
  const size_t ostride = (size_t)pr.RG * D;
  // every lane of the warp runs the same trip counts (the shuffles span the warp)
  const int np_w = __reduce_max_sync(0xffffffffu, np);

  float4 o[NB][V4];
  float lk = sub < np ? __ldg(lrow + (size_t)sub * pr.RG) : -INFINITY;
#pragma unroll
  for (int j = 0; j < NB; ++j)
#pragma unroll
    for (int v = 0; v < V4; ++v)
      o[j][v] = j < np ? __ldg(reinterpret_cast<const float4*>(obase + (size_t)j * ostride) + v)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = lk;
  for (int k = sub + LPR; k < np_w; k += LPR)
    if (k < np) M = fmaxf(M, __ldg(lrow + (size_t)k * pr.RG));
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float Ms = (M == -INFINITY) ? 0.f : M;

  float den = 0.f;
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int k0 = 0; k0 < np_w; k0 += LPR) {
    if (k0 > 0) lk = k0 + sub < np ? __ldg(lrow + (size_t)(k0 + sub) * pr.RG) : -INFINITY;
    const float wk = k0 + sub < np ? exp2f(lk - Ms) : 0.f;
    den += wk;
    for (int j0 = 0; j0 < LPR && k0 + j0 < np_w; j0 += NB) {
      if (k0 + j0 > 0) {
#pragma unroll
        for (int j = 0; j < NB; ++j)
#pragma unroll
          for (int v = 0; v < V4; ++v)
            o[j][v] = k0 + j0 + j < np
                          ? __ldg(reinterpret_cast<const float4*>(obase + (size_t)(k0 + j0 + j) * ostride) + v)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const float wj = __shfl_sync(0xffffffffu, wk, base + ((j0 + j) % LPR));
        if (j0 + j < LPR && k0 + j0 + j < np) {
#pragma unroll
          for (int v = 0; v < V4; ++v) {
            acc[4 * v + 0] = fmaf(wj, o[j][v].x, acc[4 * v + 0]);
            acc[4 * v + 1] = fmaf(wj, o[j][v].y, acc[4 * v + 1]);
            acc[4 * v + 2] = fmaf(wj, o[j][v].z, acc[4 * v + 2]);
            acc[4 * v + 3] = fmaf(wj, o[j][v].w, acc[4 * v + 3]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if (!valid) return;
  const float inv = 1.f / den;
  const size_t orow = ((size_t)n * pr.Hq + h) * D + sub * V;
  if constexpr (sizeof(T) == 4) {
    float4* out = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow);
#pragma unroll
    for (int v = 0; v < V4; ++v)
      out[v] = make_float4(acc[4 * v] * inv, acc[4 * v + 1] * inv, acc[4 * v + 2] * inv, acc[4 * v + 3] * inv);
  } else {
    uint2* out = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow);
#pragma unroll
    for (int v = 0; v < V4; ++v) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[4 * v] * inv, acc[4 * v + 1] * inv);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[4 * v + 2] * inv, acc[4 * v + 3] * inv);
      out[v] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
  if (sub == 0) a.lse[(size_t)n * pr.Hq + h] = (Ms + log2f(den)) * 0.69314718055994530942f;
}

template <typename T, int D, int LPR, int NB>
cudaError_t launch_typed(const CombineArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.pr.node_capacity * a.pr.Hq;
  const long long warps = (rows + (32 / LPR) - 1) / (32 / LPR);
  const long long blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks <= 0) return cudaSuccess;
  return check_cuda(launch_pdl(combine_kernel<T, D, LPR, NB>, dim3((unsigned)blocks),
                               dim3(32 * kWarpsPerBlock), 0, s, a),
                    "launch combine_kernel");
}

// Partials per row when every sequence is at its stated maximum size: the units of
// one row group (prefix tiles + the tree tile) spread over ceil(tiles / chunk) + 1
// workers at most.  Smaller sequences shrink the chunk and can raise the count; the
// kernel loops over any number, this only sizes its first round of loads.
int expected_partials(const Problem& pr) {
  const long long tiles = (pr.max_prefix + kKeyTile - 1) / kKeyTile + 1;
  const long long groups = ((long long)pr.max_nodes * pr.G + pr.RG - 1) / pr.RG;
  const long long T = (long long)pr.B * pr.Hkv * groups * tiles;
  const long long c = T > 0 ? (T + pr.U - 1) / pr.U : 1;
  return (int)((tiles + c - 1) / c + 1);
}

template <typename T>
cudaError_t launch_dtype(const CombineArgs& a, cudaStream_t s) {
  const int np = expected_partials(a.pr);
  if (a.pr.d == 64) {
    if (np <= 8) return launch_typed<T, 64, 8, 8>(a, s);
    return launch_typed<T, 64, 16, 16>(a, s);
  }
  if (np <= 6) return launch_typed<T, 128, 8, 6>(a, s);
  if (np <= 12) return launch_typed<T, 128, 16, 12>(a, s);
  return launch_typed<T, 128, 32, 24>(a, s);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 1) return launch_dtype<float>(a, s);
  return launch_dtype<__nv_bfloat16>(a, s);
}

}  // namespace tva
