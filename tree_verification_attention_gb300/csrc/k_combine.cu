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
// A warp takes one 32-row block of one row group and CG of its column groups (4
// columns each); lane t owns row t of the block.  The kernel is bound by load latency,
// so a warp issues the loads of up to NB partials at once; CG and NB are picked per
// launch from the expected number of partials per row group.  It is launched as a
// programmatic dependent of the partials kernel: the walk that locates the row group
// reads only the caller's cu_* arrays and runs before the wait for the partials.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

// Writes one merged row piece: out = acc / den (CG column groups from cs * CG) in T, and
// (for the first column set) lse = (Ms + log2 den) * ln 2 for row r (node `node`) of the
// row group R.
template <typename T, int D, int CG>
__device__ __forceinline__ void store_merged(const Problem& pr, const GroupLoc& R, int node, int r, int cs,
                                             const float4 (&acc)[CG], float den, float Ms, void* out_v,
                                             float* lse_out, int32_t* status) {
  const float inv = 1.f / den;
  const int head = R.g * pr.G + r % pr.G;
  if (!TVA_CHECK(R.s.n0 + node < pr.node_capacity && head < pr.Hq && (cs + 1) * CG * 4 <= D, status)) return;
  const size_t orow = ((size_t)(R.s.n0 + node) * pr.Hq + head) * D + (size_t)cs * CG * 4;
  if constexpr (sizeof(T) == 4) {
    float4* out = reinterpret_cast<float4*>(static_cast<float*>(out_v) + orow);
#pragma unroll
    for (int g = 0; g < CG; ++g)
      out[g] = make_float4(acc[g].x * inv, acc[g].y * inv, acc[g].z * inv, acc[g].w * inv);
  } else {
    uint2* out = reinterpret_cast<uint2*>(static_cast<T*>(out_v) + orow);
#pragma unroll
    for (int g = 0; g < CG; ++g) {
      uint32_t lo, hi;
      if constexpr (std::is_same<T, __half>::value) {
        const __half2 l = __floats2half2_rn(acc[g].x * inv, acc[g].y * inv);
        const __half2 h = __floats2half2_rn(acc[g].z * inv, acc[g].w * inv);
        lo = *reinterpret_cast<const uint32_t*>(&l);
        hi = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __nv_bfloat162 l = __floats2bfloat162_rn(acc[g].x * inv, acc[g].y * inv);
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[g].z * inv, acc[g].w * inv);
        lo = *reinterpret_cast<const uint32_t*>(&l);
        hi = *reinterpret_cast<const uint32_t*>(&h);
      }
      out[g] = make_uint2(lo, hi);
    }
  }
  if (cs == 0) lse_out[(size_t)(R.s.n0 + node) * pr.Hq + head] = (Ms + log2f(den)) * 0.69314718055994530942f;
}

// One warp merges one 32-row block (rb) of row group qg for CG of its column groups (4
// columns each, starting at column group cs * CG); lane t owns padded row rb * 32 + t.
// The np partials of the row group are in slots slot0 .. slot0 + np - 1 (blocked layout
// of tva_common.cuh).  Every row of a row group has the same partials (the same workers
// covered it), so all lanes run the same loops and no shuffles are needed; the loads of
// up to NB partials are issued in one round.  Lanes whose row is padding return without
// touching memory; nothing here synchronises the warp.
template <typename T, int D, int CG, int NB>
__device__ __forceinline__ void merge_rows(const Problem& pr, const float* o_part, const float* lse_part,
                                           const GroupLoc& R, size_t slot0, int np, int rb, int cs, int lane,
                                           void* out_v, float* lse_out, int32_t* status) {
  const int MT = mtile_rows(pr.G);
  const int W = pr.RG / MT;
  const int RGP = W * 128;
  const int pp = rb * 32 + lane;                // padded row of this lane
  const int mt = pp / 128, r = pp % 128;
  const int node = (R.mp * W + mt) * (MT / pr.G) + r / pr.G;  // local node id
  if (!(r < MT && node < R.s.m)) return;

  const float* lse_p = lse_part + slot0 * RGP + pp;
  const float* o_p = o_part + o_part_offset(slot0, pp, cs * CG, RGP, D);
  const size_t lstride = (size_t)RGP, ostride = (size_t)RGP * D;

  // Online over rounds of NB partials: each round's LSE and O loads are issued together
  // (no load waits on another), then the running maximum moves to the round's and the
  // sums are rescaled - the same result as one maximum over all partials, with
  // ceil(np / NB) dependent memory rounds.
  float M = -INFINITY, den = 0.f;
  float4 acc[CG];
#pragma unroll
  for (int g = 0; g < CG; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < np; k0 += NB) {
    float lk[NB];
    float4 o[NB][CG];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      lk[j] = k0 + j < np ? __ldcg(lse_p + (k0 + j) * lstride) : -INFINITY;
#pragma unroll
      for (int g = 0; g < CG; ++g)
        o[j][g] = k0 + j < np ? __ldcg(reinterpret_cast<const float4*>(o_p + (k0 + j) * ostride + g * 128))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mr = M;
#pragma unroll
    for (int j = 0; j < NB; ++j) Mr = fmaxf(Mr, lk[j]);
    const float Ms = (Mr == -INFINITY) ? 0.f : Mr;
    const float sc = (M == -INFINITY) ? 0.f : exp2f(M - Ms);  // nothing accumulated yet: 0
    den *= sc;
#pragma unroll
    for (int g = 0; g < CG; ++g) {
      acc[g].x *= sc; acc[g].y *= sc; acc[g].z *= sc; acc[g].w *= sc;
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const float wj = exp2f(lk[j] - Ms);  // exp2(-inf) = 0 for the padding entries
      den += wj;
#pragma unroll
      for (int g = 0; g < CG; ++g) {
        acc[g].x = fmaf(wj, o[j][g].x, acc[g].x);
        acc[g].y = fmaf(wj, o[j][g].y, acc[g].y);
        acc[g].z = fmaf(wj, o[j][g].z, acc[g].z);
        acc[g].w = fmaf(wj, o[j][g].w, acc[g].w);
      }
    }
    M = Mr;
  }
  const float Ms = (M == -INFINITY) ? 0.f : M;
  store_merged<T, D, CG>(pr, R, node, r, cs, acc, den, Ms, out_v, lse_out, status);
}


constexpr int kCuCap = 2048;      // ints of shared memory for the staged cu_* arrays

template <typename T, int D, int CG, int NB, int WPB>
__global__ void __launch_bounds__(32 * WPB) combine_kernel(CombineArgs a) {
  constexpr int NCG = D / 4 / CG;  // column-group sets per row block
  __shared__ int cu_buf[kCuCap];
  Problem pr = a.pr;
  stage_cu(pr, cu_buf, kCuCap);  // block-wide; reads caller inputs only
  const int lane = threadIdx.x & 31;
  const int MT = mtile_rows(pr.G);
  const int W = pr.RG / MT;
  const int RGP = W * 128;
  // Work items are dealt to the blocks round-robin (item = warp * blocks + block), so
  // that every SM ends up with the same number of items to within one per block.
  const long long wid = (long long)(threadIdx.x >> 5) * gridDim.x + blockIdx.x;
  const long long per_group = (long long)(RGP / 32) * NCG;
  const long long qg = wid / per_group;
  const int rb = (int)(wid % per_group) / NCG;  // 32-row block
  const int cs = (int)(wid % per_group) % NCG;  // column-group set
  const GroupLoc R = locate_group(pr, qg);      // uniform over the warp
  if (!R.found) return;
  // the workers that cover the group, and the slot of the first one's partial (the
  // group's partials are in consecutive slots; see partial_slot)
  long long slot0;
  int np;
  if (pr.share == 0 && pr.align > 0) {  // the group's own workers, the first min(align, tiles) busy
    const int u0 = (int)qg * pr.align;
    np = R.tiles < pr.align ? R.tiles : pr.align;
    slot0 = (long long)u0 + qg;
  } else if (pr.share == 0) {
    const long long c = chunk_units(pr, R.T);
    const int u0 = (int)(R.start / c);
    np = (int)((R.start + R.tiles - 1) / c) - u0 + 1;
    slot0 = (long long)u0 + qg;
  } else {
    const long long cc = share_columns_per_team(pr, R.tiles);
    const long long c0 = (long long)R.g * R.tiles;
    const int k0 = (int)(c0 / cc);
    np = (int)((c0 + R.tiles - 1) / cc) - k0 + 1;
    slot0 = (long long)R.mp * (share_teams(pr) + pr.Hkv) + k0 + R.g;
  }
  if (slot0 + np - 1 >= a.slots) {  // cannot happen for a consistent layout
    if (lane == 0) set_status(a.status, kStatusInvalidArg);
    return;
  }
  ptx::pdl_wait();  // the partials (and every earlier write) are visible after this
  ptx::pdl_launch_dependents();
  merge_rows<T, D, CG, NB>(pr, a.o_part, a.lse_part, R, (size_t)slot0, np, rb, cs, lane, a.out, a.lse,
                           a.status);
}

// Row groups the layout provides for (every sequence at its stated maximum size).
long long max_row_groups(const Problem& pr) {
  return (long long)pr.B * pr.Hkv * (((long long)pr.max_nodes * pr.G + pr.RG - 1) / pr.RG);
}

constexpr int kMaxDevices = 64;

// SMs of the current device (cached per device); 0 if it cannot be read.
int sm_count(int* dev_out) {
  // Filled on first use per device; concurrent first calls store the same value.
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  *dev_out = dev;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 0;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// WPB warps per block: as many as keep the registers of two blocks per SM or more.  One
// item per warp; when the items fill less than one wave of blocks, the grid is widened
// to a full wave (never past one block per item) and the round-robin deal spreads the
// items evenly over it.
template <typename T, int D, int CG, int NB>
cudaError_t launch_typed(const CombineArgs& a, cudaStream_t s) {
  constexpr int WPB = CG == 1 ? 8 : 4;
  const int RGP = padded_group_rows(a.pr.RG, a.pr.G);
  const long long warps = max_row_groups(a.pr) * (RGP / 32) * (D / 4 / CG);
  static std::atomic<int> per_sm[kMaxDevices];  // resident blocks per SM, per device (0: not yet known)
  int dev = 0;
  const int sms = sm_count(&dev);
  int resident = sms > 0 ? per_sm[dev].load(std::memory_order_relaxed) : 0;
  if (sms > 0 && resident == 0) {
    int v = 0;
    resident = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, combine_kernel<T, D, CG, NB, WPB>, 32 * WPB, 0) ==
                           cudaSuccess && v > 0 ? v : 1;
    per_sm[dev].store(resident, std::memory_order_relaxed);
  }
  const long long wave = sms > 0 ? (long long)sms * resident : 0;
  long long blocks = (warps + WPB - 1) / WPB;
  if (blocks < wave) blocks = std::min<long long>(wave, warps);
  if (blocks <= 0) return cudaSuccess;
  return check_cuda(launch_pdl(combine_kernel<T, D, CG, NB, WPB>, dim3((unsigned)blocks), dim3(32 * WPB), 0,
                               s, a),
                    "launch combine_kernel");
}

// Partials per row group when every sequence is at its stated maximum size: the units
// of one row group (prefix tiles + the tree tile) spread over ceil(tiles / chunk) + 1
// workers at most (stream-K), or over the teams that cover its KV head (shared mode).  Smaller sequences shrink the chunk and can raise the count; the
// kernel loops over any number, this only sizes its first round of loads.
int expected_partials(const Problem& pr) {
  const long long tiles = (pr.max_prefix + kKeyTile - 1) / kKeyTile + 1;
  if (pr.share == 0 && pr.align > 0) return (int)std::min<long long>(pr.align, tiles);
  if (pr.share > 0) {  // a head's columns spread over ceil(tiles / columns per team) + 1 teams
    const long long Q = pr.U / pr.share, C = (long long)pr.Hkv * tiles;
    const long long cc = Q > 0 ? (C + Q - 1) / Q : 1;
    return (int)((tiles + cc - 1) / cc + 1);
  }
  const long long T = max_row_groups(pr) * tiles;
  const long long c = T > 0 ? (T + pr.U - 1) / pr.U : 1;
  return (int)((tiles + c - 1) / c + 1);
}

template <typename T, int D>
cudaError_t launch_d(const CombineArgs& a, cudaStream_t s) {
  const int np = expected_partials(a.pr);
  if (np <= 6) return launch_typed<T, D, 4, 6>(a, s);
  if (np <= 12) return launch_typed<T, D, 2, 12>(a, s);
  return launch_typed<T, D, 2, 20>(a, s);
}

template <typename T>
cudaError_t launch_dtype(const CombineArgs& a, cudaStream_t s) {
  return a.pr.d == 64 ? launch_d<T, 64>(a, s) : launch_d<T, 128>(a, s);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 1) return launch_dtype<float>(a, s);
  if (dtype == 2) return launch_dtype<__half>(a, s);
  return launch_dtype<__nv_bfloat16>(a, s);
}

}  // namespace tva
