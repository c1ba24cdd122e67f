// k_sampling.cu - stochastic verification of a draft chain ("Faster decoding", section
// "Modified rejection sampling keeps the target distribution").
//
// Per sequence, with target distributions p (gamma + 1 rows) and draft distributions q
// (gamma rows): draft position i with token x is accepted when p(x) >= q(x) or
// u_i * q(x) < p(x) (u_i * q(x) rounded to fp32 - the test "u < p/q" without a
// division); the first rejection ends the round with a correction token drawn from the
// residual [p - q]_+ at that position, and when all gamma drafts are accepted a bonus
// token is drawn from p at position gamma.  The uniforms are inputs.
//
// Draws are inverse-CDF draws on masses quantised to 2^-40 and summed as 64-bit
// integers (W(v) = floor(w(v) * 2^40), threshold floor(U * Z) with U = floor(u * 2^24)
// / 2^24), so the drawn token does not depend on the order of the sums.  An empty
// residual (Z = 0) falls back to p.
//
// A sequence is served by a cluster of kCluster CTAs.  Every CTA repeats the cheap
// acceptance tests (so all of them take the same decisions from the same inputs and
// reach the cluster barriers together), then sums the quantised masses of the draw (the
// residual after a rejection, else p) over its slice of the vocabulary row with many
// loads in flight; a residual whose quantised total is empty is summed again as p.  The slice is cut into one contiguous
// chunk per warp, and a warp reads its chunk with coalesced 16-byte loads (lane l takes
// every 32nd group of 4 entries), so each load instruction covers 512 contiguous bytes.
// Each CTA pushes its slice sum into the shared memory of every CTA of the cluster
// (distributed shared memory) before a cluster barrier, after which no CTA reads a peer.  In the CTA whose slice holds the threshold the warp sums locate the warp chunk,
// which the whole CTA then cuts into one contiguous piece per thread: a block scan of the
// pieces' sums picks the piece, and its thread walks it entry by entry.
#include <cooperative_groups.h>

#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;
constexpr int kUnroll = 8;

__device__ __forceinline__ unsigned long long quant(float w) {
  // floor(max(w, 0) * 2^40) clamped to 64 bits (what a truncating float to u64 conversion
  // of max(w, 0) * 2^40 gives), from the bits on the integer pipe (that conversion runs on
  // the FP64 unit, which is slow here).  This exact form serves the draw and the rounds
  // that SplitSum below cannot take.  With w = m * 2^(x - 150)
  // (m the 24-bit significand, x the biased exponent), w * 2^40 = (m * 2^40) >> (150 - x),
  // where m * 2^40 fills the 64 bits exactly.  Negatives, -0 and NaN give 0, w < 2^-40
  // (denormals included) gives 0, and w >= 2^24 (+inf included) gives 2^64 - 1.
  const uint32_t b = __float_as_uint(w);
  const unsigned long long m40 = (unsigned long long)((b & 0x7fffffu) | 0x800000u) << 40;
  const unsigned long long q = m40 >> min(63u, 150u - min(150u, b >> 23));
  if (b > 0x7f800000u || b < 0x2b800000u) return 0ull;   // sign bit or NaN; below 2^-40
  return b >= 0x4b800000u ? ~0ull : q;                   // at or above 2^24
}

// The slice sums' form of quant() for w in [0, 2): floor(w * 2^40) = H * 2^23 + L with
// H = floor(w * 2^17) and L = floor(frac(w * 2^17) * 2^23), each < 2^23, found by FMAs
// that round toward zero onto the integer grid of [2^23, 2^24) (w * 2^17 + 2^23 lies in
// it, so its rounding is 2^23 + H; the fraction w * 2^17 - H is exact in fp32, and
// frac * 2^23 + 2^23 rounds to 2^23 + L).  H and L go to 32-bit sums (one 32-entry round
// stays below 2^28); a round that saw any w outside [0, 2) (sign bit or bit 30 set in
// the OR of the entries' bits) is summed again with quant().
struct SplitSum {
  uint32_t h = 0, l = 0;
  __device__ __forceinline__ void add(float w) {
    const float t = __fmaf_rz(w, 0x1p17f, 0x1p23f);                 // 2^23 + H
    const float lo = __fmaf_rz(__fmaf_rn(w, 0x1p17f, __fsub_rn(0x1p23f, t)), 0x1p23f, 0x1p23f);
    h += __float_as_uint(t) - 0x4b000000u;
    l += __float_as_uint(lo) - 0x4b000000u;
  }
  __device__ __forceinline__ unsigned long long value() const {
    return ((unsigned long long)h << 23) + l;
  }
};
constexpr uint32_t kSplitOutside = 0xc0000000u;   // sign bit or exponent >= 128: w outside [0, 2)

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

struct __align__(16) ClusterShared {
  unsigned long long red[kWarps];            // per-warp mass sums of the current pass
  unsigned long long slice[2][kCluster];     // every CTA's slice sum per pass, pushed by its owner
  unsigned long long scan[kWarps];           // the draw's per-warp piece totals
  int first, tok;
};

__global__ void __launch_bounds__(kThreads) sampling_kernel(SamplingArgs a) {
  __shared__ ClusterShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int b = blockIdx.x / kCluster;
  const int g0 = __ldg(a.cu_draft + b);
  const int gamma = __ldg(a.cu_draft + b + 1) - g0;
  const float us = __ldg(a.u_sample + b);
  bool ok = g0 >= 0 && gamma >= 0 && gamma <= a.max_draft && (long long)g0 + gamma <= a.q_rows &&
            (long long)g0 + b + gamma + 1 <= a.p_rows && us >= 0.f && us < 1.f;
  if (threadIdx.x == 0) sh.first = gamma;
  __syncthreads();
  for (int i = threadIdx.x; ok && i < gamma; i += kThreads) {
    const int x = __ldg(a.draft_tok + g0 + i);
    const float u = __ldg(a.u_accept + g0 + i);
    if (x < 0 || x >= a.V || !(u >= 0.f && u < 1.f)) { ok = false; break; }
    const float px = __ldg(a.p + (size_t)(g0 + b + i) * a.V + x);
    const float qx = __ldg(a.q + (size_t)(g0 + i) * a.V + x);
    if (!(qx > 0.f)) { ok = false; break; }   // a draft token is drawn from q
    if (!(px >= qx || __fmul_rn(u, qx) < px)) atomicMin(&sh.first, i);
  }
  // identical in every CTA of the cluster (same inputs), so all leave here together
  ok = __syncthreads_and(ok);
  if (!ok) {
    if (rank == 0 && threadIdx.x == 0) {
      set_status(a.status, kStatusInvalidArg);
      a.accept_len[b] = 0;
      a.out_token[b] = -1;
    }
    return;
  }
  const int k = sh.first;
  const float* prow = a.p + (size_t)(g0 + b + k) * a.V;
  const float* qrow = k < gamma ? a.q + (size_t)(g0 + k) * a.V : nullptr;

  // ---- this CTA's slice, cut into one contiguous chunk per warp (a multiple of 128
  // entries): per-warp sums of the draw's masses
  const int S = ((a.V + kCluster - 1) / kCluster + 3) & ~3;
  const int v0 = min(a.V, rank * S), v1 = min(a.V, v0 + S);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int WC = ((v1 - v0 + kWarps - 1) / kWarps + 127) & ~127;
  const int w0 = min(v1, v0 + warp * WC), w1 = min(v1, w0 + WC);
  // every row starts on a 16-byte boundary
  const bool vec = (a.V & 3) == 0 && ((reinterpret_cast<uintptr_t>(a.p) | reinterpret_cast<uintptr_t>(a.q)) & 15) == 0;
  auto load4 = [&](const float* row, int v, int end, float* out) {
    if (vec && v + 3 < end) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(row + v));
      out[0] = t.x; out[1] = t.y; out[2] = t.z; out[3] = t.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) out[e] = v + e < end ? __ldg(row + v + e) : 0.f;
    }
  };
  // The draw's masses are max(0, p - q) with q read as 0 when qm is null: the residual
  // [p - q]_+ after a rejection, p for the bonus.  A residual whose quantised mass is empty
  // is summed again as p in a second pass (every CTA of the cluster sees the same total,
  // so all of them take it together).
  const float* qm = qrow;
  unsigned long long Z = 0, before = 0, mine = 0;
  for (int pass = 0; pass < 2; ++pass) {
    unsigned long long c = 0;   // this lane's sum
    SplitSum hs;                // this round's split sums
    uint32_t seen = 0;          // OR of this round's masses' bits
    auto accumulate = [&](const float (&pv)[4], const float (&qv)[4]) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = fmaxf(0.f, __fsub_rn(pv[e], qv[e]));
        hs.add(m);
        seen |= __float_as_uint(m);
      }
    };
    auto accumulate_exact = [&](const float (&pv)[4], const float (&qv)[4]) {
#pragma unroll
      for (int e = 0; e < 4; ++e) c += quant(fmaxf(0.f, __fsub_rn(pv[e], qv[e])));
    };
    // end of a round: fold the 32-bit split sums in, or redo the round exactly
    auto close_round = [&](auto&& redo) {
      if (seen & kSplitOutside) redo();
      else c += hs.value();
      hs = SplitSum();
      seen = 0;
    };
    if (vec) {
      // 16-byte rows with V a multiple of 4: every group of 4 starting below w1 is whole,
      // so the loads are plain selects and all of them are issued before the first use
      const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int base = w0; base < w1; base += 128 * kUnroll) {
        float4 p4[kUnroll], q4[kUnroll];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) {
          const int v = base + 128 * j + 4 * lane;
          p4[j] = v < w1 ? __ldg(reinterpret_cast<const float4*>(prow + v)) : zero;
          q4[j] = (v < w1 && qm != nullptr) ? __ldg(reinterpret_cast<const float4*>(qm + v)) : zero;
        }
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) {
          const float pv[4] = {p4[j].x, p4[j].y, p4[j].z, p4[j].w};
          const float qv[4] = {q4[j].x, q4[j].y, q4[j].z, q4[j].w};
          accumulate(pv, qv);
        }
        close_round([&] {
          for (int j = 0; j < kUnroll; ++j) {
            const float pv[4] = {p4[j].x, p4[j].y, p4[j].z, p4[j].w};
            const float qv[4] = {q4[j].x, q4[j].y, q4[j].z, q4[j].w};
            accumulate_exact(pv, qv);
          }
        });
      }
    } else {
      for (int base = w0; base < w1; base += 128 * kUnroll) {
        float pv[kUnroll][4], qv[kUnroll][4];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) {
          const int v = base + 128 * j + 4 * lane;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            pv[j][e] = v + e < w1 ? __ldg(prow + v + e) : 0.f;
            qv[j][e] = (v + e < w1 && qm != nullptr) ? __ldg(qm + v + e) : 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) accumulate(pv[j], qv[j]);
        close_round([&] {
          for (int j = 0; j < kUnroll; ++j) accumulate_exact(pv[j], qv[j]);
        });
      }
    }
    c = warp_sum_u64(c);
    if (lane == 0) sh.red[warp] = c;
    __syncthreads();
    mine = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mine += sh.red[w];
    // push this CTA's slice sum into every CTA of the cluster (itself included), so that
    // after the barrier below nobody reads a peer's shared memory and any CTA may leave
    if (threadIdx.x < kCluster) *cluster.map_shared_rank(&sh.slice[pass][rank], (int)threadIdx.x) = mine;
    if (pass == 0 && threadIdx.x == 0) sh.tok = -1;
    cluster.sync();   // every slice sum of this pass is in every CTA's shared memory
    Z = 0;
    before = 0;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
      const unsigned long long x = sh.slice[pass][r];
      if (r < rank) before += x;
      Z += x;
    }
    if (Z > 0 || qm == nullptr) break;
    qm = nullptr;   // the residual is empty: draw from p
  }
  if (Z == 0) {   // p itself is empty (all masses below 2^-40 or invalid)
    if (rank == 0 && threadIdx.x == 0) {
      set_status(a.status, kStatusInvalidArg);
      a.accept_len[b] = k;
      a.out_token[b] = -1;
    }
    return;
  }
  // U = floor(u * 2^24) for u in [0, 1) from the bits (u = m * 2^(x - 150), so u * 2^24 =
  // m / 2^(126 - x)); -0 reads as 0
  const uint32_t ub = __float_as_uint(us) & 0x7fffffffu, ux = ub >> 23;
  const unsigned long long U = ux < 103u ? 0ull : (unsigned long long)(((ub & 0x7fffffu) | 0x800000u) >> (126u - ux));
  const unsigned long long T = (__umul64hi(U, Z) << 40) | ((U * Z) >> 24);  // floor(U * Z / 2^24)
  if (!(before <= T && T < before + mine)) return;   // another CTA's slice holds the draw

  // ---- the draw inside this slice: the warp chunk holding the threshold (a scan of the
  // warp sums across the lanes of each warp); the whole CTA then cuts that chunk into one
  // piece of E entries per thread, a block scan of the pieces' sums picks the piece, and
  // its thread walks it
  const unsigned long long wl = lane < kWarps ? sh.red[lane] : 0ull;
  const unsigned long long wincl = before + warp_incl_scan_u64(wl, lane);   // through chunk `lane`
  const unsigned hit = __ballot_sync(0xffffffffu, lane < kWarps && T < wincl);
  const int cw = hit != 0u ? __ffs(hit) - 1 : kWarps - 1;   // the first chunk ending past T
  const unsigned long long cexcl = __shfl_sync(0xffffffffu, wincl - wl, cw);
  const int c0 = min(v1, v0 + cw * WC), c1 = min(v1, c0 + WC);
  const int E = (WC + 4 * kThreads - 1) / (4 * kThreads) * 4;   // a multiple of 4
  const int e0 = min(c1, c0 + (int)threadIdx.x * E), e1 = min(c1, e0 + E);
  auto mass = [&](float pv, float qv) { return quant(fmaxf(0.f, __fsub_rn(pv, qv))); };
  unsigned long long ls = 0, m0[4] = {0ull, 0ull, 0ull, 0ull};   // m0: the first group's masses
  for (int v = e0; v < e1; v += 4) {
    float pv[4], qv[4] = {0.f, 0.f, 0.f, 0.f};
    load4(prow, v, e1, pv);   // entries past e1 read as 0, whose mass is 0
    if (qm != nullptr) load4(qm, v, e1, qv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const unsigned long long x = mass(pv[e], qv[e]);
      if (v == e0) m0[e] = x;
      ls += x;
    }
  }
  const unsigned long long incl = warp_incl_scan_u64(ls, lane);
  if (lane == 31) sh.scan[warp] = incl;
  __syncthreads();
  unsigned long long excl = cexcl + incl - ls;   // running sum before this thread's piece
#pragma unroll
  for (int w = 0; w < kWarps; ++w)
    if (w < warp) excl += sh.scan[w];
  if (excl <= T && T < excl + ls) {   // one thread: the pieces cut the chunk's mass
    unsigned long long run = excl;
    int tok = -1;
    for (int v = e0; v < e1 && tok < 0; v += 4) {
      unsigned long long x[4] = {m0[0], m0[1], m0[2], m0[3]};
      if (v != e0) {   // a piece of more than one group reads the later groups again
        float pv[4], qv[4] = {0.f, 0.f, 0.f, 0.f};
        load4(prow, v, e1, pv);
        if (qm != nullptr) load4(qm, v, e1, qv);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = mass(pv[e], qv[e]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (tok < 0 && v + e < e1) {
          run += x[e];
          if (run > T) tok = v + e;
        }
      }
    }
    sh.tok = tok;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.accept_len[b] = k;
    a.out_token[b] = sh.tok;
  }
}

}  // namespace

cudaError_t launch_sampling(const SamplingArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.B * kCluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return check_cuda(cudaLaunchKernelEx(&cfg, sampling_kernel, a), "launch sampling_kernel");
}

}  // namespace tva
