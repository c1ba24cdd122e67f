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
// One CTA per sequence.  The draw reads the row once, coalesced: warp w sums the
// quantised masses of its contiguous segment, a scan over the warp sums finds the
// segment holding the threshold, and that warp alone rescans its segment 32 entries at
// a time.
#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr float kQScale = 1099511627776.0f;  // 2^40
constexpr float kUScale = 16777216.0f;       // 2^24

__device__ __forceinline__ unsigned long long quant(float w) {
  // w * 2^40 is exact (a power-of-two scale); truncation is the floor for w >= 0
  return __float2ull_rz(fmaxf(w, 0.f) * kQScale);
}

// mass of entry v of the row being drawn from
__device__ __forceinline__ float mass(const float* prow, const float* qrow, int v) {
  const float pv = __ldg(prow + v);
  return qrow != nullptr ? fmaxf(0.f, __fsub_rn(pv, __ldg(qrow + v))) : pv;
}

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

// Inverse-CDF draw over row entries [0, V) with uniform u (block-wide; every thread
// calls it; returns the token in every thread, or -1 when the masses sum to zero).
__device__ int draw(const float* prow, const float* qrow, int V, float u, unsigned long long* s_wsum,
                    int* s_tok) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (V + kWarps - 1) / kWarps;
  const int v0 = min(V, warp * seg), v1 = min(V, v0 + seg);
  unsigned long long s = 0;
  for (int v = v0 + lane; v < v1; v += 32) s += quant(mass(prow, qrow, v));
  s = warp_sum_u64(s);
  if (lane == 0) s_wsum[warp] = s;
  if (threadIdx.x == 0) *s_tok = -1;
  __syncthreads();
  unsigned long long Z = 0, before = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += s_wsum[w];
    Z += s_wsum[w];
  }
  if (Z > 0) {
    const unsigned long long U = __float2ull_rz(u * kUScale);                 // < 2^24
    const unsigned long long T = (__umul64hi(U, Z) << 40) | ((U * Z) >> 24);  // floor(U * Z / 2^24)
    if (before <= T && T < before + s_wsum[warp]) {   // this warp's segment holds the draw
      unsigned long long run = before;
      for (int base = v0; base < v1; base += 32) {
        const int v = base + lane;
        const unsigned long long x = v < v1 ? quant(mass(prow, qrow, v)) : 0ull;
        const unsigned long long incl = run + warp_incl_scan_u64(x, lane);
        const unsigned hit = __ballot_sync(0xffffffffu, incl > T);
        if (hit != 0u) {
          if (lane == 0) *s_tok = base + __ffs(hit) - 1;
          break;
        }
        run = __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  __syncthreads();
  const int tok = *s_tok;
  __syncthreads();  // s_wsum / s_tok are reused by a second draw
  return tok;
}

__global__ void __launch_bounds__(kThreads) sampling_kernel(SamplingArgs a) {
  __shared__ unsigned long long s_wsum[kWarps];
  __shared__ int s_first, s_tok;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int b = blockIdx.x;
  const int g0 = __ldg(a.cu_draft + b);
  const int gamma = __ldg(a.cu_draft + b + 1) - g0;
  const float us = __ldg(a.u_sample + b);
  bool ok = g0 >= 0 && gamma >= 0 && gamma <= a.max_draft && (long long)g0 + gamma <= a.q_rows &&
            (long long)g0 + b + gamma + 1 <= a.p_rows && us >= 0.f && us < 1.f;
  if (threadIdx.x == 0) s_first = gamma;
  __syncthreads();
  for (int i = threadIdx.x; ok && i < gamma; i += kThreads) {
    const int x = __ldg(a.draft_tok + g0 + i);
    const float u = __ldg(a.u_accept + g0 + i);
    if (x < 0 || x >= a.V || !(u >= 0.f && u < 1.f)) { ok = false; break; }
    const float px = __ldg(a.p + (size_t)(g0 + b + i) * a.V + x);
    const float qx = __ldg(a.q + (size_t)(g0 + i) * a.V + x);
    if (!(qx > 0.f)) { ok = false; break; }   // a draft token is drawn from q
    if (!(px >= qx || __fmul_rn(u, qx) < px)) atomicMin(&s_first, i);
  }
  ok = __syncthreads_and(ok);
  if (!ok) {
    if (threadIdx.x == 0) {
      set_status(a.status, kStatusInvalidArg);
      a.accept_len[b] = 0;
      a.out_token[b] = -1;
    }
    return;
  }
  const int k = s_first;
  const float* prow = a.p + (size_t)(g0 + b + k) * a.V;
  const float* qrow = k < gamma ? a.q + (size_t)(g0 + k) * a.V : nullptr;
  int tok = draw(prow, qrow, a.V, us, s_wsum, &s_tok);
  if (tok < 0 && qrow != nullptr) tok = draw(prow, nullptr, a.V, us, s_wsum, &s_tok);
  if (threadIdx.x == 0) {
    a.accept_len[b] = k;
    a.out_token[b] = tok;
    if (tok < 0) set_status(a.status, kStatusInvalidArg);   // p itself sums to zero
  }
}

}  // namespace

cudaError_t launch_sampling(const SamplingArgs& a, cudaStream_t s) {
  return check_cuda(launch_pdl(sampling_kernel, dim3((unsigned)a.B), dim3(kThreads), 0, s, a),
                    "launch sampling_kernel");
}

}  // namespace tva
