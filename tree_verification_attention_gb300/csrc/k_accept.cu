// k_accept.cu - greedy longest accepted path ("Faster decoding", greedy
// verification contract; candidates are root-to-node paths of the draft tree).
//
// One warp per sequence (m <= 128 nodes, 4 per lane).  Node i is matched when
// draft_tok[i] equals the target's greedy token after its parent (slot parent[i]+1,
// slot 0 being the prefix end).  "Accepted" (matched with every ancestor matched) and
// the depth are found together by pointer jumping: after round r each node holds the
// AND of the match flags and the count of the 2^r nodes above it (itself included)
// and a pointer 2^r levels up, so 7 rounds cover any depth <= 128.  A warp max over
// the key (depth << 8 | 255 - i) picks the deepest accepted node, ties to the smaller
// id; one lane then writes its root-first path.
#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) accept_kernel(AcceptArgs a) {
  __shared__ int s_par[kWarps][kMaxNodes];
  __shared__ int s_ok[kWarps][kMaxNodes];
  __shared__ int s_dep[kWarps][kMaxNodes];
  __shared__ int s_anc[kWarps][kMaxNodes];
  __shared__ int s_slot[kWarps][kMaxNodes + 1];
  {
    // Before waiting for the preceding kernel: pull this block's share of the input
    // arrays into L2.  A prefetch is only a hint - no value is read here, and the loads
    // after the wait see whatever the preceding kernels wrote - so it only shortens the
    // dependent rounds of loads below.
    const long long N = a.node_capacity;
    const long long lo = N * blockIdx.x / gridDim.x, hi = N * (blockIdx.x + 1) / gridDim.x;
    for (long long i = lo + (long long)threadIdx.x * 32; i < hi; i += (long long)blockDim.x * 32) {
      ptx::prefetch_l2(a.parent + i);
      ptx::prefetch_l2(a.draft_tok + i);
      ptx::prefetch_l2(a.target_argmax + i + (long long)blockIdx.x * kWarps);
    }
    if (threadIdx.x == 0) ptx::prefetch_l2(a.cu_nodes + (long long)blockIdx.x * kWarps);
  }
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarps + w;
  if (b >= a.B) return;  // whole warp leaves; no block-wide barrier follows
  const int n0 = __ldg(a.cu_nodes + b);
  const int m = __ldg(a.cu_nodes + b + 1) - n0;
  if (m < 0 || m > kMaxNodes || n0 < 0 || n0 + m > a.node_capacity) {
    if (lane == 0) {
      set_status(a.status, kStatusInvalidArg);
      a.accept_len[b] = 0;
      a.next_token[b] = -1;
    }
    return;
  }
  // All of the sequence's inputs are fetched in one round of global loads: parents
  // and draft tokens into registers, the m+1 target slots into shared memory.
  const int32_t* slot = a.target_argmax + n0 + b;
  int par[kMaxNodes / 32], tok[kMaxNodes / 32];
#pragma unroll
  for (int k = 0; k < kMaxNodes / 32; ++k) {
    const int i = lane + 32 * k;
    par[k] = i < m ? __ldg(a.parent + n0 + i) : -1;
    tok[k] = i < m ? __ldg(a.draft_tok + n0 + i) : 0;
    if (i <= m) s_slot[w][i] = __ldg(slot + i);
  }
  if (lane == 0 && m == kMaxNodes) s_slot[w][kMaxNodes] = __ldg(slot + kMaxNodes);
  __syncwarp();
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kMaxNodes / 32; ++k) {
    const int i = lane + 32 * k;
    if (i < m) {
      const int p = par[k];
      const bool pok = p >= -1 && p < i;
      bad |= !pok;
      s_par[w][i] = pok ? p : -1;
      s_ok[w][i] = pok && tok[k] == s_slot[w][p + 1];
      s_dep[w][i] = 1;
      s_anc[w][i] = pok ? p : -1;
    }
  }
  if (__any_sync(0xffffffffu, bad)) {
#pragma unroll
    for (int k = 0; k < kMaxNodes / 32; ++k) {
      const int i = lane + 32 * k;
      if (i < m) a.accept_path[n0 + i] = -1;
    }
    if (lane == 0) {
      set_status(a.status, kStatusBadTree);
      a.accept_len[b] = 0;
      a.next_token[b] = s_slot[w][0];
    }
    return;
  }
  __syncwarp();
  for (int round = 0; round < 8; ++round) {
    int ok_n[kMaxNodes / 32], dep_n[kMaxNodes / 32], anc_n[kMaxNodes / 32];
    bool any = false;
#pragma unroll
    for (int k = 0; k < kMaxNodes / 32; ++k) {
      const int i = lane + 32 * k;
      ok_n[k] = 0; dep_n[k] = 0; anc_n[k] = -1;
      if (i < m) {
        const int up = s_anc[w][i];
        ok_n[k] = s_ok[w][i];
        dep_n[k] = s_dep[w][i];
        anc_n[k] = up;
        if (up >= 0) {
          ok_n[k] &= s_ok[w][up];
          dep_n[k] += s_dep[w][up];
          anc_n[k] = s_anc[w][up];
          any = true;
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < kMaxNodes / 32; ++k) {
      const int i = lane + 32 * k;
      if (i < m) { s_ok[w][i] = ok_n[k]; s_dep[w][i] = dep_n[k]; s_anc[w][i] = anc_n[k]; }
    }
    __syncwarp();
    if (!__any_sync(0xffffffffu, any)) break;
  }
  int key = -1;
#pragma unroll
  for (int k = 0; k < kMaxNodes / 32; ++k) {
    const int i = lane + 32 * k;
    if (i < m && s_ok[w][i]) key = max(key, (s_dep[w][i] << 8) | (255 - i));
  }
  key = __reduce_max_sync(0xffffffffu, key);
  const int best = key < 0 ? -1 : 255 - (key & 255);
  const int depth = key < 0 ? 0 : (key >> 8);
#pragma unroll
  for (int k = 0; k < kMaxNodes / 32; ++k) {
    const int i = lane + 32 * k;
    if (i < m && i >= depth) a.accept_path[n0 + i] = -1;
  }
  if (lane == 0) {
    int j = best;
    for (int pos = depth - 1; pos >= 0; --pos) {
      if (!TVA_CHECK(pos < m && j >= 0 && j < m, a.status)) break;
      a.accept_path[n0 + pos] = j;
      j = s_par[w][j];
    }
    a.accept_len[b] = depth;
    a.next_token[b] = s_slot[w][best + 1];
  }
}

}  // namespace

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
  if (a.B <= 0) return cudaSuccess;
  return check_cuda(launch_pdl(accept_kernel, dim3((a.B + kWarps - 1) / kWarps), dim3(kWarps * 32), 0, s, a),
                    "launch accept_kernel");
}

}  // namespace tva
