// k_commit.cu - commit of the accepted path's K/V into the cache ("Faster decoding",
// "The scheduler must plan speculative work": after verification only the target KV of
// the accepted draft prefix is committed; rejected branches are released, i.e. their
// rows are simply not copied).
//
// Block (b, y) copies rows j in [y * kRowsPerBlock, (y + 1) * kRowsPerBlock) of sequence
// b's accepted path: tree_k / tree_v row cu_nodes[b] + accept_path[cu_nodes[b] + j]
// goes to cache row dst_row[b] + j.  A node's row is Hkv * d contiguous elements in both
// layouts, so a row is one contiguous run of bytes, copied in 16-byte vectors.  Before
// copying, every block checks the whole sequence (its node range, the path length and
// every path id, the destination range): a sequence that fails is left untouched and
// TVA_ERR_INVALID_ARG is recorded.  The kernel reads the acceptance kernel's outputs,
// so it waits for its predecessor (programmatic dependent launch) before anything else.
#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

constexpr int kThreads = 128;
constexpr int kRowsPerBlock = 8;

__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a) {
  __shared__ int s_path[kMaxNodes];
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int b = blockIdx.x, y = blockIdx.y;
  const int n0 = __ldg(a.cu_nodes + b);
  const int m = __ldg(a.cu_nodes + b + 1) - n0;
  const int L = __ldg(a.accept_len + b);
  const long long dst = __ldg(a.dst_row + b);
  bool ok = n0 >= 0 && m >= 0 && m <= a.max_nodes && (long long)n0 + m <= a.node_capacity && L >= 0 && L <= m &&
            dst >= 0 && dst + L <= a.kv_capacity;
  // every path id of the sequence, not only this block's rows
  for (int j = threadIdx.x; ok && j < L; j += kThreads) {
    const int p = __ldg(a.accept_path + n0 + j);
    if (p < 0 || p >= m) ok = false;
    s_path[j] = p;
  }
  ok = __syncthreads_and(ok);
  if (!ok) {
    if (y == 0 && threadIdx.x == 0) set_status(a.status, kStatusInvalidArg);
    return;
  }
  const int j0 = y * kRowsPerBlock, j1 = min(L, j0 + kRowsPerBlock);
  if (j0 >= j1) return;
  const int vec_per_row = a.row_bytes / 16;
  const int total = (j1 - j0) * vec_per_row;
  for (int e = threadIdx.x; e < total; e += kThreads) {
    const int j = j0 + e / vec_per_row, c = e % vec_per_row;
    const size_t src = (size_t)(n0 + s_path[j]) * vec_per_row + c;
    const size_t dstv = (size_t)(dst + j) * vec_per_row + c;
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(a.tree_k) + src);
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(a.tree_v) + src);
    reinterpret_cast<uint4*>(a.k_cache)[dstv] = kv;
    reinterpret_cast<uint4*>(a.v_cache)[dstv] = vv;
  }
}

}  // namespace

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)a.B, (unsigned)((a.max_nodes + kRowsPerBlock - 1) / kRowsPerBlock));
  return check_cuda(launch_pdl(commit_kernel, grid, dim3(kThreads), 0, s, a), "launch commit_kernel");
}

}  // namespace tva
