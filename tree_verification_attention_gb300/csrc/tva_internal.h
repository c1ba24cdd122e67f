// tva_internal.h - launch interface between the C-ABI host code and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "tva_common.cuh"

namespace tva {

struct PartialArgs {
  Problem pr;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* tree_k;
  const void* tree_v;
  const int32_t* parent;
  float scale_log2;   // softmax_scale * log2(e): logits are kept in base 2
  float* o_part;      // [slots][RG][d] normalised partial outputs
  float* lse_part;    // [slots][RG] partial log2-sum-exp2 of the base-2 logits
  long long slots;    // slots the workspace holds (writes beyond are refused)
  int32_t* status;
};

struct CombineArgs {
  Problem pr;
  const float* o_part;
  const float* lse_part;
  long long slots;
  void* out;
  float* lse;
  int32_t* status;
};

struct AcceptArgs {
  int B;
  int node_capacity;
  const int32_t* cu_nodes;
  const int32_t* parent;
  const int32_t* draft_tok;
  const int32_t* target_argmax;
  int32_t* accept_len;
  int32_t* accept_path;
  int32_t* next_token;
  int32_t* status;
};

struct CommitArgs {
  int B;
  int row_bytes;            // bytes of one node's K (or V) row: Hkv * d * element size
  int node_capacity;
  int max_nodes;            // bound on every m_b (<= kMaxNodes); sizes the grid
  long long kv_capacity;
  const int32_t* cu_nodes;
  const int32_t* accept_len;
  const int32_t* accept_path;
  const void* tree_k;
  const void* tree_v;
  const int32_t* dst_row;
  void* k_cache;
  void* v_cache;
  int32_t* status;
};

struct SamplingArgs {
  int B, V, max_draft;
  long long p_rows, q_rows;
  const int32_t* cu_draft;
  const float* p;
  const float* q;
  const int32_t* draft_tok;
  const float* u_accept;
  const float* u_sample;
  int32_t* accept_len;
  int32_t* out_token;
  int32_t* status;
};

struct GdnArgs {
  int B, H, d, max_nodes, node_capacity;
  int bf16;                 // q, k, v and o: bf16 (1) or fp32 (0)
  const int32_t* cu_nodes;
  const int32_t* parent;
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* alpha;
  const float* S0;
  void* o;
  int32_t* status;
};

// Records a host-side failure for tva_last_error() (thread-local).
void record_error(const char* where, int code, const char* what);
// Records `e` (if it is an error) and returns it unchanged.
cudaError_t check_cuda(cudaError_t e, const char* where);

// Launches `kernel` allowing programmatic dependent launch: the kernel may become
// resident while the previous kernel in the stream still runs, and must call
// griddepcontrol.wait (ptx::pdl_wait) before touching memory that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// dtype: 0 = bf16, 1 = fp32, 2 = fp16 (tva_dtype values)
int simt_workers_per_sm();
cudaError_t launch_partials_simt(const PartialArgs& a, int dtype, cudaStream_t s);
// bf16 (bf16 = true) or fp16, head_dim 64 or 128; W M-tiles of npt nodes per row group
cudaError_t launch_partials_tc(const PartialArgs& a, bool bf16, int W, int npt, cudaStream_t s);
// Row groups of two M-tiles at head_dim 128 on CTA pairs (a.pr.U = pairs); bf16 or fp16.
cudaError_t launch_partials_pair(const PartialArgs& a, bool bf16, int npt, cudaStream_t s);
// 3-D 16-bit tensor map over [rows][heads][d] with a box of {64, box_heads, box_rows}
// (128-byte swizzle); false (and tva_last_error) if the driver rejects it.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int d, int heads, long long rows,
              int box_heads, int box_rows);
// Main-loop wait limit and test stall for the tensor-core partials kernels.
void tc_wait_settings(uint64_t* wait_ns, int* stall);
// Main-loop wait limit of the tensor-core partials kernel for later launches (0: the
// default 2 s) and the test stall (tva_diag_set_wait_limit).
void set_tc_wait_limit(unsigned long long ns, int stall);
cudaError_t launch_combine(const CombineArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s);
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s);
cudaError_t launch_sampling(const SamplingArgs& a, cudaStream_t s);
cudaError_t launch_gdn(const GdnArgs& a, cudaStream_t s);

}  // namespace tva
