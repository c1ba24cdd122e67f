// tva_host.cu - the C ABI (include/tva.h): argument checks, workspace layout and
// kernel launches.  No torch types cross this boundary.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>

#include "tva.h"
#include "tva_internal.h"

namespace {
thread_local char g_last_error[256] = "";
}  // namespace

namespace tva {
void record_error(const char* where, int code, const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, what, code);
}
cudaError_t check_cuda(cudaError_t e, const char* where) {
  if (e != cudaSuccess) record_error(where, (int)e, cudaGetErrorString(e));
  return e;
}
}  // namespace tva

namespace {

using tva::Problem;

constexpr int kMaxDevices = 64;

// tva_diag_use_cta_pair: non-zero selects the CTA-pair partials kernel where it applies.
std::atomic<int> g_use_cta_pair{0};

int device_sms(int* sms) {
  int dev = 0;
  if (tva::check_cuda(cudaGetDevice(&dev), "cudaGetDevice") != cudaSuccess || dev < 0 ||
      dev >= kMaxDevices)
    return -1;
  // Filled on first use per device; concurrent first calls store the same value.
  static std::atomic<int> cache[kMaxDevices];
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (tva::check_cuda(cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev),
                        "cudaDeviceGetAttribute") != cudaSuccess || v <= 0)
      return -1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  *sms = v;
  return 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side shape checks shared by every attention entry point.
tva_status check_shape(int B, int Hq, int Hkv, int d, int dtype, int max_prefix, int max_nodes,
                       long long kv_cap, long long node_cap) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return TVA_ERR_INVALID_ARG;
  if (Hq / Hkv > 128) return TVA_ERR_UNSUPPORTED;
  if (max_prefix < 0 || max_nodes < 1 || kv_cap < 0 || node_cap < 0) return TVA_ERR_INVALID_ARG;
  if (max_nodes > tva::kMaxNodes) return TVA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return TVA_ERR_UNSUPPORTED;
  if (dtype != TVA_BF16 && dtype != TVA_FP32 && dtype != TVA_FP16) return TVA_ERR_UNSUPPORTED;
  // index arithmetic inside the kernels is 32-bit for row counts
  if (kv_cap > (1LL << 31) - 1 - tva::kKeyTile || node_cap > (1LL << 24)) return TVA_ERR_INVALID_ARG;
  if ((long long)B * max_nodes > (1LL << 24) || (long long)B * max_prefix > (1LL << 40))
    return TVA_ERR_INVALID_ARG;
  return TVA_OK;
}

struct Layout {
  Problem pr;
  int W, npt;
  bool pair;  // row groups of two M-tiles at head_dim 128 (16-bit): the CTA-pair kernel
  size_t o_bytes, lse_bytes, total;
  long long slots;
};


size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Fills the device-visible problem and the workspace layout.  cu_* may be null for
// the single-sequence form.
tva_status make_layout(int B, int Hq, int Hkv, int d, int dtype, int max_prefix, int max_nodes,
                       int kv_cap, int node_cap, const int32_t* cu_prefix, const int32_t* cu_nodes,
                       int single_prefix, int single_nodes, Layout* L) {
  tva_status st = check_shape(B, Hq, Hkv, d, dtype, max_prefix, max_nodes, kv_cap, node_cap);
  if (st != TVA_OK) return st;
  int sms = 0;
  if (device_sms(&sms) != 0) return TVA_ERR_CUDA;
  const int G = Hq / Hkv;
  // Row groups hold whole nodes: an M-tile of 128 rows holds npt = floor(128 / G) nodes
  // (all G query heads of a node), and a row group W <= 2 M-tiles.
  const int npt = 128 / G;
  int W = (max_nodes > npt) ? 2 : 1;
  // One sequence whose tree needs several row groups: its row groups are computed by teams
  // that share K/V (Problem::share), so the group size is free; one-M-tile groups win when
  // they cover the tree with fewer M-tiles (a 68-node tree at 32 nodes per M-tile: 3
  // against 2 x 2 - the second two-M-tile group would hold 4 nodes).
  if (B == 1 && W == 2) {
    const int mt1 = (max_nodes + npt - 1) / npt;
    const int mt2 = 2 * ((max_nodes + 2 * npt - 1) / (2 * npt));
    if (mt1 < mt2) W = 1;
  }
  L->npt = npt;
  L->W = W;
  Problem& pr = L->pr;
  pr.cu_prefix = cu_prefix;
  pr.cu_nodes = cu_nodes;
  pr.single_prefix = single_prefix;
  pr.single_nodes = single_nodes;
  pr.B = B; pr.Hq = Hq; pr.Hkv = Hkv; pr.G = G; pr.d = d;
  pr.RG = W * npt * G;
  // workers: the fp32 kernel runs several CTAs per SM; the tensor-core kernel one CTA per
  // SM, the CTA-pair kernel (selected by tva_diag_use_cta_pair; two M-tiles per row group,
  // head_dim 128) one pair per two SMs
  L->pair = g_use_cta_pair.load(std::memory_order_relaxed) != 0 && dtype != TVA_FP32 && W == 2 && d == 128;
  pr.U = dtype == TVA_FP32 ? sms * tva::simt_workers_per_sm() : (L->pair ? sms / 2 : sms);
  pr.max_prefix = max_prefix; pr.max_nodes = max_nodes;
  pr.kv_capacity = kv_cap; pr.node_capacity = node_cap;
  const int mp_max = (max_nodes + W * npt - 1) / (W * npt);  // row groups per KV head
  const long long groups = (long long)B * Hkv * mp_max;
  // One sequence whose KV heads have several row groups: teams of workers, one member per
  // row group, stream the same K/V tiles together, so each is read from DRAM once.
  pr.share = (B == 1 && mp_max >= 2 && pr.U >= mp_max) ? mp_max : 0;
  // One sequence with one row group per KV head: split each head's tiles over its own
  // U / Hkv workers when Hkv divides U (see Problem::align).
  pr.align = (B == 1 && mp_max == 1 && pr.U % Hkv == 0) ? pr.U / Hkv : 0;
  L->slots = pr.U + groups;
  const size_t rgp = (size_t)W * 128;  // padded rows per slot (see o_part_offset)
  L->o_bytes = align256((size_t)L->slots * rgp * d * sizeof(float));
  L->lse_bytes = align256((size_t)L->slots * rgp * sizeof(float));
  L->total = L->o_bytes + L->lse_bytes;
  return TVA_OK;
}

tva_status layout_from_params(const tva_params* p, Layout* L) {
  if (p == nullptr) return TVA_ERR_INVALID_ARG;
  return make_layout(p->batch, p->num_q_heads, p->num_kv_heads, p->head_dim, (int)p->dtype,
                     p->max_prefix_len, p->max_nodes, p->kv_capacity, p->node_capacity,
                     p->cu_prefix, p->cu_nodes, 0, 0, L);
}

float scale_log2(float softmax_scale, int d) {
  const float s = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)d);
  return s * 1.44269504088896340736f;
}

tva_status run_partials(const Layout& L, int dtype, float softmax_scale, const void* q,
                        const void* k_cache, const void* v_cache, const void* tree_k,
                        const void* tree_v, const int32_t* parent, void* workspace,
                        int32_t* dev_status, cudaStream_t s) {
  tva::PartialArgs a;
  a.pr = L.pr;
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.tree_k = tree_k; a.tree_v = tree_v;
  a.parent = parent;
  a.scale_log2 = scale_log2(softmax_scale, L.pr.d);
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.o_bytes);
  a.slots = L.slots;
  a.status = dev_status;
  const cudaError_t e = dtype == TVA_FP32 ? tva::launch_partials_simt(a, dtype, s)
                        : L.pair           ? tva::launch_partials_pair(a, dtype == TVA_BF16, L.npt, s)
                                           : tva::launch_partials_tc(a, dtype == TVA_BF16, L.W, L.npt, s);
  return e == cudaSuccess ? TVA_OK : TVA_ERR_CUDA;
}

tva_status run_combine(const Layout& L, int dtype, const void* workspace, void* out, float* lse,
                       int32_t* dev_status, cudaStream_t s);

// The whole attention: the partials launch, then the combine launch (a programmatic
// dependent of it).
tva_status run_attention(const Layout& L, int dtype, float softmax_scale, const void* q,
                         const void* k_cache, const void* v_cache, const void* tree_k,
                         const void* tree_v, const int32_t* parent, void* workspace,
                         void* out, float* lse, int32_t* dev_status, cudaStream_t s) {
  tva_status st = run_partials(L, dtype, softmax_scale, q, k_cache, v_cache, tree_k, tree_v, parent,
                               workspace, dev_status, s);
  if (st != TVA_OK) return st;
  return run_combine(L, dtype, workspace, out, lse, dev_status, s);
}

tva_status run_combine(const Layout& L, int dtype, const void* workspace, void* out, float* lse,
                       int32_t* dev_status, cudaStream_t s) {
  tva::CombineArgs a;
  a.pr = L.pr;
  a.o_part = static_cast<const float*>(workspace);
  a.lse_part = reinterpret_cast<const float*>(static_cast<const char*>(workspace) + L.o_bytes);
  a.slots = L.slots;
  a.out = out; a.lse = lse; a.status = dev_status;
  return tva::launch_combine(a, dtype, s) == cudaSuccess ? TVA_OK : TVA_ERR_CUDA;
}

tva_status check_io_ptrs(const void* q, const void* k_cache, const void* v_cache,
                         const void* tree_k, const void* tree_v, const int32_t* parent,
                         long long kv_cap) {
  if (!q || !tree_k || !tree_v || !parent) return TVA_ERR_INVALID_ARG;
  if (kv_cap > 0 && (!k_cache || !v_cache)) return TVA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(tree_k) ||
      !aligned16(tree_v))
    return TVA_ERR_INVALID_ARG;
  return TVA_OK;
}

tva_status check_workspace(const Layout& L, const void* ws, size_t bytes) {
  if (ws == nullptr || bytes < L.total) return TVA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TVA_ERR_WORKSPACE;
  return TVA_OK;
}

// ---- convenience-form state (library-owned, per device) ----
struct OwnedState {
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int32_t* status = nullptr;
};
std::mutex g_owned_mu;
OwnedState g_owned[kMaxDevices];

}  // namespace

extern "C" {

const char* tva_last_error(void) { return g_last_error; }

const char* tva_status_string(tva_status s) {
  switch (s) {
    case TVA_OK: return "TVA_OK";
    case TVA_ERR_INVALID_ARG: return "TVA_ERR_INVALID_ARG";
    case TVA_ERR_UNSUPPORTED: return "TVA_ERR_UNSUPPORTED";
    case TVA_ERR_BAD_TREE: return "TVA_ERR_BAD_TREE";
    case TVA_ERR_WORKSPACE: return "TVA_ERR_WORKSPACE";
    case TVA_ERR_CUDA: return "TVA_ERR_CUDA";
    case TVA_ERR_TIMEOUT: return "TVA_ERR_TIMEOUT";
  }
  return "TVA_ERR_UNKNOWN";
}

size_t tva_workspace_size(const tva_params* p) {
  Layout L;
  if (layout_from_params(p, &L) != TVA_OK) return 0;
  return L.total;
}

int tva_num_workers(const tva_params* p) {
  Layout L;
  if (layout_from_params(p, &L) != TVA_OK) return -1;
  return L.pr.U;
}

tva_status tree_verify_attn_partials(const tva_params* p, const void* q, const void* k_cache,
                                     const void* v_cache, const void* tree_k,
                                     const void* tree_v, const int32_t* parent,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, void* stream) {
  if (p == nullptr || p->cu_prefix == nullptr || p->cu_nodes == nullptr || dev_status == nullptr)
    return TVA_ERR_INVALID_ARG;
  tva_status st = check_shape(p->batch, p->num_q_heads, p->num_kv_heads, p->head_dim,
                              (int)p->dtype, p->max_prefix_len, p->max_nodes, p->kv_capacity,
                              p->node_capacity);
  if (st != TVA_OK) return st;
  st = check_io_ptrs(q, k_cache, v_cache, tree_k, tree_v, parent, p->kv_capacity);
  if (st != TVA_OK) return st;
  Layout L;
  st = layout_from_params(p, &L);
  if (st != TVA_OK) return st;
  st = check_workspace(L, workspace, workspace_bytes);
  if (st != TVA_OK) return st;
  return run_partials(L, (int)p->dtype, p->softmax_scale, q, k_cache, v_cache, tree_k, tree_v,
                      parent, workspace, dev_status, static_cast<cudaStream_t>(stream));
}

tva_status tree_verify_attn_combine(const tva_params* p, const void* workspace,
                                    size_t workspace_bytes, void* out, float* lse,
                                    int32_t* dev_status, void* stream) {
  if (p == nullptr || p->cu_prefix == nullptr || p->cu_nodes == nullptr || dev_status == nullptr)
    return TVA_ERR_INVALID_ARG;
  if (out == nullptr || lse == nullptr || !aligned16(out)) return TVA_ERR_INVALID_ARG;
  Layout L;
  tva_status st = layout_from_params(p, &L);
  if (st != TVA_OK) return st;
  st = check_workspace(L, workspace, workspace_bytes);
  if (st != TVA_OK) return st;
  return run_combine(L, (int)p->dtype, workspace, out, lse, dev_status,
                     static_cast<cudaStream_t>(stream));
}

tva_status tree_verify_attn_varlen(const tva_params* p, const void* q, const void* k_cache,
                                   const void* v_cache, const void* tree_k,
                                   const void* tree_v, const int32_t* parent, void* out,
                                   float* lse, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream) {
  if (out == nullptr || lse == nullptr || !aligned16(out)) return TVA_ERR_INVALID_ARG;
  if (p == nullptr || p->cu_prefix == nullptr || p->cu_nodes == nullptr || dev_status == nullptr)
    return TVA_ERR_INVALID_ARG;
  tva_status st = check_shape(p->batch, p->num_q_heads, p->num_kv_heads, p->head_dim,
                              (int)p->dtype, p->max_prefix_len, p->max_nodes, p->kv_capacity,
                              p->node_capacity);
  if (st != TVA_OK) return st;
  st = check_io_ptrs(q, k_cache, v_cache, tree_k, tree_v, parent, p->kv_capacity);
  if (st != TVA_OK) return st;
  Layout L;
  st = layout_from_params(p, &L);
  if (st != TVA_OK) return st;
  st = check_workspace(L, workspace, workspace_bytes);
  if (st != TVA_OK) return st;
  return run_attention(L, (int)p->dtype, p->softmax_scale, q, k_cache, v_cache, tree_k, tree_v, parent,
                       workspace, out, lse, dev_status, static_cast<cudaStream_t>(stream));
}

tva_status tree_verify_attn(const void* q, const void* k_cache, const void* v_cache,
                            int prefix_len, const void* tree_k, const void* tree_v,
                            const int32_t* parent, int num_nodes, int num_q_heads,
                            int num_kv_heads, int head_dim, tva_dtype dtype, void* out,
                            float* lse, void* stream) {
  if (prefix_len < 0 || num_nodes < 1) return TVA_ERR_INVALID_ARG;
  if (out == nullptr || lse == nullptr || !aligned16(out)) return TVA_ERR_INVALID_ARG;
  tva_status st = check_io_ptrs(q, k_cache, v_cache, tree_k, tree_v, parent, prefix_len);
  if (st != TVA_OK) return st;
  Layout L;
  st = make_layout(1, num_q_heads, num_kv_heads, head_dim, (int)dtype, prefix_len, num_nodes,
                   prefix_len, num_nodes, nullptr, nullptr, prefix_len, num_nodes, &L);
  if (st != TVA_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TVA_ERR_CUDA;
  // The lock is held until both kernels are enqueued: another thread that needs a
  // larger workspace frees the old one only after synchronising the device, and it
  // cannot do so between this thread's pointer copy and its launches.
  std::lock_guard<std::mutex> lock(g_owned_mu);
  OwnedState& o = g_owned[dev];
  if (o.status == nullptr) {
    if (cudaMalloc(&o.status, sizeof(int32_t)) != cudaSuccess) return TVA_ERR_CUDA;
    if (cudaMemset(o.status, 0, sizeof(int32_t)) != cudaSuccess) return TVA_ERR_CUDA;
  }
  if (o.ws_bytes < L.total) {
    if (o.ws != nullptr) {
      cudaDeviceSynchronize();  // the old buffer may still be in use by queued work
      cudaFree(o.ws);
      o.ws = nullptr;
      o.ws_bytes = 0;
    }
    if (cudaMalloc(&o.ws, L.total) != cudaSuccess) return TVA_ERR_CUDA;
    o.ws_bytes = L.total;
  }
  return run_attention(L, (int)dtype, 0.f, q, k_cache, v_cache, tree_k, tree_v, parent, o.ws, out, lse,
                       o.status, static_cast<cudaStream_t>(stream));
}

tva_status tva_read_device_status(int32_t* host_status, void* stream) {
  if (host_status == nullptr) return TVA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TVA_ERR_CUDA;
  int32_t* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_owned_mu);
    status = g_owned[dev].status;
  }
  *host_status = 0;
  if (status == nullptr) return TVA_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return TVA_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return TVA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return TVA_ERR_CUDA;
  return TVA_OK;
}

void tva_diag_set_wait_limit(unsigned long long wait_limit_ns, int force_stall) {
  tva::set_tc_wait_limit(wait_limit_ns, force_stall);
}

void tva_diag_use_cta_pair(int enable) { g_use_cta_pair.store(enable != 0 ? 1 : 0, std::memory_order_relaxed); }

void tva_release(void) {
  std::lock_guard<std::mutex> lock(g_owned_mu);
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return;
  for (int dev = 0; dev < kMaxDevices; ++dev) {
    OwnedState& o = g_owned[dev];
    if (o.ws == nullptr && o.status == nullptr) continue;
    if (cudaSetDevice(dev) != cudaSuccess) continue;
    cudaDeviceSynchronize();
    if (o.ws) cudaFree(o.ws);
    if (o.status) cudaFree(o.status);
    o = OwnedState();
  }
  cudaSetDevice(prev);
}

tva_status accept_longest_path(int batch, int node_capacity, const int32_t* cu_nodes,
                               const int32_t* parent,
                               const int32_t* draft_tok, const int32_t* target_argmax,
                               int32_t* accept_len, int32_t* accept_path, int32_t* next_token,
                               int32_t* dev_status, void* stream) {
  if (batch < 1 || node_capacity < 0 || !cu_nodes || !parent || !draft_tok || !target_argmax || !accept_len ||
      !accept_path || !next_token || !dev_status)
    return TVA_ERR_INVALID_ARG;
  tva::AcceptArgs a;
  a.B = batch; a.node_capacity = node_capacity; a.cu_nodes = cu_nodes; a.parent = parent; a.draft_tok = draft_tok;
  a.target_argmax = target_argmax; a.accept_len = accept_len; a.accept_path = accept_path;
  a.next_token = next_token; a.status = dev_status;
  return tva::launch_accept(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TVA_OK
                                                                                 : TVA_ERR_CUDA;
}

tva_status commit_accepted_kv(int batch, int num_kv_heads, int head_dim, tva_dtype dtype, int node_capacity,
                              int max_nodes, long long kv_capacity, const int32_t* cu_nodes,
                              const int32_t* accept_len, const int32_t* accept_path, const void* tree_k,
                              const void* tree_v, const int32_t* dst_row, void* k_cache, void* v_cache,
                              int32_t* dev_status, void* stream) {
  if (batch < 1 || num_kv_heads < 1 || (head_dim != 64 && head_dim != 128) ||
      (dtype != TVA_BF16 && dtype != TVA_FP32 && dtype != TVA_FP16) || node_capacity < 0 || max_nodes < 1 ||
      max_nodes > tva::kMaxNodes || kv_capacity < 0 || !cu_nodes || !accept_len || !accept_path || !tree_k ||
      !tree_v || !dst_row || !k_cache || !v_cache || !dev_status)
    return TVA_ERR_INVALID_ARG;
  if (!aligned16(tree_k) || !aligned16(tree_v) || !aligned16(k_cache) || !aligned16(v_cache))
    return TVA_ERR_INVALID_ARG;
  const size_t row = (size_t)num_kv_heads * head_dim * (dtype == TVA_FP32 ? 4 : 2);
  // The copy has no defined order, so no source row may alias a destination row; the
  // buffers are compared over their full extents.
  auto overlap = [](const void* x, size_t nx, const void* y, size_t ny) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(x), b0 = reinterpret_cast<uintptr_t>(y);
    return nx > 0 && ny > 0 && a0 < b0 + ny && b0 < a0 + nx;
  };
  const size_t nsrc = (size_t)node_capacity * row, ndst = (size_t)kv_capacity * row;
  if (overlap(tree_k, nsrc, k_cache, ndst) || overlap(tree_k, nsrc, v_cache, ndst) ||
      overlap(tree_v, nsrc, k_cache, ndst) || overlap(tree_v, nsrc, v_cache, ndst) ||
      overlap(k_cache, ndst, v_cache, ndst))
    return TVA_ERR_INVALID_ARG;
  tva::CommitArgs a;
  a.B = batch; a.row_bytes = (int)row; a.node_capacity = node_capacity; a.max_nodes = max_nodes;
  a.kv_capacity = kv_capacity;
  a.cu_nodes = cu_nodes; a.accept_len = accept_len; a.accept_path = accept_path;
  a.tree_k = tree_k; a.tree_v = tree_v; a.dst_row = dst_row; a.k_cache = k_cache; a.v_cache = v_cache;
  a.status = dev_status;
  return tva::launch_commit(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TVA_OK
                                                                                            : TVA_ERR_CUDA;
}

tva_status verify_chain_sampling(int batch, int vocab, int max_draft, long long p_rows, long long q_rows,
                                 const int32_t* cu_draft, const float* p, const float* q,
                                 const int32_t* draft_tok, const float* u_accept, const float* u_sample,
                                 int32_t* accept_len, int32_t* out_token, int32_t* dev_status, void* stream) {
  if (batch < 1 || vocab < 1 || max_draft < 0 || p_rows < batch || q_rows < 0 || !cu_draft || !p || !q ||
      !draft_tok || !u_accept || !u_sample || !accept_len || !out_token || !dev_status)
    return TVA_ERR_INVALID_ARG;
  tva::SamplingArgs a;
  a.B = batch; a.V = vocab; a.max_draft = max_draft; a.p_rows = p_rows; a.q_rows = q_rows;
  a.cu_draft = cu_draft; a.p = p; a.q = q; a.draft_tok = draft_tok; a.u_accept = u_accept;
  a.u_sample = u_sample; a.accept_len = accept_len; a.out_token = out_token; a.status = dev_status;
  return tva::launch_sampling(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TVA_OK : TVA_ERR_CUDA;
}

tva_status gdn_tree_verify(int batch, int num_heads, int head_dim, tva_dtype dtype, int node_capacity,
                           int max_nodes, const int32_t* cu_nodes, const int32_t* parent, const void* q,
                           const void* k, const void* v, const float* beta, const float* alpha, const float* S0,
                           void* out, int32_t* dev_status, void* stream) {
  if (batch < 1 || num_heads < 1 || (head_dim != 64 && head_dim != 128) || node_capacity < 0 || max_nodes < 1 ||
      max_nodes > tva::kMaxNodes || !cu_nodes || !parent || !q || !k || !v || !beta || !alpha || !S0 || !out ||
      !dev_status)
    return TVA_ERR_INVALID_ARG;
  if (dtype != TVA_FP32 && dtype != TVA_BF16) return TVA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(S0) || !aligned16(out))
    return TVA_ERR_INVALID_ARG;
  tva::GdnArgs a;
  a.B = batch; a.H = num_heads; a.d = head_dim; a.max_nodes = max_nodes; a.node_capacity = node_capacity;
  a.bf16 = dtype == TVA_BF16 ? 1 : 0;
  a.cu_nodes = cu_nodes; a.parent = parent; a.q = q; a.k = k; a.v = v; a.beta = beta; a.alpha = alpha;
  a.S0 = S0; a.o = out; a.status = dev_status;
  return tva::launch_gdn(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TVA_OK : TVA_ERR_CUDA;
}

}  // extern "C"
