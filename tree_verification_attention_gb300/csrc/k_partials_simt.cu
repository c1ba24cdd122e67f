// k_partials_simt.cu - attention partials on the CUDA cores (float32 inputs).
//
// One CTA per worker of the unit decomposition in tva_common.cuh.  For every segment
// (a contiguous run of key tiles of one row group) the CTA walks the row group in
// blocks of 32 rows; per block it streams the segment's keys in sub-tiles of 32 (each
// thread's share fetched as 16-byte vectors one sub-tile ahead, so the loads of the
// next sub-tile overlap the work on this one) and keeps a running maximum / sum per
// row (online softmax, base 2), so each segment
// yields the partial output O and log-sum-exp LSE of the LongSpec aggregation
// ("Fast Tree Attention", Aggregation).  The tree tile is masked with the
// ancestor-or-self bits of each row's node (LongSpec's tree mask; "Faster decoding",
// "Chains and trees consume work differently").
//
// This path carries the float32 dtype (head_dim 64 or 128).  bfloat16 inputs go to
// the tensor-core kernel.
#include "tva_internal.h"

namespace tva {
namespace {

constexpr int kRB = 32;       // rows per block
constexpr int kKT = 32;       // keys per sub-tile
constexpr int kThreads = 256; // 8 threads per row: 4 keys each for QK, D/8 columns for PV

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// Four consecutive elements of a row (16-byte aligned for float: rows are D floats and
// the base pointers are 16-byte aligned).
template <typename T>
__device__ __forceinline__ float4 load4(const T* p) {
  if constexpr (sizeof(T) == 4) {
    return __ldg(reinterpret_cast<const float4*>(p));
  } else {
    return make_float4(to_f(p[0]), to_f(p[1]), to_f(p[2]), to_f(p[3]));
  }
}

template <int D>
constexpr size_t simt_smem_bytes() {
  return sizeof(float) * (kRB * (D + 1) + kKT * (D + 1) + kKT * D + kRB * (kKT + 1)) +
         sizeof(uint32_t) * kMaxNodes * 4;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 3) partials_simt_kernel(PartialArgs a) {
  extern __shared__ float smem[];
  float* qs = smem;                          // [kRB][D+1]
  float* ks = qs + kRB * (D + 1);            // [kKT][D+1]
  float* vs = ks + kKT * (D + 1);            // [kKT][D]
  float* ps = vs + kKT * D;                  // [kRB][kKT+1]
  uint32_t* masks = reinterpret_cast<uint32_t*>(ps + kRB * (kKT + 1));  // [128][4]
  __shared__ int tree_bad;
  __shared__ int par_s[kMaxNodes];           // parent ids of the current tree

  __shared__ int cu_buf[512];
  Problem pr = a.pr;
  stage_cu(pr, cu_buf, 512);
  const T* __restrict__ q = static_cast<const T*>(a.q);
  const int tid = threadIdx.x;
  const int r_loc = tid >> 3;  // row of this thread inside the block
  const int kg = tid & 7;      // key group (QK) / column phase (PV)
  const int u = blockIdx.x;
  if (u == 0 && tid == 0) validate_sequences(pr, a.status);
  long long t = 0, t_end = 0;
  worker_range(pr, u, t, t_end, pr.share != 0);
  const size_t kv_stride = (size_t)pr.Hkv * D;

  Segment S;
  while (next_segment(pr, u, t, t_end, S, pr.share != 0)) {
    const Loc L = S.L;
    const int tile0 = S.tile0;
    const int tile1 = S.tile0 + S.n;
    const bool has_tree = tile0 == 0;   // the tree tile is a row group's first unit
    const SeqInfo s = L.s;
    const long long slot = partial_slot(pr, u, L, pr.share != 0);
    const bool slot_ok = slot < a.slots;  // cannot fail for a consistent layout
    if (!slot_ok && tid == 0) set_status(a.status, kStatusInvalidArg);

    if (has_tree) {
      __syncthreads();
      if (tid == 0) tree_bad = 0;
      __syncthreads();
      for (int i = tid; i < s.m; i += kThreads) par_s[i] = __ldg(a.parent + s.n0 + i);  // one round of loads
      __syncthreads();
      for (int i = tid; i < s.m; i += kThreads) {
        uint32_t bits[4];
        if (!ancestor_bits_shared(par_s, i, bits)) tree_bad = 1;
        masks[i * 4 + 0] = bits[0]; masks[i * 4 + 1] = bits[1];
        masks[i * 4 + 2] = bits[2]; masks[i * 4 + 3] = bits[3];
      }
      __syncthreads();
      if (tid == 0 && tree_bad) set_status(a.status, kStatusBadTree);
    }

    const int rows_total = s.m * pr.G;
    const int row_begin = L.mp * pr.RG;
    const int row_end = min(rows_total, row_begin + pr.RG);
    for (int rb = row_begin; rb < row_end; rb += kRB) {
      __syncthreads();
      {
        // all of the thread's loads first (one round of latency), then the stores
        constexpr int kN = kRB * D / 4 / kThreads;
        float4 qv[kN];
#pragma unroll
        for (int i = 0; i < kN; ++i) {
          const int idx = (tid + i * kThreads) * 4, r = idx / D, dd = idx % D, row = rb + r;
          qv[i] = row < row_end
                      ? load4(q + ((size_t)(s.n0 + row / pr.G) * pr.Hq + L.g * pr.G + row % pr.G) * D + dd)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kN; ++i) {
          const int idx = (tid + i * kThreads) * 4, r = idx / D, dd = idx % D;
          float* dst = qs + r * (D + 1) + dd;
          dst[0] = qv[i].x; dst[1] = qv[i].y; dst[2] = qv[i].z; dst[3] = qv[i].w;
        }
      }
      const int my_row = rb + r_loc;
      const bool row_ok = my_row < row_end;
      const int my_node = row_ok ? my_row / pr.G : 0;
      float m_run = -INFINITY, l_run = 0.f;
      float o[D / 8];
#pragma unroll
      for (int k = 0; k < D / 8; ++k) o[k] = 0.f;

      for (int tile = tile0; tile < tile1; ++tile) {
        const bool is_tree = tile == 0;
        const int nkeys = is_tree ? s.m : min(kKeyTile, s.P - (tile - 1) * kKeyTile);
        const T* kb = static_cast<const T*>(is_tree ? a.tree_k : a.k_cache);
        const T* vb = static_cast<const T*>(is_tree ? a.tree_v : a.v_cache);
        const size_t first = is_tree ? (size_t)s.n0 : (size_t)s.p0 + (size_t)(tile - 1) * kKeyTile;
        kb += first * kv_stride + (size_t)L.g * D;
        vb += first * kv_stride + (size_t)L.g * D;
        // The sub-tile's K / V are loaded into registers one sub-tile ahead: the loads
        // of sub-tile k0 + kKT are in flight while sub-tile k0 is computed.
        constexpr int kN = kKT * D / 4 / kThreads;
        float4 kr[kN], vr[kN];
        auto fetch = [&](int k0) {
#pragma unroll
          for (int i = 0; i < kN; ++i) {
            const int idx = (tid + i * kThreads) * 4, key = idx / D, dd = idx % D;
            const bool valid = k0 + key < nkeys;
            kr[i] = valid ? load4(kb + (size_t)(k0 + key) * kv_stride + dd) : make_float4(0.f, 0.f, 0.f, 0.f);
            vr[i] = valid ? load4(vb + (size_t)(k0 + key) * kv_stride + dd) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        };
        fetch(0);
        for (int k0 = 0; k0 < nkeys; k0 += kKT) {
          __syncthreads();
#pragma unroll
          for (int i = 0; i < kN; ++i) {
            const int idx = (tid + i * kThreads) * 4, key = idx / D, dd = idx % D;
            float* kd = ks + key * (D + 1) + dd;
            kd[0] = kr[i].x; kd[1] = kr[i].y; kd[2] = kr[i].z; kd[3] = kr[i].w;
            *reinterpret_cast<float4*>(vs + key * D + dd) = vr[i];
          }
          if (k0 + kKT < nkeys) fetch(k0 + kKT);
          __syncthreads();
          float sc[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) sc[k] = 0.f;
          for (int dd = 0; dd < D; ++dd) {
            const float qv = qs[r_loc * (D + 1) + dd];
#pragma unroll
            for (int k = 0; k < 4; ++k) sc[k] = fmaf(qv, ks[(kg * 4 + k) * (D + 1) + dd], sc[k]);
          }
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int key = k0 + kg * 4 + k;
            bool vis = row_ok && key < nkeys;
            if (is_tree && vis) vis = (masks[my_node * 4 + (key >> 5)] >> (key & 31)) & 1u;
            sc[k] = vis ? sc[k] * a.scale_log2 : -INFINITY;
            mx = fmaxf(mx, sc[k]);
          }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          const float m_new = fmaxf(m_run, mx);
          const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
          float psum = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float p = (sc[k] == -INFINITY) ? 0.f : exp2f(sc[k] - m_new);
            ps[r_loc * (kKT + 1) + kg * 4 + k] = p;
            psum += p;
          }
          psum += __shfl_xor_sync(0xffffffffu, psum, 4);
          psum += __shfl_xor_sync(0xffffffffu, psum, 2);
          psum += __shfl_xor_sync(0xffffffffu, psum, 1);
          l_run = l_run * alpha + psum;
          m_run = m_new;
          __syncwarp();
#pragma unroll
          for (int k = 0; k < D / 8; ++k) o[k] *= alpha;
          for (int j = 0; j < kKT; ++j) {
            const float pj = ps[r_loc * (kKT + 1) + j];
#pragma unroll
            for (int k = 0; k < D / 8; ++k) o[k] = fmaf(pj, vs[j * D + kg + 8 * k], o[k]);
          }
        }
      }
      if (row_ok && slot_ok) {
        const float inv = 1.f / l_run;
        const int rr = my_row - row_begin, MT = mtile_rows(pr.G);
        const int pp = rr / MT * 128 + rr % MT;  // padded row (see o_part_offset)
        const int RGP = padded_group_rows(pr.RG, pr.G);
        if (TVA_CHECK(pp < RGP, a.status)) {
#pragma unroll
          for (int k = 0; k < D / 8; ++k) {
            const int c = kg + 8 * k;
            a.o_part[o_part_offset(slot, pp, c >> 2, RGP, D) + (c & 3)] = o[k] * inv;
          }
          if (kg == 0) a.lse_part[(size_t)slot * RGP + pp] = m_run + log2f(l_run);
        }
      }
    }
  }
}

template <typename T, int D>
cudaError_t launch_simt_typed(const PartialArgs& a, cudaStream_t s) {
  constexpr size_t smem = simt_smem_bytes<D>();
  cudaError_t e = check_cuda(cudaFuncSetAttribute(partials_simt_kernel<T, D>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                             "cudaFuncSetAttribute(partials_simt_kernel)");
  if (e != cudaSuccess) return e;
  partials_simt_kernel<T, D><<<a.pr.U, kThreads, smem, s>>>(a);
  return check_cuda(cudaGetLastError(), "launch partials_simt_kernel");
}

}  // namespace

int simt_workers_per_sm() { return 3; }

cudaError_t launch_partials_simt(const PartialArgs& a, int dtype, cudaStream_t s) {
  if (dtype != 1) {  // bf16 runs on the tensor-core kernel
    record_error("launch_partials_simt", 0, "float32 only");
    return cudaErrorInvalidValue;
  }
  return a.pr.d == 64 ? launch_simt_typed<float, 64>(a, s) : launch_simt_typed<float, 128>(a, s);
}

}  // namespace tva
