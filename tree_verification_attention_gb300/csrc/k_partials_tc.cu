// k_partials_tc.cu - attention partials on the 5th-generation tensor cores (bf16).
//
// What is computed: for every segment of the unit decomposition (tva_common.cuh), the
// partial output O and log-sum-exp LSE of the segment's key tiles, per query row -
// the O_cache / O_specs, LSE_cache / LSE_specs of LongSpec's Hybrid Tree Attention
// ("Fast Tree Attention": cached pairs need no mask; the speculative pairs are masked
// by the tree, each node seeing its ancestors and itself).  The tree keys are simply
// one more 128-key tile whose logits are masked with the row's ancestor bits.
//
// How (one CTA per SM, 320 threads):
//   warp 8  (producer): TMA loads, issued like the MMAs (below) by one elected lane of
//           the converged warp, of Q (once per segment; with one M-tile per row group
//           into two alternating buffers, so a worker's next segment does not wait for
//           the current one's Q to be released) and of the K / V tiles into a ring of
//           shared-memory stages, 128-byte swizzled.
//   warp 9  (MMA):      tcgen05.mma issue.  The warp runs this role converged and one
//           elected lane issues each MMA and commit (single-lane issue from a divergent
//           branch was the kernel's bottleneck).  S = Q K^T (both operands in shared
//           memory) into TMEM; O += P V with P read from TMEM (P overwrites the first
//           half of its S buffer as packed bf16) and V from shared memory.
//   warps 0-7 (softmax): two streams of 4 warps; thread r of a stream owns TMEM lane
//           (= query row) r, so row max / sum need no shuffles.  A stream's running
//           max is only moved when it grows by more than 2^8 (stale maxima cancel in
//           the final division), and then O is rescaled in TMEM.
// Streams: with 2 M-tiles per row group (W = 2) stream w owns M-tile w and sees every
// key tile; with W = 1 both streams share the M-tile and take alternate key tiles,
// and their two partials are merged in the epilogue.  Either way the MMA warp issues
//   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), ...
// so each stream's softmax overlaps the other stream's MMAs, and the commit that
// publishes S_w(j+1) also covers PV_w(j): a stream may rescale its O right after its
// S is ready.
// TMEM columns: S/P buffers at 0 and 128, O accumulators at 256 and 384 (512 total).
//
// Every wait is bounded (2 s by default; the main-loop limit is a launch argument): on
// expiry the CTA raises an abort flag, records TVA_ERR_TIMEOUT, drains its in-flight
// copies and MMAs (bounded again, always with the full 2 s), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>

#include "tc_pipeline.cuh"
#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

using namespace ptx;

constexpr int kThreadsTc = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kHalfBytes = 128 * 128;  // 128 rows of 64 bf16 (one 128-byte swizzle span)

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kStages = D == 128 ? 4 : 8;
  static constexpr int kQBytes = 2 * kHalves * kHalfBytes;
  static constexpr int kBarOff = kQBytes + kStages * kTileBytes;
  static constexpr int kCuOff = 4096;               // staged cu_* arrays inside misc
  static constexpr int kCuCap = 1024;               // ints: batches up to 511 sequences
  static constexpr int kMiscBytes = kCuOff + 4 * kCuCap;
  static constexpr int kSmemBytes = kBarOff + kMiscBytes + 1024;  // + alignment slack
};

struct TcArgs {
  PartialArgs a;
  int W;    // M-tiles per row group (1 or 2)
  int npt;  // nodes per M-tile: floor(128 / G)
  uint64_t wait_ns;  // limit of every main-loop wait
  int stall;         // test hook: the MMA thread first waits on a barrier nothing completes
};

// Process-wide diagnostic settings (tva_diag_set_wait_limit): 0 = the default limit.
std::atomic<unsigned long long> g_wait_limit_ns{0};
std::atomic<int> g_force_stall{0};

// Q buffers: with one M-tile per row group (W = 1) the Q region holds two M-tiles, so
// segments alternate between two buffers and the next segment's Q is loaded while the
// current one is still in use; with W = 2 one buffer holds both M-tiles.
__device__ __forceinline__ int q_buffer(int W, int sg) { return W == 1 ? (sg & 1) : 0; }
// Earlier segments that used the same buffer.
__device__ __forceinline__ int q_use(int W, int sg) { return W == 1 ? (sg >> 1) : sg; }

template <int D, bool kBF16, bool kShare>
__global__ void __launch_bounds__(kThreadsTc, 1)
    partials_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_tk,
                       const __grid_constant__ CUtensorMap tm_tv, const TcArgs args) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const PartialArgs& a = args.a;
  Problem* pr_s = reinterpret_cast<Problem*>(smem + C::kBarOff + C::kCuOff - 128);
  const Problem& pr = *pr_s;
  const int W = args.W, npt = args.npt, G = a.pr.G;  // kernel parameters: readable before staging
  const uint64_t wait_ns = args.wait_ns;  // main-loop waits; drains use kDrainNs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_s = sbase;
  const uint32_t kv_s = sbase + C::kQBytes;
  const uint32_t bar0 = sbase + C::kBarOff;
  const uint32_t KV_FULL = bar0;                        // [kStages]
  const uint32_t KV_EMPTY = bar0 + 8 * C::kStages;      // [kStages]
  const uint32_t Q_FULL = bar0 + 16 * C::kStages;      // [2]
  const uint32_t Q_EMPTY = Q_FULL + 16;                 // [2]
  const uint32_t S_FULL = Q_EMPTY + 16;                 // [2]
  const uint32_t P_FULL = S_FULL + 16;                  // [2]
  const uint32_t O_FULL = P_FULL + 16;                  // [2]
  const uint32_t O_FREE = O_FULL + 16;
  const uint32_t M1_READY = O_FREE + 8;
  const uint32_t DRAIN = M1_READY + 8;
  const uint32_t PAR_READY = DRAIN + 8;                 // [2]
  uint8_t* misc = smem + C::kBarOff + 16 * C::kStages + 8 * 16;
  int* par_s = reinterpret_cast<int*>(smem + C::kBarOff + 2560);   // [2][128] parent ids
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  float* m1_s = reinterpret_cast<float*>(smem + C::kBarOff + 512);  // [2][128]
  float* l1_s = m1_s + 256;                                         // [2][128]

  // ---- Set-up that reads nothing an earlier kernel may write.  This kernel is launched
  // as a programmatic dependent, so this runs while the preceding kernel finishes: the
  // tensor-map prefetches and barrier initialisation, and - when the problem is given
  // entirely by the kernel parameters (one sequence: no cu_* arrays) - the problem
  // staging and the unit schedule.  (An L2 prefetch of the first tiles here was tried:
  // slower by about 0.8 us per launch.)
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_tk);
    prefetch_tmap(&tm_tv);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(KV_FULL + 8 * s, 1);
      mbar_init(KV_EMPTY + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(Q_FULL + 8 * b, 1);
      mbar_init(Q_EMPTY + 8 * b, 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(S_FULL + 8 * w, 1);
      mbar_init(P_FULL + 8 * w, 128);
      mbar_init(O_FULL + 8 * w, 1);
    }
    mbar_init(O_FREE, 256);
    mbar_init(M1_READY, 128);
    mbar_init(DRAIN, 1);
    mbar_init(PAR_READY, 128);
    mbar_init(PAR_READY + 8, 128);
    *abort_flag = 0;
    fence_mbar_init();
    __threadfence_block();
  }
  const bool params_only = a.pr.cu_prefix == nullptr;  // uniform over the grid
  long long t_begin = 0, t_end = 0;
  auto schedule = [&]() {
    stage_problem(a.pr, pr_s, reinterpret_cast<int*>(smem + C::kBarOff + C::kCuOff), C::kCuCap);
    worker_range(pr, u, t_begin, t_end, kShare);
  };
  if (params_only) schedule();
  pdl_wait();  // launched as a programmatic dependent: inputs are final after this
  pdl_launch_dependents();
  if (!params_only) schedule();  // reads the caller's cu_* arrays
  if (u == 0 && threadIdx.x == 0) validate_sequences(pr, a.status);
  if (t_begin >= t_end) return;  // uniform over the CTA

  // The other warps wait for the barrier initialisation (made visible by the block
  // barrier inside stage_problem) and the TMEM allocation on named barrier 1, which the
  // producer warp only arrives at: it goes straight on to its first copies.
  uint32_t tmem = 0;
  if (warp == kProducerWarp) {
    __syncwarp();
    bar_arrive(1, kThreadsTc);
  } else {
    if (warp == kMmaWarp) {
      tmem_alloc(smem_u32(tmem_slot), 512);
      tmem_relinquish();
    }
    tc_fence_before();
    bar_sync(1, kThreadsTc);
    tc_fence_after();
    tmem = *tmem_slot;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    // All 32 lanes run this role; one elected lane issues each copy and expect-tx.
    {
      int ring = 0, sg = 0;
      bool ok = true;
      long long t = t_begin;
      Segment S;
      const uint32_t q_box_bytes = 64u * G * npt * 2u;
      const uint64_t evict_first = policy_evict_first();  // K/V are read once
      while (ok && next_segment(pr, u, t, t_end, S, kShare)) {
        const Loc& L = S.L;
        const int qb = q_buffer(W, sg), quse = q_use(W, sg);
        if (quse > 0 && !warp_wait(Q_EMPTY + 8 * qb, (quse - 1) & 1, abort_flag, wait_ns)) { ok = false; break; }
        mbar_expect_tx_elect(Q_FULL + 8 * qb, (uint32_t)W * C::kHalves * q_box_bytes);
        for (int mt = 0; mt < W; ++mt) {
          // an M-tile starts at a node of its own sequence, or lies wholly past the sequence's
          // nodes (padding rows: loaded - zeros past the tensor's end - but never written)
          int qrow = L.s.n0 + (L.mp * W + mt) * npt;
          if (!TVA_CHECK(qrow >= L.s.n0 && L.g >= 0 && L.g < pr.Hkv, a.status)) qrow = 0;
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_3d_elect(q_s + ((qb + mt) * C::kHalves + h) * kHalfBytes, &tm_q, 64 * h, L.g * G, qrow,
                              Q_FULL + 8 * qb);
        }
        const int n = S.n;
        auto load = [&](int k, bool is_v) -> bool {
          const int stage = ring % C::kStages, use = ring / C::kStages;
          if (use > 0 && !warp_wait(KV_EMPTY + 8 * stage, (use - 1) & 1, abort_flag, wait_ns))
            return false;
          const int tile = S.tile0 + k;
          const bool tree = tile == 0;
          const CUtensorMap* m = tree ? (is_v ? &tm_tv : &tm_tk) : (is_v ? &tm_v : &tm_k);
          int z = tree ? L.s.n0 : L.s.p0 + (tile - 1) * kKeyTile;
          // a tile starts inside its sequence's rows (loads past a tensor's end read zeros)
          if (!TVA_CHECK(z >= 0 && (tree ? z < pr.node_capacity && L.s.m > 0
                                         : z < L.s.p0 + L.s.P && z < pr.kv_capacity), a.status))
            z = 0;
          mbar_expect_tx_elect(KV_FULL + 8 * stage, C::kTileBytes);
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_3d_hint_elect(kv_s + stage * C::kTileBytes + h * kHalfBytes, m, 64 * h, L.g, z,
                             KV_FULL + 8 * stage, evict_first);
          ++ring;
          return true;
        };
        if (W == 2) {
          for (int k = 0; k < n && ok; ++k) ok = load(k, false) && load(k, true);
        } else {
          ok = load(0, false);
          if (ok && n > 1) ok = load(1, false);
          for (int j = 0; j < n && ok; ++j) {
            ok = load(j, true);
            if (ok && j + 2 < n) ok = load(j + 2, false);
          }
        }
        ++sg;
      }
      // drain: every copy this thread started has landed before TMEM / smem go away
      for (int i = max(0, ring - C::kStages); i < ring; ++i)
        drain_wait(KV_FULL + 8 * (i % C::kStages), (i / C::kStages) & 1);
      for (int b = 0; b < 2; ++b) {  // the last load into each Q buffer
        const int uses = (W == 1) ? (sg + 1 - b) / 2 : (b == 0 ? sg : 0);
        if (uses > 0) drain_wait(Q_FULL + 8 * b, (uses - 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // All 32 lanes run this role (waits and descriptor arithmetic are warp-uniform);
    // the *_elect forms issue each MMA / commit from one lane.
    {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, kBF16);
      constexpr uint32_t idesc_o = idesc_bf16(128, D, true, kBF16);
      int ring = 0, sg = 0;
      uint32_t pbits = 0;  // bit w: parity of the next P_FULL[w] phase
      bool ok = true;
      long long t = t_begin;
      Segment S;
      auto wait_kv = [&](int idx) -> bool {
        if (!warp_wait(KV_FULL + 8 * (idx % C::kStages), (idx / C::kStages) & 1, abort_flag, wait_ns))
          return false;
        tc_fence_after();
        return true;
      };
      // Operand descriptors: built once, then stepped through their low word (the issue
      // rate of this one thread bounds the tensor pipe, so each MMA costs as few
      // instructions as possible).  K / Q are K-major, V is MN-major (d contiguous).
      const uint32_t k_hi = (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32);
      const uint32_t v_hi = (uint32_t)(sdesc_sw128(0, kHalfBytes, 1024) >> 32);
      const uint32_t k_lo = (uint32_t)sdesc_sw128(kv_s, 16, 1024);
      const uint32_t v_lo = (uint32_t)sdesc_sw128(kv_s, kHalfBytes, 1024);
      const uint32_t q_lo = (uint32_t)sdesc_sw128(q_s, 16, 1024);
      int qb = 0;  // Q buffer of the current segment
      auto issue_s = [&](int w, int mt, int idx) {
        const uint32_t kl = k_lo + (uint32_t)((idx % C::kStages) * C::kTileBytes >> 4);
        const uint32_t ql = q_lo + (uint32_t)((qb + mt) * C::kHalves * kHalfBytes >> 4);
        const uint32_t dt = tmem + w * 128;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t o = (uint32_t)((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
          mma_ss_elect(dt, desc_join(ql + o, k_hi), desc_join(kl + o, k_hi), idesc_s, ks > 0);
        }
        tc_commit_elect(S_FULL + 8 * w);
      };
      auto issue_pv = [&](int w, int idx, bool acc) {
        const uint32_t vl = v_lo + (uint32_t)((idx % C::kStages) * C::kTileBytes >> 4);
        const uint32_t dt = tmem + 256 + w * 128, at = tmem + w * 128;
#pragma unroll
        for (int ks = 0; ks < kKeyTile / 16; ++ks)
          mma_ts_elect(dt, at + ks * 8, desc_join(vl + (uint32_t)(ks * 2048 >> 4), v_hi), idesc_o,
                 (acc || ks > 0) ? 1u : 0u);
      };
      auto wait_p = [&](int w) -> bool {
        if (!warp_wait(P_FULL + 8 * w, (pbits >> w) & 1u, abort_flag, wait_ns)) return false;
        tc_fence_after();
        return true;
      };
      auto wait_ofree = [&]() -> bool {
        if (sg == 0) return true;
        if (!warp_wait(O_FREE, (sg - 1) & 1, abort_flag, wait_ns)) return false;
        tc_fence_after();
        return true;
      };
      // Test hook: DRAIN's first phase completes only through this thread's own commit
      // below, so this wait runs out, exercising the timeout path (abort, drain, free).
      if (args.stall && !warp_wait(DRAIN, 0, abort_flag, wait_ns)) ok = false;
      while (ok && next_segment(pr, u, t, t_end, S, kShare)) {
        const int n = S.n;
        qb = q_buffer(W, sg);
        if (!warp_wait(Q_FULL + 8 * qb, q_use(W, sg) & 1, abort_flag, wait_ns)) { ok = false; break; }
        tc_fence_after();
        if (W == 2) {
          // ring: K_k at ring + 2k, V_k at ring + 2k + 1
          if (!(ok = wait_kv(ring))) break;
          issue_s(0, 0, ring);
          issue_s(1, 1, ring);
          tc_commit_elect(KV_EMPTY + 8 * (ring % C::kStages));
          if (n == 1) tc_commit_elect(Q_EMPTY + 8 * qb);
          for (int k = 0; k < n && ok; ++k) {
            const int vi = ring + 2 * k + 1, ki = ring + 2 * k + 2;
            if (!(ok = wait_kv(vi))) break;
            for (int w = 0; w < 2 && ok; ++w) {
              if (!(ok = wait_p(w))) break;
              if (k == 0 && w == 0 && !(ok = wait_ofree())) break;
              issue_pv(w, vi, k > 0);
              pbits ^= 1u << w;
              if (k == n - 1) tc_commit_elect(O_FULL + 8 * w);
              if (w == 1) tc_commit_elect(KV_EMPTY + 8 * (vi % C::kStages));
              if (k + 1 < n) {
                if (w == 0 && !(ok = wait_kv(ki))) break;
                issue_s(w, w, ki);
                if (w == 1) {
                  tc_commit_elect(KV_EMPTY + 8 * (ki % C::kStages));
                  if (k + 1 == n - 1) tc_commit_elect(Q_EMPTY + 8 * qb);
                }
              }
            }
          }
        } else {
          // ring order: K0, K1, then V_j followed by K_{j+2}
          auto rK = [&](int k) { return ring + (k < 2 ? k : 2 * k - 1); };
          auto rV = [&](int j) { return ring + (j <= n - 2 ? 2 + 2 * j : 2 * n - 1); };
          if (!(ok = wait_kv(rK(0)))) break;
          issue_s(0, 0, rK(0));
          tc_commit_elect(KV_EMPTY + 8 * (rK(0) % C::kStages));
          if (n > 1) {
            if (!(ok = wait_kv(rK(1)))) break;
            issue_s(1, 0, rK(1));
            tc_commit_elect(KV_EMPTY + 8 * (rK(1) % C::kStages));
          }
          if (n <= 2) tc_commit_elect(Q_EMPTY + 8 * qb);
          for (int j = 0; j < n && ok; ++j) {
            const int w = j & 1;
            if (!(ok = wait_kv(rV(j)))) break;
            if (!(ok = wait_p(w))) break;
            if (j == 0 && !(ok = wait_ofree())) break;
            issue_pv(w, rV(j), j >= 2);
            pbits ^= 1u << w;
            tc_commit_elect(KV_EMPTY + 8 * (rV(j) % C::kStages));
            if (j + 2 >= n) tc_commit_elect(O_FULL + 8 * w);
            if (j + 2 < n) {
              if (!(ok = wait_kv(rK(j + 2)))) break;
              issue_s(w, 0, rK(j + 2));
              tc_commit_elect(KV_EMPTY + 8 * (rK(j + 2) % C::kStages));
              if (j + 2 == n - 1) tc_commit_elect(Q_EMPTY + 8 * qb);
            }
          }
        }
        ring += 2 * n;
        ++sg;
      }
      // drain: every MMA issued by this thread has completed before TMEM is freed
      tc_commit_elect(DRAIN);
      drain_wait(DRAIN, 0);
    }
  } else {
    // ------------------------------------------------------------------ softmax
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = w * 128, o_col = 256 + w * 128;
    const float sl2 = a.scale_log2;
    const int RG = pr.RG;
    int cnt = 0, of0 = 0, of1 = 0, sg = 0, trees = 0;
    bool ok = true;
    long long t = t_begin;
    Segment S;
    while (ok && next_segment(pr, u, t, t_end, S, kShare)) {
      const Loc& L = S.L;
      const int n = S.n;
      const int mt = (W == 2) ? w : 0;
      const int node = (L.mp * W + mt) * npt + r / G;  // local node id of this row
      bool row_ok = r < npt * G && node < L.s.m;
      // The tree tile (a row group's first unit, taken by stream 0 when W = 1) needs the
      // row's ancestor bits.  They depend only on the parent ids, so they are found here,
      // while the first K tile is still on its way: one parent load per thread, shared
      // through shared memory, then the walk up from the row's node.
      uint32_t anc[4] = {0u, 0u, 0u, 0u};
      if (S.tile0 == 0 && (W == 2 || w == 0)) {
        int* ps = par_s + w * 128;
        if (r < L.s.m) ps[r] = __ldg(a.parent + L.s.n0 + r);
        mbar_arrive(PAR_READY + 8 * w);
        ok = __all_sync(0xffffffffu, mbar_wait(PAR_READY + 8 * w, trees & 1, abort_flag, wait_ns));
        ++trees;
        if (!ok) break;
        if (row_ok && !ancestor_bits_shared(ps, node, anc)) set_status(a.status, kStatusBadTree);
      }
      const int n_mine = (W == 2) ? n : (n - w + 1) / 2;
      float m_run = -INFINITY, l_run = 0.f;
      for (int i = 0; i < n_mine; ++i) {
        const int k = (W == 2) ? i : 2 * i + w;
        const int tile = S.tile0 + k;
        const bool is_tree = tile == 0;
        ok = __all_sync(0xffffffffu, mbar_wait(S_FULL + 8 * w, cnt & 1, abort_flag, wait_ns));
        if (!ok) break;
        tc_fence_after();
        // keys of this tile: [0, lim) exist; the tree tile also needs the ancestor bit
        const int lim = is_tree ? L.s.m : min(kKeyTile, L.s.P - (tile - 1) * kKeyTile);
        if (is_tree || lim < kKeyTile) {
          // Rare tiles (the last, partial prefix tile; the tree tile): rewrite the logits
          // the row does not see to -inf in TMEM, 32 columns at a time, so the two
          // passes below carry no masking code.
#pragma unroll 1
          for (int ck = 0; ck < 4; ++ck) {
            uint32_t sv[32];
            tmem_ld32(tl + s_col + 32 * ck, sv);
            tmem_wait_ld32(sv);
            const int rem = lim - 32 * ck;
            uint32_t vw = rem >= 32 ? 0xffffffffu : (rem <= 0 ? 0u : (1u << rem) - 1u);
            if (is_tree) {
              const uint32_t aw = ck == 0 ? anc[0] : ck == 1 ? anc[1] : ck == 2 ? anc[2] : anc[3];
              vw &= row_ok ? aw : 0u;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((vw >> e) & 1u)) sv[e] = kNegInfBits;
            tmem_st32(tl + s_col + 32 * ck, sv);
          }
          tmem_wait_st();
        }
        // pass 1: row maximum.  All 128 columns are loaded before the one wait:
        // tcgen05.wait::ld waits for every load of the thread, so each wait is a full TMEM
        // round trip on the softmax's critical path (two per pass cost 1.5-2 us a launch).
        float mx0 = -INFINITY, mx1 = -INFINITY;
        {
          uint32_t s[128];
          tmem_ld32(tl + s_col, s);
          tmem_ld32(tl + s_col + 32, s + 32);
          tmem_ld32(tl + s_col + 64, s + 64);
          tmem_ld32(tl + s_col + 96, s + 96);
          tmem_wait_ld32(s);
          tie32(s + 32);
          tie32(s + 64);
          tie32(s + 96);
#pragma unroll
          for (int c = 0; c < 128; c += 4) {
            mx0 = max3(mx0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
            mx1 = max3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
          }
        }
        const float m_new = fmaxf(m_run, fmaxf(mx0, mx1) * sl2);
        if (i == 0) {
          m_run = m_new;
        } else {
          const bool need = m_new > m_run + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2(m_run - m_new) : 1.f;
            if (need) {
              l_run *= alpha;
              m_run = m_new;
            }
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tl + o_col + c0, o);
              tmem_wait_ld32(o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(tl + o_col + c0, o);
            }
            tmem_wait_st();
          }
        }
        const float nb = (m_run == -INFINITY) ? 0.f : -m_run;
        // pass 2: p = 2^(s * scale - m), packed as bf16 pairs into the already-read
        // first half of the S buffer (P columns 32h.. come from S columns 64h..), again
        // one round trip.  The scaling and the row sum run on packed fp32 pairs.
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nbx2 = f2_pack(nb, nb);
        uint64_t lsx2 = f2_pack(0.f, 0.f);
        {
          uint32_t s[128];
          tmem_ld32(tl + s_col, s);
          tmem_ld32(tl + s_col + 32, s + 32);
          tmem_ld32(tl + s_col + 64, s + 64);
          tmem_ld32(tl + s_col + 96, s + 96);
          tmem_wait_ld32(s);
          tie32(s + 32);
          tie32(s + 64);
          tie32(s + 96);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // the packed pairs of keys 64 h .. 64 h + 63 overwrite s[32 h ..], already read
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(s[64 * h + 2 * c]), __uint_as_float(s[64 * h + 2 * c + 1])),
                               sl2x2, nbx2),
                        x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              lsx2 = f2_add(lsx2, f2_pack(p0, p1));
              s[32 * h + c] = kBF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
            }
          }
          tmem_st32(tl + s_col, s);
          tmem_st32(tl + s_col + 32, s + 32);
        }
        float ls0, ls1;
        f2_unpack(lsx2, ls0, ls1);
        l_run += ls0 + ls1;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(P_FULL + 8 * w);
        ++cnt;
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      const size_t slot = (size_t)partial_slot(pr, u, L, kShare);
      if (slot >= (size_t)a.slots) {  // cannot happen for a consistent layout; never write past it
        set_status(a.status, kStatusInvalidArg);
        row_ok = false;
      }
      const int pp = mt * 128 + r;  // padded row: lane = row within a 32-row block
      if (row_ok && !TVA_CHECK(pp < W * 128 && node >= 0 && node < L.s.m, a.status)) row_ok = false;
      float* oblk = a.o_part + o_part_offset(slot, pp, 0, W * 128, D);
      if (W == 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(O_FULL + 8 * w, (w == 0 ? of0 : of1) & 1, abort_flag, wait_ns));
        if (!ok) break;
        (w == 0 ? of0 : of1)++;
        tc_fence_after();
        const float inv = 1.f / l_run;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          // 64 columns of the row's O per TMEM round trip (one wait covers all loads in
          // flight), then their stores
          uint32_t o[64];
          tmem_ld32(tl + o_col + c0, o);
          tmem_ld32(tl + o_col + c0 + 32, o + 32);
          tmem_wait_ld32(o);
          tie32(o + 32);
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 64; e += 4)
              *reinterpret_cast<float4*>(oblk + (c0 + e) * 32) =
                  make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                              __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
          }
        }
        if (row_ok) a.lse_part[slot * (W * 128) + pp] = m_run + log2f(l_run);
        tc_fence_before();
        mbar_arrive(O_FREE);
      } else if (w == 1) {
        // Stream 1 may own no tile of this segment (or only one whose S was issued
        // before the O_FREE wait), so nothing else keeps it from arriving for
        // segment sg before segment sg-1's release completed: wait for that first.
        if (sg > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(O_FREE, (sg - 1) & 1, abort_flag, wait_ns));
          if (!ok) break;
        }
        m1_s[(sg & 1) * 128 + r] = m_run;
        l1_s[(sg & 1) * 128 + r] = l_run;
        mbar_arrive(M1_READY);
        mbar_arrive(O_FREE);
      } else {
        ok = __all_sync(0xffffffffu, mbar_wait(M1_READY, sg & 1, abort_flag, wait_ns));
        if (!ok) break;
        const float m1 = m1_s[(sg & 1) * 128 + r];
        const float l1 = l1_s[(sg & 1) * 128 + r];
        const bool has1 = n > 1;
        ok = __all_sync(0xffffffffu, mbar_wait(O_FULL, of0 & 1, abort_flag, wait_ns));
        if (!ok) break;
        ++of0;
        if (has1) {
          ok = __all_sync(0xffffffffu, mbar_wait(O_FULL + 8, of1 & 1, abort_flag, wait_ns));
          if (!ok) break;
          ++of1;
        }
        tc_fence_after();
        const float mm = has1 ? fmaxf(m_run, m1) : m_run;
        const float a0 = (m_run == -INFINITY) ? 0.f : ex2(m_run - mm);
        const float a1 = (!has1 || m1 == -INFINITY) ? 0.f : ex2(m1 - mm);
        const float lt = a0 * l_run + a1 * l1;
        const float inv = 1.f / lt;
        const float w0 = a0 * inv, w1 = a1 * inv;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32], o1[32];
          tmem_ld32(tl + 256 + c0, o);
          tmem_ld32(tl + 384 + c0, o1);
          tmem_wait_ld32(o);
          tie32(o1);
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float4 v;
              v.x = __uint_as_float(o[e]) * w0 + (has1 ? __uint_as_float(o1[e]) * w1 : 0.f);
              v.y = __uint_as_float(o[e + 1]) * w0 + (has1 ? __uint_as_float(o1[e + 1]) * w1 : 0.f);
              v.z = __uint_as_float(o[e + 2]) * w0 + (has1 ? __uint_as_float(o1[e + 2]) * w1 : 0.f);
              v.w = __uint_as_float(o[e + 3]) * w0 + (has1 ? __uint_as_float(o1[e + 3]) * w1 : 0.f);
              *reinterpret_cast<float4*>(oblk + (c0 + e) * 32) = v;
            }
          }
        }
        if (row_ok) a.lse_part[slot * (W * 128) + pp] = mm + log2f(lt);
        tc_fence_before();
        mbar_arrive(O_FREE);
      }
      ++sg;
    }
  }
  // ------------------------------------------------------------------ teardown
  __syncwarp();
  if (threadIdx.x == 0 && *abort_flag) set_status(a.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(a.status, kStatusTimeout);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
// --------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 lookup_encode_fn() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  return nullptr;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = lookup_encode_fn();  // initialised once, thread-safe
  return fn;
}

}  // namespace

// 3-D 16-bit map over [rows][heads][d] with a box of {64, box_heads, box_rows}.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int d, int heads, long long rows,
              int box_heads, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) {
    record_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", 0, "entry point not found");
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, type, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    record_error("cuTensorMapEncodeTiled", (int)r, "tensor map rejected");
    return false;
  }
  return true;
}

void tc_wait_settings(uint64_t* wait_ns, int* stall) {
  const unsigned long long lim = g_wait_limit_ns.load(std::memory_order_relaxed);
  *wait_ns = lim > 0 ? (uint64_t)lim : kDrainNs;
  *stall = g_force_stall.load(std::memory_order_relaxed);
}

namespace {

template <int D, bool kBF16, bool kShare>
cudaError_t launch_tc_typed(const PartialArgs& a, int W, int npt, cudaStream_t s) {
  constexpr CUtensorMapDataType type = kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const Problem& pr = a.pr;
  CUtensorMap mq, mk, mv, mtk, mtv;
  const void* kbase = pr.kv_capacity > 0 ? a.k_cache : a.tree_k;
  const void* vbase = pr.kv_capacity > 0 ? a.v_cache : a.tree_v;
  if (!make_map(&mq, type, a.q, D, pr.Hq, pr.node_capacity, pr.G, npt) ||
      !make_map(&mk, type, kbase, D, pr.Hkv, pr.kv_capacity, 1, kKeyTile) ||
      !make_map(&mv, type, vbase, D, pr.Hkv, pr.kv_capacity, 1, kKeyTile) ||
      !make_map(&mtk, type, a.tree_k, D, pr.Hkv, pr.node_capacity, 1, kKeyTile) ||
      !make_map(&mtv, type, a.tree_v, D, pr.Hkv, pr.node_capacity, 1, kKeyTile))
    return cudaErrorInvalidValue;
  constexpr int smem = Cfg<D>::kSmemBytes;
  cudaError_t e = check_cuda(cudaFuncSetAttribute(partials_tc_kernel<D, kBF16, kShare>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                             "cudaFuncSetAttribute(partials_tc_kernel)");
  if (e != cudaSuccess) return e;
  TcArgs ta{a, W, npt, 0, 0};
  tc_wait_settings(&ta.wait_ns, &ta.stall);
  e = launch_pdl(partials_tc_kernel<D, kBF16, kShare>, dim3(pr.U), dim3(kThreadsTc), (size_t)smem, s, mq, mk, mv, mtk,
                 mtv, ta);
  if (e != cudaSuccess) {
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, partials_tc_kernel<D, kBF16, kShare>);
    char what[160];
    snprintf(what, sizeof(what), "%s; kernel regs %d, max threads %d, smem %d+%d", cudaGetErrorString(e),
             fa.numRegs, fa.maxThreadsPerBlock, (int)fa.sharedSizeBytes, smem);
    record_error("launch partials_tc_kernel", (int)e, what);
  }
  return e;
}

}  // namespace

void set_tc_wait_limit(unsigned long long ns, int stall) {
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  g_force_stall.store(stall != 0 ? 1 : 0, std::memory_order_relaxed);
}

template <bool kShare>
cudaError_t launch_tc_mode(const PartialArgs& a, bool bf16, int W, int npt, cudaStream_t s) {
  if (bf16)
    return a.pr.d == 64 ? launch_tc_typed<64, true, kShare>(a, W, npt, s) : launch_tc_typed<128, true, kShare>(a, W, npt, s);
  return a.pr.d == 64 ? launch_tc_typed<64, false, kShare>(a, W, npt, s) : launch_tc_typed<128, false, kShare>(a, W, npt, s);
}

cudaError_t launch_partials_tc(const PartialArgs& a, bool bf16, int W, int npt, cudaStream_t s) {
  return a.pr.share != 0 ? launch_tc_mode<true>(a, bf16, W, npt, s) : launch_tc_mode<false>(a, bf16, W, npt, s);
}

}  // namespace tva
