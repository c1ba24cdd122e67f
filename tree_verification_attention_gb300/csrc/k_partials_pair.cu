// k_partials_pair.cu - attention partials for row groups of two M-tiles, on CTA pairs
// (5th-generation tensor cores, cta_group::2; bf16 or fp16, head_dim 128).
//
// What is computed: the same partials as k_partials_tc.cu (LongSpec, "Fast Tree
// Attention": O_cache / O_specs and LSE_cache / LSE_specs of every segment of the unit
// decomposition in tva_common.cuh, the tree keys being one more 128-key tile masked by
// the row's ancestor bits), for problems whose row groups hold two M-tiles.
//
// How: clusters of two CTAs.  Pair p is worker p of the unit decomposition and CTA r of
// the pair owns M-tile r of every row group in the worker's range.  The pair's first CTA
// issues M = 256 MMAs that cover both M-tiles at once:
//   S = Q K^T  A = each CTA's own Q M-tile (shared memory); B = K, the tile's 128 keys
//              split between the CTAs (keys 64 r .. 64 r + 63 in CTA r); D = S in each
//              CTA's TMEM (its 128 rows x all 128 keys);
//   O += P V   A = P from each CTA's TMEM; B = V, head_dim split between the CTAs
//              (columns 64 r .. 64 r + 63 in CTA r); D = O in each CTA's TMEM.
// Each CTA therefore loads half of every K / V tile (16 + 16 KB a unit), the shared-
// memory operand reads of an S MMA drop from 8 to 6 KB per SM, each MMA instruction
// does the work of two, and a worker's partials are written by two CTAs (64 KB each).
// Roles per CTA (320 threads):
//   warp 8    producer (both CTAs): its M-tile of Q (two buffers, alternating by
//             segment) and its halves of the K / V tiles into an 8-stage ring of 16 KB
//             stages, in the order the MMAs consume them (K0, K1, V0, K2, V1, ...).  Every
//             load completes on the first CTA's barrier (cta_group::2 TMA), to which each
//             CTA announces its own bytes.
//   warp 9    MMA issue, first CTA only (converged warp, one elected lane); in the other
//             CTA it only takes part in the TMEM allocation.
//   warps 0-7 softmax: two streams of 4 warps; stream w takes the segment's tiles j with
//             j & 1 == w, and thread r of a stream owns TMEM lane (= row of this CTA's
//             M-tile) r and all 128 keys of a tile.  The two streams' partials are merged
//             in the epilogue.
// TMEM per CTA: stream w's S buffer at columns 128 w (P overwrites its first 64 columns
// as packed 16-bit pairs) and its O accumulator at 256 + 128 w.  The MMA order is
//   S_0(0), S_1(1), PV_0(0), S_0(2), PV_1(1), S_1(3), ...
// so each stream's softmax overlaps the other stream's MMAs, and the commit that
// publishes S_w(j + 2) also covers PV_w(j): a stream may rescale its O (when its running
// max grows by more than 2^8) as soon as its S is ready.  Each CTA collects its threads'
// release of O on a local barrier; one thread per CTA passes it to the first CTA.
//
// Every wait is bounded (mbarriers and %globaltimer); a CTA whose wait expires raises its
// own and its peer's abort flag, records TVA_ERR_TIMEOUT, drains and frees TMEM.  Both
// CTAs meet at a cluster barrier before the TMEM is released, so neither leaves while
// the other's MMAs or arrivals may still touch it.
//
// Status: selected only through tva_diag_use_cta_pair.  Measured per launch it does not
// beat the one-SM kernel on the workloads it applies to (64k prefix, 64-node tree: 55.8
// vs 51.8 us; 128k prefix, 128-node tree, G = 8, tensor-bound: 381 vs 378 us; the
// 68-node beam tree: even).  Halving the shared-memory operand reads per SM did not
// lift the tensor-bound case, so those reads are not what limits the one-SM kernel
// there.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>

#include "tc_pipeline.cuh"
#include "tc_ptx.cuh"
#include "tva_internal.h"

namespace tva {
namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kD = 128;
constexpr int kHalfBytes = 128 * 128;        // 128 rows of 64 16-bit values (one swizzle span)
constexpr int kQBuf = 2 * kHalfBytes;        // one M-tile of Q: two 64-column halves
constexpr int kStageBytes = 16384;           // one half-tile of K (64 keys x 128) or V (128 keys x 64)
constexpr int kStages = 8;
constexpr int kBarOff = 2 * kQBuf + kStages * kStageBytes;   // 192 KB
// misc region (offsets from kBarOff)
constexpr int kMiscTmem = 256;               // TMEM base address, then the abort flag
constexpr int kCnt = 272;                    // int [4]: K/V copies per CTA, Q copies per CTA
constexpr int kM1 = 512;                     // float [2][128] stream 1's row maxima (segment parity, row)
constexpr int kL1 = 1536;                    // float [2][128] stream 1's row sums
constexpr int kPar = 4608;                   // int [128] parent ids of the tree tile
constexpr int kPr = 5120;                    // Problem (staged)
constexpr int kCuOff = 5376;                 // staged cu_* arrays
constexpr int kCuCap = 1024;
constexpr int kSmemBytes = kBarOff + kCuOff + 4 * kCuCap + 1024;   // + alignment slack

struct PairArgs {
  PartialArgs a;
  int npt;           // nodes per M-tile: floor(128 / G)
  uint64_t wait_ns;  // limit of every main-loop wait
  int stall;         // test hook: the MMA thread first waits on a barrier nothing completes
};

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    partials_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_tk,
                         const __grid_constant__ CUtensorMap tm_tv, const PairArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const PartialArgs& a = args.a;
  Problem* pr_s = reinterpret_cast<Problem*>(smem + kBarOff + kPr);
  const Problem& pr = *pr_s;
  const int npt = args.npt, G = a.pr.G;  // kernel parameters: readable before staging
  const uint64_t wait_ns = args.wait_ns;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int u = blockIdx.x >> 1;          // worker (pair)

  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_s = sbase;                           // [2 buffers][2 halves][128 rows][128 B]
  const uint32_t kv_s = sbase + 2 * kQBuf;              // [kStages][16 KB]
  const uint32_t bar0 = sbase + kBarOff;
  const uint32_t KV_FULL = bar0;                        // [kStages], used in the first CTA
  const uint32_t KV_EMPTY = bar0 + 64;                  // [kStages]
  const uint32_t Q_FULL = bar0 + 128;                   // [2], used in the first CTA
  const uint32_t Q_EMPTY = bar0 + 144;                  // [2]
  const uint32_t S_FULL = bar0 + 160;                   // [2] by stream
  const uint32_t P_FULL = bar0 + 176;                   // [2] by stream, used in the first CTA
  const uint32_t O_FULL = bar0 + 192;                   // [2] by stream
  const uint32_t O_FREE = bar0 + 208;                   // used in the first CTA
  const uint32_t DRAIN = bar0 + 216;                    // used in the first CTA
  const uint32_t SEG_DONE = bar0 + 224;                 // this CTA's softmax threads are done with O
  const uint32_t M1_READY = bar0 + 232;                 // stream 1's row max / sum published
  const uint32_t PAR = bar0 + 240;                      // parent ids staged
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kMiscTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + kMiscTmem + 4);
  float* m1_s = reinterpret_cast<float*>(smem + kBarOff + kM1);
  float* l1_s = reinterpret_cast<float*>(smem + kBarOff + kL1);
  int* par_s = reinterpret_cast<int*>(smem + kBarOff + kPar);
  // the first CTA's copies of the barriers it collects arrivals on, and the peer's abort flag
  const uint32_t kv_full0 = mapa_shared(KV_FULL, 0), q_full0 = mapa_shared(Q_FULL, 0);
  const uint32_t p_full0 = mapa_shared(P_FULL, 0), o_free0 = mapa_shared(O_FREE, 0);
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);

  // ---- set-up that reads nothing an earlier kernel may write (overlaps its tail)
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_tk);
    prefetch_tmap(&tm_tv);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(KV_FULL + 8 * s, 2);    // each CTA announces its half
      mbar_init(KV_EMPTY + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(Q_FULL + 8 * b, 2);
      mbar_init(Q_EMPTY + 8 * b, 1);
      mbar_init(S_FULL + 8 * b, 1);
      mbar_init(P_FULL + 8 * b, 8);     // the stream's 4 warps in each CTA
      mbar_init(O_FULL + 8 * b, 1);
    }
    mbar_init(O_FREE, 2);               // one arrival from each CTA
    mbar_init(DRAIN, 1);
    mbar_init(SEG_DONE, 256);
    mbar_init(M1_READY, 128);
    mbar_init(PAR, 128);
    *abort_flag = 0;
    fence_mbar_init();
    __threadfence_block();
  }
  const bool params_only = a.pr.cu_prefix == nullptr;  // uniform over the grid
  long long t_begin = 0, t_end = 0;
  auto schedule = [&]() {
    stage_problem(a.pr, pr_s, reinterpret_cast<int*>(smem + kBarOff + kCuOff), kCuCap);
    worker_range(pr, u, t_begin, t_end, pr.share != 0);
  };
  if (params_only) schedule();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
  pdl_wait();          // launched as a programmatic dependent: inputs are final after this
  pdl_launch_dependents();
  if (!params_only) schedule();  // reads the caller's cu_* arrays
  if (u == 0 && rank == 0 && threadIdx.x == 0) validate_sequences(pr, a.status);
  if (t_begin >= t_end) return;  // uniform over the pair

  // TMEM (both CTAs, together); the producer warp only arrives at named barrier 1 and goes
  // straight on to its first copies.
  uint32_t tmem = 0;
  if (warp == kProducerWarp) {
    __syncwarp();
    bar_arrive(1, kThreads);
  } else {
    if (warp == kMmaWarp) {
      tmem_alloc_pair(smem_u32(tmem_slot), 512);
      tmem_relinquish_pair();
    }
    tc_fence_before();
    bar_sync(1, kThreads);
    tc_fence_after();
    tmem = *tmem_slot;
  }
  // a wait of this CTA that expires raises the peer's abort flag as well
  auto wait_or_abort = [&](bool ok) {
    if (!ok) st_shared_cluster(peer_abort, 1u);
    return ok;
  };

  int copies_kv = 0, copies_q = 0;  // this CTA's producer: K/V and Q copies issued

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    int ring = 0, sg = 0;
    bool ok = true;
    long long t = t_begin;
    Segment S;
    const uint64_t evict_first = policy_evict_first();  // K / V are read once
    while (ok && next_segment(pr, u, t, t_end, S, pr.share != 0)) {
      const Loc& L = S.L;
      const int n = S.n, qb = sg & 1;
      if (sg >= 2 && !wait_or_abort(warp_wait(Q_EMPTY + 8 * qb, ((sg >> 1) - 1) & 1, abort_flag, wait_ns))) {
        ok = false;
        break;
      }
      int qrow = L.s.n0 + (L.mp * 2 + (int)rank) * npt;
      if (!TVA_CHECK(qrow >= L.s.n0 && L.g >= 0 && L.g < pr.Hkv, a.status)) qrow = 0;
      mbar_expect_tx_cluster_elect(q_full0 + 8 * qb, 2u * 64u * (uint32_t)(G * npt) * 2u);  // two boxes
      for (int h = 0; h < 2; ++h)
        tma_load_3d_pair_nohint_elect(q_s + qb * kQBuf + h * kHalfBytes, &tm_q, 64 * h, L.g * G, qrow,
                                      q_full0 + 8 * qb);
      auto load = [&](int k, bool is_v) -> bool {
        const int stage = ring % kStages, use = ring / kStages;
        if (use > 0 && !wait_or_abort(warp_wait(KV_EMPTY + 8 * stage, (use - 1) & 1, abort_flag, wait_ns)))
          return false;
        const int tile = S.tile0 + k;
        const bool tree = tile == 0;
        int z = tree ? L.s.n0 : L.s.p0 + (tile - 1) * kKeyTile;
        if (!TVA_CHECK(z >= 0 && (tree ? z < pr.node_capacity && L.s.m > 0
                                       : z < L.s.p0 + L.s.P && z < pr.kv_capacity), a.status))
          z = 0;
        const uint32_t dst = kv_s + stage * kStageBytes;
        mbar_expect_tx_cluster_elect(kv_full0 + 8 * stage, kStageBytes);
        if (!is_v) {  // keys 64 r .. 64 r + 63 of the tile, both 64-column halves
          for (int h = 0; h < 2; ++h)
            tma_load_3d_pair_elect(dst + h * (kStageBytes / 2), tree ? &tm_tk : &tm_k, 64 * h, L.g,
                                   z + 64 * (int)rank, kv_full0 + 8 * stage, evict_first);
        } else {      // columns 64 r .. 64 r + 63 of all 128 keys
          tma_load_3d_pair_elect(dst, tree ? &tm_tv : &tm_v, 64 * (int)rank, L.g, z, kv_full0 + 8 * stage,
                                 evict_first);
        }
        ++ring;
        return true;
      };
      ok = load(0, false);
      if (ok && n > 1) ok = load(1, false);
      for (int j = 0; j < n && ok; ++j) {
        ok = load(j, true);
        if (ok && j + 2 < n) ok = load(j + 2, false);
      }
      ++sg;
    }
    copies_kv = ring;
    copies_q = sg;  // drained at teardown, where both CTAs' counts are known
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issue
    if (rank == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(256, 128, false, kBF16);
      constexpr uint32_t idesc_o = idesc_bf16(256, 128, true, kBF16);
      int ring = 0, sg = 0;
      uint32_t pbits = 0;  // bit w: parity of the next P_FULL[w] phase
      bool ok = true;
      long long t = t_begin;
      Segment S;
      auto wait_kv = [&](int idx) -> bool {
        if (!wait_or_abort(warp_wait(KV_FULL + 8 * (idx % kStages), (idx / kStages) & 1, abort_flag, wait_ns)))
          return false;
        tc_fence_after();
        return true;
      };
      // operand descriptors, built once and stepped through their low word: Q and K are
      // K-major (head_dim contiguous), V is MN-major (head_dim contiguous, N = head_dim)
      const uint32_t k_hi = (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32);
      const uint32_t v_hi = (uint32_t)(sdesc_sw128(0, kStageBytes, 1024) >> 32);
      const uint32_t k_lo = (uint32_t)sdesc_sw128(kv_s, 16, 1024);
      const uint32_t v_lo = (uint32_t)sdesc_sw128(kv_s, kStageBytes, 1024);
      const uint32_t q_lo = (uint32_t)sdesc_sw128(q_s, 16, 1024);
      // S of stream w into its buffer (TMEM columns 128 w)
      auto issue_s = [&](int w, int qb, int idx) {
        const uint32_t kl = k_lo + (uint32_t)((idx % kStages) * kStageBytes >> 4);
        const uint32_t ql = q_lo + (uint32_t)(qb * kQBuf >> 4);
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t oq = (uint32_t)((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
          const uint32_t ok_ = (uint32_t)((ks >> 2) * (kStageBytes / 2) + (ks & 3) * 32) >> 4;
          mma2_ss_elect(tmem + 128 * w, desc_join(ql + oq, k_hi), desc_join(kl + ok_, k_hi), idesc_s, ks > 0);
        }
        tc_commit2_elect(S_FULL + 8 * w, 3);
        tc_commit2_elect(KV_EMPTY + 8 * (idx % kStages), 3);
      };
      // O_w += P_w V, P_w read from the first 64 columns of stream w's S buffer
      auto issue_pv = [&](int w, int idx, bool acc) {
        const uint32_t vl = v_lo + (uint32_t)((idx % kStages) * kStageBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < kKeyTile / 16; ++ks)
          mma2_ts_elect(tmem + 256 + 128 * w, tmem + 128 * w + ks * 8,
                        desc_join(vl + (uint32_t)(ks * 2048 >> 4), v_hi), idesc_o, (acc || ks > 0) ? 1u : 0u);
        tc_commit2_elect(KV_EMPTY + 8 * (idx % kStages), 3);
      };
      // Test hook: DRAIN's first phase completes only through this thread's own commit
      // below, so this wait runs out, exercising the timeout path (abort, drain, free).
      if (args.stall && !wait_or_abort(warp_wait(DRAIN, 0, abort_flag, wait_ns))) ok = false;
      while (ok && next_segment(pr, u, t, t_end, S, pr.share != 0)) {
        const int n = S.n, qb = sg & 1;
        // ring order: K0, K1, then V_j followed by K_{j+2}; tile j belongs to stream j & 1
        auto rK = [&](int k) { return ring + (k < 2 ? k : 2 * k - 1); };
        auto rV = [&](int j) { return ring + (j <= n - 2 ? 2 + 2 * j : 2 * n - 1); };
        if (!(ok = wait_or_abort(warp_wait(Q_FULL + 8 * qb, (sg >> 1) & 1, abort_flag, wait_ns)))) break;
        tc_fence_after();
        if (!(ok = wait_kv(rK(0)))) break;
        issue_s(0, qb, rK(0));
        if (n > 1) {
          if (!(ok = wait_kv(rK(1)))) break;
          issue_s(1, qb, rK(1));
        }
        if (n <= 2) tc_commit2_elect(Q_EMPTY + 8 * qb, 3);
        for (int j = 0; j < n && ok; ++j) {
          const int w = j & 1;
          if (!(ok = wait_kv(rV(j)))) break;
          if (!(ok = wait_or_abort(warp_wait(P_FULL + 8 * w, (pbits >> w) & 1u, abort_flag, wait_ns)))) break;
          tc_fence_after();
          pbits ^= 1u << w;
          if (j == 0 && sg > 0) {  // both CTAs have read the previous segment's O
            if (!(ok = wait_or_abort(warp_wait(O_FREE, (sg - 1) & 1, abort_flag, wait_ns)))) break;
            tc_fence_after();
          }
          issue_pv(w, rV(j), j >= 2);
          if (j + 2 >= n) tc_commit2_elect(O_FULL + 8 * w, 3);
          if (j + 2 < n) {
            if (!(ok = wait_kv(rK(j + 2)))) break;
            issue_s(w, qb, rK(j + 2));
            if (j + 2 == n - 1) tc_commit2_elect(Q_EMPTY + 8 * qb, 3);
          }
        }
        ring += 2 * n;
        ++sg;
      }
      // drain: every MMA issued here (on either CTA's memory) has completed
      tc_commit2_elect(DRAIN, 1);
      drain_wait(DRAIN, 0);
    }
  } else {
    // ------------------------------------------------------------------ softmax
    // Two streams of 4 warps; stream w takes the segment's tiles j with j & 1 == w, thread
    // r of a stream owns TMEM lane (= row of this CTA's M-tile) r and all 128 keys of a
    // tile.  A stream's running max moves only when it grows by more than 2^8 (stale
    // maxima cancel in the final division); then its O is rescaled in TMEM, which is
    // safe once its S is ready: the commit that publishes S_w(j + 2) follows PV_w(j).
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = 128 * w, o_col = 256 + 128 * w;
    const float sl2 = a.scale_log2;
    // phase parities: bit 0 this stream's S_FULL, 1 / 2 O_FULL[0] / O_FULL[1], 3 PAR
    uint32_t ph = 0;
    int sg = 0;
    bool ok = true;
    long long t = t_begin;
    Segment S;
    auto bwait = [&](uint32_t bar, uint32_t parity) {
      return wait_or_abort(__all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, wait_ns)));
    };
    while (ok && next_segment(pr, u, t, t_end, S, pr.share != 0)) {
      const Loc& L = S.L;
      const int n = S.n;
      const int node = (L.mp * 2 + (int)rank) * npt + r / G;  // local node id of this row
      bool row_ok = r < npt * G && node < L.s.m;
      uint32_t anc[4] = {0u, 0u, 0u, 0u};
      if (S.tile0 == 0 && w == 0) {  // the tree tile (stream 0's): ancestor bits while K0 loads
        if (r < L.s.m) par_s[r] = __ldg(a.parent + L.s.n0 + r);
        mbar_arrive(PAR);
        if (!(ok = bwait(PAR, (ph >> 3) & 1))) break;
        ph ^= 8u;
        if (row_ok && !ancestor_bits_shared(par_s, node, anc)) set_status(a.status, kStatusBadTree);
      }
      const int n_mine = (n - w + 1) / 2;
      float m_run = -INFINITY, l_run = 0.f;
      for (int i = 0; i < n_mine; ++i) {
        const int tile = S.tile0 + 2 * i + w;
        const bool is_tree = tile == 0;
        if (!(ok = bwait(S_FULL + 8 * w, ph & 1))) break;
        tc_fence_after();
        // keys of this tile: [0, lim) exist; the tree tile also needs the ancestor bit
        const int lim = is_tree ? L.s.m : min(kKeyTile, L.s.P - (tile - 1) * kKeyTile);
        if (is_tree || lim < kKeyTile) {  // rare tiles: logits the row does not see -> -inf
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
        // pass 1: row maximum; all 128 columns loaded before the one wait (each
        // tcgen05.wait::ld is a full TMEM round trip on the critical path)
        float mx0 = -INFINITY, mx1 = -INFINITY;
        {
          uint32_t sv[128];
          tmem_ld32(tl + s_col, sv);
          tmem_ld32(tl + s_col + 32, sv + 32);
          tmem_ld32(tl + s_col + 64, sv + 64);
          tmem_ld32(tl + s_col + 96, sv + 96);
          tmem_wait_ld32(sv);
          tie32(sv + 32);
          tie32(sv + 64);
          tie32(sv + 96);
#pragma unroll
          for (int c = 0; c < 128; c += 4) {
            mx0 = max3(mx0, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
            mx1 = max3(mx1, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
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
            for (int c0 = 0; c0 < kD; c0 += 32) {
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
        // pass 2: p = 2^(s * scale - m), packed as 16-bit pairs into the already-read
        // first half of the S buffer (P columns 32 h.. come from S columns 64 h..)
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nbx2 = f2_pack(nb, nb);
        uint64_t lsx2 = f2_pack(0.f, 0.f);
        {
          uint32_t sv[128];
          tmem_ld32(tl + s_col, sv);
          tmem_ld32(tl + s_col + 32, sv + 32);
          tmem_ld32(tl + s_col + 64, sv + 64);
          tmem_ld32(tl + s_col + 96, sv + 96);
          tmem_wait_ld32(sv);
          tie32(sv + 32);
          tie32(sv + 64);
          tie32(sv + 96);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // the packed pairs of keys 64 h .. 64 h + 63 overwrite sv[32 h ..], already read
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[64 * h + 2 * c]), __uint_as_float(sv[64 * h + 2 * c + 1])),
                               sl2x2, nbx2),
                        x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              lsx2 = f2_add(lsx2, f2_pack(p0, p1));
              sv[32 * h + c] = kBF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
            }
          }
          tmem_st32(tl + s_col, sv);
          tmem_st32(tl + s_col + 32, sv + 32);
        }
        float ls0, ls1;
        f2_unpack(lsx2, ls0, ls1);
        l_run += ls0 + ls1;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(p_full0 + 8 * w);
        ph ^= 1u;
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      // Stream 1 hands its row max / sum to stream 0, which merges the two O accumulators.
      // Each CTA's release of O is collected on SEG_DONE and passed to the first CTA's
      // O_FREE by one thread, so neither stream can arrive for the next segment before
      // this segment's phase is complete.
      if (w == 1) {
        if (sg > 0 && !(ok = bwait(SEG_DONE, (sg - 1) & 1))) break;
        m1_s[(sg & 1) * 128 + r] = m_run;
        l1_s[(sg & 1) * 128 + r] = l_run;
        mbar_arrive(M1_READY);
        mbar_arrive(SEG_DONE);
      } else {
        if (!(ok = bwait(M1_READY, sg & 1))) break;
        const float m1 = m1_s[(sg & 1) * 128 + r];
        const float l1 = l1_s[(sg & 1) * 128 + r];
        const bool has1 = n > 1;
        if (!(ok = bwait(O_FULL, (ph >> 1) & 1))) break;
        ph ^= 2u;
        if (has1) {
          if (!(ok = bwait(O_FULL + 8, (ph >> 2) & 1))) break;
          ph ^= 4u;
        }
        tc_fence_after();
        const float mm = has1 ? fmaxf(m_run, m1) : m_run;
        const float a0 = (m_run == -INFINITY) ? 0.f : ex2(m_run - mm);
        const float a1 = (!has1 || m1 == -INFINITY) ? 0.f : ex2(m1 - mm);
        const float lt = a0 * l_run + a1 * l1;
        const float inv = 1.f / lt;
        const float w0 = a0 * inv, w1 = a1 * inv;
        const size_t slot = (size_t)partial_slot(pr, u, L, pr.share != 0);
        if (slot >= (size_t)a.slots) {  // cannot happen for a consistent layout; never write past it
          set_status(a.status, kStatusInvalidArg);
          row_ok = false;
        }
        const int pp = (int)rank * 128 + r;  // padded row: lane = row within a 32-row block
        if (row_ok && !TVA_CHECK(node >= 0 && node < L.s.m, a.status)) row_ok = false;
        float* oblk = a.o_part + o_part_offset(slot, pp, 0, 256, kD);
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 32) {
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
        if (row_ok) a.lse_part[slot * 256 + pp] = mm + log2f(lt);
        tc_fence_before();
        mbar_arrive(SEG_DONE);
        if (warp == 0) {
          if (!(ok = bwait(SEG_DONE, sg & 1))) break;
          if (lane == 0) mbar_arrive_cluster(o_free0);
        }
      }
      ++sg;
    }
  }
  // ------------------------------------------------------------------ teardown
  // Both CTAs' copies complete on the first CTA's barriers, so that CTA drains them all.
  // In a normal run the two producers issue the same copies; after an expired wait one
  // may have stopped earlier (by at most one ring of K/V copies and two Q copies, since
  // a stage is reused only once both halves of its previous copy landed).  Each producer
  // therefore tells the other how many copies it issued, adds a plain arrival for every
  // copy the other issued beyond its own (completing those phases once their bytes land),
  // and the first CTA waits for the last phase of every stage up to the larger count.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  int* cnt = reinterpret_cast<int*>(smem + kBarOff + kCnt);
  if (warp == kProducerWarp && lane == 0) {
    cnt[rank] = copies_kv;
    cnt[2 + rank] = copies_q;
    st_shared_cluster(mapa_shared(smem_u32(cnt + rank), rank ^ 1u), (uint32_t)copies_kv);
    st_shared_cluster(mapa_shared(smem_u32(cnt + 2 + rank), rank ^ 1u), (uint32_t)copies_q);
  }
  cluster_sync_all();  // the counts are visible in both CTAs
  if (warp == kProducerWarp && lane == 0) {
    const int kv_all = max(cnt[0], cnt[1]), q_all = max(cnt[2], cnt[3]);
    for (int i = copies_kv; i < kv_all; ++i) mbar_arrive_cluster(kv_full0 + 8 * (i % kStages));
    for (int i = copies_q; i < q_all; ++i) mbar_arrive_cluster(q_full0 + 8 * (i & 1));
    if (rank == 0) {
      for (int i = max(0, kv_all - kStages); i < kv_all; ++i)
        drain_wait(KV_FULL + 8 * (i % kStages), (i / kStages) & 1);
      for (int b = 0; b < 2; ++b) {  // the last copy into each Q buffer
        const int uses = (q_all + 1 - b) / 2;
        if (uses > 0) drain_wait(Q_FULL + 8 * b, (uses - 1) & 1);
      }
    }
  }
  __syncwarp();
  if (threadIdx.x == 0 && *abort_flag) set_status(a.status, kStatusTimeout);
  cluster_sync_all();  // neither CTA leaves while the other's MMAs, copies or arrivals may touch it
  if (threadIdx.x == 0 && *abort_flag) set_status(a.status, kStatusTimeout);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

template <bool kBF16>
cudaError_t launch_pair_typed(const PartialArgs& a, int npt, cudaStream_t s) {
  constexpr CUtensorMapDataType type = kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const Problem& pr = a.pr;
  CUtensorMap mq, mk, mv, mtk, mtv;
  const void* kbase = pr.kv_capacity > 0 ? a.k_cache : a.tree_k;
  const void* vbase = pr.kv_capacity > 0 ? a.v_cache : a.tree_v;
  // K boxes hold 64 keys (half a tile), V boxes 128 keys x 64 columns
  if (!make_map(&mq, type, a.q, kD, pr.Hq, pr.node_capacity, pr.G, npt) ||
      !make_map(&mk, type, kbase, kD, pr.Hkv, pr.kv_capacity, 1, kKeyTile / 2) ||
      !make_map(&mv, type, vbase, kD, pr.Hkv, pr.kv_capacity, 1, kKeyTile) ||
      !make_map(&mtk, type, a.tree_k, kD, pr.Hkv, pr.node_capacity, 1, kKeyTile / 2) ||
      !make_map(&mtv, type, a.tree_v, kD, pr.Hkv, pr.node_capacity, 1, kKeyTile))
    return cudaErrorInvalidValue;
  cudaError_t e = check_cuda(cudaFuncSetAttribute(partials_pair_kernel<kBF16>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes),
                             "cudaFuncSetAttribute(partials_pair_kernel)");
  if (e != cudaSuccess) return e;
  PairArgs pa{a, npt, 0, 0};
  tc_wait_settings(&pa.wait_ns, &pa.stall);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pr.U);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, partials_pair_kernel<kBF16>, mq, mk, mv, mtk, mtv, pa);
  if (e != cudaSuccess) {
    char what[160];
    snprintf(what, sizeof(what), "%s; %d pairs, smem %d", cudaGetErrorString(e), pr.U, kSmemBytes);
    record_error("launch partials_pair_kernel", (int)e, what);
  }
  return e;
}

}  // namespace

cudaError_t launch_partials_pair(const PartialArgs& a, bool bf16, int npt, cudaStream_t s) {
  return bf16 ? launch_pair_typed<true>(a, npt, s) : launch_pair_typed<false>(a, npt, s);
}

}  // namespace tva
