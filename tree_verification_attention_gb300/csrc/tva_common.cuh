// tva_common.cuh - work decomposition and small helpers shared by the kernels.
//
// Work decomposition ("units")
// ----------------------------
// Rows: for KV head g of sequence b, the m_b * G query rows (node i, query head
// g*G + j) are numbered r = i*G + j and cut into row groups of RG = 128 * W rows.
// Keys: each row group sees the P_b prefix keys, cut into tiles of 128, plus ONE more
// tile holding the sequence's tree keys (masked to ancestors-and-self), which comes
// first: tile 0 is the tree tile and tile t >= 1 holds prefix keys [128 (t-1), 128 t).
// (Its masking work then falls where a worker's pipeline is still filling instead of
// at the end of the launch.)
// A unit is one (row group, key tile) pair.  Units are numbered sequence by sequence,
// KV head by KV head, row group by row group, tile by tile (the tree tile first).  The
// U workers (CTAs) take equal contiguous ranges of c = ceil(T / U) units, so a
// worker's range can cross row-group boundaries; each maximal piece of a range inside
// one row group is a "segment" and produces one partial (O, LSE) per row.  The
// segment of worker u in row group q is stored in slot u + q: distinct pieces never
// share a slot, because worker u+1 starting inside group q-1 would contradict worker
// u reaching group q.  Partials therefore need at most U + Q slots (Q row groups).
//
// Two refinements for one sequence (see Problem::align and Problem::share): with one
// row group per KV head, each head's tiles are split evenly over its own workers (no
// range crosses a group); with several, workers form teams, one member per row group,
// that walk the same (KV head, key tile) columns side by side, so the K/V tiles come
// from DRAM once; a member's partials go to slots r (Q + Hkv) + k + g.
//
// Both the partials kernels and the combine kernel recompute this map from
// cu_prefix / cu_nodes, so no schedule table is stored.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace tva {

constexpr int kKeyTile = 128;   // keys per unit
constexpr int kMaxNodes = 128;  // tree nodes per sequence (ancestor mask = 4 words)

enum : int {
  kStatusOk = 0,
  kStatusInvalidArg = 1,
  kStatusBadTree = 3,
  kStatusTimeout = 6,
};

struct Problem {
  const int32_t* cu_prefix;  // null: single sequence of single_prefix keys
  const int32_t* cu_nodes;   // null: single sequence of single_nodes nodes
  int single_prefix, single_nodes;
  int B, Hq, Hkv, G, d;
  int RG;                    // rows per row group
  int U;                     // workers
  int max_prefix, max_nodes, kv_capacity, node_capacity;
  // 0: workers take contiguous ranges of units (stream-K).  S >= 2 (one sequence whose
  // KV heads have S row groups): workers form teams of S; team k takes a contiguous
  // range of (KV head, key tile) columns and its member r computes row group r over it,
  // so the team's S workers stream the same K/V tiles together and DRAM serves each
  // tile once (the others read it from L2).
  int share;
  // 0, or (one sequence, one row group per KV head, Hkv dividing U) the workers per row
  // group: each row group's tiles are split evenly over its own workers, so no worker's
  // range crosses into another row group (stream-K ranges do, and such a worker pays a
  // second segment - epilogue, Q copy, tree tile - in the middle of its stream).
  int align;
};

struct SeqInfo {
  int p0, P;   // first k_cache row, prefix length
  int n0, m;   // first node row, tree size
  bool ok;     // false: bounds violated (sequence treated as empty)
};

__device__ __forceinline__ void set_status(int32_t* st, int code) {
  if (st != nullptr) atomicCAS(reinterpret_cast<int*>(st), 0, code);
}

// Checked build (compiled with -DTVA_CHECKED; libtva_checked.so).  TVA_CHECK(cond, st)
// guards an index the kernels compute themselves - a TMA tile coordinate, a partial slot,
// an output row, a position on an accepted path - that a consistent schedule keeps in
// bounds.  In the checked build a failed check records TVA_ERR_INVALID_ARG in *st and
// evaluates to false, so the access is skipped (or its coordinate clamped); nothing
// traps.  In the normal build the checks compile to `true`.
__device__ __forceinline__ bool checked_ok(bool cond, int32_t* st) {
  if (!cond) set_status(st, kStatusInvalidArg);
  return cond;
}
#ifdef TVA_CHECKED
#define TVA_CHECK(cond, st) (::tva::checked_ok((cond), (st)))
#else
#define TVA_CHECK(cond, st) (true)
#endif

__device__ __forceinline__ SeqInfo seq_info(const Problem& pr, int b) {
  SeqInfo s;
  if (pr.cu_prefix == nullptr) {
    s.p0 = 0; s.P = pr.single_prefix; s.n0 = 0; s.m = pr.single_nodes;
  } else {
    // plain (generic) loads: the arrays may have been staged in shared memory
    s.p0 = pr.cu_prefix[b];
    s.P = pr.cu_prefix[b + 1] - s.p0;
    s.n0 = pr.cu_nodes[b];
    s.m = pr.cu_nodes[b + 1] - s.n0;
  }
  s.ok = s.p0 >= 0 && s.P >= 0 && s.P <= pr.max_prefix && s.p0 + s.P <= pr.kv_capacity &&
         s.n0 >= 0 && s.m >= 0 && s.m <= pr.max_nodes && s.n0 + s.m <= pr.node_capacity;
  if (!s.ok) { s.P = 0; s.m = 0; }
  return s;
}

// Copies cu_prefix / cu_nodes into `buf` (2 * (B + 1) ints of shared memory) when they
// fit in `cap` ints, and points `pr` at the copies, so that the sequence walks below
// cost shared-memory loads instead of one round of global loads per sequence.  Every
// thread of the block must call it; it ends with a block barrier.
__device__ __forceinline__ void stage_cu(Problem& pr, int* buf, int cap) {
  const bool fits = pr.cu_prefix != nullptr && 2 * (pr.B + 1) <= cap;
  if (fits) {
    for (int i = threadIdx.x; i <= pr.B; i += blockDim.x) {
      buf[i] = __ldg(pr.cu_prefix + i);
      buf[pr.B + 1 + i] = __ldg(pr.cu_nodes + i);
    }
  }
  __syncthreads();
  if (fits) {
    pr.cu_prefix = buf;
    pr.cu_nodes = buf + pr.B + 1;
  }
}

// Same, but the resulting problem description is also placed in shared memory (`dst`),
// so that kernels short of registers can read its fields from there.
__device__ __forceinline__ void stage_problem(const Problem& src, Problem* dst, int* buf, int cap) {
  const bool fits = src.cu_prefix != nullptr && 2 * (src.B + 1) <= cap;
  if (fits) {
    for (int i = threadIdx.x; i <= src.B; i += blockDim.x) {
      buf[i] = __ldg(src.cu_prefix + i);
      buf[src.B + 1 + i] = __ldg(src.cu_nodes + i);
    }
  }
  if (threadIdx.x == 0) {
    *dst = src;
    if (fits) {
      dst->cu_prefix = buf;
      dst->cu_nodes = buf + src.B + 1;
    }
  }
  __syncthreads();
}

// Reports (once, from one thread) a cu_* entry outside the stated bounds.  The
// offending sequence is treated as empty by every kernel.
__device__ __forceinline__ void validate_sequences(const Problem& pr, int32_t* status) {
  for (int b = 0; b < pr.B; ++b) {
    if (!seq_info(pr, b).ok) {
      set_status(status, kStatusInvalidArg);
      return;
    }
  }
}

__device__ __forceinline__ int seq_tiles(int P) { return (P + kKeyTile - 1) / kKeyTile + 1; }
__device__ __forceinline__ int seq_groups(const Problem& pr, int m) {
  return (m * pr.G + pr.RG - 1) / pr.RG;
}

// Total units T and the chunk size c = ceil(T / U).
__device__ __forceinline__ long long total_units(const Problem& pr) {
  long long T = 0;
  for (int b = 0; b < pr.B; ++b) {
    SeqInfo s = seq_info(pr, b);
    T += (long long)pr.Hkv * seq_groups(pr, s.m) * seq_tiles(s.P);
  }
  return T;
}

__device__ __forceinline__ long long chunk_units(const Problem& pr, long long T) {
  return (T + pr.U - 1) / pr.U;
}

// Where unit t lives.
struct Loc {
  SeqInfo s;
  int b;
  int g, mp;          // KV head, row group within (b, g)
  int MP;             // row groups per (b, g)
  int tiles;          // units per row group (prefix tiles + 1 tree tile)
  int tile;           // tile index of unit t inside its row group
  int q;              // global row-group index
  long long start;    // global index of the row group's first unit
};

__device__ __forceinline__ Loc locate_unit(const Problem& pr, long long t) {
  Loc L;
  long long acc = 0;
  int qacc = 0;
  for (int b = 0; b < pr.B; ++b) {
    SeqInfo s = seq_info(pr, b);
    int MP = seq_groups(pr, s.m);
    int tiles = seq_tiles(s.P);
    long long units = (long long)pr.Hkv * MP * tiles;
    if (t < acc + units) {
      long long local = t - acc;
      int gi = (int)(local / tiles);
      L.s = s; L.b = b; L.MP = MP; L.tiles = tiles;
      L.g = gi / MP; L.mp = gi % MP;
      L.tile = (int)(local % tiles);
      L.q = qacc + gi;
      L.start = acc + (long long)gi * tiles;
      return L;
    }
    acc += units;
    qacc += pr.Hkv * MP;
  }
  L.b = -1;  // not reached for t < T
  return L;
}

// Row group of query row (node n, head h), for the combine.
struct RowLoc {
  SeqInfo s;
  int b, q, r;        // sequence, global row group, row inside the group
  int tiles;
  long long start;    // first unit of the row group
  long long T;        // total units
};

__device__ __forceinline__ bool locate_row(const Problem& pr, int n, int h, RowLoc& R) {
  long long acc = 0;
  int qacc = 0;
  bool found = false;
  for (int b = 0; b < pr.B; ++b) {
    SeqInfo s = seq_info(pr, b);
    int MP = seq_groups(pr, s.m);
    int tiles = seq_tiles(s.P);
    if (!found && n >= s.n0 && n < s.n0 + s.m) {
      int g = h / pr.G, j = h % pr.G;
      int rs = (n - s.n0) * pr.G + j;
      int mp = rs / pr.RG;
      R.s = s; R.b = b; R.r = rs % pr.RG; R.tiles = tiles;
      R.q = qacc + g * MP + mp;
      R.start = acc + (long long)(g * MP + mp) * tiles;
      found = true;
    }
    acc += (long long)pr.Hkv * MP * tiles;
    qacc += pr.Hkv * MP;
  }
  R.T = acc;
  return found;
}

// ---- A worker's work.  Walk positions are units in stream-K mode and (KV head, key
// tile) columns of the one sequence in shared mode; a segment is a maximal run of a
// worker's positions inside one row group.
struct Segment {
  Loc L;
  int tile0, n;
};

// Shared mode: teams, and the columns a team takes.
__device__ __forceinline__ int share_teams(const Problem& pr) { return pr.U / pr.share; }
__device__ __forceinline__ long long share_columns_per_team(const Problem& pr, int tiles) {
  const long long C = (long long)pr.Hkv * tiles;
  const int Q = share_teams(pr);
  return (C + Q - 1) / Q;
}

// Worker u's walk positions [t0, t1).  `shared` is pr.share != 0; kernels that know it
// at compile time pass a constant, so the other mode's code is not in them.
__device__ __forceinline__ void worker_range(const Problem& pr, int u, long long& t0, long long& t1, bool shared) {
  if (!shared) {
    if (pr.align > 0) {  // worker j of row group q: its share of the group's tiles
      const SeqInfo s = seq_info(pr, 0);
      const int tiles = seq_tiles(s.P), q = u / pr.align, j = u - q * pr.align;
      t0 = t1 = 0;
      if (q >= pr.Hkv * seq_groups(pr, s.m)) return;
      const int base = tiles / pr.align, extra = tiles - base * pr.align;
      const long long start = (long long)q * tiles + (long long)j * base + (j < extra ? j : extra);
      t0 = start;
      t1 = start + base + (j < extra ? 1 : 0);
      return;
    }
    const long long T = total_units(pr);
    const long long c = chunk_units(pr, T);
    t0 = (long long)u * c;
    t1 = t0 + c < T ? t0 + c : T;
    return;
  }
  const SeqInfo s = seq_info(pr, 0);
  const int MP = seq_groups(pr, s.m), tiles = seq_tiles(s.P);
  const int k = u / pr.share, r = u - k * pr.share;
  t0 = t1 = 0;
  if (k >= share_teams(pr) || r >= MP) return;  // no such row group, or a spare worker
  const long long C = (long long)pr.Hkv * tiles, cc = share_columns_per_team(pr, tiles);
  t0 = k * cc < C ? k * cc : C;
  t1 = t0 + cc < C ? t0 + cc : C;
}

// The segment of worker u's walk that starts at t; advances t past it.
__device__ __forceinline__ bool next_segment(const Problem& pr, int u, long long& t, long long t_end, Segment& seg,
                                             bool shared) {
  if (t >= t_end) return false;
  long long end;
  if (!shared) {
    seg.L = locate_unit(pr, t);
    end = seg.L.start + seg.L.tiles;
  } else {
    Loc& L = seg.L;
    L.s = seq_info(pr, 0);
    L.b = 0;
    L.MP = seq_groups(pr, L.s.m);
    L.tiles = seq_tiles(L.s.P);
    L.g = (int)(t / L.tiles);
    L.mp = u % pr.share;
    L.tile = (int)(t - (long long)L.g * L.tiles);
    L.q = L.g * L.MP + L.mp;
    L.start = (long long)L.q * L.tiles;
    end = (long long)(L.g + 1) * L.tiles;
  }
  if (end > t_end) end = t_end;
  seg.tile0 = seg.L.tile;
  seg.n = (int)(end - t);
  t = end;
  return true;
}

// The workspace slot of worker u's partial for the row group of L.  Stream-K: u + q
// (a worker's row groups are consecutive, so no two (worker, group) pairs collide).
// Shared mode, team k, member r, KV head g: r (Q + Hkv) + k + g (the teams covering a head
// are consecutive, so k + g is unique for each r, and a group's partials are adjacent).
__device__ __forceinline__ long long partial_slot(const Problem& pr, int u, const Loc& L, bool shared) {
  if (!shared) return (long long)u + L.q;
  const int k = u / pr.share, r = u - k * pr.share;
  return (long long)r * (share_teams(pr) + pr.Hkv) + k + L.g;
}

// Partial-output layout.  A row group of RG = W * MT rows (W M-tiles of MT =
// floor(128 / G) * G rows) occupies W * 128 padded rows per slot: row r of M-tile mt is
// padded row mt * 128 + r.  LSE partials are [slot][padded row].  O partials are stored
// in 32-row blocks, each column-group major - [block][d / 4][32 rows][4 floats] - so that
// a warp whose lanes hold 32 consecutive rows writes, and the combine reads, 512
// contiguous bytes per 16-byte access.
__host__ __device__ __forceinline__ int mtile_rows(int G) { return (128 / G) * G; }
__host__ __device__ __forceinline__ int padded_group_rows(int RG, int G) { return RG / mtile_rows(G) * 128; }
// float offset of column group cg (4 floats) of padded row pp in slot `slot`
__host__ __device__ __forceinline__ size_t o_part_offset(size_t slot, int pp, int cg, int RGP, int D) {
  return (slot * RGP + (pp & ~31)) * D + (size_t)cg * 128 + (pp & 31) * 4;
}

// Where row group qg lives, for the combine.
struct GroupLoc {
  SeqInfo s;
  int b, g, mp;       // sequence, KV head, row group within (b, g)
  int tiles;          // units of the row group
  long long start;    // first unit of the row group
  long long T;        // total units
  bool found;
};

__device__ __forceinline__ GroupLoc locate_group(const Problem& pr, long long qg) {
  GroupLoc R;
  R.found = false;
  R.b = R.g = R.mp = R.tiles = 0;
  R.start = 0;
  long long acc = 0, qacc = 0;
  for (int b = 0; b < pr.B; ++b) {
    const SeqInfo s = seq_info(pr, b);
    const int MP = seq_groups(pr, s.m);
    const int tiles = seq_tiles(s.P);
    const long long nq = (long long)pr.Hkv * MP;
    if (!R.found && qg >= qacc && qg < qacc + nq) {
      const long long gi = qg - qacc;
      R.s = s; R.b = b; R.g = (int)(gi / MP); R.mp = (int)(gi % MP); R.tiles = tiles;
      R.start = acc + gi * tiles;
      R.found = true;
    }
    acc += nq * tiles;
    qacc += nq;
  }
  R.T = acc;
  return R;
}

// Ancestor-or-self bit mask of tree node i (local id) over local ids 0..127, from the
// sequence's parent ids staged in shared memory (`par`): bit c set iff node c is i or an
// ancestor of i.  Returns false if a parent id met on the walk is outside [-1, node)
// (then only i's own bit is set).
__device__ __forceinline__ bool ancestor_bits_shared(const int* par, int i, uint32_t bits[4]) {
  bits[0] = bits[1] = bits[2] = bits[3] = 0u;
  bits[i >> 5] |= 1u << (i & 31);
  int j = i;
  for (int steps = 0; steps < kMaxNodes; ++steps) {
    const int p = par[j];
    if (p < -1 || p >= j) {
      bits[0] = bits[1] = bits[2] = bits[3] = 0u;
      bits[i >> 5] |= 1u << (i & 31);
      return false;
    }
    if (p < 0) return true;
    bits[p >> 5] |= 1u << (p & 31);
    j = p;
  }
  return true;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace tva
