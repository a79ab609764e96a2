// Persistent, warp-specialised K-grouped weight-gradient kernel for sm_103a,
// run by CTA pairs (clusters of two CTAs on two SMs) with the 2-SM tensor-core
// MMA (tcgen05 cta_group::2).
//
//   D[e] (+)= A_e^T B_e,   A_e = A[off_e : off_e + K_e, :],  B_e likewise.
//
// A pair computes a 256 x BN tile: each CTA holds 128 rows of the A operand
// (its half of M) and BN/2 columns of the B operand in its shared memory, and
// its 128 x BN half of the accumulator in its tensor memory.  The even CTA's
// MMA thread issues every MMA for both; the operands of one stage are thus
// loaded once per pair, halving each SM's B traffic.
//
// Pairs own one tile of every round of R tiles of the list (expert entry,
// 256-row M tile, BN-column N tile), which the host sorts longest entry first,
// in snake order.  A pair's two tensor-memory
// accumulators serve as two lanes: lane 0 takes its tiles from the head of its
// list, lane 1 from the tail, and the MMA stream alternates `chunk` stages of
// lane 0's (long) tile with the whole of lane 1's (short) tile, so the
// epilogue drains short tiles while a long one accumulates.
//
// Roles per CTA (224 threads; 352 with transposed tiles):
//   warp 0      TMA producer (one thread): A/B stages of 128 (FP8) or 64
//               (BF16) tokens; both CTAs' bytes complete on the even CTA's
//               `full` barrier.
//   warp 1      tensor-memory allocation (collective over the pair); in the
//               even CTA the warp walks the schedule and one elected lane
//               issues tcgen05.cp per scale group and four tcgen05.mma per
//               stage, committing to both CTAs' barriers.
//   warps 2..5  epilogue, one warp per tensor-memory lane quadrant (32 rows),
//               each on its own: tensor memory -> registers -> swizzled
//               shared-memory staging -> TMA store (or TMA reduce-add for
//               in-place D += acc) of 32-row x kEpiCols boxes.  Transposed
//               tiles add warps 7..10: two warps per quadrant, each over
//               every other 32-column chunk.
//   warp 6      FP8: scale loader -- fetches each scale group's packed
//               records (written beforehand by the scale pack pass in the
//               layout tcgen05.cp copies into tensor memory) up to five groups
//               ahead.  BF16: stage gate -- each CTA zeroes the token rows
//               past an expert's slice in its own tiles of that expert's last
//               stage.
// Two accumulators live in tensor memory (the two lanes), so the epilogue of
// one tile overlaps the MMAs of others.
//
// Operands are MN-major (the token axis is K and is the slow axis in memory):
// an operand tile for one stage is BK token rows x 128-byte swizzle atoms.
// With kKMajor both are K-major (rows of BK bytes of K).
//
// M-grouped mode (kMG, the FP8 data gradient dx_e = dy_e W_e): the schedule
// entries are the experts with tokens, a tile is (256-token chunk, BN columns)
// of one expert, A is K-major (dy's token rows, [sum_m, K]) and B the expert's
// weight, MN-major [K, N] or, with kKMajor, K-major [N, K]; every tile runs
// the same K, so both lanes take tiles in order and k loops are not rotated.
//
// Every role reads the schedule table once per chunk; it is copied into
// shared memory at kernel start when it fits.
//
// Building with -DDG_KERNEL_TIMERS adds per-role cycle counters written to
// WgradParams::timers (profiling builds only).
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

// The MMA issuer runs as a whole warp with warp-uniform control flow; one
// lane, elected once, issues every tcgen05 instruction, and every wait result
// is made warp-uniform (a single thread issuing from divergent code kept the
// tensor pipe less than half busy).
#define DG_ISSUE if (mma_el)
#define DG_MMA_OK(x) (__all_sync(0xffffffffu, (x)))

#include "wgrad_params.h"

namespace dg {

template <bool kFP8, int kBN, bool kKMajor = false, bool kMG = false, bool kTransD = false>
struct WgradCfg {
  // Epilogue warps: one per tensor-memory lane quadrant (warps 2..5), or, for
  // transposed tiles (whose staging is a scattered 4-byte write per element),
  // two per quadrant (warps 2..5 and 7..10) each draining every other
  // 32-column chunk with one staging buffer, which releases an accumulator in
  // about half the time.  Roles: warp 0 producer, 1 MMA, 6 scale loader /
  // BF16 gate, the rest epilogue.
  // Register-held drain (weight gradient): each of two warps per quadrant
  // reads its whole share of a finished accumulator (every other 32-column
  // chunk) into registers, releases the accumulator at once, and only then
  // stages and stores those chunks; the accumulator is busy for the MMAs and
  // one tensor-memory read instead of the whole drain.
  static constexpr bool REG_EPI = kFP8 && !kMG;
  static constexpr int EPI_WARPS = (kTransD || REG_EPI) ? 8 : 4;
  static constexpr int EPI_CH = (kBN / kEpiCols + 1) / 2;   // chunks a warp holds (at most)
  static constexpr int THREADS = 32 * (3 + EPI_WARPS);
  static_assert(!kKMajor || kFP8, "K-major operands: FP8 only");
  static_assert(!kMG || kFP8, "M-grouped: FP8");
  // Mixed tile widths (FP8 weight gradient, block_n 256): the first accumulator is 256 columns wide and takes the wide tiles
  // (the longest experts) and narrow ones; the second is BN1 = 224 wide and
  // takes narrow tiles only.  256 + 224 columns leave room for two scale
  // slots in tensor memory.
  static constexpr bool kMixed = kFP8 && !kMG && kBN == kWideBN;
  static_assert(!(kFP8 && kBN == kWideBN) || kMixed, "FP8 block_n 256: mixed widths only");
  static constexpr int BN1 = kMixed ? kNarrowBN : kBN;   // second accumulator's width
  // Operand majorness: kKMajor makes both operands K-major (NT weight
  // gradient; the data gradient with the weight stored [N, K]); the M-grouped
  // data gradient otherwise has a K-major A (token rows of dy) and an
  // MN-major B (the expert weight [K, N]).
  static constexpr bool A_KM = kKMajor || kMG;
  static constexpr bool B_KM = kKMajor;
  static constexpr int BM = 128;                        // rows per CTA (pair: 256)
  static constexpr int ELEM = kFP8 ? 1 : 2;
  static constexpr int BK = kFP8 ? 128 : 64;            // tokens per stage
  static constexpr int ATOM = 128 / ELEM;               // elements per swizzle row
  static constexpr int MMA_K = kFP8 ? 32 : 16;          // K of one tcgen05.mma
  static constexpr int KSTEPS = BK / MMA_K;             // 4
  // k-loop rotation step (stages); M-grouped tiles are not rotated (a unit
  // longer than any k loop): their operand slices all stay in L2.
  static constexpr int ROT_UNIT = kMG ? (1 << 24) : kFP8 ? 8 : 16;
  static constexpr int BN_CTA = kBN / 2;                // B columns held per CTA
  static constexpr int A_ATOMS = BM / ATOM;
  static constexpr int B_ATOMS = (BN_CTA + ATOM - 1) / ATOM;
  static constexpr int ATOM_BYTES = BK * 128;           // BK rows x 128 bytes
  // MN-major tiles are BK token rows of 128-byte swizzle atoms; K-major tiles
  // (NT operands, [M, sum_k] / [N, sum_k]) are BM or BN_CTA rows of BK bytes,
  // 128-byte swizzled in groups of eight rows.
  static constexpr int A_BYTES = A_KM ? BM * BK * ELEM : A_ATOMS * ATOM_BYTES;
  static constexpr int B_BYTES = B_KM ? BN_CTA * BK * ELEM : B_ATOMS * ATOM_BYTES;
  // Bytes a stage's B loads bring in: each box is min(ATOM, BN_CTA) columns
  // wide, so a CTA's 112-column half of a 224-wide tile is loaded exactly
  // (its 128-byte swizzled rows keep their 128-byte pitch in shared memory).
  static constexpr int B_BOX_COLS = BN_CTA < ATOM ? BN_CTA : ATOM;
  static constexpr int B_LOAD_BYTES = B_KM ? B_BYTES : B_ATOMS * BK * B_BOX_COLS * ELEM;
  static constexpr int B_LOAD_BYTES_N = kMixed ? BK * (BN1 / 2) * ELEM : B_LOAD_BYTES;   // narrow tiles
  // Descriptor start-address step of one MMA along K: MN-major, MMA_K token
  // rows of 128 bytes; K-major, MMA_K elements inside the 128-byte row.
  static constexpr int A_KSTEP = A_KM ? MMA_K * ELEM : MMA_K * 128;
  static constexpr int B_KSTEP = B_KM ? MMA_K * ELEM : MMA_K * 128;
  // Descriptor strides: SBO = 1024 (8 token rows x 128 B) between K groups,
  // LBO = ATOM_BYTES between 128-byte atoms along M/N.  A single-atom operand
  // never steps along M/N, so its LBO is set to the K-group stride as well.
  static constexpr int A_LBO = A_ATOMS > 1 ? ATOM_BYTES : 1024;
  static constexpr int B_LBO = B_ATOMS > 1 ? ATOM_BYTES : 1024;
  // all-K-major 224-wide stages are 30 KB, others 32 KB (with mixed widths
  // the K-major B stage holds 128 rows)
  static constexpr int STAGES = (A_KM && B_KM && !kMixed) ? 6 : 5;
  static constexpr int NUM_ACC = 2;
  // FP8 scale groups: four UE8M0 rows (four k-blocks at gran_k 128, the four
  // 32-token sub-blocks of one k-block at gran_k 32), in a ring of SF_SLOTS.
  // Each slot holds the group's packed records (UT_A for this CTA's 128 rows
  // of A, UT_B for the tile's BN columns of B) as tcgen05.cp reads them.
  static constexpr int SF_SLOTS = kFP8 ? 5 : 0;
  static constexpr int SF_CHUNKS_B = kFP8 ? (kBN + 127) / 128 : 0;
  static constexpr int UT_A = 512;                      // 32 rows x 16 bytes
  static constexpr int UT_B = 512 * SF_CHUNKS_B;
  static constexpr int SF_COLS = 4 + 4 * SF_CHUNKS_B;   // tensor-memory columns per slot
  static constexpr int SF_COL0 = kBN + BN1;              // after the two accumulators
  // Tensor-memory scale slots, a ring of SF_TSLOTS (two with mixed widths,
  // whose accumulators leave room for no more).  The copy of a group's scales
  // into a slot is issued only once the MMAs of the group that last read the
  // slot have completed: the tensor pipe orders a copy before later MMAs, but
  // not after earlier ones.
  static constexpr int SF_TSLOTS = kMixed ? 2 : SF_SLOTS;
  static constexpr int EC = kEpiCols;                   // output columns per epilogue chunk
  static constexpr int WSTG_BYTES = 32 * EC * 4;        // per epilogue warp and buffer: 32 FP32 rows
  static constexpr int EPI_BUFS = 8 / EPI_WARPS;        // staging buffers per epilogue warp
  static constexpr int TMEM_COLS = 512;
  static_assert(SF_COL0 + SF_TSLOTS * SF_COLS <= TMEM_COLS, "tmem budget");
  static_assert(kBN % 32 == 0 && kBN <= 256, "block N");

  static constexpr int OFF_B = 0;
  static constexpr int OFF_A = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_STG = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_UTA = OFF_STG + EPI_WARPS * EPI_BUFS * WSTG_BYTES;
  static_assert(EPI_WARPS * EPI_BUFS == 8, "eight staging buffers and separate-C barriers");
  static constexpr int OFF_UTB = OFF_UTA + SF_SLOTS * UT_A;
  static constexpr int OFF_BAR = (OFF_UTB + SF_SLOTS * UT_B + 7) / 8 * 8;
  // barriers: full[S], empty[S], gate[S], tfull[S], accf[2], acce[2],
  // cbar[4 warps x 2], sfr/sfe[SLOTS], drain
  static constexpr int NUM_BARS = 4 * STAGES + 2 * NUM_ACC + 8 + 2 * SF_SLOTS + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // The schedule table is read once per chunk by every role; indexed reads
  // of the kernel parameters miss the constant cache, so it is copied here
  // when it fits (up to SCHED_CAP entries, from the space left over).
  static constexpr int OFF_SCHED = OFF_MISC + 16;
  static constexpr int SCHED_LEFT = (232448 - 1024 - OFF_SCHED) / static_cast<int>(sizeof(SchedEntry));
  static constexpr int SCHED_CAP = SCHED_LEFT < 256 ? SCHED_LEFT : 256;
  static constexpr int SMEM_BYTES = OFF_SCHED + SCHED_CAP * static_cast<int>(sizeof(SchedEntry)) + 1024;
  static_assert(SCHED_CAP >= 64, "schedule table in shared memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};


// Roles' wait sites, reported in DevStatus::where.
enum : int { W_PROD_EMPTY = 0x01, W_PROD_DRAIN = 0x02, W_PROD_SFE = 0x03, W_MMA_ACCE = 0x11,
             W_MMA_FULL = 0x12, W_MMA_DRAIN = 0x13, W_MMA_SFR = 0x14, W_MMA_SFD = 0x15, W_EPI_ACCF = 0x21,
             W_EPI_C = 0x22, W_SF_FULL = 0x31 };

struct TileCoord {
  int expert, k_off, k_len, m0, n0;   // m0: this CTA's first row; n0: the pair's first column
  int mt, nt, g_off;                  // M- and N-tile index; first packed scale group of the entry
  int ka_off;                         // A's offset along K (k_off, or 0 when M-grouped)
  int rows;                           // M-grouped: this CTA's rows inside the expert (<= 0: none)
  int k_exp;                          // the entry's k_exp (checked against ks_dev)
  int bn;                             // the tile's width
};

// Weight gradient: entry u / tiles_per_group, tiles (M tile, N tile) of the
// expert's [M, N] output; with mixed widths the first wide_tiles tiles are the
// wide entries' (kWideBN columns, tpg_w per entry) and the rest follow with
// width bn.  M-grouped data gradient: the entry whose tile_off
// range holds u; its tiles are (256-token chunk, N tile) of the expert's rows,
// N tiles fastest, and A's rows are the tokens (m0 is a row of the [sum_m, K]
// operand), B's rows the expert's K rows of W.
template <bool kMG>
__device__ __forceinline__ TileCoord tile_coord(const WgradParams &p, const SchedEntry *sched,
                                                int u, int bn, uint32_t rank) {
  TileCoord c;
  if constexpr (kMG) {
    int lo = 0, hi = p.n_entries - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sched[mid].tile_off <= u) lo = mid; else hi = mid - 1;
    }
    const SchedEntry se = sched[lo];
    const int lt = u - se.tile_off;
    const int mt = fast_div(lt, p.div_nt), nt = lt - mt * p.n_tiles;
    const int r0 = mt * 256 + static_cast<int>(rank) * 128;
    c.expert = se.expert; c.k_off = se.k_off; c.k_len = se.k_len;
    c.m0 = se.row_off + r0; c.n0 = nt * bn; c.mt = mt; c.nt = nt; c.g_off = se.g_off;
    c.ka_off = 0; c.rows = se.k_exp - r0; c.k_exp = se.k_exp; c.bn = bn;
  } else {
    int gi, lt, ntn;
    FastDiv dnt;
    if (u < p.wide_tiles) {
      gi = fast_div(u, p.div_tpg_w);
      lt = u - gi * p.tpg_w;
      ntn = p.n_tiles_w;
      dnt = p.div_nt_w;
      bn = kWideBN;
    } else {
      const int v = u - p.wide_tiles;
      const int gq = fast_div(v, p.div_tpg);
      gi = p.n_wide + gq;
      lt = v - gq * p.tiles_per_group;
      ntn = p.n_tiles;
      dnt = p.div_nt;
    }
    const SchedEntry se = sched[gi];
    const int q = fast_div(lt, p.m_fastest ? p.div_mt : dnt);
    const int r = lt - q * (p.m_fastest ? p.m_tiles : ntn);
    const int mt = p.m_fastest ? r : q;
    const int nt = p.m_fastest ? q : r;
    c.expert = se.expert; c.k_off = se.k_off; c.k_len = se.k_len;
    c.m0 = mt * 256 + static_cast<int>(rank) * 128; c.n0 = nt * bn; c.mt = mt; c.nt = nt;
    c.g_off = se.g_off; c.ka_off = se.k_off; c.rows = 128; c.k_exp = se.k_exp; c.bn = bn;
  }
  return c;
}

// Rotation of a tile's k loop.  Tiles running at the same time that share an
// operand slice (same expert, same M tile or same N tile) start their k loops
// `unit` stages apart, so each k-block of the slice is first read (from HBM)
// by one of them and found in L2 by the others, instead of all of them
// waiting on the same HBM fetch.  Only the first F = nk rounded down to a
// multiple of 4 stages rotate; a last partial scale group stays at the end.
// With `unit` a multiple of 4, every scale group is visited whole and starts at
// a position that is a multiple of 4, as in the unrotated loop, so lane
// chunks (multiples of 4 stages) always begin with a new group.
struct KRot {
  int rot, F;
};
__device__ __forceinline__ KRot tile_rot(int mt, int nt, int nk, int unit) {
  const int F = nk & ~3;
  const int nu = F / unit;
  // start unit: (mt + nt) modulo the largest power of two <= nu (no division)
  const int mask = nu >= 2 ? (1 << (31 - __clz(nu))) - 1 : 0;
  return KRot{unit * ((mt + nt) & mask), F};
}
// Stage of the tile's k range visited at loop position j.
__device__ __forceinline__ int rot_stage(int j, KRot r) {
  if (j >= r.F) return j;
  const int x = j + r.rot;
  return x < r.F ? x : x - r.F;
}

// ---------------------------------------------------------------- schedule
// A pair owns one tile of every round of R tiles of the longest-first list,
// in snake order (round i: position pid when i is even, R - 1 - pid when odd),
// which balances the pairs' totals better than the same position every round
// while keeping each pair's list longest first.
__device__ __forceinline__ int owned_tile(int i, int pid, int R) {
  return i * R + ((i & 1) ? R - 1 - pid : pid);
}
__device__ __forceinline__ int owned_count(int num_tiles, int pid, int R) {
  const int full = num_tiles / R;
  const int off = (full & 1) ? R - 1 - pid : pid;
  return full + (off < num_tiles - full * R ? 1 : 0);
}

// A pair owns the tiles u = owned_tile(i) (i = 0, 1, ...) of the longest-first
// tile list.  Its two accumulator buffers work as two lanes: lane 0 takes
// tiles from the head of its list (long, MMA-heavy) and lane 1 from the tail
// (short or output-only, store-heavy).  The MMA stream alternates between the
// lanes: `chunk` stages of lane 0's tile, then all of lane 1's tile, and so
// on, so that while a long tile accumulates the epilogue drains a stream of
// short ones.  Every role walks the same sequence of chunks.
struct Chunk {
  int u;        // tile
  int j0, j1;   // its stages [j0, j1) (BK tokens each)
  int nk;       // stages of the whole tile; 0 = output-only tile
  int lane;     // accumulator buffer
};

struct LaneSched {
  const SchedEntry *sched;   // the schedule table (shared memory, or the parameters)
  int head, tail;   // list positions not yet taken: [head, tail]
  int u0, nk0, j0;  // lane 0: tile (-1: none), its stages, next stage
  int u1, nk1, j1;  // lane 1
  int turn;
};

__device__ __forceinline__ void lane_init(LaneSched &L, const WgradParams &p, int pid, int R,
                                          const SchedEntry *sched) {
  L.sched = sched;
  L.head = 0;
  L.tail = owned_count(p.num_tiles, pid, R) - 1;
  L.u0 = L.u1 = -1;
  L.nk0 = L.nk1 = L.j0 = L.j1 = 0;
  L.turn = 0;
}

// One lane's turn: a chunk of its current tile, taking the next tile from its
// end of the list first if it has none.  Returns false if the lane has no
// tile and the list is used up.
__device__ __forceinline__ bool lane_turn(LaneSched &L, const WgradParams &p, int pid, int R,
                                          int bk, int l, int &u, int &nk, int &j, Chunk &c) {
  if (u < 0) {
    if (L.head > L.tail) return false;
    // M-grouped tiles all have the same length: both lanes take the next tile
    // in order, so the running tiles share one expert's weight in L2.
    const int i = (l == 0 || p.mgroup) ? L.head++ : L.tail--;
    u = owned_tile(i, pid, R);
    if (l == 1 && u < p.wide_tiles) {   // a wide tile does not fit the second accumulator
      ++L.tail;
      u = -1;
      return false;
    }
    // (M-grouped: every entry's K is the same, sched[0].k_len)
    const int ei = u < p.wide_tiles ? fast_div(u, p.div_tpg_w)
                                    : p.n_wide + fast_div(u - p.wide_tiles, p.div_tpg);
    const int kl = p.mgroup ? L.sched[0].k_len : L.sched[ei].k_len;
    nk = (u < p.num_mma_tiles) ? (kl + bk - 1) / bk : 0;
    j = 0;
    if (nk == 0) {   // output-only tile: a completion without MMAs
      c = Chunk{u, 0, 0, 0, l};
      u = -1;
      return true;
    }
  }
  const int rem = nk - j;
  const int len = (l == 0) ? min(p.chunk, rem) : rem;
  c = Chunk{u, j, j + len, nk, l};
  j += len;
  if (j == nk) u = -1;
  return true;
}

__device__ __forceinline__ bool lane_next(LaneSched &L, const WgradParams &p, int pid, int R,
                                          int bk, Chunk &c) {
  const int first = L.turn;
  L.turn ^= 1;
  if (first == 0) {
    if (lane_turn(L, p, pid, R, bk, 0, L.u0, L.nk0, L.j0, c)) return true;
    L.turn = 0;
    return lane_turn(L, p, pid, R, bk, 1, L.u1, L.nk1, L.j1, c);
  }
  if (lane_turn(L, p, pid, R, bk, 1, L.u1, L.nk1, L.j1, c)) return true;
  L.turn = 1;
  return lane_turn(L, p, pid, R, bk, 0, L.u0, L.nk0, L.j0, c);
}

// 16-byte chunk i of staging row `row` (rows of RB = 32, 64 or 128 bytes) under
// the TMA swizzle of that width: the chunk index is XORed with address bits
// 7.. of the row start.
template <int RB>
__device__ __forceinline__ int swz_chunk(int i, int row) {
  return i ^ (((row * RB) >> 7) & (RB / 16 - 1));
}

#ifdef DG_KERNEL_TIMERS
#define DG_T0(v) const unsigned long long v = clock64()
#define DG_TACC(slot, v) (tm[slot] += clock64() - (v))
#else
#define DG_T0(v)
#define DG_TACC(slot, v)
#endif

template <bool kFP8, int kBN, int kOut, bool kKMajor, bool kTransD, bool kMG = false>
__global__ void __launch_bounds__((WgradCfg<kFP8, kBN, kKMajor, kMG, kTransD>::THREADS), 1)
    kgrouped_wgrad_kernel(const __grid_constant__ WgradParams p) {
  using Cfg = WgradCfg<kFP8, kBN, kKMajor, kMG, kTransD>;
  static_assert(!kMG || (!kTransD && (kOut == OUT_F32 || kOut == OUT_BF16)),
                "M-grouped: direct tiles, no accumulator");
  constexpr int S = Cfg::STAGES;
  constexpr int NS = Cfg::SF_SLOTS;
  extern __shared__ uint8_t smem_raw[];
  // The dynamic shared window starts at the same offset in both CTAs, so the
  // aligned base (and every buffer offset) matches across the pair.
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
  uint64_t *full = bars;           // even CTA: both CTAs' stage bytes landed
  uint64_t *empty = bars + S;      // stage consumed by the pair's MMAs
  uint64_t *gate = bars + 2 * S;   // BF16, even CTA: tail rows masked in both CTAs
  uint64_t *tfull = bars + 3 * S;  // BF16, odd CTA: its bytes of an expert's last stage landed
  uint64_t *accf = bars + 4 * S;   // accumulator ready (multicast commit)
  uint64_t *acce = accf + 2;       // even CTA: accumulator drained by both epilogues
  uint64_t *cbar = acce + 2;       // separate-C box landed (per epilogue warp and buffer)
  uint64_t *sfr = cbar + 8;        // even CTA: both CTAs' records of a scale group landed
  uint64_t *sfe = sfr + NS;        // scale slot free (its tcgen05.cp completed)
  uint64_t *drain = sfe + NS;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t rank = cluster_ctarank();          // 0 = even CTA (issues the MMAs)
  const bool leader = (rank == 0);
  const int pid = blockIdx.x >> 1;                  // pair index
  const int R = gridDim.x >> 1;                     // number of pairs
  // k-blocks covered by one scale group
  const int gs = kFP8 ? (p.gran_k == 128 ? 4 : 1) : 1;
  // gs is 1 or 4: group tests by mask and shift (no runtime division per stage)
  const int gs_mask = gs - 1, gs_shift = (gs == 4) ? 2 : 0;
#ifdef DG_KERNEL_TIMERS
  unsigned long long tm[7] = {0, 0, 0, 0, 0, 0, 0};
  const unsigned long long t_start = clock64();
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&gate[i], 2);       // BF16: the stage gate of each CTA
      mbar_init(&tfull[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 2 * Cfg::EPI_WARPS);   // every epilogue warp of both CTAs
    }
    for (int i = 0; i < Cfg::EPI_WARPS * Cfg::EPI_BUFS; ++i) mbar_init(&cbar[i], 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sfr[i], 1);
      mbar_init(&sfe[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  const bool sched_smem = p.n_sched <= Cfg::SCHED_CAP;
  SchedEntry *sched_s = reinterpret_cast<SchedEntry *>(smem + Cfg::OFF_SCHED);
  if (sched_smem) {
    const int *src = reinterpret_cast<const int *>(p.sched);
    int *dst = reinterpret_cast<int *>(sched_s);
    constexpr int W = static_cast<int>(sizeof(SchedEntry) / sizeof(int));
    for (int i = threadIdx.x; i < p.n_sched * W; i += blockDim.x) dst[i] = src[i];
  }
  const SchedEntry *sched = sched_smem ? sched_s : p.sched;
  tc_fence_before();
  cluster_sync();                   // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
      if constexpr (Cfg::kMixed) prefetch_tmap(&p.tmBn);
      const uint64_t keep = l2_policy_evict_last();   // operands are re-read by other tiles
      int s = 0;
      uint32_t ph = 0, armed = 0;
      bool ok = true;
      LaneSched L;
      lane_init(L, p, pid, R, sched);
      Chunk ch;
      while (ok && lane_next(L, p, pid, R, Cfg::BK, ch)) {
        if (ch.nk == 0) continue;
        const TileCoord tc = tile_coord<kMG>(p, sched, ch.u, Cfg::BN1, rank);
        const int t = ch.u;
        // both CTAs' bytes of a stage; a narrow tile's B boxes (mixed widths)
        const bool narrow = Cfg::kMixed && tc.bn != kBN;
        const uint32_t tx = 2 * (Cfg::A_BYTES + (narrow ? Cfg::B_LOAD_BYTES_N : Cfg::B_LOAD_BYTES));
        const CUtensorMap *tmb = narrow ? &p.tmBn : &p.tmB;
        if (leader && ch.j0 == 0 && p.ks_dev != nullptr && tc.mt == 0 && tc.nt == 0 &&
            p.ks_dev[tc.expert] != tc.k_exp)
          atomicCAS(&p.status->code, DEV_OK, DEV_KS_MISMATCH);
        const int nb = tc.n0 + static_cast<int>(rank) * (tc.bn / 2);   // this CTA's B columns
        const KRot rot = tile_rot(tc.mt, tc.nt, ch.nk, Cfg::ROT_UNIT);
        for (int j = ch.j0; j < ch.j1; ++j) {
          const int jj = rot_stage(j, rot);   // stage of the tile's k range at position j
          const int k = tc.k_off + jj * Cfg::BK;      // B's row (token) coordinate
          const int ka = tc.ka_off + jj * Cfg::BK;    // A's (the same unless M-grouped)
          DG_T0(w1);
          ok = mbar_wait(&empty[s], ph ^ 1, abort_flag, lim, p.status, W_PROD_EMPTY, t);
          DG_TACC(0, w1);
          if (!ok) break;
          // BF16: the odd CTA's bytes of an expert's last, partial stage
          // complete on its own `tfull`, so that its gate can mask the rows
          // past the slice once they land; every other stage of both CTAs
          // completes on the even CTA's `full`.
          const bool tail_stage = !kFP8 && jj == ch.nk - 1 && tc.k_len - jj * Cfg::BK < Cfg::BK;
          if (leader) mbar_arrive_expect_tx(&full[s], tail_stage ? tx / 2 : tx);
          uint8_t *sa = smem + Cfg::OFF_A + s * Cfg::A_BYTES;
          uint8_t *sb = smem + Cfg::OFF_B + s * Cfg::B_BYTES;
          if (tail_stage && !leader) {
            mbar_arrive_expect_tx(&tfull[s], tx / 2);
#pragma unroll
            for (int a = 0; a < Cfg::A_ATOMS; ++a)
              tma_load_2d_hint(sa + a * Cfg::ATOM_BYTES, &p.tmA, &tfull[s], tc.m0 + a * Cfg::ATOM,
                               k, keep);
#pragma unroll
            for (int b = 0; b < Cfg::B_ATOMS; ++b)
              tma_load_2d_hint(sb + b * Cfg::ATOM_BYTES, &p.tmB, &tfull[s], nb + b * Cfg::ATOM, k,
                               keep);
          } else {
            // K-major operand: one box of BK bytes along K x this CTA's rows;
            // MN-major: BK rows along K of 128-byte atoms.
            const uint32_t fbar = mapa_shared(smem_u32(&full[s]), 0);
            if constexpr (Cfg::A_KM) {
              tma_load_2d_pair(sa, &p.tmA, fbar, ka, tc.m0, keep);
            } else {
#pragma unroll
              for (int a = 0; a < Cfg::A_ATOMS; ++a)
                tma_load_2d_pair(sa + a * Cfg::ATOM_BYTES, &p.tmA, fbar, tc.m0 + a * Cfg::ATOM,
                                 ka, keep);
            }
            if constexpr (Cfg::B_KM && kMG) {
              // the weight stored [G N, K]: K from 0, rows from the expert's first (k_off = e N)
              tma_load_2d_pair(sb, &p.tmB, fbar, ka, nb + tc.k_off, keep);
            } else if constexpr (Cfg::B_KM) {
              tma_load_2d_pair(sb, tmb, fbar, k, nb, keep);
            } else {
#pragma unroll
              for (int b = 0; b < Cfg::B_ATOMS; ++b)
                tma_load_2d_pair(sb + b * Cfg::ATOM_BYTES, tmb, fbar, nb + b * Cfg::ATOM, k, keep);
            }
          }
          ++armed;
          if (++s == S) { s = 0; ph ^= 1; }
        }
      }
      // Let every load this CTA started land before the pair can exit: the
      // even CTA sees them on `full`; its partner sees the stages released.
      for (uint32_t i = (armed > static_cast<uint32_t>(S) ? armed - S : 0); i < armed; ++i) {
        const bool landed =
            leader ? mbar_wait(&full[i % S], (i / S) & 1, abort_flag, drain_limit_ns(lim),
                               p.status, W_PROD_DRAIN, static_cast<int>(i), false)
                   : mbar_wait(&empty[i % S], (i / S) & 1, abort_flag, drain_limit_ns(lim),
                               p.status, W_PROD_DRAIN, static_cast<int>(i), false);
        if (!landed) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    // The whole warp walks the schedule in lockstep (waits made warp-uniform);
    // one lane, elected once, issues the copies, MMAs and commits.  Per stage
    // only constant-offset descriptor updates and the four MMAs, so that issue
    // keeps ahead of the tensor pipe.
    const bool mma_el = elect_one();   // the issuing lane
    if (leader) {
      int s = 0, g = 0;
      uint32_t ph = 0, gph = 0;
      uint32_t sfa_t = 0, sfb_t = 0;
      bool ok = true;
      // A K-major operand clears its transpose bit (15: A, 16: B).
      constexpr uint32_t kKMajorMask = (Cfg::A_KM ? ~(1u << 15) : ~0u) & (Cfg::B_KM ? ~(1u << 16) : ~0u);
      constexpr uint32_t kIdescBase =
          (kFP8 ? idesc_mxf8(2 * Cfg::BM, kBN, 0, 0) : idesc_bf16(2 * Cfg::BM, kBN)) & kKMajorMask;
      // mixed widths: the narrow tiles' MMAs (N = BN1)
      constexpr uint32_t kIdescNarrow =
          kFP8 ? (idesc_mxf8(2 * Cfg::BM, Cfg::BN1, 0, 0) & kKMajorMask) : kIdescBase;
      uint32_t ig = 0;             // scale groups issued
      int ts = 0;                  // tensor-memory slot of the next group (ig mod SF_TSLOTS)
      int n_st = 0;                // stages issued (stage n_st uses `empty[n_st % S]`, phase n_st / S)
      int gstart = 0;              // first stage of the current scale group
      uint32_t glens = 0;          // lengths (at most 7) of the last SF_TSLOTS - 1 groups, 3 bits each
      // Descriptors of stage 0 / scale slot 0; later stages and k-steps add
      // their byte offset >> 4 to the start-address field (shared addresses
      // stay below 256 KB, so the field never carries out).
      // K-major 128-byte swizzle: SBO = 1024 between groups of eight rows
      // (the leading offset is unused there).
      const uint64_t a_desc0 =
          smem_desc(smem_u32(smem + Cfg::OFF_A), Cfg::A_KM ? 16 : Cfg::A_LBO, 1024, 2);
      const uint64_t b_desc0 =
          smem_desc(smem_u32(smem + Cfg::OFF_B), Cfg::B_KM ? 16 : Cfg::B_LBO, 1024, 2);
      const uint64_t uta_desc0 = smem_desc(smem_u32(smem + Cfg::OFF_UTA), 0, 128, 0);
      const uint64_t utb_desc0 = smem_desc(smem_u32(smem + Cfg::OFF_UTB), 0, 128, 0);
      uint64_t a_desc = a_desc0, b_desc = b_desc0;
      uint32_t uses[2] = {0, 0};   // tiles completed per accumulator buffer
      uint32_t gate_ph = 0;        // BF16: phase bit of each slot's `gate` (tail stages only)
      LaneSched L;
      lane_init(L, p, pid, R, sched);
      Chunk ch;
      while (ok && lane_next(L, p, pid, R, Cfg::BK, ch)) {
        if (ch.nk == 0) continue;
        const int t = ch.u;
        const int b = ch.lane;
        if (ch.j0 == 0) {
          // the buffer's previous tile has been drained by both epilogues
          DG_T0(w0);
          ok = DG_MMA_OK(mbar_wait(&acce[b], (uses[b] & 1) ^ 1, abort_flag, lim, p.status, W_MMA_ACCE, t));
          DG_TACC(1, w0);
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t d_tmem = tmem_base + b * kBN;
        const TileCoord tcm = tile_coord<kMG>(p, sched, ch.u, Cfg::BN1, 0);
        const KRot rot = tile_rot(tcm.mt, tcm.nt, ch.nk, Cfg::ROT_UNIT);
        // The chunk's stages, with the tile's instruction descriptor as a
        // compile-time constant: one selected at run time slowed the MMA
        // stream by about 40 % (measured), so mixed widths run one of two
        // copies of this loop.
        auto stages = [&](auto id_c) {
          constexpr uint32_t idesc_t = decltype(id_c)::value;
          for (int j = ch.j0; j < ch.j1; ++j) {
            const int jj = rot_stage(j, rot);   // k-block of this position
            DG_T0(w2);
            // A stage is complete once both CTAs' bytes land (`full`); an
            // expert's last, partial BF16 stage once warp 6 has also masked the
            // rows past the slice in both CTAs (`gate`, used by tail stages only).
            const bool tail = !kFP8 && jj == ch.nk - 1 && tcm.k_len - jj * Cfg::BK < Cfg::BK;
            // (the gate's phase is completed by a cluster-scope release from the
            // odd CTA, whose zeroed rows the MMA reads: cluster-scope acquire)
            ok = DG_MMA_OK(tail ? mbar_wait<true>(&gate[s], (gate_ph >> s) & 1u, abort_flag, lim,
                                                  p.status, W_MMA_FULL, t)
                                : mbar_wait(&full[s], ph, abort_flag, lim, p.status, W_MMA_FULL, t));
            if (tail) gate_ph ^= 1u << s;
            DG_TACC(2, w2);
            if (!ok) break;
            tc_fence_after();
            if constexpr (kFP8) {
              if ((jj & gs_mask) == 0) {
                DG_T0(w1);
                ok = DG_MMA_OK(mbar_wait(&sfr[g], gph, abort_flag, lim, p.status, W_MMA_SFR, t));
                DG_TACC(2, w1);
                if (!ok) break;
                // This group's copy overwrites tensor-memory slot ts, last read
                // by the MMAs of group ig - SF_TSLOTS, which ended `between`
                // stages before this one (the lengths of the groups since).
                // Stage n_st's bytes have landed, so the producer has seen
                // stage n_st - S consumed (its `empty` commit), and with it
                // every earlier MMA: with between >= S - 1 the slot is free.
                // Otherwise (short groups) wait for the `empty` phase of that
                // group's last stage, which cannot have been reused yet (the
                // stage's next use is not issued).
                constexpr int T = Cfg::SF_TSLOTS;
                constexpr uint32_t kLenMask = (1u << (3 * (T - 1))) - 1u;
                if (ig >= 1) {
                  const int len = min(n_st - gstart, 7);
                  glens = ((glens << 3) | static_cast<uint32_t>(len)) & kLenMask;
                }
                gstart = n_st;
                if (ig >= static_cast<uint32_t>(T)) {
                  int between = 0;
#pragma unroll
                  for (int i = 0; i < T - 1; ++i) between += static_cast<int>((glens >> (3 * i)) & 7u);
                  if (between < S - 1) {
                    const int last = n_st - 1 - between;
                    ok = DG_MMA_OK(mbar_wait(&empty[last % S], static_cast<uint32_t>(last / S) & 1u,
                                             abort_flag, lim, p.status, W_MMA_SFD, t));
                  }
                }
                if (!ok) break;
                tc_fence_after();
                sfa_t = tmem_base + Cfg::SF_COL0 + ts * Cfg::SF_COLS;
                ++ig;
                if (++ts == T) ts = 0;
                sfb_t = sfa_t + 4;
                DG_ISSUE tmem_cp_32x128b_warpx4_pair(sfa_t, uta_desc0 + static_cast<uint64_t>(g * (Cfg::UT_A >> 4)));
#pragma unroll
                for (int c = 0; c < Cfg::SF_CHUNKS_B; ++c)
                  DG_ISSUE tmem_cp_32x128b_warpx4_pair(
                      sfb_t + 4 * c,
                      utb_desc0 + static_cast<uint64_t>(g * (Cfg::UT_B >> 4) + c * (512 >> 4)));
                DG_ISSUE mma_commit_pair(&sfe[g], 0x3);
                if (++g == NS) { g = 0; gph ^= 1; }
              }
            }
            // gran_k 128: byte j%4 of each scale word holds this k-block's
            // scale; gran_k 32: byte ks holds this 32-token sub-block's.
            const uint32_t idesc_j = idesc_t | ((gs == 4) ? (static_cast<uint32_t>(jj & 3) * 0x20000010u) : 0u);
#pragma unroll
            for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
              const uint64_t ad = a_desc + static_cast<uint64_t>(ks * (Cfg::A_KSTEP >> 4));
              const uint64_t bd = b_desc + static_cast<uint64_t>(ks * (Cfg::B_KSTEP >> 4));
              if constexpr (kFP8) {
                const uint32_t idesc = (gs == 4) ? idesc_j : (idesc_t | (static_cast<uint32_t>(ks) * 0x20000010u));
                DG_ISSUE mma_mxf8_pair(d_tmem, ad, bd, idesc, sfa_t, sfb_t, (j | ks) != 0);
              } else {
                DG_ISSUE mma_bf16_pair(d_tmem, ad, bd, idesc_t, (j | ks) != 0);
              }
            }
            DG_ISSUE mma_commit_pair(&empty[s], 0x3);
            ++n_st;
            if (++s == S) {
              s = 0;
              ph ^= 1;
              a_desc = a_desc0;
              b_desc = b_desc0;
            } else {
              a_desc += Cfg::A_BYTES >> 4;
              b_desc += Cfg::B_BYTES >> 4;
            }
          }
        };
        if constexpr (Cfg::kMixed) {
          if (tcm.bn != kBN)
            stages(std::integral_constant<uint32_t, kIdescNarrow>{});
          else
            stages(std::integral_constant<uint32_t, kIdescBase>{});
        } else {
          stages(std::integral_constant<uint32_t, kIdescBase>{});
        }
        if (!ok) break;
        if (ch.j1 == ch.nk) {
          DG_ISSUE mma_commit_pair(&accf[b], 0x3);
          ++uses[b];
        }
      }
      // Drain: every tcgen05 op issued here completes before tensor memory
      // is released.
      DG_ISSUE mma_commit_pair(drain, 0x1);
      mbar_wait(drain, 0, abort_flag, drain_limit_ns(lim), p.status, W_MMA_DRAIN, 0, false);
    }
  } else if (warp == 6) {
    if constexpr (!kFP8) {
      // ---------------------------------------------------------- BF16 stage gate
      // An expert's last stage may run past its slice: each CTA zeroes those
      // token rows of its own operand tiles (row k of an atom is bytes
      // [k*128, k*128 + 128)) once they have landed, makes the writes visible
      // to the tensor core (CTA-scope proxy fence) and arrives on the even
      // CTA's `gate`, which the MMA thread waits on for such stages only.
      // Every stage is walked in order and waited on through `empty`, so this
      // warp is never more than one use of a slot ahead.
      {
        int s = 0;
        uint32_t ph = 0;
        uint32_t tph = 0;   // odd CTA: phase bit of each slot's `tfull` (advances on tail stages only)
        bool ok = true;
        const uint32_t gate_leader = mapa_shared(smem_u32(&gate[0]), 0);
        LaneSched L;
        lane_init(L, p, pid, R, sched);
        Chunk ch;
        while (ok && lane_next(L, p, pid, R, Cfg::BK, ch)) {
          if (ch.nk == 0) continue;
          const int t = ch.u;
          const int nk = ch.nk;
          const int tail = sched[fast_div(ch.u, p.div_tpg)].k_len - (nk - 1) * Cfg::BK;
          const TileCoord tcg = tile_coord<kMG>(p, sched, ch.u, Cfg::BN1, 0);
          const KRot rot = tile_rot(tcg.mt, tcg.nt, nk, Cfg::ROT_UNIT);
          for (int j = ch.j0; j < ch.j1; ++j) {
            const int jj = rot_stage(j, rot);
            const bool tail_stage = (jj == nk - 1 && tail < Cfg::BK);
            // the slot's previous use has been consumed (keeps phases in order)
            ok = mbar_wait(&empty[s], ph ^ 1, abort_flag, lim, p.status, W_SF_FULL, t);
            if (ok && tail_stage) {
              if (leader) {
                ok = mbar_wait(&full[s], ph, abort_flag, lim, p.status, W_SF_FULL, t);
              } else {
                ok = mbar_wait(&tfull[s], (tph >> s) & 1, abort_flag, lim, p.status, W_SF_FULL, t);
                tph ^= 1u << s;
              }
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (tail_stage) {
              uint8_t *sa = smem + Cfg::OFF_A + s * Cfg::A_BYTES;
              uint8_t *sb = smem + Cfg::OFF_B + s * Cfg::B_BYTES;
              const int per_atom = (Cfg::BK - tail) * 8;   // 16-byte chunks per atom
              const int n_chunks = per_atom * (Cfg::A_ATOMS + Cfg::B_ATOMS);
              for (int i = lane; i < n_chunks; i += 32) {
                const int atom = i / per_atom;
                const int r = i - atom * per_atom;
                uint8_t *base = atom < Cfg::A_ATOMS ? sa + atom * Cfg::ATOM_BYTES
                                                    : sb + (atom - Cfg::A_ATOMS) * Cfg::ATOM_BYTES;
                *reinterpret_cast<uint4 *>(base + tail * 128 + r * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (leader)
                  mbar_arrive(&gate[s]);
                else
                  mbar_arrive_cluster(gate_leader + 8 * s);   // publishes the zeroed rows
              }
            }
            if (++s == S) { s = 0; ph ^= 1; }
          }
        }
      }
    } else {
      // ---------------------------------------------------------- scale loader
      // Each CTA fetches, per scale group, its packed records (its 128 rows
      // of A, the tile's BN columns of B) into the group's slot once the
      // tcgen05.cp of the slot's previous group has completed; both CTAs'
      // bytes complete on the even CTA's `sfr`.
      if (lane == 0) {
        prefetch_tmap(&p.tmSFA);
        prefetch_tmap(&p.tmSFB);
        // the records come from the pack pass this grid may have started beside
        griddep_wait();
        const uint64_t keep = l2_policy_evict_last();   // B's records serve every M tile
        const uint32_t sfr_leader = mapa_shared(smem_u32(&sfr[0]), 0);
        LaneSched L;
        lane_init(L, p, pid, R, sched);
        Chunk ch;
        TileCoord tc{};
        int j = 0, jj = 0;            // position in the current chunk, its k-block
        KRot rot{0, 0};
        bool have = false;            // a chunk with positions left is current
        uint32_t ig = 0;
        bool ok = true;
        while (ok) {
          // next scale group: the next position whose k-block starts a group
          bool found = false;
          while (!found) {
            if (!have || j >= ch.j1) {
              have = lane_next(L, p, pid, R, Cfg::BK, ch);
              if (!have) break;
              if (ch.nk == 0) { have = false; continue; }
              tc = tile_coord<kMG>(p, sched, ch.u, Cfg::BN1, rank);
              rot = tile_rot(tc.mt, tc.nt, ch.nk, Cfg::ROT_UNIT);
              j = ch.j0;
              continue;
            }
            jj = rot_stage(j, rot);
            if ((jj & gs_mask) == 0) found = true; else ++j;
          }
          if (!found) break;
          const int g = ig % NS;
          DG_T0(w0);
          ok = mbar_wait(&sfe[g], ((ig / NS) & 1) ^ 1, abort_flag, lim, p.status, W_PROD_SFE,
                         ch.u);
          DG_TACC(2, w0);
          if (!ok) break;
          if (leader) mbar_arrive_expect_tx(&sfr[g], 2 * (Cfg::UT_A + Cfg::UT_B));
          const int grp = tc.g_off + (jj >> gs_shift);
          // A's records: per (group, 128-row chunk); M-grouped, the chunk is a
          // 128-token chunk of the whole [sum_m, K] operand and the group one
          // of K's, shared by every expert.
          const int grp_a = kMG ? (jj >> gs_shift) : grp;
          tma_load_2d_pair(smem + Cfg::OFF_UTA + g * Cfg::UT_A, &p.tmSFA, sfr_leader + 8 * g, 0,
                           grp_a * p.sf_mc + tc.m0 / 128, keep);
          // B's records: the wide entries' groups (n_tiles_w tiles each) first
          const int brec = grp < p.sf_gw ? grp * p.n_tiles_w + tc.nt
                                         : p.sf_gw * p.n_tiles_w + (grp - p.sf_gw) * p.n_tiles + tc.nt;
          tma_load_2d_pair(smem + Cfg::OFF_UTB + g * Cfg::UT_B, &p.tmSFB, sfr_leader + 8 * g, 0,
                           brec * Cfg::SF_CHUNKS_B, keep);
          ++ig;
          ++j;
        }
        // Let every record this CTA requested land before the pair can exit:
        // the even CTA sees them on `sfr`; its partner sees the slots' copies
        // complete.
        for (uint32_t i = (ig > static_cast<uint32_t>(NS) ? ig - NS : 0); i < ig; ++i) {
          const bool landed =
              leader ? mbar_wait(&sfr[i % NS], (i / NS) & 1, abort_flag, drain_limit_ns(lim),
                                 p.status, W_PROD_DRAIN, static_cast<int>(i), false)
                     : mbar_wait(&sfe[i % NS], (i / NS) & 1, abort_flag, drain_limit_ns(lim),
                                 p.status, W_PROD_DRAIN, static_cast<int>(i), false);
          if (!landed) break;
        }
      }
    }
  } else if constexpr (Cfg::REG_EPI) {
    // ------------------------------------------------------------ epilogue (register-held)
    // Two warps per tensor-memory lane quadrant; each takes every other
    // 32-column chunk of a finished tile (the two swap sets from tile to tile,
    // so each stores half the columns on average).  A warp reads up to three
    // of its chunks into registers with one tcgen05.wait (a fourth after its
    // first chunk is staged) and releases the accumulator as soon as every
    // read of it has completed, then stages and stores the chunks from
    // registers: the accumulator is held for the MMAs and its read-out, not
    // for the whole drain.
    const int q = warp & 3;
    const int ew = warp < 6 ? warp - 2 : warp - 3;
    const int half = ew >> 2;
    uint32_t uses[2] = {0, 0};
    uint32_t cuse = 0, ntile = 0;
    bool stg_busy = false;
    constexpr bool kHasC = (kOut == OUT_F32_C);
    constexpr int EC = Cfg::EC;
    constexpr int NCH = Cfg::EPI_CH;           // chunks of this warp per tile (at most)
    constexpr int H = NCH < 2 ? NCH : 2;       // chunks held in registers at once
    static_assert(Cfg::EPI_BUFS == 1, "one staging buffer per warp");
    const uint64_t stream_out = l2_policy_evict_first();
    const uint32_t acce_leader = mapa_shared(smem_u32(&acce[0]), 0);
    uint8_t *stg = smem + Cfg::OFF_STG + ew * Cfg::WSTG_BYTES;
    uint64_t *wcbar = cbar + ew;
    uint32_t r[H][EC];
    LaneSched L;
    lane_init(L, p, pid, R, sched);
    Chunk ch;
    bool ok = true;
    // Stage chunk c of the current tile from registers rr and store it.
    auto emit = [&](uint32_t(&rr)[EC], int c, int row0, int n0, int expert, int t) -> bool {
      DG_T0(w1);
      if (lane == 0 && stg_busy) bulk_wait_read<0>();   // the previous store has read stg
      __syncwarp();
      DG_TACC(2, w1);
      const int bx = kTransD ? row0 : n0 + EC * c;
      const int by = kTransD ? n0 + EC * c : row0;
      if constexpr (kHasC) {
        if (lane == 0) {
          mbar_arrive_expect_tx(wcbar, 32 * EC * 4);
          tma_load_3d(stg, &p.tmC, wcbar, bx, by, expert);
        }
        bool got = mbar_wait(wcbar, cuse & 1, abort_flag, lim, p.status, W_EPI_C, t);
        ++cuse;
        if (!__all_sync(0xffffffffu, got)) return false;
        if constexpr (kTransD) {
#pragma unroll
          for (int j = 0; j < EC; ++j)
            rr[j] = __float_as_uint(__uint_as_float(rr[j]) + *reinterpret_cast<const float *>(
                stg + j * (32 * 4) + (swz_chunk<32 * 4>(lane >> 2, j) << 4) + (lane & 3) * 4));
        } else {
          const uint8_t *rowp = stg + lane * (EC * 4);
#pragma unroll
          for (int j = 0; j < EC / 4; ++j) {
            const float4 cv = *reinterpret_cast<const float4 *>(rowp + (swz_chunk<EC * 4>(j, lane) << 4));
            rr[4 * j + 0] = __float_as_uint(__uint_as_float(rr[4 * j + 0]) + cv.x);
            rr[4 * j + 1] = __float_as_uint(__uint_as_float(rr[4 * j + 1]) + cv.y);
            rr[4 * j + 2] = __float_as_uint(__uint_as_float(rr[4 * j + 2]) + cv.z);
            rr[4 * j + 3] = __float_as_uint(__uint_as_float(rr[4 * j + 3]) + cv.w);
          }
        }
        __syncwarp();   // every lane has read the C box before it is overwritten
      }
      if constexpr (kTransD) {
        static_assert(EC == 32, "transposed boxes are 32 x 32");
        if constexpr (kOut == OUT_BF16) {
#pragma unroll
          for (int j = 0; j < EC; ++j)
            *reinterpret_cast<__nv_bfloat16 *>(stg + j * 64 + (swz_chunk<64>(lane >> 3, j) << 4) +
                                               (lane & 7) * 2) =
                __float2bfloat16_rn(__uint_as_float(rr[j]));
        } else {
#pragma unroll
          for (int j = 0; j < EC; ++j)
            *reinterpret_cast<uint32_t *>(stg + j * 128 + (swz_chunk<128>(lane >> 2, j) << 4) +
                                          (lane & 3) * 4) = rr[j];
        }
      } else if constexpr (kOut == OUT_BF16) {
        uint8_t *rowp = stg + lane * (EC * 2);
#pragma unroll
        for (int j = 0; j < EC / 8; ++j) {
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(rr[8 * j + 2 * h]),
                                                            __uint_as_float(rr[8 * j + 2 * h + 1]));
            w[h] = *reinterpret_cast<const uint32_t *>(&pr);
          }
          *reinterpret_cast<uint4 *>(rowp + (swz_chunk<EC * 2>(j, lane) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        uint8_t *rowp = stg + lane * (EC * 4);
#pragma unroll
        for (int j = 0; j < EC / 4; ++j)
          *reinterpret_cast<uint4 *>(rowp + (swz_chunk<EC * 4>(j, lane) << 4)) =
              make_uint4(rr[4 * j], rr[4 * j + 1], rr[4 * j + 2], rr[4 * j + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kOut == OUT_F32_REDUCE)
          tma_reduce_add_3d_hint(&p.tmD, stg, bx, by, expert, stream_out);
        else
          tma_store_3d_hint(&p.tmD, stg, bx, by, expert, stream_out);
        bulk_commit();
      }
      stg_busy = true;
      return true;
    };
    while (ok && lane_next(L, p, pid, R, Cfg::BK, ch)) {
      if (ch.nk > 0 && ch.j1 != ch.nk) continue;   // only tile completions
      const int t = ch.u;
      const TileCoord tc = tile_coord<kMG>(p, sched, ch.u, Cfg::BN1, rank);
      const bool mma_tile = ch.nk > 0;
      const int b = ch.lane;
      const int sel = half ^ static_cast<int>(ntile & 1);   // this tile's chunk set
      ++ntile;
      const int ncols = min(tc.bn, p.N - tc.n0);
      const int nch = (ncols + EC - 1) / EC;
      const int mine = nch > sel ? (nch - sel + 1) / 2 : 0;   // chunks sel, sel + 2, ...
      const int row0 = tc.m0 + 32 * q;
      const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * kBN;
      if (mma_tile) {
        DG_T0(w0);
        bool got = mbar_wait(&accf[b], uses[b] & 1, abort_flag, lim, p.status, W_EPI_ACCF, t);
        DG_TACC(1, w0);
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < H; ++i)
          if (i < mine) tmem_ld_row<EC>(tmem_row + EC * (sel + 2 * i), r[i]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < H; ++i) tmem_reg_fence_n<EC>(r[i]);
        if (mine <= H) {
          // every read of this buffer has completed: release it (CTA-scope arrive)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acce_leader + 8 * b);
        }
      } else {
#pragma unroll
        for (int i = 0; i < H; ++i)
#pragma unroll
          for (int j = 0; j < EC; ++j) r[i][j] = 0u;
      }
      // chunk i sits in slot i % H; once it is stored, the slot takes chunk
      // i + H, and the accumulator is released after its last chunk's read
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        if (!ok || i >= mine) break;
        ok = emit(r[i % H], sel + 2 * i, row0, tc.n0, tc.expert, t);
        if (ok && i + H < NCH && i + H < mine) {
          if (mma_tile) {
            tmem_ld_row<EC>(tmem_row + EC * (sel + 2 * (i + H)), r[i % H]);
            tmem_wait_ld();
            tmem_reg_fence_n<EC>(r[i % H]);
            if (i + H == mine - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_remote(acce_leader + 8 * b);
            }
          } else {
#pragma unroll
            for (int j = 0; j < EC; ++j) r[i % H][j] = 0u;
          }
        }
      }
      if (!ok) break;
      if (mma_tile) ++uses[b];
    }
    if (lane == 0) bulk_wait<0>();
  } else {
    // ------------------------------------------------------------ epilogue
    // Each warp owns one tensor-memory lane quadrant (32 rows of this CTA's
    // 128) and runs its own pipeline, so the four warps never wait on one
    // another: tcgen05.ld of EC columns -> one of its EPI_BUFS swizzled
    // staging buffers -> TMA store (or reduce-add) of that 32-row box.
    const int q = warp & 3;               // tensor-memory lane quadrant of this warp
    const int ew = warp < 6 ? warp - 2 : warp - 3;   // epilogue warp index
    constexpr int CSTEP = Cfg::EPI_WARPS / 4;         // warps per quadrant
    const int half = ew >> 2;                         // first chunk of this warp
    uint32_t uses[2] = {0, 0}, nchunk = 0;
    uint32_t cuse[2] = {0, 0};
    constexpr bool kHasC = (kOut == OUT_F32_C);
    const uint64_t stream_out = l2_policy_evict_first();   // D is written once
    const uint32_t acce_leader = mapa_shared(smem_u32(&acce[0]), 0);
    uint8_t *wstg = smem + Cfg::OFF_STG + ew * Cfg::EPI_BUFS * Cfg::WSTG_BYTES;
    uint64_t *wcbar = cbar + Cfg::EPI_BUFS * ew;
    constexpr int EC = Cfg::EC;
    uint32_t r[EC];   // tensor-memory chunk in flight
    LaneSched L;
    lane_init(L, p, pid, R, sched);
    Chunk ch;
    while (lane_next(L, p, pid, R, Cfg::BK, ch)) {
      if (ch.nk > 0 && ch.j1 != ch.nk) continue;   // only tile completions
      const int t = ch.u;
      const TileCoord tc = tile_coord<kMG>(p, sched, ch.u, Cfg::BN1, rank);
      const bool mma_tile = ch.nk > 0;
      // M-grouped: a CTA whose 128 rows lie past its expert's last token
      // (the second half of an expert's last 256-row chunk) stores nothing.
      const bool store = !kMG || tc.rows > 0;
      const int dz = kMG ? 0 : tc.expert;   // D's third coordinate
      const int b = ch.lane;
      if (mma_tile) {
        DG_T0(w0);
        bool got = mbar_wait(&accf[b], uses[b] & 1, abort_flag, lim, p.status, W_EPI_ACCF, t);
        DG_TACC(1, w0);
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
      }
      const int ncols = min(tc.bn, p.N - tc.n0);
      const int nch = (ncols + EC - 1) / EC;
      const int row0 = tc.m0 + 32 * q;    // first output row of this warp's boxes
      const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * kBN;
      if (mma_tile && half < nch) tmem_ld_row<EC>(tmem_row + EC * half, r);
      if (mma_tile && half >= nch) {
        // no chunk of this tile for this warp: release the accumulator now
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acce_leader + 8 * b);
      }
      bool ok = true;
      for (int c = half; c < nch; c += CSTEP, ++nchunk) {
        const int sbuf = static_cast<int>(nchunk % Cfg::EPI_BUFS);
        uint8_t *stg = wstg + sbuf * Cfg::WSTG_BYTES;
        DG_T0(w1);
        if (lane == 0) bulk_wait_read<Cfg::EPI_BUFS - 1>();   // the store that last used stg is done reading
        __syncwarp();
        DG_TACC(2, w1);
        // Output box: 32 rows x EC columns of D, or (transposed tiles) the
        // box whose rows are this chunk's EC columns and whose columns are
        // this warp's 32 rows.
        const int bx = kTransD ? row0 : tc.n0 + EC * c;
        const int by = kTransD ? tc.n0 + EC * c : row0;
        if (kHasC && lane == 0) {
          mbar_arrive_expect_tx(&wcbar[sbuf], 32 * EC * 4);
          tma_load_3d(stg, &p.tmC, &wcbar[sbuf], bx, by, tc.expert);
        }
        float v[EC];
        if (mma_tile) {
          // Chunk c was requested one iteration earlier; request this warp's
          // next chunk now so that it streams in while this one is staged.
          tmem_wait_ld();
          tmem_reg_fence_n<EC>(r);
#pragma unroll
          for (int i = 0; i < EC; ++i) v[i] = __uint_as_float(r[i]);
          if (c + CSTEP < nch) {
            tmem_ld_row<EC>(tmem_row + EC * (c + CSTEP), r);
          } else {
            // Every read of this buffer has completed (tcgen05.wait::ld above);
            // the tcgen05 fence orders them before the release, so a CTA-scope
            // arrive suffices (a cluster-scope release costs thousands of cycles).
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acce_leader + 8 * b);
          }
        } else {
#pragma unroll
          for (int i = 0; i < EC; ++i) v[i] = 0.f;
        }
        if constexpr (kHasC) {
          ok = mbar_wait(&wcbar[sbuf], cuse[sbuf] & 1, abort_flag, lim, p.status, W_EPI_C, t);
          cuse[sbuf]++;
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          if constexpr (kTransD) {
            // element (row i, column lane) of the staged FP32 box
#pragma unroll
            for (int i = 0; i < EC; ++i)
              v[i] += *reinterpret_cast<const float *>(
                  stg + i * (32 * 4) + (swz_chunk<32 * 4>(lane >> 2, i) << 4) + (lane & 3) * 4);
          } else {
            const uint8_t *rowp = stg + lane * (EC * 4);
#pragma unroll
            for (int i = 0; i < EC / 4; ++i) {
              const float4 cv = *reinterpret_cast<const float4 *>(rowp + (swz_chunk<EC * 4>(i, lane) << 4));
              v[4 * i + 0] += cv.x;
              v[4 * i + 1] += cv.y;
              v[4 * i + 2] += cv.z;
              v[4 * i + 3] += cv.w;
            }
          }
        }
        if constexpr (kTransD) {
          // Transposed tile: register i of lane l is D[row i of the box][column l];
          // each i writes one staged row (a warp-wide contiguous row, swizzled).
          static_assert(EC == 32, "transposed boxes are 32 x 32");
          if constexpr (kOut == OUT_BF16) {
#pragma unroll
            for (int i = 0; i < EC; ++i)
              *reinterpret_cast<__nv_bfloat16 *>(stg + i * 64 + (swz_chunk<64>(lane >> 3, i) << 4) +
                                                 (lane & 7) * 2) = __float2bfloat16_rn(v[i]);
          } else {
#pragma unroll
            for (int i = 0; i < EC; ++i)
              *reinterpret_cast<float *>(stg + i * 128 + (swz_chunk<128>(lane >> 2, i) << 4) +
                                         (lane & 3) * 4) = v[i];
          }
        } else if constexpr (kOut == OUT_BF16) {
          uint8_t *rowp = stg + lane * (EC * 2);
#pragma unroll
          for (int i = 0; i < EC / 8; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const __nv_bfloat162 pr =
                  __floats2bfloat162_rn(v[8 * i + 2 * h], v[8 * i + 2 * h + 1]);
              w[h] = *reinterpret_cast<const uint32_t *>(&pr);
            }
            *reinterpret_cast<uint4 *>(rowp + (swz_chunk<EC * 2>(i, lane) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          uint8_t *rowp = stg + lane * (EC * 4);
#pragma unroll
          for (int i = 0; i < EC / 4; ++i)
            *reinterpret_cast<float4 *>(rowp + (swz_chunk<EC * 4>(i, lane) << 4)) =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && store) {
          if constexpr (kOut == OUT_F32_REDUCE)
            tma_reduce_add_3d_hint(&p.tmD, stg, bx, by, dz, stream_out);
          else
            tma_store_3d_hint(&p.tmD, stg, bx, by, dz, stream_out);
          bulk_commit();
        }
      }
      if (!ok) break;
      if (mma_tile) ++uses[b];
    }
    if (lane == 0) bulk_wait<0>();
  }

#ifdef DG_KERNEL_TIMERS
  // Per CTA 32 counters, 8 per role (producer, MMA, warp 6, epilogue warp 2):
  // the role's counters tm[0..3], its total cycles, then tm[4..6].
  if (lane == 0 && p.timers != nullptr && (warp <= 2 || warp == 6)) {
    const int role = warp == 0 ? 0 : warp == 1 ? 1 : warp == 6 ? 2 : 3;
    unsigned long long *o = p.timers + blockIdx.x * 32 + role * 8;
    for (int i = 0; i < 4; ++i) o[i] = tm[i];
    o[4] = clock64() - t_start;
    for (int i = 4; i < 7; ++i) o[i + 1] = tm[i];
  }
#endif

  // Neither CTA may release its shared or tensor memory while the pair's MMAs
  // or the partner's remote arrivals may still touch it.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

template <bool kFP8, int kBN, int kOut, bool kKMajor, bool kTransD, bool kMG = false>
cudaError_t launch_wgrad_variant(const WgradParams &p, int pairs, cudaStream_t stream) {
  using Cfg = WgradCfg<kFP8, kBN, kKMajor, kMG, kTransD>;
  auto kern = kgrouped_wgrad_kernel<kFP8, kBN, kOut, kKMajor, kTransD, kMG>;
  // the schedule length and the division constants come from set_derived()
  if (p.num_tiles > 0 && (p.n_sched <= 0 || p.n_sched > kMaxGroups)) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // After the scale-pack pass: start while it runs (only the scale loader
  // waits for its records, griddepcontrol.wait).
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Shared-memory attribute and the number of co-resident pairs, once per
  // process (thread-safe static initialisation).
  struct Setup {
    cudaError_t err;
    int max_pairs;
  };
  static const Setup setup = [&] {
    Setup st{cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Cfg::SMEM_BYTES), 0};
    if (st.err != cudaSuccess) return st;
    cudaLaunchConfig_t c = cfg;
    c.gridDim = dim3(2 * (pairs > 0 ? pairs : 1), 1, 1);
    st.err = cudaOccupancyMaxActiveClusters(&st.max_pairs, kern, &c);
    return st;
  }();
  if (setup.err != cudaSuccess) return setup.err;
  if (setup.max_pairs > 0) pairs = min(pairs, setup.max_pairs);
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  if (kFP8 && p.pdl) cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// kTransD: the kernel computes D^T tiles (the host passes B as the kernel's A
// and A as its B, with M and N swapped) and writes them transposed into D.
template <bool kFP8, int kBN, bool kKMajor = false, bool kTransD = false>
cudaError_t launch_wgrad_bn(const WgradParams &p, int pairs, cudaStream_t stream) {
  switch (p.out_mode) {
    case OUT_F32:
      return launch_wgrad_variant<kFP8, kBN, OUT_F32, kKMajor, kTransD>(p, pairs, stream);
    case OUT_F32_REDUCE:
      return launch_wgrad_variant<kFP8, kBN, OUT_F32_REDUCE, kKMajor, kTransD>(p, pairs, stream);
    case OUT_F32_C:
      return launch_wgrad_variant<kFP8, kBN, OUT_F32_C, kKMajor, kTransD>(p, pairs, stream);
    case OUT_BF16:
      return launch_wgrad_variant<kFP8, kBN, OUT_BF16, kKMajor, kTransD>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

// M-grouped FP8 data gradient: A K-major (token rows of dy), B MN-major (the
// expert weights), direct tiles, FP32 or BF16 output.
// kKMajor: the weights stored K-major, [G, N, K].
template <int kBN, bool kKMajor = false>
cudaError_t launch_mgrouped_bn(const WgradParams &p, int pairs, cudaStream_t stream) {
  switch (p.out_mode) {
    case OUT_F32:
      return launch_wgrad_variant<true, kBN, OUT_F32, kKMajor, false, true>(p, pairs, stream);
    case OUT_BF16:
      return launch_wgrad_variant<true, kBN, OUT_BF16, kKMajor, false, true>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
