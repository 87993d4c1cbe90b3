// Pieces shared by the host planner and the device kernel: tile geometry, the
// grouped tile order, and the tcgen05 descriptor encoders.  Plain integer code,
// callable on both sides (host tests exercise it without a GPU).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define GEMM_HD __host__ __device__ __forceinline__
#else
#define GEMM_HD inline
#endif

namespace gemm_tc {

constexpr int BM = 128;      // output rows per CTA tile = MMA M: one TMEM lane per row
constexpr int BK = 64;       // K per pipeline stage: 64 x 16-bit = one 128-byte swizzle row
constexpr int UMMA_K = 16;   // K of one tcgen05.mma of kind::f16
constexpr int SW = 128;      // swizzle width in bytes (TMA and MMA agree on the 128B pattern)
constexpr int ATOM_MN = 64;  // 16-bit elements across one swizzle row (MN-major operands)

// ---------------------------------------------------------------- tile order
//
// Grouped ("walk a few rows of the tile grid at a time") order from the lecture
// "The Asynchronous Kernel: Tensor Cores & TMA" (linearly.space), section
// "Scheduling is geometry", and the Ada GEMM page's CTA-rasterisation table
// (kd.iw.mk): tiles are taken group_m tile-rows at a time, column by column
// inside the group, so the tiles in flight share few A and B panels in L2.
GEMM_HD void tile_coord(int t, int m_tiles, int n_tiles, int group_m, int* m_blk, int* n_blk) {
  const int group_size = group_m * n_tiles;
  const int g = t / group_size;
  const int first_m = g * group_m;
  const int rows_in_group = (m_tiles - first_m) < group_m ? (m_tiles - first_m) : group_m;
  const int r = t - g * group_size;
  *m_blk = first_m + r % rows_in_group;
  *n_blk = r / rows_in_group;
}

// Division by a run-time constant d (1 <= d < 2^31) of numerators n in
// [0, 2^31) by a multiply and a shift, the constants worked out once on the host
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994: l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
// q = (mulhi(m, n) + n) >> l; with n < 2^31 the sum cannot overflow 32 bits).
// The device's own integer division is a long dependent instruction sequence,
// and the tile order divides on the producer's path to its first copy.
struct FastDiv {
  uint32_t d, mul, shift;
};

GEMM_HD FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  f.shift = l;
  f.mul = static_cast<uint32_t>((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
  return f;
}

GEMM_HD uint32_t fastdiv(uint32_t n, uint32_t mul, uint32_t shift) {
#if defined(__CUDA_ARCH__)
  const uint32_t t = __umulhi(n, mul);
#else
  const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(n) * mul) >> 32);
#endif
  return (t + n) >> shift;
}

// The grouped order of tile_coord with its divisions by the group size (in
// tiles) and by a group's row count (group_m, or the last group's rows) done by
// fastdiv; gs, gm and gl are make_fastdiv of those three.
GEMM_HD void tile_coord_fast(int t, int m_tiles, int group_m, const FastDiv& gs, const FastDiv& gm,
                             const FastDiv& gl, int* m_blk, int* n_blk) {
  const int g = static_cast<int>(fastdiv(static_cast<uint32_t>(t), gs.mul, gs.shift));
  const int first_m = g * group_m;
  const int r = t - g * static_cast<int>(gs.d);
  const bool last = m_tiles - first_m < group_m;
  const uint32_t rows = last ? gl.d : gm.d;
  const int n = static_cast<int>(fastdiv(static_cast<uint32_t>(r), last ? gl.mul : gm.mul,
                                         last ? gl.shift : gm.shift));
  *m_blk = first_m + (r - n * static_cast<int>(rows));
  *n_blk = n;
}

// Cell (x, y) at index d of the Hilbert curve over a 2^k x 2^k grid (the order the
// lecture "The Asynchronous Kernel: Tensor Cores & TMA" compares in "Scheduling
// is geometry": a space-filling curve whose every prefix stays compact).  Built
// one level at a time from the lowest: two bits of d pick the quadrant, and the
// cells placed so far are turned into that quadrant's orientation (a transpose,
// plus a reflection in the last quadrant) so consecutive indices stay adjacent.
GEMM_HD void hilbert_cell(int k, long long d, int* x, int* y) {
  int cx = 0, cy = 0;
  for (int lvl = 0; lvl < k; ++lvl) {
    const int s = 1 << lvl;
    const int qx = static_cast<int>((d >> 1) & 1);
    const int qy = static_cast<int>((d ^ qx) & 1);
    if (qy == 0) {
      if (qx == 1) {
        cx = s - 1 - cx;
        cy = s - 1 - cy;
      }
      const int t = cx;
      cx = cy;
      cy = t;
    }
    cx += s * qx;
    cy += s * qy;
    d >>= 2;
  }
  *x = cx;
  *y = cy;
}

// -------------------------------------------------------- tcgen05 descriptors
//
// Instruction descriptor of tcgen05.mma kind::f16 and kind::f8f6f4 (32 bits, public
// PTX ISA; the same layout for both kinds):
//   [4,6) D format (1 = f32)   [7,10) A format   [10,13) B format (kind::f16: 0 = f16,
//   1 = bf16; kind::f8f6f4: 0 = E4M3, 1 = E5M2; in_is_bf16 carries that code)
//   [15] A major   [16] B major (0 = K-major, 1 = MN-major)
//   [17,23) N >> 3   [24,29) M >> 4     (everything else 0: dense, no negate)
GEMM_HD uint32_t make_idesc_f16(int in_is_bf16, int a_mn, int b_mn, int m, int n) {
  return (1u << 4) | ((uint32_t)in_is_bf16 << 7) | ((uint32_t)in_is_bf16 << 10) |
         ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// Shared-memory matrix descriptor (64 bits, public PTX ISA):
//   [0,14) start address >> 4   [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4   [46,48) = 1 (descriptor version)
//   [49,52) base offset (0: atoms are 1024-byte aligned)   [61,64) swizzle (2 = 128B)
//
// Canonical 128B-swizzled layouts (units: 16-bit elements):
//  * K-major: rows of 64 K-elements (128 B), 8-row core groups 1024 B apart
//    -> SBO = 1024, LBO unused (encoded 1).  Advancing K by 16 inside the row
//    adds 32 bytes to the start address (the swizzle is applied on address bits).
//  * MN-major: 64 MN-elements per 128-byte row, one row per K index, 8-row core
//    groups 1024 B apart along K (SBO) and 64-element MN atoms LBO bytes apart.
GEMM_HD uint64_t make_sdesc_sw128(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// ------------------------------------------------------------- work split
//
// A launch's work is a list of tiles, each a sequence of `groups` k-groups (ring
// stages).  Data-parallel tiles: unit u (a CTA, or a CTA pair) takes whole tiles
// u, u + units, ... below dp_tiles.  Stream-K tiles: the remaining tiles'
// k-groups form one iteration space of sk_iters = (num_tiles - dp_tiles) *
// groups entries, split evenly: unit u takes [u * sk_iters / units,
// (u + 1) * sk_iters / units), walked tile by tile from its top down.  A unit
// walks its stream-K share first and its data-parallel tiles after it, so the
// stream-K fix-ups (below) run while data-parallel mainloops keep the tensor
// cores busy, and the launch ends on plain tiles.  The unit holding a tile's
// last k-groups owns the tile (for it that is the last segment of its stream-K
// share); every earlier unit touching the tile leaves its share as a partial
// sum in its first (or only) segment, so partials are ready long before their
// owner needs them and no unit waits on a chain.  A unit's data-parallel tiles
// alternate the direction of their k loop (up, down, up, ...): the units run
// their data-parallel rounds side by side, so each round starts with the
// k-blocks the previous round loaded last, which are the ones still in L2
// (the rows of A are shared by the rounds of one group of the grouped order).
// Walking its stream-K share down, the first
// segment of every unit whose share spans tiles starts at k-group 0 of a tile,
// as the first tiles of a data-parallel launch do: the neighbouring units'
// first copies share operand panels in L2 rather than all coming from DRAM at
// once.
struct WorkItem {
  int tile, g0, g1;   // tile index and k-group range [g0, g1)
  int down;           // 1: the k-groups are walked from g1 - 1 down to g0
};

// Split-tile schedule (tile_split = s >= 2, instead of the two kinds above):
// unit u works on tile u / s alone.  Part u % s = 0 takes k-groups
// [0, owner_groups) and owns the tile; parts 1 .. s-1 split the remaining
// k-groups evenly and leave partial sums.  The owner's share is the larger one,
// so the other parts finish (and publish) while it is still accumulating.
//
// The stream-K range is worked out without 64-bit divisions (slow on the
// device, and on the producer's path to its first copy): sk_iters < 2^31 (the
// planner's limit), and with sk_iters = q * units + r, u * sk_iters / units =
// u * q + (u * r) / units, all 32-bit; a position i is split into tile and
// k-group by fastdiv (fg: make_fastdiv of groups).
struct WorkIter {
  int units, dp_tiles, groups, next_dp, dp_round;
  long long i, hi;
  FastDiv fg;
  int st_tile, st_g0, st_g1;   // split-tile: the unit's one item (st_tile < 0: taken)
  GEMM_HD void init(int unit, int units_, int dp_tiles_, long long sk_iters, int groups_,
                    const FastDiv& fg_, int tile_split = 0, int owner_groups = 0) {
    units = units_;
    dp_tiles = dp_tiles_;
    groups = groups_;
    next_dp = unit;
    dp_round = 0;
    fg = fg_;
    i = hi = 0;
    st_tile = -1;
    st_g0 = st_g1 = 0;
    if (tile_split > 1) {
      const int part = unit % tile_split;
      st_tile = unit / tile_split;
      if (part == 0) {
        st_g1 = owner_groups;
      } else {
        const int rest = groups_ - owner_groups, np = tile_split - 1;
        st_g0 = owner_groups + ((part - 1) * rest) / np;
        st_g1 = owner_groups + (part * rest) / np;
      }
      dp_tiles = 0;
    } else if (sk_iters != 0) {
      const uint32_t u = static_cast<uint32_t>(units_);
      const uint32_t q = static_cast<uint32_t>(sk_iters) / u;
      const uint32_t r = static_cast<uint32_t>(sk_iters) - q * u;
      const uint32_t ur = static_cast<uint32_t>(unit) * r;
      i = static_cast<long long>(unit) * q + ur / u;
      hi = static_cast<long long>(unit + 1) * q + (ur + r) / u;
    }
  }
  GEMM_HD bool next(WorkItem* w) {
    if (st_tile >= 0) {
      w->tile = st_tile;
      w->g0 = st_g0;
      w->g1 = st_g1;
      w->down = 0;
      st_tile = -1;
      return true;
    }
    if (i < hi) {   // the stream-K share first, from its last tile down
      const int t = static_cast<int>(fastdiv(static_cast<uint32_t>(hi - 1), fg.mul, fg.shift));
      const long long start = static_cast<long long>(t) * groups;
      const long long lo = i > start ? i : start;
      w->tile = dp_tiles + t;
      w->g0 = static_cast<int>(lo - start);
      w->g1 = static_cast<int>(hi - start);
      w->down = 0;
      hi = lo;
      return true;
    }
    if (next_dp < dp_tiles) {
      w->tile = next_dp;
      w->g0 = 0;
      w->g1 = groups;
      w->down = dp_round & 1;
      next_dp += units;
      ++dp_round;
      return true;
    }
    return false;
  }
};

// Stream-K unit whose iteration range contains iteration i (0 <= i < sk_iters).
GEMM_HD int sk_unit_of(long long i, int units, long long sk_iters) {
  int u = static_cast<int>((i * units) / sk_iters);
  while (u + 1 < units && ((static_cast<long long>(u) + 1) * sk_iters) / units <= i) ++u;
  while (u > 0 && (static_cast<long long>(u) * sk_iters) / units > i) --u;
  return u;
}

// Fused epilogue kinds (same values as the public GEMM_BIAS_* / GEMM_ACT_*).
enum { EPI_BIAS_NONE = 0, EPI_BIAS_COL = 1, EPI_BIAS_ROW = 2 };
enum { EPI_ACT_NONE = 0, EPI_ACT_RELU = 1 };

// Kernel arguments (plain data, built on the host).
struct KernelArgs {
  // The fields the producer and the MMA issuer read before their first copy and
  // first MMA come first, so that those reads touch few constant-cache lines
  // (each line a kernel's CTAs first read costs a round trip to memory).
  int m_tiles, n_tiles, group_m, k_blocks;
  // Work split (see WorkIter): k-groups per tile, whole tiles of the
  // data-parallel phase, stream-K iterations after it; or the split-tile
  // schedule's parts per tile (0: not used) and the k-groups of its owning part.
  int groups, dp_tiles, tile_split, owner_groups;
  int a_hint, b_hint;    // L2 policy of the operand loads: 0 default, 1 evict first, 2 evict last
  int a_mn, b_mn;        // 1: operand is MN-major in memory (A column-major / B row-major)
  // Extent of the 3-D operand maps in whole 64-element blocks (0: no 3-D map):
  // K-major operand -> full k-blocks (K / 64); MN-major -> full 64-wide atoms.
  int a_full3d, b_full3d;
  // K elements of one k-block (64 for 16-bit operands, 128 for 8-bit ones: one
  // 128-byte swizzled row either way).
  int kblock_elems;
  // Rows of A each k-block copy brings (BM, or fewer for a single row of tiles
  // with M < BM: the rows of smem beyond them only feed accumulator rows >= M,
  // which are never stored).
  int a_box_rows;
  long long sk_iters;    // < 2^31
  FastDiv fd_groups;     // make_fastdiv(groups), for WorkIter
  unsigned long long timeout_ns;
  int* status;           // device status word (0 = ok)
  // Tile order: NULL = grouped (tile_coord), else (m block, n block) of tile t
  // in Hilbert-curve order, num_tiles entries.
  const int2* tile_map;
  // The grouped order's divisors (tile_coord_fast): group size in tiles
  // (group_m * n_tiles), group_m, and the last group's row count.
  FastDiv fd_group, fd_rows, fd_last_rows;
  uint32_t idesc;        // tcgen05 instruction descriptor (formats, majors, M, N)
  int read_c;            // beta != 0
  // 1: beta * C is written into a tile's TMEM accumulator before its first MMA
  // (alpha == 1 only, so the accumulator then holds alpha*AB + beta*C), for every
  // work item after a unit's first two that finishes its tile (item_preloads_c).
  int pre_c;
  int inject_skip;       // debug: the producer leaves ring iteration (inject_skip - 1) unarmed
  int num_tiles;
  int M, N, K;
  float alpha, beta;
  void* c_ptr;           // C base (for the ragged right edge, written with plain stores)
  long long ldc;         // C leading dimension in elements
  int n_ragged;          // 1 when N * sizeof(out) is not a multiple of 16 bytes
  // Stream-K scratch: one fp32 partial tile slot and one ready flag per CTA;
  // a flag holds the epoch of the launch whose partial is in the slot.
  unsigned int epoch;
  float* ws;
  unsigned int* ws_flags;
  // Fused epilogue: out = act(alpha*acc + beta*C + bias) before the rounding.
  const float* bias;     // N floats (EPI_BIAS_COL) or M floats (EPI_BIAS_ROW), 16-byte aligned
  int bias_kind;         // EPI_BIAS_*
  int act;               // EPI_ACT_*
  int epi;               // 1 when bias_kind or act is set (selects the fused epilogue)
};

// Whether work item w finishes its tile: a whole tile, or the owner's segment
// (the last k-groups for stream-K, the first for a split-tile part), which adds
// the other units' partial sums and stores the output.  Every other item leaves
// a partial sum.
GEMM_HD bool item_finishes(const KernelArgs& a, const WorkItem& w) {
  return a.tile_split > 1 ? w.g0 == 0 : w.g1 >= a.groups;
}

// Whether work item number `tl` of a unit (item `w`) starts from an accumulator
// holding beta * C rather than zero (see KernelArgs::pre_c): only an item that
// finishes its tile takes the C term.  The MMA issuer and the epilogue warps
// evaluate it on the same item sequence.
GEMM_HD bool item_preloads_c(const KernelArgs& a, uint32_t tl, const WorkItem& w) {
  return a.pre_c && a.read_c && tl >= 2 && item_finishes(a, w);
}

// Units whose partial sums the owner of work item w (unit `unit` of `units`;
// w finishes its tile but does not hold all of its k-groups) adds, in unit
// order: [*c0, *c1).  Stream-K: the units before it, down to the one holding
// the tile's first k-group; split-tile: the tile's other parts, after it.
GEMM_HD void owner_contributors(const KernelArgs& a, int unit, int units, const WorkItem& w,
                                int* c0, int* c1) {
  if (a.tile_split > 1) {
    *c0 = unit + 1;
    *c1 = unit + a.tile_split;
  } else {
    const long long base = static_cast<long long>(w.tile - a.dp_tiles) * a.groups;
    *c0 = sk_unit_of(base, units, a.sk_iters);
    *c1 = unit;
  }
}

#if defined(__CUDACC__)
// Output block (m_blk, n_blk) of tile index t in the launch's tile order.
__device__ __forceinline__ void tile_of(const KernelArgs& a, int t, int* m_blk, int* n_blk) {
  if (a.tile_map) {
    const int2 v = __ldg(a.tile_map + t);
    *m_blk = v.x;
    *n_blk = v.y;
  } else {
    tile_coord_fast(t, a.m_tiles, a.group_m, a.fd_group, a.fd_rows, a.fd_last_rows, m_blk, n_blk);
  }
}
#endif

}  // namespace gemm_tc
