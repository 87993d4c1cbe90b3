// Host side of the C ABI declared in include/gemm_tcgen05.h: argument checks,
// launch planning, TMA tensor-map encoding and kernel launch.
//
// The tensor map is the host-built copy descriptor of the lecture "The
// Asynchronous Kernel: Tensor Cores & TMA" (linearly.space), section "One thread
// orders the groceries": element type, base pointer, matrix shape, row pitch,
// tile shape and the 128B swizzle the tile gets on arrival ("The XOR that unties
// the banks").  cuTensorMapEncodeTiled is reached through the runtime's driver
// entry-point query, so the library does not link libcuda.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "gemm_common.h"
#include "gemm_kernel.cuh"
#include "gemm_launch.h"
#include "gemm_tcgen05.h"

using namespace gemm_tc;

// Wait-timeout status word of every GEMM kernel launched on a device.
__device__ int g_gemm_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int cc_major = 0, cc_minor = 0, num_sms = 0;
  int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<int32_t> g_inject_skip{0};

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

const DeviceInfo* device_info(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, [&d, dev]() {
    cudaDeviceProp p;
    d.err = cudaGetDeviceProperties(&p, dev);
    if (d.err != cudaSuccess) return;
    d.cc_major = p.major;
    d.cc_minor = p.minor;
    d.num_sms = p.multiProcessorCount;
    d.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_gemm_status_word);
  });
  return &d;
}

// Stream-K scratch, one per (device, stream) so that launches on different
// streams never share it: a fixed region of kMaxSkCtas ready flags (so a flag's
// address never depends on the launch shape), then one fp32 partial tile slot
// per CTA.  Grown on demand (the old buffer is freed after the stream drains),
// zeroed on the stream when allocated; every launch gets the next epoch, so a
// flag equal to the current epoch can only have been written by this launch.
constexpr int kMaxSkCtas = 1024;
constexpr size_t kFlagBytes = sizeof(unsigned int) * kMaxSkCtas;

struct Scratch {
  void* ptr = nullptr;
  size_t bytes = 0;
  unsigned int epoch = 0;
};
std::mutex g_scratch_mu;
std::map<std::pair<int, cudaStream_t>, Scratch> g_scratch;

gemm_status_t scratch_for(int dev, cudaStream_t st, size_t slot_bytes, int ctas, float** ws,
                          unsigned int** flags, unsigned int* epoch) {
  if (ctas > kMaxSkCtas) return GEMM_ERR_INVALID_ARG;
  const size_t need = kFlagBytes + slot_bytes * static_cast<size_t>(ctas);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  Scratch& sc = g_scratch[std::make_pair(dev, st)];
  if (sc.bytes < need) {
    if (sc.ptr) {
      if (cudaStreamSynchronize(st) != cudaSuccess) return GEMM_ERR_CUDA;
      cudaFree(sc.ptr);
      sc.ptr = nullptr;
      sc.bytes = 0;
    }
    if (cudaMalloc(&sc.ptr, need) != cudaSuccess) return GEMM_ERR_CUDA;
    sc.bytes = need;
    if (cudaMemsetAsync(sc.ptr, 0, kFlagBytes, st) != cudaSuccess) return GEMM_ERR_CUDA;
    sc.epoch = 0;
  }
  *flags = static_cast<unsigned int*>(sc.ptr);
  *ws = reinterpret_cast<float*>(static_cast<char*>(sc.ptr) + kFlagBytes);
  if (++sc.epoch == 0) {   // wrapped: old flags could match again, so clear them
    if (cudaMemsetAsync(sc.ptr, 0, kFlagBytes, st) != cudaSuccess) return GEMM_ERR_CUDA;
    sc.epoch = 1;
  }
  *epoch = sc.epoch;
  return GEMM_OK;
}

// Fixed stream-K scratch of gemm_ex_noalloc, for callers that must not
// allocate device memory on the call path (their memory is held by another
// allocator, or their loop must not synchronise or fail on cudaMalloc): a
// file-scope device array, one per device, laid out like the cached scratch
// (kFlagBytes of ready flags, then the fp32 partial slots).  Every call on a
// device shares it, so calls that overlap on the device race.
constexpr size_t kNoAllocScratchBytes = GEMM_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes > kFlagBytes, "the fixed scratch must hold the flags");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocScratch {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  void* ptr = nullptr;
  bool cleared = false;
  unsigned int epoch = 0;
};
NoAllocScratch g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Set-up, once per device with that device current: the array's device
// address.  The flags are cleared on the stream of the first launch that uses
// them (and again when the epoch wraps), then every launch takes the next epoch.
gemm_status_t noalloc_scratch(int dev, cudaStream_t st, size_t slot_bytes, int ctas, float** ws,
                              unsigned int** flags, unsigned int* epoch) {
  // the flag region holds kMaxSkCtas flags: a wider grid would index past it
  if (ctas > kMaxSkCtas) return GEMM_ERR_INVALID_ARG;
  const size_t need = kFlagBytes + slot_bytes * static_cast<size_t>(ctas);
  if (need > kNoAllocScratchBytes) return GEMM_ERR_SCRATCH;
  NoAllocScratch& n = g_noalloc[dev];
  std::call_once(n.once, [&n]() {
    n.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&n.ptr), g_noalloc_scratch);
  });
  if (n.err != cudaSuccess || n.ptr == nullptr) return GEMM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!n.cleared || ++n.epoch == 0) {
    if (cudaMemsetAsync(n.ptr, 0, kFlagBytes, st) != cudaSuccess) return GEMM_ERR_CUDA;
    n.cleared = true;
    n.epoch = 1;
  }
  *flags = static_cast<unsigned int*>(n.ptr);
  *ws = reinterpret_cast<float*>(static_cast<char*>(n.ptr) + kFlagBytes);
  *epoch = n.epoch;
  return GEMM_OK;
}

// Tiles of an m_tiles x n_tiles grid in Hilbert-curve order: the curve over the
// smallest power-of-two square holding the grid, keeping the cells inside it
// (x = n block, y = m block).  False (nothing written) when the square would hold
// more than 16 times the grid's tiles, or the grid more than 2^22 tiles.
bool hilbert_tiles(int m_tiles, int n_tiles, std::vector<int2>* out) {
  const int64_t tiles = int64_t(m_tiles) * n_tiles;
  if (m_tiles <= 0 || n_tiles <= 0 || tiles > (int64_t(1) << 22)) return false;
  int k = 0;
  while ((int64_t(1) << k) < std::max(m_tiles, n_tiles)) ++k;
  const int64_t cells = int64_t(1) << (2 * k);
  if (cells > 16 * tiles) return false;
  out->clear();
  out->reserve(static_cast<size_t>(tiles));
  for (int64_t d = 0; d < cells; ++d) {
    int x, y;
    hilbert_cell(k, d, &x, &y);
    if (x < n_tiles && y < m_tiles) out->push_back(make_int2(y, x));
  }
  return true;
}

// Device copies of Hilbert tile tables, one per (device, grid shape), built on
// first use and kept for the life of the process.
std::mutex g_map_mu;
std::map<std::tuple<int, int, int>, int2*> g_maps;

gemm_status_t hilbert_map_for(int dev, int m_tiles, int n_tiles, const int2** table) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  const auto key = std::make_tuple(dev, m_tiles, n_tiles);
  auto it = g_maps.find(key);
  if (it != g_maps.end()) {
    *table = it->second;
    return GEMM_OK;
  }
  std::vector<int2> host;
  if (!hilbert_tiles(m_tiles, n_tiles, &host)) return GEMM_ERR_INVALID_ARG;
  int2* d = nullptr;
  if (cudaMalloc(&d, host.size() * sizeof(int2)) != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaMemcpy(d, host.data(), host.size() * sizeof(int2), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(d);
    return GEMM_ERR_CUDA;
  }
  g_maps[key] = d;
  *table = d;
  return GEMM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

int out_size(int out_dtype) { return out_dtype == GEMM_F32 ? 4 : 2; }

bool is_fp8(int in_dtype) { return in_dtype == GEMM_E4M3 || in_dtype == GEMM_E5M2; }

// Bytes per input element, and K elements per k-block (one 128-byte swizzled row).
int in_size(int in_dtype) { return is_fp8(in_dtype) ? 1 : 2; }
int kblock_elems(int in_dtype) { return is_fp8(in_dtype) ? 2 * BK : BK; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks on sizes, formats and layout only (no pointers): shared by gemm() and
// gemm_plan().  *quick is set when M == 0 or N == 0 (nothing to do).
gemm_status_t check_shape(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int layout,
                          bool* quick) {
  *quick = false;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (layout & ~(GEMM_A_COL | GEMM_B_COL)) return GEMM_ERR_INVALID_ARG;
  if (in_dtype != GEMM_F16 && in_dtype != GEMM_BF16 && !is_fp8(in_dtype))
    return GEMM_ERR_UNSUPPORTED;
  // 8-bit operands: K-major only (A row-major, B column-major)
  if (is_fp8(in_dtype) && layout != (GEMM_A_ROW | GEMM_B_COL)) return GEMM_ERR_UNSUPPORTED;
  if (out_dtype != GEMM_F32 && out_dtype != GEMM_BF16 && out_dtype != GEMM_F16)
    return GEMM_ERR_UNSUPPORTED;
  // tile indices and TMA coordinates are 32-bit signed on the device
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return GEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) *quick = true;
  return GEMM_OK;
}

// Full argument check of gemm(); pointers may be device or host (gemm_host).
gemm_status_t check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, const void* C, int64_t ldc, int in_dtype,
                         int out_dtype, int layout, bool* quick) {
  gemm_status_t s = check_shape(M, N, K, in_dtype, out_dtype, layout, quick);
  if (s != GEMM_OK || *quick) return s;
  const bool a_col = (layout & GEMM_A_COL) != 0, b_col = (layout & GEMM_B_COL) != 0;
  if (ldc < N) return GEMM_ERR_INVALID_ARG;
  if (C == nullptr) return GEMM_ERR_INVALID_ARG;
  const int osz = out_size(out_dtype);
  // byte extents must fit comfortably in 63 bits and TMA strides below 2^40 bytes
  if (ldc > (int64_t(1) << 36) || M > (int64_t(1) << 62) / (ldc * osz + 1))
    return GEMM_ERR_INVALID_ARG;
  if (!aligned16(C) || (ldc * osz) % 16 != 0) return GEMM_ERR_UNSUPPORTED;
  if (K > 0) {
    const int64_t lda_min = a_col ? M : K, ldb_min = b_col ? K : N;
    if (lda < lda_min || ldb < ldb_min) return GEMM_ERR_INVALID_ARG;
    if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_ARG;
    if (lda > (int64_t(1) << 36) || ldb > (int64_t(1) << 36)) return GEMM_ERR_INVALID_ARG;
    const int64_t a_rows = a_col ? K : M, b_rows = b_col ? N : K;
    const int isz = in_size(in_dtype);
    if (a_rows > (int64_t(1) << 62) / (lda * isz + 1) || b_rows > (int64_t(1) << 62) / (ldb * isz + 1))
      return GEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || (lda * isz) % 16 != 0 || (ldb * isz) % 16 != 0)
      return GEMM_ERR_UNSUPPORTED;
  }
  return GEMM_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Work-unit choice.  Per k-block a CTA's tensor core needs 2*W cycles for a
// 128 x W tile, while its shared memory must receive (128 + W') * 128 bytes
// (W' = B columns it loads: W, or W/2 for a CTA pair); measured on GB300 the
// delivery is ~64 B per SM clock, so a k-block costs max(2W, bytes/64) cycles.
// A launch costs waves * k-block cost (a wave = one unit per SM, or per SM pair),
// so the choice weighs tile efficiency against wave quantisation.  Pairs need
// more than 128 rows.  Ties go to the earlier candidate (single CTA first, then
// the wider tile: fewer clusters to launch, fewer tiles to store).
void choose_unit(int64_t M, int64_t N, int num_sms, int* bn_out, bool* pair_out) {
  struct Cand { int bn; bool pair; };
  const Cand cands[5] = {{256, false}, {128, false}, {64, false}, {256, true}, {128, true}};
  int64_t best_cost = -1;
  *bn_out = 256;
  *pair_out = false;
  for (const Cand& c : cands) {
    if (c.pair && (M <= BM || num_sms < 2)) continue;
    const int64_t rows = c.pair ? 2 * BM : BM;
    const int64_t units = ceil_div(M, rows) * ceil_div(N, c.bn);
    const int64_t slots = c.pair ? num_sms / 2 : num_sms;
    const int64_t waves = ceil_div(units, slots);
    const int64_t bytes = int64_t(BM + b_cols_per_cta(c.bn, c.pair)) * BK * 2;
    const int64_t per_kblock = std::max<int64_t>(2 * c.bn, bytes / 64);
    const int64_t cost = waves * per_kblock;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      *bn_out = c.bn;
      *pair_out = c.pair;
    }
  }
}

// Tile and split-K choice for a single 128-row panel (M <= 128), where output
// tiles alone cannot occupy the GPU: a tile width and a cluster of `split` CTAs
// per tile, each accumulating 1/split of K.  The choice that puts the most CTAs
// in one wave, each with at least 8 k-blocks; on a tie the earlier of this list:
// 128-wide tiles first (their 3-stage ring hides HBM latency better than the
// 2-stage ring of 256-wide ones: 8 x 14336 x 4096 runs 30.7 us unsplit at 128
// against 35.4 us split 2 at 256; 128 x 8192 x 8192 36.9 vs 45 us split 4),
// fewer splits first (less partial-sum exchange), 64-wide before 256-wide.
// Unsplit tiles only for panels of at most 32 rows: each CTA then reads all of
// A's K, which for taller panels outweighs the exchange a split saves.
// Returns 0 (no opinion: the general unit choice applies) when M > 128 or when
// no choice reaches the parallelism of 64-wide unsplit tiles; otherwise the
// split (1 = unsplit) with the tile width in *bn_out.
int choose_split(int64_t M, int64_t N, int64_t K, int kbe, int num_sms, int* bn_out) {
  if (M > BM) return 0;
  const int64_t kb = ceil_div(K, kbe);
  const struct { int bn, s; } cands[] = {{128, 1}, {128, 2}, {64, 2}, {256, 2},
                                         {128, 4}, {64, 4}, {256, 4}, {128, 8}};
  int best = -1;
  int64_t best_ctas = 0;
  for (int i = 0; i < static_cast<int>(sizeof(cands) / sizeof(cands[0])); ++i) {
    const int64_t ctas = ceil_div(N, cands[i].bn) * cands[i].s;
    if (cands[i].s == 1 && M > 32) continue;
    if (ctas <= num_sms && kb >= 8 * cands[i].s && ctas > best_ctas) {
      best = i;
      best_ctas = ctas;
    }
  }
  if (best < 0 || best_ctas < std::min<int64_t>(ceil_div(N, 64), num_sms / 2)) return 0;
  *bn_out = cands[best].bn;
  return cands[best].s;
}

// k-groups of a split tile's first part, the one that finishes the tile: a
// larger share than each of the others' (by about a tenth of the tile's
// k-groups), so they finish first and their partial sums are in its spare
// accumulator before its own MMAs end.  Every other part keeps at least one
// k-group.
int split_owner_groups(int groups, int parts) {
  const int extra = std::max(1, groups / 10);
  int owner = (groups + (parts - 1) * extra) / parts;
  owner = std::min(owner, groups - (parts - 1));
  return std::max(owner, 1);
}

gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int layout,
                        int num_sms, const gemm_config_t* cfg, gemm_plan_t* p) {
  const int kbe = kblock_elems(in_dtype);
  if (num_sms <= 0) return GEMM_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  if (cfg && (cfg->general < 0 || cfg->general > 1)) return GEMM_ERR_INVALID_ARG;
  if (cfg && (cfg->order < GEMM_ORDER_AUTO || cfg->order > GEMM_ORDER_HILBERT))
    return GEMM_ERR_INVALID_ARG;
  int bn = 0;
  bool pair = false;
  choose_unit(M, N, num_sms, &bn, &pair);
  int split = choose_split(M, N, K, kbe, num_sms, &bn);
  if (split > 0) pair = false;   // the single panel's choice: single-CTA tiles
  if (split == 0) split = 1;
  // a manual tile setting without an explicit split_k turns the automatic split off
  if (cfg && (cfg->cta_group || cfg->bn) && !cfg->split_k) split = 1;
  if (cfg && cfg->cta_group) {
    if (cfg->cta_group != 1 && cfg->cta_group != 2) return GEMM_ERR_INVALID_ARG;
    pair = cfg->cta_group == 2;
    if (!cfg->bn) bn = 256;
  }
  const int sk_mode = cfg ? cfg->stream_k : 0;
  if (sk_mode < 0 || sk_mode > 3) return GEMM_ERR_INVALID_ARG;
  // split-tile (stream_k 3): split_k parts per tile through the scratch buffer,
  // single-CTA tiles, no cluster
  int tile_split = 0;
  if (sk_mode == 3) {
    tile_split = cfg->split_k ? cfg->split_k : 2;
    if (tile_split < 2 || tile_split > 16 || cfg->cta_group == 2) return GEMM_ERR_INVALID_ARG;
    pair = false;
    split = 1;
    if (!cfg->bn) bn = 128;
  } else if (cfg && cfg->split_k) {
    if (cfg->split_k < 1) return GEMM_ERR_INVALID_ARG;
    split = cfg->split_k;
    if (!cfg->bn) bn = 256;
    if (split > 1 && !cfg->cta_group) pair = false;   // split-K clusters are single-CTA tiles
  }
  if (cfg && cfg->bn) bn = cfg->bn;
  if (pair ? (bn != 128 && bn != 256) : (bn != 64 && bn != 128 && bn != 256))
    return GEMM_ERR_INVALID_ARG;
  if (split > 1 && (pair || !split_supported(bn, split) || ceil_div(K, kbe) < split))
    return GEMM_ERR_INVALID_ARG;
  const int rows = pair ? 2 * BM : BM;
  p->bm = rows;
  p->bn = bn;
  p->bk = kbe * ko_for(bn, pair);   // K elements per ring stage
  p->stages = stages_for(bn, pair);
  const int64_t mt = ceil_div(M, rows), nt = ceil_div(N, bn), kb = ceil_div(K, kbe);
  if (mt * nt >= (int64_t(1) << 30)) return GEMM_ERR_UNSUPPORTED;
  p->m_tiles = static_cast<int32_t>(mt);
  p->n_tiles = static_cast<int32_t>(nt);
  p->k_blocks = static_cast<int32_t>(kb);
  p->num_tiles = static_cast<int32_t>(mt * nt);
  int gm = (cfg && cfg->group_m) ? cfg->group_m : (bn == 256 ? 16 : 8);
  if (pair && !(cfg && cfg->group_m)) gm = 8;
  if (gm < 0) return GEMM_ERR_INVALID_ARG;
  if (gm > p->m_tiles) gm = p->m_tiles > 0 ? p->m_tiles : 1;
  p->group_m = gm;
  // tile order: grouped unless the Hilbert curve is asked for and usable here
  p->order = GEMM_ORDER_GROUPED;
  if (cfg && cfg->order == GEMM_ORDER_HILBERT) {
    const int64_t cells_side = std::max(mt, nt);
    int k = 0;
    while ((int64_t(1) << k) < cells_side) ++k;
    if (mt * nt <= (int64_t(1) << 22) && (int64_t(1) << (2 * k)) <= 16 * mt * nt)
      p->order = GEMM_ORDER_HILBERT;
  }
  const int per_unit = pair ? 2 : 1;
  int grid = (cfg && cfg->grid) ? cfg->grid : (pair ? (num_sms / 2) * 2 : num_sms);
  if (grid < 0) return GEMM_ERR_INVALID_ARG;
  if (pair) grid = std::max(2, grid & ~1);
  // Work split: k-groups per tile, then stream-K for the last wave(s).  All but
  // the last whole wave stay data-parallel; the rest of the tiles' k-groups are
  // shared evenly by all units.  Chosen automatically when the run is at least
  // 2 waves long and the last wave would leave at least a quarter of the units
  // idle: with less than 2 waves every tile is split and the partial-sum
  // traffic costs more than the tail saves, and an almost full last wave has
  // little to balance (measured on GB300, same runs, us: 4096^3 76.5 / 78.6
  // data-parallel, 6144^2 x 4096 164.5 / 172.7, 8192^3 615.6 / 619.1 with
  // stream-K; 2048^3 27.3 / 21.1 and 3072^2 x 4096 51.8 / 47.8 without).
  const int ko = ko_for(bn, pair);
  p->groups = static_cast<int32_t>(ceil_div(kb, ko));
  p->dp_tiles = p->num_tiles;
  p->sk_iters = 0;
  // Owners wait for partials of higher-numbered units, so stream-K and
  // split-tile work need every unit resident at once: at most one CTA per SM.
  if (tile_split) {
    if (p->groups < tile_split) return GEMM_ERR_INVALID_ARG;   // a k-group per part at least
    if (int64_t(p->num_tiles) * tile_split > std::min(num_sms, kMaxSkCtas))
      return GEMM_ERR_UNSUPPORTED;
    p->dp_tiles = 0;
    p->tile_split = tile_split;
    p->owner_groups = split_owner_groups(p->groups, tile_split);
    grid = p->num_tiles * tile_split;
  } else if (split == 1 && sk_mode != 1 && grid <= kMaxSkCtas && grid <= num_sms) {
    const int64_t units = grid / per_unit;
    const int64_t waves = p->num_tiles / units, rem = p->num_tiles % units;
    const bool worth = rem != 0 && 4 * rem <= 3 * units && waves >= 2 && p->groups >= 4;
    if (sk_mode == 2 || worth) {
      const int64_t dp = (waves > 0 ? waves - 1 : 0) * units;
      const int64_t sk = (p->num_tiles - dp) * int64_t(p->groups);
      if (sk >= units && sk < (int64_t(1) << 31)) {   // the kernel's 32-bit stream-K range
        p->dp_tiles = static_cast<int32_t>(dp);
        p->sk_iters = sk;
      }
    }
  }
  // a data-parallel launch needs no more units than tiles
  if (!p->sk_iters && !tile_split && grid > p->num_tiles * per_unit) grid = p->num_tiles * per_unit;
  if (split > 1) {
    if (int64_t(p->num_tiles) * split >= (int64_t(1) << 31)) return GEMM_ERR_UNSUPPORTED;
    grid = p->num_tiles * split;   // exactly one tile per split-K cluster
  }
  p->grid = grid;
  p->split_k = split;
  p->scratch_bytes = (p->sk_iters || tile_split) ? int64_t(kFlagBytes) + int64_t(grid) * BM * int64_t(bn) * 4
                                                 : 0;
  p->threads = NUM_THREADS;
  p->smem_bytes = smem_alloc_bytes(bn, pair);
  p->tmem_cols = 2 * bn;
  p->a_mn = (layout & GEMM_A_COL) ? 1 : 0;
  p->b_mn = (layout & GEMM_B_COL) ? 0 : 1;
  p->epi_chunk_cols = out_dtype == GEMM_F32 ? 32 : 64;
  p->cta_group = pair ? 2 : 1;
  // the conditions of run_gemm's plain path that the plan itself fixes
  p->specialised = (p->order == GEMM_ORDER_GROUPED && !(cfg && cfg->general) &&
                    spec_supported(bn, pair, split, layout, is_fp8(in_dtype),
                                   p->sk_iters != 0 || tile_split != 0, false, false,
                                   (N * out_size(out_dtype)) % 16 != 0))
                       ? 1
                       : 0;
  return GEMM_OK;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D operand map: (64 elements, `d1` rows, `d2` whole 64-element blocks), the
// blocks 128 B apart along the row, so one box {64, box1, box2} covers box2
// consecutive blocks of each of its rows.  Only whole blocks are mapped: the
// kernel uses it for copies that stay inside them and the 2-D map otherwise.
// 3-D map (block, d1, d2): `inner` elements make the 128-byte block (64 16-bit or
// 128 8-bit elements), whole blocks 128 B apart along d2.
bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d1, uint64_t d2,
               uint64_t row_bytes, uint32_t box1, uint32_t box2, uint32_t inner = 64) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, d1, d2};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {inner, box1, box2};
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

CUtensorMapDataType tma_dtype(int dt) {
  switch (dt) {
    case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case GEMM_E4M3:
    case GEMM_E5M2: return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // raw bytes; the MMA knows the format
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  }
}

template <int OUT>
gemm_status_t launch_scale(void* C, int64_t ldc, int64_t M, int64_t N, float beta, const float* bias,
                           int bias_kind, int act, int num_sms, cudaStream_t stream) {
  const int64_t total = M * N;
  int64_t blocks = ceil_div(total, 256);
  if (blocks > int64_t(num_sms) * 8) blocks = int64_t(num_sms) * 8;
  scale_c_kernel<OUT><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      C, ldc, static_cast<int>(M), static_cast<int>(N), beta, bias, bias_kind, act);
  return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_status_t run_gemm(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                       const void* B, int64_t ldb, float beta, void* C, int64_t ldc, int in_dtype,
                       int out_dtype, int layout, void* stream_v, const gemm_config_t* cfg,
                       bool fixed_scratch = false, const float* bias = nullptr,
                       int bias_kind = GEMM_BIAS_NONE, int act = GEMM_ACT_NONE) {
  bool quick = false;
  gemm_status_t s = check_args(M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, layout, &quick);
  if (s != GEMM_OK) return s;
  if (bias_kind < GEMM_BIAS_NONE || bias_kind > GEMM_BIAS_ROW || act < GEMM_ACT_NONE ||
      act > GEMM_ACT_RELU)
    return GEMM_ERR_INVALID_ARG;
  if (bias_kind != GEMM_BIAS_NONE && !quick) {
    if (bias == nullptr) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(bias)) return GEMM_ERR_UNSUPPORTED;
  }
  if (quick) return GEMM_OK;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  const DeviceInfo* di = device_info(dev);
  if (!di || di->err != cudaSuccess) return GEMM_ERR_CUDA;
  if (di->cc_major != 10 || di->cc_minor != 3) return GEMM_ERR_ARCH;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

  if (K == 0) {
    switch (out_dtype) {
      case GEMM_F32:
        return launch_scale<OUT_F32>(C, ldc, M, N, beta, bias, bias_kind, act, di->num_sms, stream);
      case GEMM_BF16:
        return launch_scale<OUT_BF16>(C, ldc, M, N, beta, bias, bias_kind, act, di->num_sms, stream);
      default:
        return launch_scale<OUT_F16>(C, ldc, M, N, beta, bias, bias_kind, act, di->num_sms, stream);
    }
  }

  gemm_plan_t p;
  s = make_plan(M, N, K, in_dtype, out_dtype, layout, di->num_sms, cfg, &p);
  if (s != GEMM_OK) return s;

  OperandMaps mp;
  const bool a_col = (layout & GEMM_A_COL) != 0, b_col = (layout & GEMM_B_COL) != 0;
  const CUtensorMapDataType din = tma_dtype(in_dtype);
  const bool pair = p.cta_group == 2;
  const int ko = ko_for(p.bn, pair);
  const int b_cols = b_cols_per_cta(p.bn, pair);
  // A single row of tiles with M < BM (K-major A): copy only the first
  // ceil8(M) rows of A per k-block (a box of whole 8-row swizzle atoms); the
  // smem rows beyond feed only accumulator rows >= M, which are never stored.
  // Saves the zero-fill of the other rows, and TMA is slow on a box whose first
  // swizzle atom is only partly inside the tensor.
  const int a_box_rows = (!pair && !a_col && p.m_tiles == 1 && M < BM)
                             ? static_cast<int>((M + 7) / 8 * 8) : BM;
  const int isz = in_size(in_dtype), kbe = kblock_elems(in_dtype);   // MN-major: 16-bit only
  bool ok = a_col ? encode_2d(&mp.a, din, A, M, K, lda * isz, ATOM_MN, BK)
                  : encode_2d(&mp.a, din, A, K, M, lda * isz, kbe, a_box_rows);
  ok = ok && (b_col ? encode_2d(&mp.b, din, B, K, N, ldb * isz, kbe, b_cols)
                    : encode_2d(&mp.b, din, B, N, K, ldb * isz, ATOM_MN, BK));
  ok = ok && encode_2d(&mp.c, tma_dtype(out_dtype), C, N, M, ldc * out_size(out_dtype),
                       p.epi_chunk_cols, EPI_ROWS);
  if (!ok) return GEMM_ERR_CUDA;
  // 3-D maps over whole 64-element blocks: K-major (A row-major, B column-major)
  // -> blocks along K; MN-major (A column-major, B row-major) -> 64-wide atoms.
  const int64_t a_full = a_col ? M / ATOM_MN : K / kbe;
  const int64_t b_full = b_col ? K / kbe : N / ATOM_MN;
  int a_full3d = 0, b_full3d = 0;
  if (a_full > 0 && a_box_rows == BM &&
      (a_col ? encode_3d(&mp.a3, din, A, K, a_full, lda * isz, ko * BK, BM / ATOM_MN)
             : encode_3d(&mp.a3, din, A, M, a_full, lda * isz, BM, ko, kbe)))
    a_full3d = static_cast<int>(a_full);
  else
    mp.a3 = mp.a;
  if (b_full > 0 && (b_col ? encode_3d(&mp.b3, din, B, N, b_full, ldb * isz, b_cols, ko, kbe)
                           : encode_3d(&mp.b3, din, B, K, b_full, ldb * isz, ko * BK, b_cols / ATOM_MN)))
    b_full3d = static_cast<int>(b_full);
  else
    mp.b3 = mp.b;

  KernelArgs ka;
  std::memset(&ka, 0, sizeof(ka));
  ka.M = static_cast<int>(M);
  ka.N = static_cast<int>(N);
  ka.K = static_cast<int>(K);
  ka.m_tiles = p.m_tiles;
  ka.n_tiles = p.n_tiles;
  ka.k_blocks = p.k_blocks;
  ka.num_tiles = p.num_tiles;
  ka.group_m = p.group_m;
  ka.alpha = alpha;
  ka.beta = beta;
  // format code 1: bf16 (kind::f16) or E5M2 (kind::f8f6f4); 0: f16 or E4M3
  ka.idesc = make_idesc_f16((in_dtype == GEMM_BF16 || in_dtype == GEMM_E5M2) ? 1 : 0, p.a_mn,
                            p.b_mn, p.bm, p.bn);
  ka.kblock_elems = kblock_elems(in_dtype);
  ka.a_mn = p.a_mn;
  ka.b_mn = p.b_mn;
  ka.read_c = beta != 0.0f ? 1 : 0;
  ka.status = di->status;
  const uint64_t tmo = g_timeout_ns.load(std::memory_order_relaxed);
  ka.timeout_ns = tmo ? tmo : kDefaultTimeoutNs;
  ka.inject_skip = g_inject_skip.load(std::memory_order_relaxed);
  ka.c_ptr = C;
  ka.ldc = ldc;
  ka.n_ragged = ((N * out_size(out_dtype)) % 16) != 0 ? 1 : 0;
  // An operand every work unit re-reads (the single A panel when there is one
  // row of tiles, or the single B panel) is kept in L2; the other one streams.
  ka.a_hint = p.m_tiles == 1 && p.n_tiles > 1 ? 2 : (p.n_tiles == 1 && p.m_tiles > 1 ? 1 : 0);
  ka.b_hint = p.m_tiles == 1 && p.n_tiles > 1 ? 1 : (p.n_tiles == 1 && p.m_tiles > 1 ? 2 : 0);
  ka.a_full3d = a_full3d;
  ka.a_box_rows = a_box_rows;
  ka.b_full3d = b_full3d;
  ka.groups = p.groups;
  ka.dp_tiles = p.dp_tiles;
  ka.sk_iters = p.sk_iters;
  ka.fd_groups = make_fastdiv(static_cast<uint32_t>(p.groups));
  ka.tile_split = p.tile_split;
  ka.owner_groups = p.owner_groups;
  ka.bias = bias;
  ka.bias_kind = bias_kind;
  ka.act = act;
  ka.epi = (bias_kind != GEMM_BIAS_NONE || act != GEMM_ACT_NONE) ? 1 : 0;
  ka.tile_map = nullptr;
  {
    const int64_t groups_m = ceil_div(p.m_tiles, p.group_m);
    ka.fd_group = make_fastdiv(static_cast<uint32_t>(p.group_m) * static_cast<uint32_t>(p.n_tiles));
    ka.fd_rows = make_fastdiv(static_cast<uint32_t>(p.group_m));
    ka.fd_last_rows = make_fastdiv(static_cast<uint32_t>(p.m_tiles - (groups_m - 1) * p.group_m));
  }
  // beta * C goes into the accumulator ahead of the MMAs (persistent launches
  // with alpha == 1; a split-K cluster's CTAs each hold only part of the sum)
  ka.pre_c = (alpha == 1.0f && beta != 0.0f && p.split_k == 1) ? 1 : 0;
  if (p.order == GEMM_ORDER_HILBERT && !fixed_scratch) {   // the fixed-scratch path allocates nothing
    s = hilbert_map_for(dev, p.m_tiles, p.n_tiles, &ka.tile_map);
    if (s != GEMM_OK) return s;
  }
  if (p.sk_iters || p.tile_split) {
    s = fixed_scratch ? noalloc_scratch(dev, stream, size_t(BM) * p.bn * 4, p.grid, &ka.ws,
                                        &ka.ws_flags, &ka.epoch)
                      : scratch_for(dev, stream, size_t(BM) * p.bn * 4, p.grid, &ka.ws,
                                    &ka.ws_flags, &ka.epoch);
    if (s != GEMM_OK) return s;
  }

  // A call on the plain path takes the specialised instance of its
  // configuration and layout when there is one (cfg->general = 1 forbids it).
  const bool plain = !(cfg && cfg->general) && ka.inject_skip == 0 && ka.tile_map == nullptr;
  const bool sk = ka.sk_iters != 0 || ka.tile_split != 0, readc = ka.read_c != 0, epi = ka.epi != 0;
  const bool ragged = ka.n_ragged != 0;
  cudaError_t e = cudaErrorNotSupported;
  if (plain) {
    using SpecLaunch = cudaError_t (*)(int, bool, int, int, bool, bool, bool, bool,
                                       const OperandMaps&, const KernelArgs&, int, cudaStream_t, int);
    const bool f8 = is_fp8(in_dtype);
    const int set = spec_set(p.bn, pair, p.split_k, sk, readc, epi, ragged);
    const SpecLaunch launch =
        f8 ? (out_dtype == GEMM_F32    ? launch_gemm_f8_spec_f32
              : out_dtype == GEMM_BF16 ? launch_gemm_f8_spec_bf16
                                       : launch_gemm_f8_spec_f16)
        : set == 4 ? (out_dtype == GEMM_F32    ? launch_gemm_spec4_f32
                      : out_dtype == GEMM_BF16 ? launch_gemm_spec4_bf16
                                               : launch_gemm_spec4_f16)
        : set == 3 ? (out_dtype == GEMM_F32    ? launch_gemm_spec3_f32
                      : out_dtype == GEMM_BF16 ? launch_gemm_spec3_bf16
                                               : launch_gemm_spec3_f16)
        : set == 2 ? (out_dtype == GEMM_F32    ? launch_gemm_spec2_f32
                      : out_dtype == GEMM_BF16 ? launch_gemm_spec2_bf16
                                               : launch_gemm_spec2_f16)
                   : (out_dtype == GEMM_F32    ? launch_gemm_spec_f32
                      : out_dtype == GEMM_BF16 ? launch_gemm_spec_bf16
                                               : launch_gemm_spec_f16);
    e = launch(p.bn, pair, p.split_k, layout, sk, readc, epi, ragged, mp, ka, p.grid, stream, dev);
    if (e != cudaErrorNotSupported) return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  switch (out_dtype) {
    case GEMM_F32:
      e = is_fp8(in_dtype) ? launch_gemm_f8_f32(p.bn, pair, p.split_k, mp, ka, p.grid, stream, dev)
                           : launch_gemm_f32(p.bn, pair, p.split_k, mp, ka, p.grid, stream, dev);
      break;
    case GEMM_BF16:
      e = is_fp8(in_dtype) ? launch_gemm_f8_bf16(p.bn, pair, p.split_k, mp, ka, p.grid, stream, dev)
                           : launch_gemm_bf16(p.bn, pair, p.split_k, mp, ka, p.grid, stream, dev);
      break;
    default:
      e = is_fp8(in_dtype) ? launch_gemm_f8_f16(p.bn, pair, p.split_k, mp, ka, p.grid, stream, dev)
                           : launch_gemm_f16(p.bn, pair, p.split_k, mp, ka, p.grid, stream, dev);
      break;
  }
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Rows of C per panel of gemm_host's pipeline; M itself means one panel (the
// copies and the GEMM in sequence).  A problem that moves at least 64 MiB over
// the host link and has at least 2048 rows is cut into about 8 panels, each a
// multiple of 256 rows (the CTA pair's tile height), so that one panel's copies
// overlap the GEMMs of the panels before it and the copy-out of those after.
int64_t host_panel_rows(int64_t M, int64_t link_bytes) {
  if (link_bytes < (int64_t(64) << 20) || M < 2048) return M;
  const int64_t rows = ceil_div(ceil_div(M, 8), 256) * 256;
  return rows < M ? rows : M;
}

// One row panel [r0, r0 + rows) of a stored matrix (rows x cols elements of
// esz bytes in the caller's view, leading dimension ld) between host and
// device.  col_major: the matrix is stored column by column, so the panel is a
// band of every stored column.
cudaError_t copy_rows(void* dst, const void* src, int64_t ld, int64_t esz, int64_t r0, int64_t rows,
                      int64_t cols, bool col_major, cudaMemcpyKind kind, cudaStream_t st) {
  const size_t pitch = static_cast<size_t>(ld * esz);
  const int64_t off = col_major ? r0 * esz : r0 * ld * esz;
  char* d = static_cast<char*>(dst) + off;
  const char* h = static_cast<const char*>(src) + off;
  if (col_major)
    return cudaMemcpy2DAsync(d, pitch, h, pitch, static_cast<size_t>(rows * esz),
                             static_cast<size_t>(cols), kind, st);
  return cudaMemcpy2DAsync(d, pitch, h, pitch, static_cast<size_t>(cols * esz),
                           static_cast<size_t>(rows), kind, st);
}

}  // namespace

namespace gemm_tc {
int smem_alloc_bytes(int bn, bool pair) {
#define GEMM_SMEM(BN_, PAIR_) \
  SmemLayout<BN_, stages_for(BN_, PAIR_), PAIR_, ko_for(BN_, PAIR_)>::ALLOC
  if (pair) {
    switch (bn) {
      case 128: return GEMM_SMEM(128, true);
      case 256: return GEMM_SMEM(256, true);
      default: return 0;
    }
  }
  switch (bn) {
    case 64: return GEMM_SMEM(64, false);
    case 128: return GEMM_SMEM(128, false);
    case 256: return GEMM_SMEM(256, false);
    default: return 0;
  }
#undef GEMM_SMEM
}
}  // namespace gemm_tc

extern "C" {

gemm_status_t gemm(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                   const void* B, int64_t ldb, float beta, void* C, int64_t ldc, int in_dtype,
                   int out_dtype, int layout, void* stream) {
  return run_gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                  stream, nullptr);
}

gemm_status_t gemm_ex(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                      const void* B, int64_t ldb, float beta, void* C, int64_t ldc, int in_dtype,
                      int out_dtype, int layout, void* stream, const gemm_config_t* cfg) {
  return run_gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                  stream, cfg);
}

gemm_status_t gemm_bias_act(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                            int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                            int64_t ldc, int in_dtype, int out_dtype, int layout, const float* bias,
                            int bias_kind, int act, void* stream, const gemm_config_t* cfg) {
  return run_gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                  stream, cfg, /*fixed_scratch=*/false, bias, bias_kind, act);
}

gemm_status_t gemm_ex_noalloc(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                              int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                              int64_t ldc, int in_dtype, int out_dtype, int layout, void* stream,
                              const gemm_config_t* cfg) {
  return run_gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                  stream, cfg, /*fixed_scratch=*/true);
}

gemm_status_t gemm_host(int64_t M, int64_t N, int64_t K, float alpha, const void* hA, int64_t lda,
                        const void* hB, int64_t ldb, float beta, void* hC, int64_t ldc,
                        int in_dtype, int out_dtype, int layout, void* dA, void* dB, void* dC,
                        void* stream_v) {
  bool quick = false;
  gemm_status_t s =
      check_args(M, N, K, hA, lda, hB, ldb, hC, ldc, in_dtype, out_dtype, layout, &quick);
  if (s != GEMM_OK || quick) return s;
  s = check_args(M, N, K, dA, lda, dB, ldb, dC, ldc, in_dtype, out_dtype, layout, &quick);
  if (s != GEMM_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  const bool a_col = (layout & GEMM_A_COL) != 0, b_col = (layout & GEMM_B_COL) != 0;
  const int64_t osz = out_size(out_dtype), isz = in_size(in_dtype);
  const bool read_c = beta != 0.0f;
  // B's stored extent: K rows of N (row-major) or N rows of K (column-major)
  const int64_t b_rows = b_col ? N : K, b_cols = b_col ? K : N;
  const int64_t link = (K > 0 ? (M + N) * K * isz : 0) + M * N * osz * (read_c ? 2 : 1);
  const int64_t pr = K > 0 ? host_panel_rows(M, link) : M;
  if (pr >= M) {
    // one panel: copies in, GEMM, copy out, in order on the caller's stream
    if (K > 0 && (copy_rows(dA, hA, lda, isz, 0, M, K, a_col, cudaMemcpyHostToDevice, st) != cudaSuccess ||
                  cudaMemcpy2DAsync(dB, ldb * isz, hB, ldb * isz, b_cols * isz, b_rows,
                                    cudaMemcpyHostToDevice, st) != cudaSuccess))
      return GEMM_ERR_CUDA;
    if (read_c && copy_rows(dC, hC, ldc, osz, 0, M, N, false, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return GEMM_ERR_CUDA;
    s = run_gemm(M, N, K, alpha, dA, lda, dB, ldb, beta, dC, ldc, in_dtype, out_dtype, layout,
                 stream_v, nullptr);
    if (s != GEMM_OK) return s;
    if (copy_rows(hC, dC, ldc, osz, 0, M, N, false, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return GEMM_ERR_CUDA;
    return GEMM_OK;
  }
  // Row panels.  A copy-in stream carries B, then each panel's rows of A (and
  // of C when beta != 0); the caller's stream runs each panel's GEMM once its
  // rows are in; a copy-out stream returns each panel's rows of C once its GEMM
  // is done.  Events order the three; the caller's stream finally waits for the
  // copy-out stream, so synchronising it covers the whole call.  The internal
  // streams and events are released once their work completes.
  cudaStream_t s_in = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> evs;
  evs.reserve(static_cast<size_t>(2 * ceil_div(M, pr) + 3));
  auto mark = [&](cudaStream_t on, cudaStream_t waiter) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    evs.push_back(e);
    return cudaEventRecord(e, on) == cudaSuccess && cudaStreamWaitEvent(waiter, e, 0) == cudaSuccess;
  };
  bool ok = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) == cudaSuccess &&
            mark(st, s_in) &&   // after whatever the caller queued before
            cudaMemcpy2DAsync(dB, ldb * isz, hB, ldb * isz, b_cols * isz, b_rows,
                              cudaMemcpyHostToDevice, s_in) == cudaSuccess;
  gemm_status_t result = ok ? GEMM_OK : GEMM_ERR_CUDA;
  for (int64_t r0 = 0; ok && r0 < M; r0 += pr) {
    const int64_t rows = std::min(pr, M - r0);
    ok = copy_rows(dA, hA, lda, isz, r0, rows, K, a_col, cudaMemcpyHostToDevice, s_in) == cudaSuccess &&
         (!read_c || copy_rows(dC, hC, ldc, osz, r0, rows, N, false, cudaMemcpyHostToDevice, s_in) ==
                         cudaSuccess) &&
         mark(s_in, st);
    if (!ok) {
      result = GEMM_ERR_CUDA;
      break;
    }
    const void* a_panel = static_cast<const char*>(dA) + (a_col ? r0 * isz : r0 * lda * isz);
    void* c_panel = static_cast<char*>(dC) + r0 * ldc * osz;
    result = run_gemm(rows, N, K, alpha, a_panel, lda, dB, ldb, beta, c_panel, ldc, in_dtype,
                      out_dtype, layout, stream_v, nullptr);
    ok = result == GEMM_OK && mark(st, s_out) &&
         copy_rows(hC, dC, ldc, osz, r0, rows, N, false, cudaMemcpyDeviceToHost, s_out) == cudaSuccess;
    if (!ok && result == GEMM_OK) result = GEMM_ERR_CUDA;
  }
  // the caller's stream waits for both internal streams, also after a failure
  // (work already queued on them still touches the caller's buffers)
  if (s_in && !mark(s_in, st) && result == GEMM_OK) result = GEMM_ERR_CUDA;
  if (s_out && !mark(s_out, st) && result == GEMM_OK) result = GEMM_ERR_CUDA;
  for (cudaEvent_t e : evs) cudaEventDestroy(e);
  if (s_in) cudaStreamDestroy(s_in);
  if (s_out) cudaStreamDestroy(s_out);
  return result;
}

const char* gemm_status_string(gemm_status_t status) {
  switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported argument (dtype, alignment or stride)";
    case GEMM_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case GEMM_ERR_CUDA: return "CUDA runtime or driver error";
    case GEMM_ERR_TIMEOUT: return "a kernel wait timed out";
    case GEMM_ERR_SCRATCH:
      return "the launch needs more stream-K scratch than gemm_ex_noalloc's fixed buffer holds";
    default: return "unknown status";
  }
}

gemm_status_t gemm_sync_status(void* stream, int* site) {
  if (site) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_status_word, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
  if (v == 0) return GEMM_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_gemm_status_word, &zero, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
  if (site) *site = v;
  return GEMM_ERR_TIMEOUT;
}

void gemm_debug_set(uint64_t wait_timeout_ns, int32_t inject_skip) {
  g_timeout_ns.store(wait_timeout_ns, std::memory_order_relaxed);
  g_inject_skip.store(inject_skip > 0 ? inject_skip : 0, std::memory_order_relaxed);
}

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int layout,
                        int32_t num_sms, const gemm_config_t* cfg, gemm_plan_t* plan) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  bool quick = false;
  gemm_status_t s = check_shape(M, N, K, in_dtype, out_dtype, layout, &quick);
  if (s != GEMM_OK) return s;
  return make_plan(M, N, K, in_dtype, out_dtype, layout, num_sms, cfg, plan);
}

void gemm_tile_coord(int32_t t, int32_t m_tiles, int32_t n_tiles, int32_t group_m, int32_t* m_blk,
                     int32_t* n_blk) {
  int m = 0, n = 0;
  tile_coord(t, m_tiles, n_tiles, group_m, &m, &n);
  *m_blk = m;
  *n_blk = n;
}

int32_t gemm_tile_order(int order, int32_t m_tiles, int32_t n_tiles, int32_t group_m,
                        int32_t* m_blk, int32_t* n_blk, int32_t max_tiles) {
  if (m_tiles <= 0 || n_tiles <= 0 || !m_blk || !n_blk || max_tiles < 0) return -1;
  const int64_t tiles = int64_t(m_tiles) * n_tiles;
  if (order == GEMM_ORDER_GROUPED) {
    if (group_m <= 0 || tiles >= (int64_t(1) << 31)) return -1;
    // the device's walk: the divisions by the group size and row counts done by
    // fastdiv (a group_m above m_tiles orders the tiles as m_tiles does)
    const int gmc = std::min(group_m, m_tiles);
    const FastDiv gs = make_fastdiv(static_cast<uint32_t>(gmc) * static_cast<uint32_t>(n_tiles));
    const FastDiv gm = make_fastdiv(static_cast<uint32_t>(gmc));
    const FastDiv gl = make_fastdiv(static_cast<uint32_t>(m_tiles - (ceil_div(m_tiles, gmc) - 1) * gmc));
    for (int64_t t = 0; t < tiles && t < max_tiles; ++t) {
      int m = 0, n = 0;
      tile_coord_fast(static_cast<int>(t), m_tiles, gmc, gs, gm, gl, &m, &n);
      m_blk[t] = m;
      n_blk[t] = n;
    }
    return static_cast<int32_t>(tiles);
  }
  if (order == GEMM_ORDER_HILBERT) {
    std::vector<int2> v;
    if (!hilbert_tiles(m_tiles, n_tiles, &v)) return -1;
    for (size_t t = 0; t < v.size() && t < static_cast<size_t>(max_tiles); ++t) {
      m_blk[t] = v[t].x;
      n_blk[t] = v[t].y;
    }
    return static_cast<int32_t>(v.size());
  }
  return -1;
}

int32_t gemm_work_items(int32_t unit, int32_t units, int32_t dp_tiles, int64_t sk_iters,
                        int32_t groups, int32_t* items, int32_t max_items) {
  if (unit < 0 || units <= 0 || unit >= units || groups <= 0 || dp_tiles < 0 || sk_iters < 0)
    return 0;
  if (sk_iters >= (int64_t(1) << 31)) return 0;
  WorkIter wi;
  wi.init(unit, units, dp_tiles, sk_iters, groups, make_fastdiv(static_cast<uint32_t>(groups)));
  WorkItem w;
  int32_t n = 0;
  while (wi.next(&w)) {
    if (items && n < max_items) {
      items[3 * n] = w.tile;
      items[3 * n + 1] = w.g0;
      items[3 * n + 2] = w.g1;
    }
    ++n;
  }
  return n;
}

int32_t gemm_split_tile_item(int32_t unit, int32_t tile_split, int32_t owner_groups,
                             int32_t groups, int32_t* item) {
  if (unit < 0 || tile_split < 2 || groups < tile_split || owner_groups < 1 ||
      groups - owner_groups < tile_split - 1 || item == nullptr)
    return 0;
  WorkIter wi;
  wi.init(unit, 1, 0, 0, groups, make_fastdiv(static_cast<uint32_t>(groups)), tile_split, owner_groups);
  WorkItem w;
  if (!wi.next(&w)) return 0;
  item[0] = w.tile;
  item[1] = w.g0;
  item[2] = w.g1;
  int32_t n = 1;
  while (wi.next(&w)) ++n;
  return n;
}

uint32_t gemm_fastdiv(uint32_t n, uint32_t d) {
  if (d == 0 || d >= (1u << 31) || n >= (1u << 31)) return 0xFFFFFFFFu;
  const FastDiv f = make_fastdiv(d);
  return fastdiv(n, f.mul, f.shift);
}

uint32_t gemm_encode_idesc(int in_dtype, int a_mn, int b_mn, int m, int n) {
  return make_idesc_f16(in_dtype == GEMM_BF16 ? 1 : 0, a_mn, b_mn, m, n);
}

uint64_t gemm_encode_sdesc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return make_sdesc_sw128(smem_addr, lbo_bytes, sbo_bytes);
}

int32_t gemm_version(void) { return 100; }

}  // extern "C"
