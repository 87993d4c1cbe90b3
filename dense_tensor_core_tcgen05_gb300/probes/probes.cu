// Hardware probes behind the GEMM's design choices (measurement only; not on the
// GEMM path):
//  * mma_rate: back-to-back tcgen05.mma (kind::f16, K = 16) from one thread per CTA
//    (or per CTA pair), timed with clock64 -> cycles per instruction and dense
//    FLOP/clk/SM for a given N.  The tensor-core peak used by the roofline is this
//    rate times the SM count times the clock (the Ada GEMM page's advice to measure
//    FLOP/clk/SM with an in-kernel clock and convert with the clock seen under load).
//  * tma_stream: one producer thread per CTA streams a K-major [N, K] bf16 matrix
//    through a ring of TMA tile copies of `R` rows x `KO` consecutive 64-element
//    blocks (a 3-D map whose third dimension walks blocks along the row) -> the DRAM
//    bandwidth a tile-copy access pattern reaches.  Grouped mode: a 4-D map
//    (64 elements, 8 rows, KO blocks, row groups) fetches the KO blocks of each
//    group of 8 rows back to back, landing as the same 128B-swizzled K-major tile
//    with 8-row atoms KO * 1024 B apart.  The L2 promotion of the map is a knob.
//    Variant bits: 1 waits through a shared helper, 2 keeps the slot, k-group and
//    row-block indices incrementally (the default divides by run-time values, which
//    costs the single issuing thread ~0.3 us per copy and bounds the copy rate), 4
//    runs the problem through the intake kernel instead; variant >> 8 adds KB of
//    unused dynamic shared memory.
//  * store_rate: every CTA writes a 128 x 256 fp32 block of C (the share of one CTA
//    of a 256 x 256 pair tile) from registers, by one of five routes: tensor stores
//    of 32 x 32 chunks through two staging buffers per warp (the GEMM epilogue),
//    the same with a buffer per chunk, plain 16-byte global stores by row,
//    coalesced 16-byte global stores through the swizzled staging buffer, or one
//    3-D tensor store of the warp's whole 32 x 256 block -> the time the output
//    of a one-wave GEMM takes to leave the SMs.
//  * intake: an SM taking in L2-resident data by TMA copies (one thread, a ring of
//    128-row x 2-block copies) and, at the same time, by cp.async 16-byte copies
//    from up to 4 other warps -> whether a second load path adds to what TMA
//    alone brings into an SM.
// Every wait is bounded (1-2 s, %globaltimer); a CTA that gives up writes ~0.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_common.h"
#include "ptx.cuh"

using namespace gemm_tc;

namespace {

template <int N, bool PAIR>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 64 * 1024);
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + 64 * 1024 + 64);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  // operands: 64 KB of finite bf16 values (the contents do not matter for timing)
  for (int i = threadIdx.x; i < 16 * 1024; i += blockDim.x) reinterpret_cast<uint32_t*>(smem)[i] = 0x3f803f80u;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    if (PAIR) {
      tmem_alloc_pair(slot, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(slot, 512);
      tmem_relinquish();
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  if (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (warp == 0 && lane == 0 && rank == 0) {
    const uint32_t idesc = make_idesc_f16(1, 0, 0, PAIR ? 256 : 128, N);
    const uint64_t da = make_sdesc_sw128(smem_u32(smem), 16, 1024);
    const uint64_t db = make_sdesc_sw128(smem_u32(smem + 32 * 1024), 16, 1024);
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (PAIR) umma_f16_pair(tmem, da + 2 * kk, db + 2 * kk, idesc, 1);
        else umma_f16(tmem, da + 2 * kk, db + 2 * kk, idesc, 1);
      }
    }
    if (PAIR) umma_commit_pair_multicast(bar, 0x1); else umma_commit(bar);
    const uint64_t g0 = globaltimer_ns();
    bool done = false;
    while (!(done = mbar_try_wait(bar, 0)) && globaltimer_ns() - g0 < 2000000000ull) {
    }
    out[blockIdx.x] = done ? static_cast<unsigned long long>(clock64() - t0) : ~0ull;
  }
  tc_fence_before();
  if (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    if (PAIR) tmem_dealloc_pair(tmem, 512); else tmem_dealloc(tmem, 512);
  }
}

__device__ bool probe_wait_fn(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait<false>(bar, parity))
    if (globaltimer_ns() - t0 > 1000000000ull) return false;
  return true;
}

__global__ void __launch_bounds__(160, 1)
    tma_stream_kernel(const __grid_constant__ CUtensorMap tm, int rows_per_cta, int R, int KO, int S,
                      int K, int grouped, int reps, int variant, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int box_bytes = R * 128 * KO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * box_bytes);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const int row0 = blockIdx.x * rows_per_cta;
  const int kgroups = K / (64 * KO), rblocks = rows_per_cta / R, pass = kgroups * rblocks;
  const int total = pass * reps;
  int ns = 0, nkg = 0, nrb = 0, ws = 0;   // next slot, k-group, row block; slot waited for next
  uint32_t wph = 0;                        // its phase parity
  const uint64_t t0 = globaltimer_ns();
  for (int i = 0; i < total + S; ++i) {
    if (i >= S && (variant & 2)) {   // the wait with incremental slot and parity
      if (!probe_wait_fn(&bars[ws], wph)) {
        const uint64_t g1 = globaltimer_ns();
        while (globaltimer_ns() - g1 < 1000000ull) {
        }
        out[blockIdx.x] = ~0ull;
        return;
      }
      if (++ws == S) {
        ws = 0;
        wph ^= 1;
      }
    } else if (i >= S && (variant & 1)) {   // the same wait through the shared helper
      const int j = i - S;
      if (!probe_wait_fn(&bars[j % S], (j / S) & 1)) {
        const uint64_t g1 = globaltimer_ns();
        while (globaltimer_ns() - g1 < 1000000ull) {
        }
        out[blockIdx.x] = ~0ull;
        return;
      }
    } else if (i >= S) {   // the copy issued S iterations ago must have landed before its slot is reused
      const int j = i - S, s = j % S;
      const uint64_t g0 = globaltimer_ns();
      while (!mbar_try_wait(&bars[s], (j / S) & 1)) {
        if (globaltimer_ns() - g0 > 1000000000ull) {
          // give the copies still in flight a bounded moment to land, then report failure
          const uint64_t g1 = globaltimer_ns();
          while (globaltimer_ns() - g1 < 1000000ull) {
          }
          out[blockIdx.x] = ~0ull;
          return;
        }
      }
    }
    if (i < total) {
      int s, kg, rb;
      if (variant & 2) {   // indices kept incrementally (no division by run-time values)
        s = ns;
        kg = nkg;
        rb = nrb;
        if (++ns == S) ns = 0;
        if (++nkg == kgroups) {
          nkg = 0;
          if (++nrb == rblocks) nrb = 0;
        }
      } else {
        s = i % S;
        kg = i % kgroups;
        rb = (i % pass) / kgroups;
      }
      mbar_arrive_expect_tx(&bars[s], box_bytes);
      if (grouped)
        tma_load_4d(smem + s * box_bytes, &tm, 0, 0, kg * KO, (row0 + rb * R) / 8, &bars[s]);
      else
        tma_load_3d(smem + s * box_bytes, &tm, 0, row0 + rb * R, kg * KO, &bars[s]);
    }
  }
  out[blockIdx.x] = globaltimer_ns() - t0;
}

// Bounded wait for a phase (1 s); false if it gave up.
template <bool CLUSTER>
__device__ bool probe_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait<CLUSTER>(bar, parity))
    if (globaltimer_ns() - t0 > 1000000000ull) return false;
  return true;
}

// Multicast streaming: clusters of C CTAs share every copy of R rows x KO
// blocks; cluster rank k issues rows [k R/C, (k+1) R/C) of it, multicast to all
// C CTAs, so each CTA receives whole boxes while issuing 1/C of them.  A slot is
// refilled only after every CTA of the cluster has seen it full (empty[s],
// C arrivals).  Thread 0 issues, thread 32 consumes; every thread meets at the
// final cluster barrier, so no CTA exits while a peer may still write into it.
// A producer that gives up stops issuing; the consumers then give up too.
__global__ void __launch_bounds__(64, 1)
    tma_mcast_kernel(const __grid_constant__ CUtensorMap tm, int rows_per_cluster, int R, int KO,
                     int S, int K, int C, int reps, int batched, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int box_bytes = R * 128 * KO;
  const int piece_rows = R / C;
  const int piece_bytes = piece_rows * 128 * KO;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * box_bytes);
  uint64_t* empty = full + S;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C);
    }
    fence_barrier_init();
  }
  cluster_sync();
  const int cluster = blockIdx.x / C;
  const int kgroups = K / (64 * KO), rblocks = rows_per_cluster / R, pass = kgroups * rblocks;
  const int total = pass * reps;
  if (batched) {
    // batches of S copies into distinct slots, the cluster meeting at a
    // barrier between batches (no per-slot hand-off)
    const uint16_t mask = static_cast<uint16_t>((1u << C) - 1);
    const int batches = total / S;
    bool failed = false;
    const uint64_t t0 = globaltimer_ns();
    for (int b = 0; b < batches; ++b) {
      if (threadIdx.x == 0 && !failed) {
        for (int s = 0; s < S; ++s) {
          const int i = b * S + s;
          mbar_arrive_expect_tx(&full[s], box_bytes);
          const int kg = i % kgroups, rb = (i % pass) / kgroups;
          tma_load_3d_mcast(smem + s * box_bytes + rank * piece_bytes, &tm, 0,
                            cluster * rows_per_cluster + rb * R + static_cast<int>(rank) * piece_rows,
                            kg * KO, &full[s], mask);
        }
        for (int s = 0; s < S && !failed; ++s)
          if (!probe_wait<true>(&full[s], b & 1)) failed = true;
      }
      __syncthreads();
      cluster_sync();
    }
    if (threadIdx.x == 0) {
      if (failed) {
        const uint64_t g1 = globaltimer_ns();
        while (globaltimer_ns() - g1 < 1000000ull) {
        }
      }
      out[blockIdx.x] = failed ? ~0ull : globaltimer_ns() - t0;
    }
  } else if (threadIdx.x == 0) {
    // producer: refill slot s once every CTA of the cluster has consumed it
    const uint16_t mask = static_cast<uint16_t>((1u << C) - 1);
    for (int i = 0; i < total; ++i) {
      const int s = i % S;
      if (i >= S && !probe_wait<true>(&empty[s], ((i / S) - 1) & 1)) break;
      mbar_arrive_expect_tx(&full[s], box_bytes);
      const int kg = i % kgroups, rb = (i % pass) / kgroups;
      tma_load_3d_mcast(smem + s * box_bytes + rank * piece_bytes, &tm, 0,
                        cluster * rows_per_cluster + rb * R + static_cast<int>(rank) * piece_rows,
                        kg * KO, &full[s], mask);
    }
  } else if (threadIdx.x == 32) {
    // consumer: every copy that lands here releases its slot in all C CTAs
    bool failed = false;
    const uint64_t t0 = globaltimer_ns();
    for (int j = 0; j < total; ++j) {
      const int s = j % S;
      if (!probe_wait<false>(&full[s], (j / S) & 1)) {
        failed = true;
        break;
      }
      for (int q = 0; q < C; ++q) mbar_arrive_cluster(map_to_rank(&empty[s], q));
    }
    if (failed) {
      // let copies already in flight land before the CTA can exit
      const uint64_t g1 = globaltimer_ns();
      while (globaltimer_ns() - g1 < 1000000ull) {
      }
      out[blockIdx.x] = ~0ull;
    } else {
      out[blockIdx.x] = globaltimer_ns() - t0;
    }
  }
  __syncthreads();
  cluster_sync();
}


// ------------------------------------------------------------------- intake
constexpr int CP_BUFS = 6;   // 4 KB cp.async buffers per warp (CP_BUFS - 1 rounds in flight)

// Warp 0, lane 0: `tma_copies` copies of 128 rows x 2 blocks from rows
// [128 g, 128 g + 128) of A ([rows, cols] bf16, L2-resident), g = b / share
// (`share` consecutive CTAs read the same rows), walking the row's columns
// cyclically, through S = 3 slots.  Warps 1..W: each re-reads its own 24 KB
// slice of P `cp_iters` times 4 KB with cp.async.cg (16 B per lane and copy),
// or with cp_iters < 0 reads its 24 KB of shared memory -cp_iters times 4 KB.
// out[8 b] = TMA ns, out[8 b + w] = warp w's ns (~0 if the TMA thread gave up).
__global__ void __launch_bounds__(160, 1)
    intake_kernel(const __grid_constant__ CUtensorMap tm, int cols, int share, const uint8_t* P, int W,
                  int tma_copies, int cp_iters, int bars_after_ring, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  constexpr int S = 3, BOX = 128 * 128 * 2;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * BOX + (bars_after_ring ? 0 : 4 * CP_BUFS * 4096));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    if (lane != 0 || tma_copies == 0) return;
    const int groups = cols / 128;   // copies per pass over the row's columns
    const int y = (static_cast<int>(blockIdx.x) / share) * 128;
    const uint64_t t0 = globaltimer_ns();
    for (int i = 0; i < tma_copies + S; ++i) {
      if (i >= S) {
        const int j = i - S;
        if (!probe_wait<false>(&bars[j % S], (j / S) & 1)) {
          const uint64_t g1 = globaltimer_ns();
          while (globaltimer_ns() - g1 < 1000000ull) {
          }
          out[8 * blockIdx.x] = ~0ull;
          return;
        }
      }
      if (i < tma_copies) {
        const int s = i % S;
        mbar_arrive_expect_tx(&bars[s], BOX);
        tma_load_3d(smem + s * BOX, &tm, 0, y, (i % groups) * 2, &bars[s]);
      }
    }
    out[8 * blockIdx.x] = globaltimer_ns() - t0;
    return;
  }
  if (warp > W) return;
  const uint8_t* src = P + (static_cast<size_t>(blockIdx.x) * 4 + (warp - 1)) * (CP_BUFS * 4096);
  const uint32_t dst = smem_u32(smem + S * BOX + (warp - 1) * CP_BUFS * 4096);
  const uint64_t t0 = globaltimer_ns();
  if (cp_iters < 0) {
    // shared-memory reads only: 16 bytes per lane and load over the warp's
    // 24 KB, -cp_iters passes of 4 KB; the sum keeps the loads alive
    uint32_t acc = 0;
    for (int it = 0; it < -cp_iters; ++it) {
      const int b = it % CP_BUFS;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 q = ld_shared_v4(dst + b * 4096 + (j * 32 + lane) * 16);
        acc += q.x ^ q.y ^ q.z ^ q.w;
      }
    }
    __syncwarp();
    if (lane == 0) out[8 * blockIdx.x + warp] = (globaltimer_ns() - t0) | (acc == 0x9e3779b9u ? 1ull : 0ull);
    return;
  }
  for (int it = 0; it < cp_iters; ++it) {
    const int b = it % CP_BUFS;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int off = b * 4096 + (j * 32 + lane) * 16;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + off), "l"(src + off) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(CP_BUFS - 1) : "memory");
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncwarp();
  if (lane == 0) out[8 * blockIdx.x + warp] = globaltimer_ns() - t0;
}

template <int N, bool PAIR>
int launch_mma(int grid, int iters, unsigned long long* dout) {
  auto k = mma_rate_kernel<N, PAIR>;
  const int smem = 64 * 1024 + 2048;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&cfg, k, iters, dout) != cudaSuccess) return -2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}


// ---------------------------------------------------------------- store_rate
__device__ __forceinline__ void tma_store_3d_probe(const CUtensorMap* m, const void* src, int32_t x,
                                                   int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void st_global_v4_probe(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// 4 warps; warp w writes rows [32 w, 32 w + 32) of the CTA's 128 x 256 block,
// as 8 chunks of 32 columns.  Element (r, c) of C holds 0.5 r + c.  out[5 b] =
// start, out[5 b + 1 + w] = the time warp w's writes were complete.
__global__ void __launch_bounds__(128, 1)
    store_rate_kernel(const __grid_constant__ CUtensorMap tm2, const __grid_constant__ CUtensorMap tm3,
                      float* C, int ldc, int grid_n, int mode, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row0 = (blockIdx.x / grid_n) * 128 + warp * 32;
  const int col0 = (blockIdx.x % grid_n) * 256;
  uint8_t* wbuf = smem + warp * 32768;
  __syncthreads();
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.5f * static_cast<float>(row0 + lane) + static_cast<float>(col0 + c * 32 + i);
    if (mode == 2) {
      float* dst = C + static_cast<size_t>(row0 + lane) * ldc + col0 + c * 32;
#pragma unroll
      for (int j = 0; j < 8; ++j) st_global_v4_probe(dst + 4 * j, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      continue;
    }
    uint8_t* buf = wbuf + (mode == 0 ? (c & 1) : c) * 4096;
    if (mode == 0) {
      if (lane == 0) bulk_wait_group_read<1>();
      __syncwarp();
    }
    const uint32_t rowp = smem_u32(buf) + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a = rowp + ((j ^ (lane & 7)) << 4);
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v[4 * j]), "f"(v[4 * j + 1]),
                   "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                   : "memory");
    }
    if (mode == 3) {
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = i * 4 + (lane >> 3), piece = lane & 7;
        const uint4 q = ld_shared_v4(smem_u32(buf) + r * 128 + ((piece ^ (r & 7)) << 4));
        st_global_v4_probe(C + static_cast<size_t>(row0 + r) * ldc + col0 + c * 32 + piece * 4,
                           __uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z),
                           __uint_as_float(q.w));
      }
      __syncwarp();
      continue;
    }
    if (mode == 4) continue;   // stored at once after the loop
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&tm2, buf, col0 + c * 32, row0);
      bulk_commit_group();
    }
  }
  if (mode == 4) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d_probe(&tm3, wbuf, 0, row0, col0 / 32);
      bulk_commit_group();
    }
  }
  if (mode == 2 || mode == 3) {
    __threadfence();
  } else if (lane == 0) {
    bulk_wait_group<0>();
  }
  __syncwarp();
  const uint64_t t1 = globaltimer_ns();
  if (lane == 0) {
    if (warp == 0) out[5 * blockIdx.x] = t0;
    out[5 * blockIdx.x + 1 + warp] = t1;
  }
}

}  // namespace

// Cycles for `iters` x 4 back-to-back MMAs (M = 128, or 256 over a pair; K = 16;
// the given N) per issuing CTA, written to dout[blockIdx.x] (~0 if a wait gave up).
// grid must be even when pair != 0.  Returns 0 or a negative error.
extern "C" int probe_mma_rate(int n, int pair, int grid, int iters, unsigned long long* dout) {
  if (grid <= 0 || iters <= 0 || (pair && (grid & 1))) return -10;
#define GEMM_PROBE_CASE(NN, PP) \
  if (n == NN && pair == PP) return launch_mma<NN, PP>(grid, iters, dout);
  GEMM_PROBE_CASE(64, 0) GEMM_PROBE_CASE(128, 0) GEMM_PROBE_CASE(256, 0)
  GEMM_PROBE_CASE(128, 1) GEMM_PROBE_CASE(256, 1)
#undef GEMM_PROBE_CASE
  return -11;
}

// Nanoseconds per CTA to stream B ([N, K] bf16, row pitch K, 16-byte aligned) with
// copies of R rows x KO blocks of 64 elements, S copies in flight per CTA, grid
// CTAs each owning N / grid rows.  grouped: 4-D map in 8-row groups (see top);
// promo: L2 promotion 0 none, 1 64 B, 2 128 B, 3 256 B; reps: passes over the
// CTA's rows (reps > 1 on a matrix that fits in L2 measures L2 -> shared).  Requires
// K % (64 * KO) == 0, (N / grid) % R == 0, R % 8 == 0, R <= 256, the ring within
// 227 KB.  Returns 0 or a negative error.
extern "C" int probe_tma_stream(const void* B, int N, int K, int grid, int R, int KO, int S,
                                int grouped, int promo, int reps, int variant, int threads,
                                unsigned long long* dout) {
  if (threads != 64 && threads != 160) return -10;
  if (grid <= 0 || N % grid || (N / grid) % R || R > 256 || R % 8 || KO < 1 || K % (64 * KO) ||
      S < 1 || promo < 0 || promo > 3 || N % 8 || reps < 1)
    return -10;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return -1;
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  CUtensorMap tm;
  const CUtensorMapL2promotion pr[4] = {CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B};
  const cuuint64_t ld = static_cast<cuuint64_t>(K) * 2;
  cuuint64_t dims3[3] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / 64)};
  cuuint64_t strides3[2] = {ld, 128};
  cuuint32_t box3[3] = {64, static_cast<cuuint32_t>(R), static_cast<cuuint32_t>(KO)};
  cuuint64_t dims4[4] = {64, 8, static_cast<cuuint64_t>(K / 64), static_cast<cuuint64_t>(N / 8)};
  cuuint64_t strides4[3] = {ld, 128, 8 * ld};
  cuuint32_t box4[4] = {64, 8, static_cast<cuuint32_t>(KO), static_cast<cuuint32_t>(R / 8)};
  cuuint32_t es[4] = {1, 1, 1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, grouped ? 4 : 3, const_cast<void*>(B),
          grouped ? dims4 : dims3, grouped ? strides4 : strides3, grouped ? box4 : box3, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, pr[promo],
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -2;
  // variant >> 8: extra KB of dynamic shared memory (unused; sizes the carveout)
  const int smem = S * R * 128 * KO + 1024 + 8 * S + 64 + (variant >> 8) * 1024;
  if (smem > 232448) return -12;
  if (cudaFuncSetAttribute(tma_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -3;
  if (variant & 4) {
    // this map and problem through the intake kernel (R = 128, KO = 2, S = 3 only)
    if (R != 128 || KO != 2 || S != 3 || grouped || N / grid != 128) return -13;
    const int ismem = 3 * 32768 + 4 * CP_BUFS * 4096 + 1024 + 64;
    if (cudaFuncSetAttribute(intake_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ismem) !=
        cudaSuccess)
      return -3;
    intake_kernel<<<grid, 160, ismem>>>(tm, K, 1, nullptr, 0, reps * (K / 128), 0, 0, dout);
  } else {
    tma_stream_kernel<<<grid, threads, smem>>>(tm, N / grid, R, KO, S, K, grouped, reps, variant, dout);
  }
  if (cudaGetLastError() != cudaSuccess) return -4;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -5;
}

// Nanoseconds per CTA to receive `reps` passes over its cluster's rows of B
// ([N, K] bf16) as copies of R rows x KO blocks, each issued in C pieces by the
// C CTAs of a cluster and multicast to all of them (C = 1: no multicast), S
// copies in flight.  Requires grid % C == 0, N % (grid / C) == 0, the cluster's
// rows a multiple of R, R % (8 C) == 0, K % (64 KO) == 0, C in {1, 2, 4}.
// batched: S copies at a time into distinct slots, a cluster barrier between
// batches, instead of per-slot release (reps * passes must be a multiple of S).
extern "C" int probe_tma_mcast(const void* B, int N, int K, int grid, int R, int KO, int S, int C,
                               int reps, int batched, unsigned long long* dout) {
  if (C != 1 && C != 2 && C != 4) return -10;
  if (grid <= 0 || grid % C || N % (grid / C) || (N / (grid / C)) % R || R % (8 * C) ||
      R / C > 256 || KO < 1 || K % (64 * KO) || S < 1 || reps < 1)
    return -10;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return -1;
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  CUtensorMap tm;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(R / C), static_cast<cuuint32_t>(KO)};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(B), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -2;
  const int smem = S * R * 128 * KO + 1024 + 16 * S + 64;
  if (smem > 232448) return -12;
  if (cudaFuncSetAttribute(tma_mcast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -3;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(64);
  cfg.dynamicSmemBytes = smem;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tma_mcast_kernel, tm, N / (grid / C), R, KO, S, K, C, reps, batched,
                         dout) !=
      cudaSuccess)
    return -4;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -5;
}

// Start and per-warp completion times (globaltimer ns, 5 per CTA) of store_rate:
// grid_m x grid_n CTAs each writing a 128 x 256 fp32 block of C ([M, N] row
// major, ldc elements, base 16-byte aligned) by route `mode` (0..4, see top).
// Requires grid_m * 128 <= M, grid_n * 256 <= N, ldc % 4 == 0.  Returns 0 or a
// negative error.
extern "C" int probe_store_rate(float* C, int M, int N, int ldc, int grid_m, int grid_n, int mode,
                                unsigned long long* dout) {
  if (mode < 0 || mode > 4 || grid_m < 1 || grid_n < 1 || grid_m * 128 > M || grid_n * 256 > N ||
      ldc < N || ldc % 4 || (reinterpret_cast<uintptr_t>(C) & 15))
    return -10;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return -1;
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  CUtensorMap tm2, tm3;
  cuuint64_t dims2[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides2[1] = {static_cast<cuuint64_t>(ldc) * 4};
  cuuint32_t box2[2] = {32, 32};
  cuuint64_t dims3[3] = {32, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(N / 32)};
  cuuint64_t strides3[2] = {static_cast<cuuint64_t>(ldc) * 4, 128};
  cuuint32_t box3[3] = {32, 32, 8};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(&tm2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims2, strides2, box2, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -2;
  if (enc(&tm3, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, C, dims3, strides3, box3, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -2;
  const int smem = 4 * 32768 + 1024;
  if (cudaFuncSetAttribute(store_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -3;
  store_rate_kernel<<<grid_m * grid_n, 128, smem>>>(tm2, tm3, C, ldc, grid_n, mode, dout);
  if (cudaGetLastError() != cudaSuccess) return -4;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -5;
}

// Per-CTA nanoseconds of intake_kernel (8 per CTA: TMA, then cp.async warps
// 1..W): grid CTAs; A [rows, cols] bf16 with cols % 128 == 0 and
// rows >= 128 * ceil(grid / share); P at least grid * 4 * 24 KB, 16-byte
// aligned.  tma_copies = 0 turns the TMA stream off, W = 0 the cp.async warps.
// Returns 0 or a negative error.
extern "C" int probe_intake(const void* A, int rows, int cols, int share, const void* P,
                            long long p_bytes, int grid, int W, int tma_copies, int cp_iters,
                            int bars_after_ring, unsigned long long* dout) {
  // barriers right after the TMA ring overlap the cp.async buffers
  if (W > 0 && bars_after_ring) return -10;
  if (grid < 1 || share < 1 || cols < 128 || cols % 128 || rows < 128 * ((grid + share - 1) / share) ||
      W < 0 || W > 4 || tma_copies < 0 ||
      p_bytes < static_cast<long long>(grid) * 4 * CP_BUFS * 4096 || (reinterpret_cast<uintptr_t>(P) & 15))
    return -10;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return -1;
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  CUtensorMap tm;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
  cuuint32_t box[3] = {64, 128, 2};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(A), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -2;
  const int smem = 3 * 32768 + 4 * CP_BUFS * 4096 + 1024 + 64;
  if (cudaFuncSetAttribute(intake_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -3;
  if (bars_after_ring == 2) {
    // this map and problem through the streaming kernel (S = 3, one row block)
    if (share != 1 || W != 0 || tma_copies % (cols / 128)) return -13;
    const int ssmem = 3 * 32768 + 1024 + 24 + 64;
    if (cudaFuncSetAttribute(tma_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ssmem) !=
        cudaSuccess)
      return -3;
    tma_stream_kernel<<<grid, 64, ssmem>>>(tm, 128, 128, 2, 3, cols, 0, tma_copies / (cols / 128), 1,
                                           dout);
  } else {
    intake_kernel<<<grid, 160, smem>>>(tm, cols, share, static_cast<const uint8_t*>(P), W, tma_copies,
                                       cp_iters, bars_after_ring, dout);
  }
  if (cudaGetLastError() != cudaSuccess) return -4;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -5;
}
