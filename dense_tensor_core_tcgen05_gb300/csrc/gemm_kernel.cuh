// Persistent tcgen05 GEMM kernel for sm_103a:  C <- alpha * A * B + beta * C.
//
// One CTA per SM, 6 warps with fixed roles ("warp specialisation", the
// producer/consumer split of the lecture "The Asynchronous Kernel: Tensor Cores &
// TMA", section "The factory"), re-expressed for the fifth-generation tensor core:
//
//   warp 0, one lane   TMA producer: for every k-block of every tile it waits for
//                      a free ring slot (empty[s]), arms full[s] with the slot's
//                      byte count and issues the A and B tile copies.
//   warp 1             allocates Tensor Memory; one lane issues tcgen05.mma
//                      (4 per k-block, K = 16 each) into one of two TMEM
//                      accumulators and releases each slot with tcgen05.commit,
//                      i.e. only after the MMAs reading it have *completed*
//                      (the leetllm page's "releasing a stage at instruction
//                      issue is unsafe").
//   warps 2..5         epilogue: TMEM -> registers (tcgen05.ld, each warp its
//                      own 32-lane quarter) -> alpha*acc + beta*C in fp32 ->
//                      output cast -> 128B-swizzled shared memory -> TMA store.
//                      The accumulator is handed back right after the last
//                      TMEM read, so the epilogue of tile i overlaps the
//                      mainloop of tile i+1 (the "ping-pong" of the lecture).
//
// Every wait is bounded (nanosecond timer); on expiry the waiter records an
// error code in the status word, raises a CTA-wide abort flag, the roles drain
// their own asynchronous work, TMEM is freed and the kernel returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gemm_common.h"
#include "ptx.cuh"

namespace gemm_tc {

constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 4;
constexpr int EPI_ROWS = 32;     // rows per epilogue warp = its TMEM lane quarter
constexpr int EPI_BUFS = 2;      // staging buffers per epilogue warp

enum OutKind { OUT_F32 = 0, OUT_BF16 = 1, OUT_F16 = 2 };

template <bool B>
struct BoolC {
  static constexpr bool value = B;
};

// Where a bounded wait gave up (written to the status word, first error wins).
enum WaitSite {
  SITE_PRODUCER_EMPTY = 1,
  SITE_MMA_TMEM_EMPTY = 2,
  SITE_MMA_FULL = 3,
  SITE_EPI_TMEM_FULL = 4,
  SITE_EPI_C_LOAD = 5,
  SITE_DRAIN = 6,
  SITE_STREAMK_FLAG = 7,
  SITE_SPLITK_SLICES = 8,
};

// Shared-memory map of one CTA.  A ring stage holds KO consecutive k-blocks
// (one TMA copy per operand fetches all of them).  In pair mode (two CTAs
// computing a 256-row tile with one cta_group::2 MMA) each CTA holds its own
// 128 rows of A and half of the tile's B columns.
//   K-major operand tile of a stage:  [KO k-blocks][rows][128 B]
//   MN-major operand tile of a stage: [64-wide atoms][KO * 64 K-rows][128 B]
template <int BN, int STAGES, bool PAIR, int KO>
struct SmemLayout {
  static constexpr int B_COLS = PAIR ? BN / 2 : BN;   // B columns (N) held by this CTA
  static constexpr int KB_A_BYTES = BM * BK * 2;      // one k-block of A
  static constexpr int KB_B_BYTES = B_COLS * BK * 2;  // one k-block of B
  static constexpr int KB_BYTES = KB_A_BYTES + KB_B_BYTES;
  static constexpr int A_BYTES = KO * KB_A_BYTES;
  static constexpr int B_BYTES = KO * KB_B_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_BUF_BYTES = EPI_ROWS * SW;
  static constexpr int off_a = 0;
  static constexpr int off_b = STAGES * A_BYTES;
  static constexpr int off_epi = off_b + STAGES * B_BYTES;
  static constexpr int off_bar = off_epi + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
  static constexpr int RING_BYTES = off_epi;
  // full[STAGES], empty[STAGES], tfull[2], tempty[2], cload[EPI_WARPS*EPI_BUFS], drain, esync,
  // rfull
  static constexpr int NUM_BARS = 2 * STAGES + 4 + EPI_WARPS * EPI_BUFS + 2 + 1;
  static constexpr int off_tmem = off_bar + NUM_BARS * 8;
  static constexpr int off_flag = off_tmem + 8;
  static constexpr int BYTES = off_flag + 8;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 B
  static constexpr int TMEM_COLS = 2 * BN;    // two fp32 accumulators of BN columns
  static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                "TMEM allocation must be a power of two in [32, 512]");
  static_assert(ALLOC <= 232448, "exceeds the 227 KB per-block shared memory limit");
  static_assert(B_COLS % ATOM_MN == 0, "B half-tiles are whole 64-column swizzle atoms");
  static_assert(KO >= 1 && KO * BK <= 256, "a stage's K-rows must fit one copy box");
  static_assert(STAGES >= 2, "the ring needs at least two stages");
};

__device__ __forceinline__ void record_error(int* status, int code) {
  atomicCAS(status, 0, code);
}

// Bounded wait by one thread.  Returns false on timeout or when another role
// has raised the abort flag.  CLUSTER: acquire at cluster scope (pair mode).
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_one(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         const KernelArgs& a, int site) {
  if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    if ((i & 15) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > a.timeout_ns) {
        record_error(a.status, site);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait by a whole warp, with a warp-uniform result: it succeeds once
// every lane has observed the phase (a phase cannot advance again before this
// warp acts on it), and lane 0 alone decides to give up.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const KernelArgs& a, int site) {
  const int lane = threadIdx.x & 31;
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    const bool done = mbar_try_wait<CLUSTER>(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((i & 15) == 15) {
      int give_up = 0;
      if (lane == 0) {
        const uint64_t now = globaltimer_ns();
        if (t0 == 0) t0 = now;
        if (*abort_flag) {
          give_up = 1;
        } else if (now - t0 > a.timeout_ns) {
          record_error(a.status, site);
          *abort_flag = 1;
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
  }
}

// Wait used only while draining after an abort: ignores the abort flag.
template <bool CLUSTER = false>
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, const KernelArgs& a) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait<CLUSTER>(bar, parity)) {
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      record_error(a.status, SITE_DRAIN);
      return;
    }
  }
}

template <int OUT>
struct OutTraits;
template <>
struct OutTraits<OUT_F32> {
  static constexpr int CHUNK_COLS = 32;  // 32 x 4 B = one 128-byte row per chunk
};
template <>
struct OutTraits<OUT_BF16> {
  static constexpr int CHUNK_COLS = 64;  // 64 x 2 B
};
template <>
struct OutTraits<OUT_F16> {
  static constexpr int CHUNK_COLS = 64;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int out_kind) {
  if (out_kind == OUT_BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack2(uint32_t w, int out_kind) {
  if (out_kind == OUT_BF16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(h);
  }
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

// Bias values of one output chunk, loaded before the chunk's waits: lane l holds
// the column bias of chunk columns l and 32 + l (c0, c1; 0 without a column
// bias) and the row bias of its row (row; 0 without a row bias); lo is the ReLU
// floor (0, or -infinity without ReLU).  Pieces pick their columns' values by
// shuffle, so no piece waits on memory, and the step has no branch.
struct EpiBias {
  float c0, c1, row, lo;
};

// Load them (every lane of the warp; columns past N and a row past M read 0).
template <int CHUNK>
__device__ __forceinline__ EpiBias load_epi_bias(const KernelArgs& args, int col0, int grow) {
  const int lane = threadIdx.x & 31;
  EpiBias b{0.0f, 0.0f, 0.0f, args.act == EPI_ACT_RELU ? 0.0f : -__int_as_float(0x7f800000)};
  if (args.bias_kind == EPI_BIAS_COL) {
    if (col0 + lane < args.N) b.c0 = __ldg(args.bias + col0 + lane);
    if (CHUNK == 64 && col0 + 32 + lane < args.N) b.c1 = __ldg(args.bias + col0 + 32 + lane);
  } else if (args.bias_kind == EPI_BIAS_ROW) {
    if (grow < args.M) b.row = __ldg(args.bias + grow);
  }
  return b;
}

// The fused epilogue of one piece (E outputs from chunk column pc, a multiple of
// 4), on fp32 values that already hold alpha*acc + beta*c: add the bias (the
// column and row terms, at most one of them nonzero, so the sum is that bias
// exactly), then the ReLU floor (x < lo -> +0; NaN kept).  All 32 lanes call it.
template <int E>
__device__ __forceinline__ void bias_act(float* x, const EpiBias& b, int pc) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int t = pc + e;
    const float bias = __shfl_sync(0xffffffffu, t < 32 ? b.c0 : b.c1, t & 31) + b.row;
    const float y = x[e] + bias;
    x[e] = y < b.lo ? 0.0f : y;
  }
}

// One 16-byte piece of an output row: x holds its accumulator values (4 for
// fp32 output, 8 for 16-bit output, alpha not yet applied).  Applies
// alpha*acc + beta*c (c read from the staged C chunk at p when rc), then
// (FUSED) the bias and activation, casts, and either writes the piece to the
// swizzled staging buffer (p) or, for a chunk crossing the ragged right edge of
// C, stores its in-range elements straight to global memory.
template <int OUT>
__device__ __forceinline__ void store_piece(const float* x, uint4* p, const KernelArgs& args,
                                            bool ragged, bool store_row, int grow, int gcol);

template <int OUT, bool FUSED = false>
__device__ __forceinline__ void finish_piece(float* x, uint4* p, const KernelArgs& args, bool rc,
                                             bool ragged, bool store_row, int grow, int gcol,
                                             const EpiBias& eb = EpiBias{0.0f, 0.0f, 0.0f, 0.0f},
                                             int pc = 0) {
  constexpr int E = OUT == OUT_F32 ? 4 : 8;
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] *= args.alpha;
  if (rc) {
    const uint4 ci = *p;
    if (OUT == OUT_F32) {
      x[0] = fmaf(args.beta, __uint_as_float(ci.x), x[0]);
      x[1] = fmaf(args.beta, __uint_as_float(ci.y), x[1]);
      x[2] = fmaf(args.beta, __uint_as_float(ci.z), x[2]);
      x[3] = fmaf(args.beta, __uint_as_float(ci.w), x[3]);
    } else {
      const uint32_t cw[4] = {ci.x, ci.y, ci.z, ci.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack2(cw[e], OUT);
        x[2 * e] = fmaf(args.beta, f.x, x[2 * e]);
        x[2 * e + 1] = fmaf(args.beta, f.y, x[2 * e + 1]);
      }
    }
  }
  if (FUSED) bias_act<E>(x, eb, pc);
  store_piece<OUT>(x, p, args, ragged, store_row, grow, gcol);
}

// The fused epilogue on a whole output chunk held in registers (this thread's
// row, CHUNK columns from col0: v0 = columns 0..31, v1 = 32..63), before any of
// it is stored: x = alpha*acc, + beta*c (c from the staged C chunk at rowp when
// rc), + bias, then ReLU (negative -> 0, NaN kept); written back into v0/v1.
// The bias was loaded before the accumulator was ready: with a column bias,
// lane l holds columns l (cb0) and 32 + l (cb1) of the chunk (0 past N) and the
// values go round by shuffle; with a row bias, rb is this thread's row's value.
// The branches are taken once per chunk.
template <int OUT, int CHUNK>
__device__ __forceinline__ void fused_chunk(uint32_t* v0, uint32_t* v1, const uint8_t* rowp,
                                            const KernelArgs& args, bool rc, float cb0, float cb1,
                                            float rb, int r) {
  constexpr int E = OUT == OUT_F32 ? 4 : 8;
  float x[CHUNK];
#pragma unroll
  for (int i = 0; i < CHUNK; ++i) x[i] = __uint_as_float(i < 32 ? v0[i] : v1[i - 32]) * args.alpha;
  if (rc) {
#pragma unroll
    for (int j = 0; j < CHUNK / E; ++j) {
      const uint4 ci = *reinterpret_cast<const uint4*>(rowp + ((j ^ (r & 7)) << 4));
      const uint32_t cw[4] = {ci.x, ci.y, ci.z, ci.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (OUT == OUT_F32) {
          x[4 * j + e] = fmaf(args.beta, __uint_as_float(cw[e]), x[4 * j + e]);
        } else {
          const float2 f = unpack2(cw[e], OUT);
          x[8 * j + 2 * e] = fmaf(args.beta, f.x, x[8 * j + 2 * e]);
          x[8 * j + 2 * e + 1] = fmaf(args.beta, f.y, x[8 * j + 2 * e + 1]);
        }
      }
    }
  }
  if (args.bias_kind == EPI_BIAS_COL) {
#pragma unroll
    for (int i = 0; i < CHUNK; ++i) x[i] += __shfl_sync(0xffffffffu, i < 32 ? cb0 : cb1, i & 31);
  } else if (args.bias_kind == EPI_BIAS_ROW) {
#pragma unroll
    for (int i = 0; i < CHUNK; ++i) x[i] += rb;
  }
  if (args.act == EPI_ACT_RELU) {
#pragma unroll
    for (int i = 0; i < CHUNK; ++i) x[i] = x[i] < 0.0f ? 0.0f : x[i];
  }
#pragma unroll
  for (int i = 0; i < CHUNK; ++i) {
    if (i < 32)
      v0[i] = __float_as_uint(x[i]);
    else
      v1[i - 32] = __float_as_uint(x[i]);
  }
}

// Cast a finished piece (E fp32 values) to the output format and store it: into
// the swizzled staging buffer (p), or for a chunk crossing the ragged right edge
// of C, its in-range elements straight to global memory.
template <int OUT>
__device__ __forceinline__ void store_piece(const float* x, uint4* p, const KernelArgs& args,
                                            bool ragged, bool store_row, int grow, int gcol) {
  uint4 o;
  if (OUT == OUT_F32) {
    o = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                   __float_as_uint(x[3]));
  } else {
    o = make_uint4(pack2(x[0], x[1], OUT), pack2(x[2], x[3], OUT), pack2(x[4], x[5], OUT),
                   pack2(x[6], x[7], OUT));
  }
  if (!ragged) {
    *p = o;
  } else if (store_row) {
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
    if (OUT == OUT_F32) {
      float* dst = static_cast<float*>(args.c_ptr) + static_cast<long long>(grow) * args.ldc + gcol;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (gcol + e < args.N) dst[e] = __uint_as_float(ow[e]);
    } else {
      uint16_t* dst =
          static_cast<uint16_t*>(args.c_ptr) + static_cast<long long>(grow) * args.ldc + gcol;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (gcol + e < args.N) dst[e] = static_cast<uint16_t>(ow[e >> 1] >> (16 * (e & 1)));
    }
  }
}

// A ragged 16-bit chunk of the main epilogue (N * sizeof(out) not a multiple of
// 16 bytes and the chunk crossing column N) is staged like any other and then
// written from the staging buffer with plain stores, row by row: 8 lanes per
// 128-byte staged row, 4 rows per step, whole 16-byte pieces where they lie
// inside C and element by element at the edge (a tensor store writes whole
// 16-byte pieces and would touch the columns just past N).  Every row of C
// starts 16-byte aligned (ldc * sizeof(out) is a multiple of 16).
template <int OUT>
__device__ __forceinline__ void copy_out_ragged(const uint8_t* stg, const KernelArgs& args, int row0,
                                                int col0) {
  constexpr int E = OUT == OUT_F32 ? 4 : 8;   // elements per 16-byte piece
  constexpr int OSZ = OUT == OUT_F32 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int piece = lane & 7;
  const int gcol = col0 + piece * E;
  __syncwarp();   // every lane's staged row is written
  // all 8 of this lane's pieces read first (the loads' latency overlaps), then stored
  uint4 pv[EPI_ROWS / 4];
#pragma unroll
  for (int i = 0; i < EPI_ROWS / 4; ++i) {
    const int r = 4 * i + (lane >> 3);
    pv[i] = ld_shared_v4(smem_u32(stg) + static_cast<uint32_t>(r * SW + ((piece ^ (r & 7)) << 4)));
  }
#pragma unroll
  for (int i = 0; i < EPI_ROWS / 4; ++i) {
    const int r = 4 * i + (lane >> 3);
    const int grow = row0 + r;
    if (grow < args.M && gcol < args.N) {
      const uint4 v = pv[i];
      char* dst = static_cast<char*>(args.c_ptr) +
                  (static_cast<long long>(grow) * args.ldc + gcol) * OSZ;
      if (gcol + E <= args.N) {
        *reinterpret_cast<uint4*>(dst) = v;
      } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (gcol + e >= args.N) break;
          if (OUT == OUT_F32)
            reinterpret_cast<uint32_t*>(dst)[e] = w[e];
          else
            reinterpret_cast<uint16_t*>(dst)[e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
        }
      }
    }
  }
}

// Epilogue bookkeeping shared by the chunk loops of one epilogue warp.
struct EpiState {
  uint8_t* stage0;        // this warp's staging buffers
  uint64_t* cload;        // this warp's C-load barriers
  uint32_t chunk_ctr;     // chunks finished so far (alternates the two buffers)
  int pending_cload;      // buffer with a C load in flight (abort drain), or -1
  uint32_t pending_phase;
};

// Prepare the next staging buffer for an output chunk at (row0, col0): wait
// until the store that last read it has finished, and when rc (beta != 0 and C
// not already in the accumulator) fetch the C chunk into it.  Returns false if
// a wait gave up.
template <bool CLUSTER, int EPI_BUF_BYTES>
__device__ __forceinline__ bool begin_chunk(EpiState& st, uint8_t*& stg, const CUtensorMap* tmC,
                                            int row0, int col0, volatile int* abort_flag,
                                            const KernelArgs& args, bool rc) {
  const int lane = threadIdx.x & 31;
  const int sbuf = st.chunk_ctr & 1;
  stg = st.stage0 + sbuf * EPI_BUF_BYTES;
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  if (rc) {
    uint64_t* cb = &st.cload[sbuf];
    const uint32_t cph = (st.chunk_ctr >> 1) & 1;
    if (lane == 0) {
      mbar_arrive_expect_tx(cb, EPI_BUF_BYTES);
      tma_load_2d(stg, tmC, col0, row0, cb);
    }
    st.pending_cload = sbuf;
    st.pending_phase = cph;
    if (!wait_warp<CLUSTER>(cb, cph, abort_flag, args, SITE_EPI_C_LOAD)) return false;
    st.pending_cload = -1;
  }
  return true;
}

// Issue the tensor store of a finished chunk (unless it was ragged or entirely
// outside C) and commit exactly one bulk group per chunk, so that "at most one
// group still reading" in begin_chunk always means "the other buffer".
__device__ __forceinline__ void end_chunk(EpiState& st, const uint8_t* stg, const CUtensorMap* tmC,
                                          int row0, int col0, bool ragged, bool skip_store) {
  const int lane = threadIdx.x & 31;
  if (!ragged && !skip_store) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_2d(tmC, stg, col0, row0);
  }
  if (lane == 0) bulk_commit_group();
  __syncwarp();
  ++st.chunk_ctr;
}

// Shared-memory address of 16-byte piece `piece` of row `row` in a split-K
// slice block (128 rows of SLICE floats; pieces XOR-swizzled by row so that the
// 8 rows sharing a 1 KB span use all 8 bank groups: by row & 7 with 8 or more
// pieces per row, by (row / (8 / P)) & (P - 1) with P < 8 pieces per row).
template <int SLICE>
__device__ __forceinline__ uint32_t slice_addr(uint32_t base, int row, int piece) {
  constexpr int P = SLICE / 4;
  const int sw = P >= 8 ? (row & 7) : ((row / (8 / P)) & (P - 1));
  return base + static_cast<uint32_t>(row * (SLICE * 4) + ((piece ^ sw) << 4));
}

// Stream-K hand-off: a CTA publishes its partial tile with a release store of
// the launch epoch into its flag; the owner of the tile acquires it.
__device__ __forceinline__ void flag_release(unsigned int* f, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int flag_acquire(const unsigned int* f) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}


// Specialised instances.  Most launches take the plain path: no C read (or,
// with SPEC_READC, always a C read), no bias or activation (or, with SPEC_EPI,
// the fused epilogue, its kinds chosen at run time), N * sizeof(out) a
// multiple of 16 bytes, tiles in grouped order, no fault injection, and
// data-parallel tiles only (or, with SPEC_STREAMK, a stream-K tail as well);
// and each operand's major-ness is fixed by the call's layout.  Folding those parameters into constants drops
// the code of the other paths from the kernel, which roughly halves its
// instruction-cache misses and shortens the one-off start-up and epilogue code
// (2048^3: about 10% of the launch).  The host launches a specialised instance
// only for a call that matches it; every other call takes the general kernel.
enum : int {
  SPEC_PLAIN = 1,          // plain epilogue and scheduling (see above)
  SPEC_LAYOUT = 2,         // operand layout fixed: bits 2..3 hold GEMM_A_* | GEMM_B_*
  SPEC_LAYOUT_SHIFT = 2,
  SPEC_STREAMK = 16,       // with SPEC_PLAIN: stream-K or split-tile work stays a run-time choice
  SPEC_READC = 32,         // with SPEC_PLAIN: C is read (beta != 0)
  SPEC_EPI = 64,           // with SPEC_PLAIN: a bias and/or an activation is applied
  SPEC_RAGGED = 128,       // with SPEC_PLAIN: the ragged right edge stays a run-time choice
};
// the specialisation of a plain call with `layout` (stream-K work when sk, a C
// read when readc, the fused epilogue when epi, a ragged right edge possible when
// ragged)
constexpr int spec_bits(int layout, bool sk, bool readc, bool epi = false, bool ragged = false) {
  return SPEC_PLAIN | SPEC_LAYOUT | (layout << SPEC_LAYOUT_SHIFT) | (sk ? SPEC_STREAMK : 0) |
         (readc ? SPEC_READC : 0) | (epi ? SPEC_EPI : 0) | (ragged ? SPEC_RAGGED : 0);
}
template <int SPEC, bool F8>
__device__ __forceinline__ KernelArgs specialise_args(const KernelArgs& in) {
  KernelArgs a = in;
  if (SPEC & SPEC_PLAIN) {
    a.read_c = (SPEC & SPEC_READC) ? 1 : 0;
    if (SPEC & SPEC_EPI) {
      a.epi = 1;   // bias_kind and act stay run-time values
    } else {
      a.epi = 0;
      a.bias_kind = EPI_BIAS_NONE;
      a.act = EPI_ACT_NONE;
    }
    if (!(SPEC & SPEC_RAGGED)) a.n_ragged = 0;
    if (!(SPEC & SPEC_STREAMK)) {
      a.sk_iters = 0;
      a.tile_split = 0;
    }
    a.inject_skip = 0;
    a.tile_map = nullptr;
  }
  if (SPEC & SPEC_LAYOUT) {
    constexpr int layout = SPEC >> SPEC_LAYOUT_SHIFT;
    a.a_mn = (layout & 1) ? 1 : 0;   // A column-major: M-major
    a.b_mn = (layout & 2) ? 0 : 1;   // B row-major: N-major
    a.kblock_elems = F8 ? 128 : 64;
  }
  return a;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Stage one output chunk row (this thread's row r, registers v0 = columns 0..31,
// v1 = 32..63) as alpha * acc (SCALE) or as the finished values themselves
// (!SCALE: bits kept as they are), cast to the output format, into the swizzled
// staging row at shared address `row`: 16-byte piece j at (j ^ (r & 7)) * 16.
template <int OUT, bool SCALE = true>
__device__ __forceinline__ void stage_chunk_scaled(const uint32_t* v0, const uint32_t* v1,
                                                   uint32_t row, float alpha, int r) {
  auto f = [&](uint32_t w) { return SCALE ? __uint_as_float(w) * alpha : __uint_as_float(w); };
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 o;
    if (OUT == OUT_F32) {
      const uint32_t* s = v0 + 4 * j;
      o = SCALE ? make_uint4(__float_as_uint(f(s[0])), __float_as_uint(f(s[1])),
                             __float_as_uint(f(s[2])), __float_as_uint(f(s[3])))
                : make_uint4(s[0], s[1], s[2], s[3]);
    } else {
      const uint32_t* s = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
      o = make_uint4(pack2(f(s[0]), f(s[1]), OUT), pack2(f(s[2]), f(s[3]), OUT),
                     pack2(f(s[4]), f(s[5]), OUT), pack2(f(s[6]), f(s[7]), OUT));
    }
    st_shared_v4(row + ((j ^ (r & 7)) << 4), o);
  }
}

// beta * C[grow][col0 .. col0 + 32) as fp32 bits (0 outside C), read with plain
// loads: the initial accumulator value of a tile whose C term is added by the
// MMAs.  Rows are 16-byte aligned (ldc times the element size is a multiple of
// 16) and col0 is a multiple of 32.
template <int OUT>
__device__ __forceinline__ void load_c32(const KernelArgs& a, int grow, int col0, uint32_t (&v)[32]) {
  if (grow >= a.M || col0 >= a.N) {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = 0u;
    return;
  }
  const bool full = col0 + 32 <= a.N;
  if (OUT == OUT_F32) {
    const float* src = static_cast<const float*>(a.c_ptr) + static_cast<long long>(grow) * a.ldc + col0;
    if (full) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 f = reinterpret_cast<const float4*>(src)[j];
        v[4 * j] = __float_as_uint(a.beta * f.x);
        v[4 * j + 1] = __float_as_uint(a.beta * f.y);
        v[4 * j + 2] = __float_as_uint(a.beta * f.z);
        v[4 * j + 3] = __float_as_uint(a.beta * f.w);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = col0 + e < a.N ? __float_as_uint(a.beta * src[e]) : 0u;
    }
  } else {
    const uint16_t* src =
        static_cast<const uint16_t*>(a.c_ptr) + static_cast<long long>(grow) * a.ldc + col0;
    if (full) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = reinterpret_cast<const uint4*>(src)[j];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack2(ws[e], OUT);
          v[8 * j + 2 * e] = __float_as_uint(a.beta * f.x);
          v[8 * j + 2 * e + 1] = __float_as_uint(a.beta * f.y);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float f = col0 + e < a.N ? unpack2(src[e], OUT).x : 0.0f;
        v[e] = __float_as_uint(a.beta * f);
      }
    }
  }
}

// PAIR: two CTAs per 256-row tile (cta_group::2).  SPLIT > 1: a cluster of
// SPLIT CTAs shares one 128-row tile, each accumulating 1/SPLIT of the K range;
// the partial sums meet in distributed shared memory (split-K without a global
// workspace; one tile per cluster).
// F8: 8-bit operands (tcgen05.mma kind::f8f6f4) instead of 16-bit ones; a
// compile-time choice, as a branch between MMA kinds in the issue loop slows it.
// SPEC: SPEC_* bits folding run-time parameters into constants (see
// specialise_args); 0 for the general kernel.
template <int BN, int STAGES, int OUT, bool PAIR, int SPLIT, int KO, bool F8 = false, int SPEC = 0>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmA3,
                        const __grid_constant__ CUtensorMap tmB3,
                        const __grid_constant__ CUtensorMap tmC, const KernelArgs args_in) {
  const KernelArgs args = specialise_args<SPEC, F8>(args_in);
  using L = SmemLayout<BN, STAGES, PAIR, KO>;
  constexpr int CHUNK = OutTraits<OUT>::CHUNK_COLS;
  constexpr int CHUNKS = BN / CHUNK;
  constexpr int TILE_M = PAIR ? 2 * BM : BM;       // rows of one work unit
  constexpr bool SPLITK = SPLIT > 1;
  constexpr bool CLUSTERED = PAIR || SPLITK;
  constexpr int SLICE = BN / SPLIT;                // output columns each split CTA reduces
  static_assert(BN % CHUNK == 0, "tile width must be a whole number of epilogue chunks");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N must be in [16,256], N%16==0");
  static_assert(!(PAIR && SPLITK), "pair and split-K modes are exclusive");
  static_assert(!SPLITK || (SLICE >= 16 && (SLICE % CHUNK == 0 || CHUNK % SLICE == 0)),
                "a split CTA finishes whole epilogue chunks or one narrower slice");
  // split-K: the fp32 slices a CTA sends to its SPLIT-1 peers and the ones it
  // receives from them share the (idle) ring
  constexpr int SLICE_BYTES = BM * SLICE * 4;
  static_assert(!SPLITK || 2 * (SPLIT - 1) * SLICE_BYTES <= STAGES * L::STAGE_BYTES,
                "the split-K slices must fit in the ring's shared memory");
  // Two-CTA split-K whose peer slice fits the epilogue staging area (unused by a
  // split-K CTA until its final chunks): each epilogue warp pushes its rows of
  // the peer's slice into that area as soon as they are staged, with no cluster
  // barrier in between; the final chunks then stage in the idle ring, after
  // the send area.  Wider slices and more peers meet in the ring after a
  // cluster barrier instead.
  constexpr bool EARLY = SPLIT == 2 && SLICE_BYTES <= L::off_bar - L::off_epi;
  static_assert(!EARLY || SLICE_BYTES + EPI_WARPS * EPI_BUFS * L::EPI_BUF_BYTES <= L::RING_BYTES,
                "final-chunk staging must fit in the ring after the send area");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bar);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* cload = tempty + 2;
  uint64_t* drain = cload + EPI_WARPS * EPI_BUFS;
  uint64_t* esync = drain + 1;   // rendezvous of the four epilogue warps (stream-K hand-off)
  uint64_t* rfull = esync + 1;   // split-K: the peers' slices have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::off_tmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_flag);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Pair mode: the even CTA of the cluster (rank 0) issues the MMAs and owns the
  // "full" and "tmem empty" barriers both CTAs signal; each CTA computes rows
  // [rank * 128, rank * 128 + 128) of the 256-row unit.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  const uint32_t srank = SPLITK ? cluster_ctarank() : 0;  // K slice of a split-K CTA
  const bool leader = rank == 0;
  constexpr int UNIT_CTAS = PAIR ? 2 : SPLIT;
  const int unit0 = static_cast<int>(blockIdx.x) / UNIT_CTAS;
  const int unit_stride = static_cast<int>(gridDim.x) / UNIT_CTAS;
  // K range of a work item, in k-blocks: a split-K CTA's fixed slice, otherwise
  // the item's k-groups.
  const int split_kb0 = SPLITK ? (args.k_blocks * static_cast<int>(srank)) / SPLIT : 0;
  const int split_kb1 = SPLITK ? (args.k_blocks * static_cast<int>(srank + 1)) / SPLIT : 0;
  auto kb_range = [&](const WorkItem& w, int* b, int* e) {
    if (SPLITK) {
      *b = split_kb0;
      *e = split_kb1;
    } else {
      *b = w.g0 * KO;
      *e = w.g1 * KO < args.k_blocks ? w.g1 * KO : args.k_blocks;
    }
  };
  auto work_begin = [&](WorkIter& wi) {
    wi.init(unit0, unit_stride, args.dp_tiles, args.sk_iters, args.groups, args.fd_groups,
            args.tile_split, args.owner_groups);
  };
  uint32_t producer_iters = 0;  // ring iterations armed (producer thread only)
  // Start-up.  The lanes of warp 0 initialise the barriers (one each) while
  // warp 1 allocates TMEM and warp 2 prefetches the tensor maps (on warp 0's
  // path the prefetches delayed the first copy by ~0.4 us).  The start-up barrier
  // is split: warp 0 arrives, works out the producer's first work item and L2
  // policies, and waits only where it must (pair mode: the odd CTA's copies
  // signal the leader's barrier), so the first copies go out as soon as it opens.
  if (warp == 0) {
    for (int i = lane; i < L::NUM_BARS; i += 32) {
      const uint64_t* b = bars + i;
      const uint32_t count = (b == tempty || b == tempty + 1) ? (PAIR ? 2 * EPI_WARPS : EPI_WARPS)
                             : b == esync                    ? EPI_WARPS
                                                             : 1;
      mbar_init(bars + i, count);
    }
    if (lane == 0) *abort_flag = 0;
    fence_barrier_init();
    __syncwarp();
    // early split-K exchange: the peer's block is expected from the start; the
    // cluster barrier below orders this before the peer's copy
    if (EARLY && lane == 0) mbar_arrive_expect_tx(rfull, SLICE_BYTES);
  }
  // Pair mode, phase 1 of the cluster barrier: both CTAs' mbarriers exist (the
  // odd CTA's copies and the MMA commits signal the leader's and the peer's).
  // Warp 0 arrives after initialising them (relaxed: fence.mbarrier_init has
  // published them), every other warp at once, before the TMEM allocation.
  if (PAIR) cluster_arrive_relaxed();
  if (warp == 2) {
    if (lane == 0) prefetch_tensormap(&tmA);
    if (lane == 1) prefetch_tensormap(&tmB);
    if (lane == 2 && args.a_full3d) prefetch_tensormap(&tmA3);
    if (lane == 3 && args.b_full3d) prefetch_tensormap(&tmB3);
    if (lane == 4) prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, L::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, L::TMEM_COLS);
      tmem_relinquish();
    }
  }
  __syncwarp();
  tc_fence_before();
  // The barriers (and, for every role but the producer, the TMEM address) are
  // visible before use.  Pair mode, phase 2: TMEM is allocated in both CTAs
  // (the leader's MMAs write both); warp 1 arrives after allocating, with
  // release for the address it wrote.  The producer waits for phase 1 only and
  // for phase 2 at the end, so its first copies do not wait for the allocation.
  if (PAIR) {
    cluster_wait();
    if (warp == 1)
      cluster_arrive();
    else
      cluster_arrive_relaxed();
    if (warp != 0) cluster_wait();
  } else if (warp == 0) {
    named_bar_arrive(1, NUM_THREADS);
  } else {
    named_bar_sync(1, NUM_THREADS);
  }
  // early split-K exchange: every CTA's barriers exist before a peer copies into
  // it (waited for by the epilogue warps before their copies, by the others at
  // the end)
  if (EARLY) {
    if (warp == 0)
      cluster_arrive_relaxed();
    else
      cluster_arrive();
  }
  tc_fence_after();
  const uint32_t tmem_base = warp == 0 ? 0u : *tmem_slot;   // warp 0 never touches TMEM

  if (warp == 0) {
    // L2 policies: 0 = default, 1 = evict first (streamed once), 2 = evict last (reused)
    uint64_t pol_a = 0, pol_b = 0;
    WorkIter wi;
    WorkItem w;
    bool have = false;
    int mb = 0, nb = 0;
    if (lane == 0) {
      work_begin(wi);
      have = wi.next(&w);
      if (have) tile_of(args, w.tile, &mb, &nb);
    }
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      uint32_t it = 0;
      bool ok = true;
      while (ok && have) {
        int kb_begin, kb_end;
        kb_range(w, &kb_begin, &kb_end);
        const int a_row = mb * TILE_M + static_cast<int>(rank) * BM;
        const int b_col = nb * BN + static_cast<int>(rank) * L::B_COLS;
        const int steps = (kb_end - kb_begin + KO - 1) / KO;
        const bool down = !SPLITK && w.down;
        for (int q = 0; q < steps; ++q, ++it) {
          const int kb0 = kb_begin + (down ? steps - 1 - q : q) * KO;
          const int nkb = kb_end - kb0 < KO ? kb_end - kb0 : KO;
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (it == 1) {   // the L2 policies of every copy after the first stage's
            if (args.a_hint) pol_a = args.a_hint == 1 ? policy_evict_first() : policy_evict_last();
            if (args.b_hint) pol_b = args.b_hint == 1 ? policy_evict_first() : policy_evict_last();
          }
          if (!wait_one<PAIR>(&empty[s], ph ^ 1, abort_flag, args, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          if (args.inject_skip != 0 && it + 1 == static_cast<uint32_t>(args.inject_skip)) continue;
          // the leader's full[s] counts the bytes of both CTAs of a pair
          if (leader)
            mbar_arrive_expect_tx(&full[s], PAIR ? 2 * nkb * L::KB_BYTES
                                                 : nkb * (args.a_box_rows * BK * 2 + L::KB_B_BYTES));
          uint8_t* sa = smem + L::off_a + s * L::A_BYTES;
          uint8_t* sb = smem + L::off_b + s * L::B_BYTES;
          const uint32_t bar_c = PAIR ? map_to_rank(&full[s], 0) : 0;
          auto load2 = [&](void* dst, const CUtensorMap* m, int x, int y, int hint, uint64_t pol) {
            if (PAIR)
              tma_load_2d_pair(dst, m, x, y, bar_c);
            else if (hint)
              tma_load_2d_hint(dst, m, x, y, &full[s], pol);
            else
              tma_load_2d(dst, m, x, y, &full[s]);
          };
          auto load3 = [&](void* dst, const CUtensorMap* m, int y, int z, int hint, uint64_t pol) {
            if (PAIR)
              tma_load_3d_pair(dst, m, 0, y, z, bar_c);
            else if (hint)
              tma_load_3d_hint(dst, m, 0, y, z, &full[s], pol);
            else
              tma_load_3d(dst, m, 0, y, z, &full[s]);
          };
          // One operand's share of the stage.  The 3-D map fetches all KO k-blocks
          // (K-major) or all atoms (MN-major) in one copy; it only covers whole
          // 64-element blocks, so a group touching a ragged edge takes the 2-D
          // map, whose out-of-range elements read as zero.
          auto load_operand = [&](uint8_t* dst, const CUtensorMap* m2, const CUtensorMap* m3,
                                  int mn, int rows, int row0, int full3d, int hint, uint64_t pol) {
            if (!mn) {
              if (nkb == KO && kb0 + KO <= full3d) {
                load3(dst, m3, row0, kb0, hint, pol);
              } else {
                for (int j = 0; j < nkb; ++j)
                  load2(dst + j * rows * SW, m2, (kb0 + j) * args.kblock_elems, row0, hint, pol);
              }
            } else {
              const int atoms = rows / ATOM_MN;
              if (nkb == KO && row0 / ATOM_MN + atoms <= full3d) {
                load3(dst, m3, kb0 * BK, row0 / ATOM_MN, hint, pol);
              } else {
                for (int a = 0; a < atoms; ++a)
                  for (int j = 0; j < nkb; ++j)
                    load2(dst + a * (KO * BK * SW) + j * (BK * SW), m2, row0 + a * ATOM_MN,
                          (kb0 + j) * BK, hint, pol);
              }
            }
          };
          // the first stage goes out without L2 hints: their policies are made
          // after it is issued (createpolicy is slow enough to delay the first copy)
          const bool hinted = it != 0;
          load_operand(sa, &tmA, &tmA3, args.a_mn, BM, a_row, args.a_full3d, hinted ? args.a_hint : 0,
                       pol_a);
          load_operand(sb, &tmB, &tmB3, args.b_mn, L::B_COLS, b_col, args.b_full3d,
                       hinted ? args.b_hint : 0, pol_b);

        }
        have = wi.next(&w);
        if (have) tile_of(args, w.tile, &mb, &nb);
      }
      producer_iters = it;
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------ MMA issuer
      uint32_t it = 0, tl = 0;
      bool ok = true;
      // Per k-block j of a stage: K-major tiles are rows*128 B apart and a K16
      // slice moves the start address 32 B inside the swizzled row; MN-major
      // operands step 64 K-rows (8 KB) per k-block and 16 rows (2 KB) per K16
      // slice, their 64-wide atoms KO*8 KB apart (LBO).
      const uint32_t a_lbo = args.a_mn ? KO * BK * SW : 16, b_lbo = args.b_mn ? KO * BK * SW : 16;
      const uint32_t a_kb = args.a_mn ? BK * SW : BM * SW;
      const uint32_t b_kb = args.b_mn ? BK * SW : L::B_COLS * SW;
      const uint32_t a_step = (args.a_mn ? UMMA_K * SW : UMMA_K * 2) >> 4;
      const uint32_t b_step = (args.b_mn ? UMMA_K * SW : UMMA_K * 2) >> 4;
      auto mma = [&](uint32_t d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
        if (F8) {
          if (PAIR)
            umma_f8_pair(d, da, db, idesc, acc);
          else
            umma_f8(d, da, db, idesc, acc);
        } else {
          if (PAIR)
            umma_f16_pair(d, da, db, idesc, acc);
          else
            umma_f16(d, da, db, idesc, acc);
        }
      };
      // The MMAs of one ring stage (slot s, nkb k-blocks, the item's stage si).
      auto issue_stage = [&](int s, int nkb, int si, uint32_t d_tmem, bool pre) {
        const uint32_t sa = smem_u32(smem + L::off_a + s * L::A_BYTES);
        const uint32_t sb = smem_u32(smem + L::off_b + s * L::B_BYTES);
#pragma unroll
        for (int j = 0; j < KO; ++j) {
          if (j < nkb) {
            const uint64_t da0 = make_sdesc_sw128(sa + j * a_kb, a_lbo, 8 * SW);
            const uint64_t db0 = make_sdesc_sw128(sb + j * b_kb, b_lbo, 8 * SW);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {   // 4 x 32 bytes of each row
              const uint64_t da = da0 + static_cast<uint64_t>(kk) * a_step;
              const uint64_t db = db0 + static_cast<uint64_t>(kk) * b_step;
              const uint32_t acc = (pre || si != 0 || j != 0 || kk != 0) ? 1u : 0u;
              mma(d_tmem, da, db, args.idesc, acc);
            }
          }
        }
      };
      auto commit_to = [&](uint64_t* bar) {
        if (PAIR)
          umma_commit_pair_multicast(bar, 0x3);   // in both CTAs
        else
          umma_commit(bar);
      };
      WorkIter wi;
      WorkItem w;
      work_begin(wi);
      for (; ok && wi.next(&w); ++tl) {
        int kb_begin, kb_end;
        kb_range(w, &kb_begin, &kb_end);
        const int buf = tl & 1;
        const uint32_t aph = (tl >> 1) & 1;
        // the epilogue warps may have written beta * C into the accumulator
        const bool pre = item_preloads_c(args, tl, w);
        if (!wait_one<PAIR>(&tempty[buf], aph ^ 1, abort_flag, args, SITE_MMA_TMEM_EMPTY)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        const int steps = (kb_end - kb_begin + KO - 1) / KO;
        const bool down = !SPLITK && w.down;
        for (int si = 0; si < steps; ++si, ++it) {
          const int kb0 = kb_begin + (down ? steps - 1 - si : si) * KO;
          const int nkb = kb_end - kb0 < KO ? kb_end - kb0 : KO;
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_one<PAIR>(&full[s], ph, abort_flag, args, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_stage(s, nkb, si, d_tmem, pre);
          commit_to(&empty[s]);   // free slot s once these MMAs have completed
        }
        if (!ok) break;
        commit_to(&tfull[buf]);   // accumulator ready
      }
    }
  } else {
    // -------------------------------------------------------- epilogue
    const int ew = warp - EPI_WARP0;     // 0..3
    const int quarter = warp & 3;        // the TMEM lane quarter this warp may access
    if (EARLY) cluster_wait();           // the peer's barriers exist (long before it is needed)
    bool pushed = false;                 // early split-K: this warp's rows were sent
    // early split-K: copy this warp's 32 rows of the staged peer slice (ring
    // offset 0) into the peer's staging area, counted on the peer's rfull
    auto push_rows = [&]() {
      __syncwarp();
      if (lane == 0) {
        const uint32_t peer = 1u - srank;
        const uint32_t part = static_cast<uint32_t>(quarter * 32 * SLICE * 4);
        bulk_copy_s2cluster(map_addr_to_rank(smem_u32(smem + L::off_epi) + part, peer),
                            smem_u32(smem) + part, 32 * SLICE * 4,
                            map_addr_to_rank(smem_u32(rfull), peer));
      }
      pushed = true;
    };
    EpiState st{smem + L::off_epi + ew * EPI_BUFS * L::EPI_BUF_BYTES, &cload[ew * EPI_BUFS], 0,
                -1, 0};
    uint32_t tl = 0, esync_uses = 0;
    bool ok = true;
    const int r = lane;                  // this thread's row inside the warp's 32-row block
    // Rendezvous of the four epilogue warps, bounded like every other wait.
    auto epilogue_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(esync);
      return wait_warp<PAIR>(esync, (esync_uses++) & 1, abort_flag, args, SITE_STREAMK_FLAG);
    };
    // Bounded wait by the whole warp for a contributing unit's ready flag (its
    // partial sum published with this launch's epoch).  Every lane acquires the
    // flag itself, so every lane's later loads of the partial see it.
    auto wait_flag_warp = [&](const unsigned int* f) -> bool {
      uint64_t t0 = 0;
      for (uint32_t i = 0;; ++i) {
        const bool done = flag_acquire(f) == args.epoch;
        if (__all_sync(0xffffffffu, done)) return true;
        __nanosleep(64);
        if ((i & 7) == 7) {
          int give_up = 0;
          if (lane == 0) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            if (*abort_flag) {
              give_up = 1;
            } else if (now - t0 > args.timeout_ns) {
              record_error(args.status, SITE_STREAMK_FLAG);
              *abort_flag = 1;
              give_up = 1;
            }
          }
          if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
      }
    };
    // Owner of a tile whose other k-groups other units hold: once their flags
    // are up, sum their partials of this warp's 32 rows (unit order c0, c0+1,
    // ...) into the TMEM accumulator buffer at t_part, which the unit no longer
    // uses (the owner item is the unit's last), while the item's own MMAs are
    // still running.  A contributor's slot holds each 32-column group of a
    // warp's rows as [8 pieces][32 rows][16 B], so one 16-byte load per lane and
    // piece reads 512 contiguous bytes.  Returns false if a wait gave up.
    auto preload_partials = [&](int c0, int n, uint32_t t_part) -> bool {
      for (int k = 0; k < n; ++k)
        if (!wait_flag_warp(args.ws_flags + (c0 + k) * UNIT_CTAS + rank)) return false;
      // Each round loads GR 32-column groups (8 x 16 B per lane each) before
      // writing any to TMEM, so 128 B per lane and group are in flight: the
      // partials come from L2 while it serves the mainloop's operand traffic.
      // Contributor 0 is stored, the later ones are added to what is stored.
      constexpr int GR = BN / 32 < 4 ? BN / 32 : 4;
#pragma unroll 1
      for (int k = 0; k < n; ++k) {
        const float4* src = reinterpret_cast<const float4*>(
            args.ws + static_cast<size_t>((c0 + k) * UNIT_CTAS + rank) * BM * BN +
            static_cast<size_t>(quarter) * BN * EPI_ROWS) + lane;
#pragma unroll 1
        for (int c = 0; c < BN / 32; c += GR) {
          float4 v[8 * GR];
#pragma unroll
          for (int j = 0; j < 8 * GR; ++j) v[j] = __ldcg(src + static_cast<size_t>(c * 8 + j) * EPI_ROWS);
#pragma unroll
          for (int q = 0; q < GR; ++q) {
            uint32_t r[32];
            if (k > 0) {
              tmem_ld_32x32b_x32(t_part, r, (c + q) * 32);
              tmem_ld_wait();
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 f = v[8 * q + j];
              if (k == 0) {
                r[4 * j] = __float_as_uint(f.x);
                r[4 * j + 1] = __float_as_uint(f.y);
                r[4 * j + 2] = __float_as_uint(f.z);
                r[4 * j + 3] = __float_as_uint(f.w);
              } else {
                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + f.x);
                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + f.y);
                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + f.z);
                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + f.w);
              }
            }
            tmem_st_32x32b_x32(t_part, r, (c + q) * 32);
          }
        }
        tmem_st_wait();   // stored before the next contributor's sums read them back
      }
      return true;
    };

    // Owner whose item is not its unit's last, with one contributor (flag up):
    // that unit's partial of this warp's 32 rows added onto the accumulator in
    // TMEM at t_acc, GR 32-column groups per round (the same loads as
    // preload_partials), so the tile is then stored like a whole one.  The
    // sum is acc + partial, as the chunk loop's would be.
    auto add_partial = [&](int c0, uint32_t t_acc) {
      constexpr int GR = BN / 32 < 4 ? BN / 32 : 4;
      const float4* src = reinterpret_cast<const float4*>(
          args.ws + static_cast<size_t>(c0 * UNIT_CTAS + rank) * BM * BN +
          static_cast<size_t>(quarter) * BN * EPI_ROWS) + lane;
#pragma unroll 1
      for (int c = 0; c < BN / 32; c += GR) {
        float4 v[8 * GR];
#pragma unroll
        for (int j = 0; j < 8 * GR; ++j) v[j] = __ldcg(src + static_cast<size_t>(c * 8 + j) * EPI_ROWS);
#pragma unroll
        for (int q = 0; q < GR; ++q) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_acc, r, (c + q) * 32);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f = v[8 * q + j];
            r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + f.x);
            r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + f.y);
            r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + f.z);
            r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + f.w);
          }
          tmem_st_32x32b_x32(t_acc, r, (c + q) * 32);
        }
      }
      tmem_st_wait();   // stored before the chunk loop reads the accumulator
    };

    float tb[BN / 32] = {};   // the current tile's column bias (see the tile loop)
    float trb = 0.0f;         // ... or this thread's row bias
    // Write one finished tile: TMEM -> registers (+ the other units' partial
    // sums when ADD: already summed in unit order in the TMEM buffer at t_part
    // when part_tmem, else loaded here from the scratch slots of units oc0 ..
    // oc0 + ncontrib - 1, whose flags are up, and summed in the same order) ->
    // alpha * acc + beta * C (C read here when rc) -> output.  hold: the
    // accumulator is not handed back here (the caller first writes the next
    // item's initial value into it).  Returns false if a wait gave up.
    auto store_tile = [&](auto add_tag, auto fused_tag, uint32_t t_row, uint32_t t_part, int nb,
                          int row0, int buf, bool rc, bool hold, bool part_tmem, int oc0,
                          int ncontrib) -> bool {
      constexpr bool ADD = decltype(add_tag)::value;
      constexpr bool FUSED = decltype(fused_tag)::value;   // bias / activation
#pragma unroll 1
      for (int c = 0; c < CHUNKS; ++c) {
        const int pc = c * CHUNK;   // column inside the tile (and in TMEM)
        const int col0 = nb * BN + pc;
        uint8_t* stg;
        if (!begin_chunk<PAIR, L::EPI_BUF_BYTES>(st, stg, &tmC, row0, col0, abort_flag, args, rc))
          return false;
        // A chunk that crosses the right edge of C when N * sizeof(out) is not a
        // multiple of 16 bytes is written with predicated plain stores (below):
        // the tensor store writes whole 16-byte pieces and would touch the
        // columns just past N.  Chunks entirely right of N are not stored at all.
        const bool ragged = args.n_ragged && (col0 + CHUNK > args.N);
        const bool skip_store = col0 >= args.N || row0 >= args.M;
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_row, v0, pc);
        if (CHUNK == 64) tmem_ld_32x32b_x32(t_row, v1, pc + 32);
        if (ADD && part_tmem) {
          uint32_t p0[32], p1[32];
          tmem_ld_32x32b_x32(t_part, p0, pc);
          if (CHUNK == 64) tmem_ld_32x32b_x32(t_part, p1, pc + 32);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v0[i] = __float_as_uint(__uint_as_float(v0[i]) + __uint_as_float(p0[i]));
            if (CHUNK == 64) v1[i] = __float_as_uint(__uint_as_float(v1[i]) + __uint_as_float(p1[i]));
          }
        } else if (ADD) {
          tmem_ld_wait();
          // this chunk's columns of the partials (slot layout [quarter][BN/4
          // pieces][32 rows][16 B]: 512 contiguous bytes per piece), 16 columns
          // at a time (few registers: the next tile's mainloop hides this
          // epilogue), summed in unit order and then added
          const float4* base = reinterpret_cast<const float4*>(args.ws) +
                               static_cast<size_t>(quarter) * BN * EPI_ROWS / 4 + lane;
#pragma unroll
          for (int h = 0; h < CHUNK / 16; ++h) {
            float4 sp[4];
#pragma unroll 1
            for (int k = 0; k < ncontrib; ++k) {
              const float4* src = base + static_cast<size_t>((oc0 + k) * UNIT_CTAS + rank) * (BM * BN / 4) +
                                  static_cast<size_t>(pc / 4 + 4 * h) * EPI_ROWS;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 f = __ldcg(src + j * EPI_ROWS);
                if (k == 0) {
                  sp[j] = f;
                } else {
                  sp[j].x += f.x;
                  sp[j].y += f.y;
                  sp[j].z += f.z;
                  sp[j].w += f.w;
                }
              }
            }
            uint32_t* vv = h < 2 ? v0 + 16 * h : v1 + 16 * (h - 2);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              vv[4 * j] = __float_as_uint(__uint_as_float(vv[4 * j]) + sp[j].x);
              vv[4 * j + 1] = __float_as_uint(__uint_as_float(vv[4 * j + 1]) + sp[j].y);
              vv[4 * j + 2] = __float_as_uint(__uint_as_float(vv[4 * j + 2]) + sp[j].z);
              vv[4 * j + 3] = __float_as_uint(__uint_as_float(vv[4 * j + 3]) + sp[j].w);
            }
          }
        } else {
          tmem_ld_wait();
        }
        if (c == CHUNKS - 1 && !hold) {
          // accumulator fully read: hand it back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader)
              mbar_arrive(&tempty[buf]);
            else
              mbar_arrive_cluster(map_to_rank(&tempty[buf], 0));
          }
        }
        uint8_t* rowp = stg + r * SW;
        if (FUSED) {
          // this chunk's column-bias registers (static selects: no local memory)
          float cb0 = 0.0f, cb1 = 0.0f;
#pragma unroll
          for (int q = 0; q < BN / 32; ++q) {
            if (q == pc / 32) cb0 = tb[q];
            if (CHUNK == 64 && q == pc / 32 + 1) cb1 = tb[q];
          }
          fused_chunk<OUT, CHUNK>(v0, v1, rowp, args, rc, cb0, cb1, trb, r);
        }
        // A ragged fp32 chunk is stored element by element from registers; a
        // ragged 16-bit one is staged like the others and copied out by rows
        // (copy_out_ragged): per-element 16-bit stores took 73 x 61 x 67 bf16
        // from 8.9 to 12.0 us, while for fp32 the direct stores measured as fast.
        const bool direct = OUT == OUT_F32 && ragged;
        if (FUSED && !direct) {
          // finished values (alpha, beta * C, bias and activation applied in
          // registers): cast and staged by the same branch-free shared stores
          stage_chunk_scaled<OUT, false>(v0, v1, smem_u32(rowp), 1.0f, r);
        } else if (!FUSED && !ADD && !rc && !direct) {
          // the common case, branch-free: alpha * acc, cast, one 16-byte
          // shared store per piece (per-piece branches slowed the stores ~1.6x)
          stage_chunk_scaled<OUT>(v0, v1, smem_u32(rowp), args.alpha, r);
        } else
#pragma unroll
        for (int j = 0; j < 8; ++j) {   // 16-byte pieces of the 128-byte row
          uint4* p = reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) << 4));
          constexpr int E = OUT == OUT_F32 ? 4 : 8;
          float x[E];
          const uint32_t* src = (OUT == OUT_F32) ? (v0 + 4 * j) : ((j < 4) ? (v0 + 8 * j) : (v1 + 8 * (j - 4)));
#pragma unroll
          for (int e = 0; e < E; ++e) x[e] = __uint_as_float(src[e]);
          if (FUSED)
            store_piece<OUT>(x, p, args, direct, !skip_store && row0 + r < args.M, row0 + r,
                             col0 + E * j);
          else
            finish_piece<OUT>(x, p, args, rc, direct, !skip_store && row0 + r < args.M, row0 + r,
                              col0 + E * j);
        }
        if (ragged && !direct && !skip_store) copy_out_ragged<OUT>(stg, args, row0, col0);
        end_chunk(st, stg, &tmC, row0, col0, ragged, skip_store);
      }
      return true;
    };
    // Hand accumulator buffer b back to the MMA issuer (after this warp's last
    // TMEM access to it).
    auto release_acc = [&](int b) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty[b]);
        else
          mbar_arrive_cluster(map_to_rank(&tempty[b], 0));
      }
    };
    // beta * C of item wp's tile (this warp's 32 rows) into accumulator buffer b,
    // the value its MMAs then accumulate onto.  Two column groups in flight.
    auto preload_c = [&](const WorkItem& wp, int b) {
      int mbp, nbp;
      tile_of(args, wp.tile, &mbp, &nbp);
      const int grow = mbp * TILE_M + static_cast<int>(rank) * BM + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(b * BN);
      constexpr int NQ = BN / 32;
      uint32_t va[32], vb[32];
      load_c32<OUT>(args, grow, nbp * BN, va);
#pragma unroll 1
      for (int q = 0; q < NQ; q += 2) {
        if (q + 1 < NQ) load_c32<OUT>(args, grow, nbp * BN + (q + 1) * 32, vb);
        tmem_st_32x32b_x32(taddr, va, q * 32);
        if (q + 2 < NQ) load_c32<OUT>(args, grow, nbp * BN + (q + 2) * 32, va);
        if (q + 1 < NQ) tmem_st_32x32b_x32(taddr, vb, (q + 1) * 32);
      }
      tmem_st_wait();
    };
    // The unit's items in order, looked at two ahead: item tl + 2 uses the same
    // accumulator buffer as item tl, and when it starts from beta * C this warp
    // writes that into the buffer after finishing item tl.
    WorkIter wq;
    work_begin(wq);
    WorkItem w, w1, w2;
    bool h0 = wq.next(&w);
    bool h1 = h0 && wq.next(&w1);
    bool h2 = false;
    for (; ok && h0; ++tl, w = w1, h0 = h1, w1 = w2, h1 = h2) {
      h2 = h1 && wq.next(&w2);
      const bool hold = h2 && item_preloads_c(args, tl + 2, w2);
      const bool rc = args.read_c && !item_preloads_c(args, tl, w);
      int mb, nb;
      tile_of(args, w.tile, &mb, &nb);
      const int buf = tl & 1;
      const uint32_t aph = (tl >> 1) & 1;
      if (args.epi) {
        // the tile's bias into registers while its mainloop runs: lane l holds
        // column nb * BN + 32 q + l in tb[q] (0 past N), or its row's value
        if (args.bias_kind == EPI_BIAS_COL) {
#pragma unroll
          for (int q = 0; q < BN / 32; ++q) {
            const int c = nb * BN + q * 32 + lane;
            tb[q] = c < args.N ? __ldg(args.bias + c) : 0.0f;
          }
        } else if (args.bias_kind == EPI_BIAS_ROW) {
          const int rr = mb * TILE_M + static_cast<int>(rank) * BM + quarter * 32 + lane;
          trb = rr < args.M ? __ldg(args.bias + rr) : 0.0f;
        }
      }
      // A work item that finishes its tile without holding all of its k-groups
      // owns the tile: the other units touching it leave partial sums, summed
      // in unit order and added to this item's accumulator.  When
      // the item is its unit's last (no data-parallel tiles follow, or a
      // split-tile unit), the other accumulator buffer is free: the partials
      // are summed into it while this item's MMAs run, and the chunk loop adds
      // them from there.  Otherwise the chunk loop loads them itself, in an
      // epilogue that the next tile's mainloop hides.
      const uint32_t t_part = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>((buf ^ 1) * BN);
      int ncontrib = 0, oc0 = 0;
      bool part_tmem = false;
      if (!SPLITK && item_finishes(args, w) && (w.g0 > 0 || w.g1 < args.groups)) {
        int c1;
        owner_contributors(args, unit0, unit_stride, w, &oc0, &c1);
        ncontrib = c1 - oc0;
        if (ncontrib > 0 && !h1) {
          if (!preload_partials(oc0, ncontrib, t_part)) {
            ok = false;
            break;
          }
          part_tmem = true;
        }
      }
      if (!wait_warp<PAIR>(&tfull[buf], aph, abort_flag, args, SITE_EPI_TMEM_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the C map's descriptor back in the TMA unit's cache before this tile's
      // stores (its prefetch at start-up may have been evicted long ago)
      if (ew == 0 && lane == 0) prefetch_tensormap(&tmC);
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(buf * BN);
      const int row0 = mb * TILE_M + static_cast<int>(rank) * BM + quarter * 32;
      if (SPLITK) {
        // Phase 1: this CTA's fp32 partial of every peer's column slice ->
        // this CTA's ring (idle: every MMA that read it has completed), one
        // contiguous [128 rows][SLICE] block per peer, 16-byte pieces
        // XOR-swizzled by row; the blocks are bulk-copied to the peers after
        // the cluster barrier (early exchange: each warp sends its rows at
        // once).  The CTA's own slice stays in TMEM.
        const int prow = quarter * 32 + r;
#pragma unroll 1
        for (int qi = 0; qi < SPLIT - 1; ++qi) {
          const int q = qi < static_cast<int>(srank) ? qi : qi + 1;
          const uint32_t sbase = smem_u32(smem) + static_cast<uint32_t>(qi * SLICE_BYTES);
          // 32 columns per TMEM load; a 16-column slice takes the first half of
          // one (the load stays inside the 2 x BN allocated columns)
          constexpr int LOADS = SLICE >= 32 ? SLICE / 32 : 1;
          constexpr int PIECES = SLICE >= 32 ? 8 : SLICE / 4;
#pragma unroll 1
          for (int c = 0; c < LOADS; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row, v, q * SLICE + c * 32);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < PIECES; ++j)
              st_shared_v4(slice_addr<SLICE>(sbase, prow, c * 8 + j),
                           make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
          }
        }
        fence_proxy_async_smem();   // read next by the bulk copies
        if (EARLY) push_rows();
        continue;   // one tile per split-K cluster; phase 2 follows
      }
      if (!item_finishes(args, w)) {
        // Stream-K segment (or split-tile part) that does not finish its tile: publish
        // the fp32 partial sum in this CTA's scratch slot, hand the accumulator
        // back, then release the CTA's flag with the launch epoch.  Such a
        // segment is the first (or only) one of its unit, so it is published
        // early.  Slot layout [quarter][BN/4 pieces][32 rows][4 floats]: each
        // group of 32 columns of a warp's rows is one contiguous 4 KB block,
        // staged in the warp's epilogue buffers (conflict-free rows) and written
        // with a bulk copy; each epilogue warp's rows form one contiguous span,
        // which the owner fetches with bulk copies.
        float* slot = args.ws + static_cast<size_t>(blockIdx.x) * BM * BN +
                      static_cast<size_t>(quarter) * BN * EPI_ROWS;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row, v, c * 32);
          tmem_ld_wait();
          uint8_t* stg = st.stage0 + (st.chunk_ctr & 1) * L::EPI_BUF_BYTES;
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
          const uint32_t sb = smem_u32(stg) + static_cast<uint32_t>(r * 16);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(sb + j * EPI_ROWS * 16, make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            bulk_store_s2g(slot + c * 32 * EPI_ROWS, smem_u32(stg), 32 * EPI_ROWS * 4);
            bulk_commit_group();
          }
          __syncwarp();
          ++st.chunk_ctr;
        }
        if (!hold) release_acc(buf);
        if (lane == 0) {
          bulk_wait_group<0>();          // the partial is written
          fence_proxy_async_global();    // the owner reads it with bulk copies
        }
        __threadfence();
        if (!epilogue_sync()) {
          ok = false;
          break;
        }
        if (ew == 0 && lane == 0) flag_release(args.ws_flags + blockIdx.x, args.epoch);
        if (hold) {
          preload_c(w2, buf);
          release_acc(buf);
        }
        continue;
      }
      if (ncontrib > 0 && !part_tmem) {   // the partials the chunk loop will load
        bool got = true;
        for (int k = 0; k < ncontrib && got; ++k)
          got = wait_flag_warp(args.ws_flags + (oc0 + k) * UNIT_CTAS + rank);
        if (!got) {
          ok = false;
          break;
        }
        if (ncontrib == 1) {   // one contributor: added in TMEM, in batched loads
          add_partial(oc0, t_row);
          ncontrib = 0;
        }
      }
      // one specialised chunk loop per case, chosen once per tile
      const BoolC<false> no;
      const BoolC<true> yes;
      if (ncontrib == 0)
        ok = args.epi ? store_tile(no, yes, t_row, 0u, nb, row0, buf, rc, hold, false, 0, 0)
                      : store_tile(no, no, t_row, 0u, nb, row0, buf, rc, hold, false, 0, 0);
      else
        ok = args.epi ? store_tile(yes, yes, t_row, t_part, nb, row0, buf, rc, hold, part_tmem, oc0, ncontrib)
                      : store_tile(yes, no, t_row, t_part, nb, row0, buf, rc, hold, part_tmem, oc0, ncontrib);
      if (ok && hold) {
        preload_c(w2, buf);
        release_acc(buf);
      }
    }
    // after an abort the rows are sent all the same, so the peer never waits
    // for a block that will not come
    if (EARLY && !pushed) push_rows();
    if (!SPLITK) {
      if (!ok && st.pending_cload >= 0 && lane == 0)
        wait_drain<PAIR>(&st.cload[st.pending_cload], st.pending_phase, args);
      // the staging buffers must be read out before the CTA exits; the grid's
      // completion makes the stores themselves visible
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
    }
  }

  if (EARLY && warp < EPI_WARP0) {   // the start-up cluster barrier, for the other roles
    __syncwarp();
    cluster_wait();
  }
  if (PAIR && warp == 0) {   // phase 2 of the start-up barrier, for the producer
    __syncwarp();
    cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (SPLITK) {
    // Phase 2.  CTA `srank` finishes columns [srank*SLICE, (srank+1)*SLICE) of
    // the tile: after the cluster barrier (every CTA's blocks staged and its ring
    // idle) each CTA bulk-copies its block for every peer into that peer's
    // receive area, counted on the peer's rfull; then it sums its own slice
    // (from TMEM) and the received ones in rank order (deterministic) and
    // finishes them like the plain epilogue.  The copies are sent even after an
    // abort, so a peer never waits for a block that will not come.
    // (The early exchange has sent its block already: its receive area is the
    // staging area, and the final chunks stage in the ring after the send area.)
    constexpr uint32_t RECV0 = EARLY ? static_cast<uint32_t>(L::off_epi)
                                     : (SPLIT - 1) * SLICE_BYTES;   // receive area
    if (!EARLY && threadIdx.x == 0) mbar_arrive_expect_tx(rfull, (SPLIT - 1) * SLICE_BYTES);
    if (!EARLY) cluster_sync();
    if (!EARLY && threadIdx.x == 0) {
      const uint32_t base = smem_u32(smem);
      for (int qi = 0; qi < SPLIT - 1; ++qi) {
        const uint32_t q = qi < static_cast<int>(srank) ? qi : qi + 1;
        const uint32_t slot = srank < q ? srank : srank - 1;   // this CTA among q's peers
        bulk_copy_s2cluster(map_addr_to_rank(base + RECV0 + slot * SLICE_BYTES, q),
                            base + static_cast<uint32_t>(qi) * SLICE_BYTES, SLICE_BYTES,
                            map_addr_to_rank(smem_u32(rfull), q));
      }
    }
    bool received = false;
    if (warp >= EPI_WARP0 && !*abort_flag && unit0 < args.num_tiles) {
      const int ew = warp - EPI_WARP0;
      const int quarter = warp & 3;
      const int r = lane;
      uint8_t* const stage0 = EARLY ? smem + SLICE_BYTES : smem + L::off_epi;
      EpiState st{stage0 + ew * EPI_BUFS * L::EPI_BUF_BYTES, &cload[ew * EPI_BUFS], 0, -1, 0};
      int mb, nb;
      tile_of(args, unit0, &mb, &nb);
      const int row0 = mb * BM + quarter * 32;
      const int prow = quarter * 32 + r;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      const uint32_t rbase = smem_u32(smem) + RECV0;
      // the first chunk's bias is loaded before the wait for the peers' slices
      // (the loads' round trip overlaps it)
      EpiBias eb0{0.0f, 0.0f, 0.0f, 0.0f};
      if (args.epi) eb0 = load_epi_bias<CHUNK>(args, nb * BN + static_cast<int>(srank) * SLICE, row0 + r);
      bool ok = wait_warp<true>(rfull, 0, abort_flag, args, SITE_SPLITK_SLICES);
      received = ok;
      // chunks of PCH columns: whole epilogue chunks, or one slice narrower than a
      // chunk, finished through the predicated direct stores of a ragged edge
      constexpr int PCH = SLICE < CHUNK ? SLICE : CHUNK;
      constexpr bool NARROW = PCH < CHUNK;
      constexpr int PIECES = PCH * (OUT == OUT_F32 ? 4 : 2) / 16;   // 16-byte pieces per row
#pragma unroll 1
      for (int c = 0; ok && c < SLICE / PCH; ++c) {
        const int tcol = static_cast<int>(srank) * SLICE + c * PCH;   // column inside the tile
        const int col0 = nb * BN + tcol;
        EpiBias eb = eb0;
        if (args.epi && c > 0) eb = load_epi_bias<CHUNK>(args, col0, row0 + r);
        uint8_t* stg;
        if (!begin_chunk<true, L::EPI_BUF_BYTES>(st, stg, &tmC, row0, col0, abort_flag, args,
                                                 args.read_c)) {
          ok = false;
          break;
        }
        const bool ragged = NARROW || (args.n_ragged && (col0 + CHUNK > args.N));
        const bool skip_store = col0 >= args.N || row0 >= args.M;
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_row, v0, tcol);
        if (PCH == 64) tmem_ld_32x32b_x32(t_row, v1, tcol + 32);
        tmem_ld_wait();
        uint8_t* rowp = stg + r * SW;
        constexpr int E = OUT == OUT_F32 ? 4 : 8;   // outputs per 16-byte piece
#pragma unroll
        for (int j = 0; j < PIECES; ++j) {
          const uint32_t* own = (OUT == OUT_F32) ? (v0 + 4 * j) : ((j < 4) ? (v0 + 8 * j) : (v1 + 8 * (j - 4)));
          float x[E];
#pragma unroll
          for (int e = 0; e < E; ++e) x[e] = 0.0f;
#pragma unroll
          for (int q = 0; q < SPLIT; ++q) {
            if (q == static_cast<int>(srank)) {
#pragma unroll
              for (int e = 0; e < E; ++e) x[e] += __uint_as_float(own[e]);
            } else {
              const uint32_t blk = rbase + static_cast<uint32_t>((q < static_cast<int>(srank) ? q : q - 1) * SLICE_BYTES);
#pragma unroll
              for (int h = 0; h < E / 4; ++h) {
                const uint4 pv = ld_shared_v4(slice_addr<SLICE>(blk, prow, (c * PCH + E * j) / 4 + h));
                x[4 * h + 0] += __uint_as_float(pv.x);
                x[4 * h + 1] += __uint_as_float(pv.y);
                x[4 * h + 2] += __uint_as_float(pv.z);
                x[4 * h + 3] += __uint_as_float(pv.w);
              }
            }
          }
          uint4* p = reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) << 4));
          if (args.epi)
            finish_piece<OUT, true>(x, p, args, args.read_c, ragged, !skip_store && row0 + r < args.M,
                                    row0 + r, col0 + E * j, eb, E * j);
          else
            finish_piece<OUT, false>(x, p, args, args.read_c, ragged,
                                     !skip_store && row0 + r < args.M, row0 + r, col0 + E * j);
        }
        end_chunk(st, stg, &tmC, row0, col0, ragged, skip_store);
      }
      if (!ok && st.pending_cload >= 0 && lane == 0)
        wait_drain<true>(&st.cload[st.pending_cload], st.pending_phase, args);
      // the staging buffers must be read out before the CTA exits; the grid's
      // completion makes the stores themselves visible
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
    }
    // blocks still landing in this CTA's ring must arrive before it exits
    if (warp == EPI_WARP0 && lane == 0 && !received) wait_drain<true>(rfull, 0, args);
    tc_fence_before();
    __syncthreads();
  }
  if (*abort_flag) {
    // Some role gave up.  Before TMEM is freed and the CTA exits, every
    // asynchronous operation this CTA started must have finished:
    if (warp == 0 && lane == 0) {
      if (leader) {
        // the copies of the last STAGES ring iterations (older slots were
        // consumed and re-armed), except an iteration deliberately left unarmed;
        // in pair mode these phases also count the peer's copies
        const uint32_t it = producer_iters;
        const uint32_t lo = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0;
        for (uint32_t j = lo; j < it; ++j) {
          if (args.inject_skip != 0 && j + 1 == static_cast<uint32_t>(args.inject_skip)) continue;
          wait_drain<PAIR>(&full[j % STAGES], (j / STAGES) & 1, args);
        }
      } else {
        // the odd CTA's copies complete on the leader's barrier, which it cannot
        // wait on: give copies in flight a bounded grace period to land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    if (warp == 1 && lane == 0 && leader) {
      // every MMA already issued (a commit with nothing pending arrives at once)
      if (PAIR)
        umma_commit_pair_multicast(drain, 0x1);
      else
        umma_commit(drain);
      wait_drain<PAIR>(drain, 0, args);
    }
  }
  if (CLUSTERED) {
    // no CTA may free TMEM or exit while a peer can still signal its barriers
    // or read its shared memory
    tc_fence_before();
    cluster_sync();
  }
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// C <- act(beta * C + bias) (beta * C taken as 0 when beta == 0, without reading
// C): the K == 0 case.
template <int OUT>
__global__ void scale_c_kernel(void* C, long long ldc, int M, int N, float beta, const float* bias,
                               int bias_kind, int act) {
  const long long total = static_cast<long long>(M) * N;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / N, c = i % N;
    const long long o = r * ldc + c;
    float x = 0.0f;
    if (beta != 0.0f) {
      if (OUT == OUT_F32)
        x = beta * static_cast<const float*>(C)[o];
      else if (OUT == OUT_BF16)
        x = beta * __bfloat162float(static_cast<const __nv_bfloat16*>(C)[o]);
      else
        x = beta * __half2float(static_cast<const __half*>(C)[o]);
    }
    if (bias_kind == EPI_BIAS_COL) x += bias[c];
    else if (bias_kind == EPI_BIAS_ROW) x += bias[r];
    if (act == EPI_ACT_RELU) x = x < 0.0f ? 0.0f : x;
    if (OUT == OUT_F32)
      static_cast<float*>(C)[o] = x;
    else if (OUT == OUT_BF16)
      static_cast<__nv_bfloat16*>(C)[o] = __float2bfloat16_rn(x);
    else
      static_cast<__half*>(C)[o] = __float2half_rn(x);
  }
}

}  // namespace gemm_tc
