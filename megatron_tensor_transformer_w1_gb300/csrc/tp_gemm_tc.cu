// tp_gemm_tc.cu -- the tensor-core GEMM of every bf16 shard computation.
//
// Blackwell (sm_103a) design, written for this library:
//   * one persistent CTA per SM, 192 or 320 threads in three roles:
//       warp 0      : TMA producer (one elected lane) -- cp.async.bulk.tensor
//                     3-D tiled loads, 128-byte swizzle, into a STAGES-deep
//                     shared-memory ring guarded by mbarriers;
//       warp 1      : allocates tensor memory, and one lane issues
//                     tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M=128,
//                     N=BN, K=16 per instruction) and tcgen05.commit;
//       warps 2..   : epilogue (4, or 8 for the backward epilogues) --
//                     tcgen05.ld of the fp32 accumulator (warp w reads TMEM
//                     lanes 32*(w%4)..; with 8, two warps per lane quarter
//                     split the columns), fused activation or derivative,
//                     then the results: staged in shared memory and written
//                     with TMA stores (the two-SM pair kernel's epilogues,
//                     except the GELU backward one), or 16-byte stores from
//                     the threads (the one-SM kernel, the GELU backward
//                     epilogue, and TPFFN_TMA_STORE=0);
//   * the accumulator is double-buffered in tensor memory (2 x BN columns),
//     so the epilogue of one tile overlaps the MMA K-loop of the next;
//   * every wait on an mbarrier is bounded: after the time limit the waiting
//     thread sets the device error word and a CTA-wide abort flag, every role
//     leaves its loop, in-flight copies and MMAs are drained with bounded
//     waits, and tensor memory is freed before the CTA exits.
//
// Operand majorness: K-major tiles are one TMA box {64 (K), rows} and use the
// canonical 128B-swizzle K-major layout (8-row atoms of 1024 B, SBO = 1024,
// K advanced inside the atom by 32 B per MMA).  MN-major tiles are boxes
// {64 (M or N), 64 (K)}: 128-byte rows along M/N, one 8 KB box per 64 M/N
// (LBO = 8192 between boxes, SBO = 1024 between 8-row K groups, K advanced by
// 2048 B per MMA).  MN-major serves the backward GEMMs that contract over the
// hidden or token dimension without transposing any buffer.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"
#include "tp_act.cuh"
#include "tp_internal.h"
#include "tpffn.h"

namespace tpffn {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;
// Epilogue warps per CTA: 8 (two per TMEM lane quarter, each taking half the
// columns) for the backward epilogues, whose global loads of the saved
// activations are latency-bound; 4 for the others, whose arithmetic would
// otherwise take issue slots from the producer and MMA threads.
template <int EPI>
__host__ __device__ constexpr int epi_warps() {
  return (EPI == EPI_SWIGLU_BWD || EPI == EPI_GELU_BWD) ? 8 : 4;
}
template <int EPI>
__host__ __device__ constexpr int threads_for() {
  return 64 + 32 * epi_warps<EPI>();  // producer, MMA, epilogue
}

struct Params {
  int M, N, K;
  int NB, G;
  int tiles_m, tiles_n, k_blocks;
  int a_bsel, a_gsel, b_bsel, b_gsel;
  int a_swap, b_swap;  // 0: {inner, rows, batch}; 1: {inner, batch, rows}; 2: 4-D MN-major groups
  void* out;
  long long out_bs, out_rs;
  void* out2;
  long long out2_bs, out2_rs;
  const void* aux;
  long long aux_bs, aux_rs;
  const __nv_bfloat16* bias;
  long long bias_bs, bias_len;
  long long n_store;
  int* err;
  unsigned long long timeout_ns;
  int debug_skip;
  int dbg_slot;  // launch slot of the optional wait counters (instrumented builds only)
  int ksplit;    // K split into this many parts (1: none; fp32 parts only)
  int raster;    // pair kernel tile order (RASTER_*)
  int o_swap;    // pair kernel TMA stores: output maps are {cols, batch, rows} (batch stride < row stride)
  int out_cs, b_cs;  // pair kernel: shards merged along N (see GemmSpec), 0: off
  int tail_tiles, tail_parts;  // pair kernel: the last tail_tiles tiles run as tail_parts K parts (0: off)
  int dep_mode;  // programmatic dependent launch: 1 wait for the previous kernel, then let the next
                 // one launch; 2 no wait at the start (reads nothing the previous kernel writes),
                 // wait before exit; 0 let the next one launch, then wait (for comparisons)
  int keep_op;   // pair kernel: operand every batch shares (1: A, 2: B, 0: none); the other one
                 // streams through L2 with evict_first priority
};

// Pair-kernel tile orders.  Grouped raster order (the default) lets the
// roughly 8 x 9.5 tiles that run at the same time share both operands' K
// slabs through L2.  The other two orders walk the operand that every shard
// shares fastest, over its whole extent, hoping it stays resident in L2 across
// the launch; measured on the Llama-3-8B step they read more from DRAM, not
// less (up 1.23 -> 2.12 GB, dh 1.71 -> 2.44 GB: the shared operand does not
// survive a wave in L2) and were slower for up and dh (1648 -> 1598,
// 1448 -> 1338 TFLOP/s), so they are opt-in (TPFFN_RASTER=1) for comparisons.
// Programmatic dependent launch.  A dependent grid launches once every CTA
// of this grid has called launch_dependents (or exited).  Mode 1 (default):
// wait until the previous kernel has completed and its writes are visible,
// then let the next kernel launch -- so that whenever a kernel starts, every
// kernel before its predecessor has completed.  Mode 2, for a GEMM that
// neither reads nor writes anything written by its predecessor or by
// another mode-2 GEMM right before it (the weight gradients after the dx
// GEMM): let the next kernel launch and start without waiting, so that its
// CTAs fill the SMs the predecessor's last wave leaves idle; one thread per
// CTA waits before the CTA exits, so that its completion still implies its
// predecessor's.  Mode 0: the former order (next kernel first, then wait),
// for comparisons.
__device__ __forceinline__ void dep_prologue(int mode) {
  if (mode == 1) {
    grid_dep_wait();
    grid_dep_launch();
  } else {
    grid_dep_launch();
    if (mode == 0) grid_dep_wait();
  }
}
__device__ __forceinline__ void dep_epilogue(int mode) {
  if (mode == 2 && threadIdx.x == 0) grid_dep_wait();
}

constexpr int RASTER_GROUPED = 0;  // groups of 8 M blocks, N within a group
constexpr int RASTER_M_FAST = 1;   // A shared by every batch: all M blocks of one N block in turn
constexpr int RASTER_N_FAST = 2;   // B shared by every batch: all N blocks of one M block in turn

// Work unit u of the one-SM kernel: tile u mod (tiles per split) over its
// part u / (tiles per split) of the K blocks -- [kb0, kb0 + nkb).
__device__ __forceinline__ int unit_split(const Params& p, int u, int& tile, int& kb0, int& nkb) {
  const int per = p.tiles_m * p.tiles_n * p.NB;
  const int kh = p.ksplit > 1 ? u / per : 0;
  tile = u - kh * per;
  const int kbs = (p.k_blocks + p.ksplit - 1) / p.ksplit;
  kb0 = kh * kbs;
  nkb = min(p.k_blocks - kb0, kbs);
  return kh;
}

// Bounded wait (see wait_bounded_raw).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             const Params& p, bool honour_abort = true) {
  return wait_bounded_raw(bar, parity, abort_flag, p.err, p.timeout_ns, honour_abort);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9, 10-12 = 1), transpose (MN-major) bits 15/16, N>>3 at 17, M>>4 at 24.
template <int BN, bool AMN, bool BMN>
__device__ __forceinline__ constexpr uint32_t instr_desc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(AMN) << 15) |
         (static_cast<uint32_t>(BMN) << 16) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* dst, const float* v) {
  uint4 q;
  q.x = pack_bf16x2(v[0], v[1]);
  q.y = pack_bf16x2(v[2], v[3]);
  q.z = pack_bf16x2(v[4], v[5]);
  q.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(dst) = q;
}
__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* src, float* v) {
  uint4 q = *reinterpret_cast<const uint4*>(src);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 q, float* v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// ------------------------------------------------------------ tile order
__device__ __forceinline__ void decode_tile(const Params& p, int tile, int& b, int& mb, int& nb) {
  const int tpb = p.tiles_m * p.tiles_n;
  b = tile / tpb;
  const int r = tile - b * tpb;
  constexpr int GM = 8;  // m-blocks per raster group (L2 reuse of B tiles)
  const int group = r / (GM * p.tiles_n);
  const int first_m = group * GM;
  const int gm = min(p.tiles_m - first_m, GM);
  const int in_group = r - group * GM * p.tiles_n;
  mb = first_m + in_group % gm;
  nb = in_group / gm;
}

// ------------------------------------------------------------ epilogues
// One thread owns one output row of the tile; `taddr` points at its TMEM
// lane and the first column of the accumulator buffer.
// `part` selects which share of the tile's columns this warp handles when a
// TMEM lane quarter is served by two epilogue warps (part is 0 with one).
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(const Params& p, int b, int row, bool row_ok, int n0, int nb,
                                              uint32_t taddr, int part) {
  constexpr int NSPLIT = epi_warps<EPI>() / 4;
  if constexpr (EPI == EPI_SWIGLU_FWD) {
    static_assert(BN == 256, "SwiGLU forward tiles hold 128 a-columns then 128 g-columns");
    __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(p.out) + b * p.out_bs + (long long)row * p.out_rs;
    __nv_bfloat16* sv = p.out2 ? static_cast<__nv_bfloat16*>(p.out2) + b * p.out2_bs + (long long)row * p.out2_rs
                               : nullptr;
#pragma unroll 1
    for (int c = part * (4 / NSPLIT); c < (part + 1) * (4 / NSPLIT); ++c) {
      uint32_t ra[32], rg[32];
      __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
      tmem_ld32(taddr + c * 32, ra);
      tmem_ld32(taddr + 128 + c * 32, rg);
      tmem_wait_ld();
      if (row_ok) {
        const int hcol = nb * 128 + c * 32;  // hidden unit within the shard
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float h[8], a[8], g[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            a[j] = __uint_as_float(ra[q * 8 + j]);
            g[j] = __uint_as_float(rg[q * 8 + j]);
            h[j] = a[j] * sigmoid_f(a[j]) * g[j];
          }
          store_bf16x8(hout + hcol + q * 8, h);
          if (sv) {
            store_bf16x8(sv + nb * 256 + c * 32 + q * 8, a);
            store_bf16x8(sv + nb * 256 + 128 + c * 32 + q * 8, g);
          }
        }
      }
    }
    return;
  } else {
#pragma unroll 1
    for (int c = part * (BN / 32 / NSPLIT); c < (part + 1) * (BN / 32 / NSPLIT); ++c) {
      uint32_t r[32];
      __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
      tmem_ld32(taddr + c * 32, r);
      tmem_wait_ld();
      const int nc = n0 + c * 32;
      if (!row_ok || nc >= p.n_store) continue;  // no warp-collective op follows in this iteration
      // the chunk's 32 bias values, read once (one round trip per chunk)
      float bv[32];
      if constexpr (EPI == EPI_OUT || EPI == EPI_GELU_FWD) {
        if (p.bias) {
          const __nv_bfloat16* bp = p.bias + b * p.bias_bs + nc;
          if (nc + 32 <= p.bias_len && (reinterpret_cast<uintptr_t>(bp) & 15) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) load_bf16x8(bp + q * 8, bv + q * 8);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) bv[j] = nc + j < p.bias_len ? __bfloat162float(bp[j]) : 0.f;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = nc + q * 8;
        if (n >= p.n_store) break;  // n_store is a multiple of 8
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[q * 8 + j]);
        if constexpr (EPI == EPI_F32) {
          float* o = static_cast<float*>(p.out) + b * p.out_bs + (long long)row * p.out_rs + n;
          *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4*>(o + 4) = make_float4(v[4], v[5], v[6], v[7]);
        } else if constexpr (EPI == EPI_OUT) {
          if (p.bias) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] += bv[q * 8 + j];
          }
          store_bf16x8(static_cast<__nv_bfloat16*>(p.out) + b * p.out_bs + (long long)row * p.out_rs + n, v);
        } else if constexpr (EPI == EPI_GELU_FWD) {
          if (p.bias) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] += bv[q * 8 + j];
          }
          if (p.out2)
            store_bf16x8(static_cast<__nv_bfloat16*>(p.out2) + b * p.out2_bs + (long long)row * p.out2_rs + n, v);
          float h[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) h[j] = gelu_tanh_f(v[j]);
          store_bf16x8(static_cast<__nv_bfloat16*>(p.out) + b * p.out_bs + (long long)row * p.out_rs + n, h);
        } else if constexpr (EPI == EPI_GELU_BWD) {
          float z[8];
          load_bf16x8(static_cast<const __nv_bfloat16*>(p.aux) + b * p.aux_bs + (long long)row * p.aux_rs + n, z);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] *= gelu_tanh_grad_f(z[j]);
          store_bf16x8(static_cast<__nv_bfloat16*>(p.out) + b * p.out_bs + (long long)row * p.out_rs + n, v);
        } else if constexpr (EPI == EPI_SWIGLU_BWD) {
          // hidden unit n lives in 128-block n>>7 of the interleaved [a|g] rows
          const long long col = (long long)(n >> 7) * 256 + (n & 127);
          const __nv_bfloat16* ag =
              static_cast<const __nv_bfloat16*>(p.aux) + b * p.aux_bs + (long long)row * p.aux_rs + col;
          float a[8], g[8], da[8], dg[8];
          load_bf16x8(ag, a);
          load_bf16x8(ag + 128, g);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float sg = sigmoid_f(a[j]);
            dg[j] = v[j] * a[j] * sg;                          // dh * silu(a)
            da[j] = v[j] * g[j] * sg * (1.0f + a[j] * (1.0f - sg));  // dh * g * silu'(a)
          }
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + b * p.out_bs + (long long)row * p.out_rs + col;
          store_bf16x8(o, da);
          store_bf16x8(o + 128, dg);
        }
      }
    }
  }
}

// ------------------------------------------------------------ the kernel
// AR: rows of A staged per K block.  Decode-sized token counts stage only
// their 32 rows; the M = 128 product still reads 128 rows of A, and rows
// 32..127 then come from the B tile that follows in the same stage -- rows
// whose outputs are never stored (each output row depends on its A row
// only).  The stage shrinks from 48 to 36 KB, so six stages instead of four
// keep 50 % more weight bytes in flight per SM.
template <int BN, int STAGES, int AR = BM>
struct Layout {
  static constexpr int A_BYTES = AR * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert((2 * STAGES + 5) * 8 <= 232, "barrier area");
  static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM columns");
};

template <int BN, int STAGES, int EPI, bool AMN, bool BMN, int AR = BM>
__global__ void __launch_bounds__(threads_for<EPI>(), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const Params p) {
  using L = Layout<BN, STAGES, AR>;
  static_assert(AR == BM || (!AMN && AR % 8 == 0 && L::STAGE_BYTES >= BM * BK * 2),
                "a short A tile is K-major and the product's 128 rows stay inside the stage");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 244);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], epi_warps<EPI>());  // one arrive per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // launched as a programmatic dependent of the previous kernel (decode-sized
  // GEMMs): everything above overlapped its tail; no global memory is touched
  // before its results are visible
  dep_prologue(p.dep_mode);

  const int num_tiles = p.tiles_m * p.tiles_n * p.NB * p.ksplit;  // work units
  const int k_iters_all = p.G * p.k_blocks;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_issue_phase[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) last_issue_phase[s] = -1;
      bool ok = true;
      const uint64_t pol_stream = l2_policy_evict_first();
      for (int unit = blockIdx.x; unit < num_tiles && ok; unit += gridDim.x) {
        int tile, kb0, k_iters;
        unit_split(p, unit, tile, kb0, k_iters);
        if (p.ksplit == 1) k_iters = k_iters_all;
        int b, mb, nb;
        decode_tile(p, tile, b, mb, nb);
        const int m0 = mb * BM, n0 = nb * BN;
        for (int it = 0; it < k_iters; ++it) {
          const int g = it / p.k_blocks;
          const int k0 = (kb0 + it - g * p.k_blocks) * BK;
          if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p)) {
            ok = false;
            break;
          }
          const bool skip = p.debug_skip && unit == (int)blockIdx.x && it == 0;
          if (!skip) {
            uint8_t* sA = smem + stage * L::STAGE_BYTES;
            uint8_t* sB = sA + L::A_BYTES;
            mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
            const int ab = b * p.a_bsel + g * p.a_gsel;
            const int bb = b * p.b_bsel + g * p.b_gsel;
            if (!AMN) {
              tma_load_3d(sA, &tmA, &full[stage], k0, p.a_swap ? ab : m0, p.a_swap ? m0 : ab);
            } else {
              if (p.a_swap == 2)
                tma_load_4d(sA, &tmA, &full[stage], 0, k0, m0 / 64, ab);
              else
#pragma unroll
                for (int i = 0; i < BM / 64; ++i)
                  tma_load_3d(sA + i * 8192, &tmA, &full[stage], m0 + 64 * i, p.a_swap ? ab : k0,
                              p.a_swap ? k0 : ab);
            }
            if (!BMN && p.keep_op == 1) {
              // weights read once (decode): evicted from L2 first
              tma_load_3d_hint(sB, &tmB, &full[stage], k0, p.b_swap ? bb : n0, p.b_swap ? n0 : bb, pol_stream);
            } else if (!BMN) {
              tma_load_3d(sB, &tmB, &full[stage], k0, p.b_swap ? bb : n0, p.b_swap ? n0 : bb);
            } else {
              if (p.b_swap == 2)
                tma_load_4d(sB, &tmB, &full[stage], 0, k0, n0 / 64, bb);
              else
#pragma unroll
                for (int i = 0; i < BN / 64; ++i)
                  tma_load_3d(sB + i * 8192, &tmB, &full[stage], n0 + 64 * i, p.b_swap ? bb : k0,
                              p.b_swap ? k0 : bb);
            }
            last_issue_phase[stage] = static_cast<int>(phase);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every issued copy must have landed before the CTA may exit.
#pragma unroll 1
      for (int s = 0; s < STAGES; ++s)
        if (last_issue_phase[s] >= 0)
          wait_bounded(&full[s], static_cast<uint32_t>(last_issue_phase[s]), abort_flag, p, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = instr_desc<BN, AMN, BMN>();
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < num_tiles && ok; unit += gridDim.x, ++local) {
        int tile, kb0, k_iters;
        unit_split(p, unit, tile, kb0, k_iters);
        if (p.ksplit == 1) k_iters = k_iters_all;
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!wait_bounded(&tempty[buf], (use & 1u) ^ 1u, abort_flag, p)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int it = 0; it < k_iters; ++it) {
          if (!wait_bounded(&full[stage], phase, abort_flag, p)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * L::STAGE_BYTES);
          const uint32_t b_addr = a_addr + L::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d_tmem, smem_desc<AMN>(a_addr, k), smem_desc<BMN>(b_addr, k), IDESC,
                      (it > 0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);  // accumulator ready for the epilogue
      }
      // Drain: all issued MMAs complete before tensor memory is released.
      umma_commit(drain);
      wait_bounded(drain, 0u, abort_flag, p, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps 2..9
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    int local = 0;
    for (int unit = blockIdx.x; unit < num_tiles; unit += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!wait_bounded(&tfull[buf], use & 1u, abort_flag, p)) break;
      tc_fence_after();
      int tile, kb0, nkb;
      const int kh = unit_split(p, unit, tile, kb0, nkb);
      int b, mb, nb;
      decode_tile(p, tile, b, mb, nb);
      b += kh * p.NB;  // K part kh: fp32 batch kh * NB + b (EPI_F32 only)
      const int row = mb * BM + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(buf * BN);
      epilogue_tile<BN, EPI>(p, b, row, row < p.M, nb * BN, nb, taddr, (warp - 2) >> 2);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
  dep_epilogue(p.dep_mode);
}

// ------------------------------------------------------------ 2-SM pair kernel
//
// Two CTAs of a cluster (one per SM) compute one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): CTA r holds rows
// [128r, 128r + 128) of the A tile and rows [128r, 128r + 128) of the B tile
// (its half of N) in its own shared memory; the leader CTA (rank 0) issues the
// MMAs, which read A from both CTAs and B from both halves and write each
// CTA's 128 output rows into that CTA's tensor memory.  Each SM therefore
// stages 32 KB per K step of 64 instead of 48 KB, which leaves room for 7
// stages (more latency hidden) and reads a third less from L2 per SM.
//
// Barriers: TMA copies of both CTAs complete on the leader's full[] barrier
// (cp.async.bulk.tensor .cta_group::2 with the leader's barrier address),
// which only the leader arms (expect-tx for both CTAs' bytes);
// the leader's commits arrive on empty[] and tfull[] of both CTAs
// (multicast); both CTAs' epilogue warps arrive on the leader's tempty[].
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_smem), "r"(rank));
  return remote;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(void* dst, const CUtensorMap* tm, uint32_t leader_bar, int c0,
                                                 int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(leader_bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* tm, uint32_t leader_bar, int c0,
                                                 int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(leader_bar)
      : "memory");
}
// The same copies with an L2 cache policy (createpolicy) attached.
__device__ __forceinline__ void tma_load_4d_pair_hint(void* dst, const CUtensorMap* tm, uint32_t leader_bar, int c0,
                                                      int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(leader_bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair_hint(void* dst, const CUtensorMap* tm, uint32_t leader_bar, int c0,
                                                      int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(leader_bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {  // arrive on bar in both CTAs
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void umma_commit_pair_local(uint64_t* bar) {  // arrive on this CTA's bar
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

#ifdef TPFFN_INSTRUMENT
// Per-CTA cycle counters for performance investigations (not in normal builds):
// [0] MMA wait on full, [1] MMA wait on tempty, [2] MMA thread total,
// [3] producer wait on empty, [4] epilogue wait on tfull, [5] epilogue total, [6] k-iterations
__device__ unsigned long long g_tpffn_dbg[8][256][8];  // [launch slot][CTA][counter]
static int g_dbg_launch = 0;                           // pair-GEMM launches since the last clear
#define DBG_T0() const long long _t0 = clock64()
#define DBG_ADD(slot, since) \
  atomicAdd(&g_tpffn_dbg[p.dbg_slot & 7][blockIdx.x & 255][slot], (unsigned long long)(clock64() - (since)))
#else
#define DBG_T0()
#define DBG_ADD(slot, since)
#endif

constexpr int PAIR_BN = 256;   // N of the pair tile (each CTA stages half of it)

// The backward epilogues read saved activations (z, or a|g) for every output
// element.  Fetched by the epilogue threads themselves, one row per thread,
// those loads slowed the tensor pipe of the same SM by ~15 % (measured: the
// same kernel with the loads removed ran 1250 -> 1480 TFLOP/s, with the
// arithmetic kept); staged by TMA into shared memory they cost little.  Each
// epilogue warp owns a 4 KB slot: per 32-column chunk of its 32 rows, the
// 32 x 32 bf16 block of z (2 KB), or of a and of g (2 x 2 KB), with 64-byte
// swizzle.  The slots take one operand stage.
template <int EPI>
__host__ __device__ constexpr bool aux_staged() {
  return EPI == EPI_SWIGLU_BWD || EPI == EPI_GELU_BWD;
}

// Pair-kernel store modes: TM 0 stores from registers, TM 1 stages boxes for
// TMA stores, TM 2 does so with eight epilogue warps (two per TMEM lane
// quarter, each taking half of a tile's columns) for the forward epilogues of
// GEMMs whose K loop is too short to hide a four-warp epilogue.
template <int EPI, int TM>
__host__ __device__ constexpr int pair_epi_warps() {
  return TM == 2 ? 8 : epi_warps<EPI>();
}
template <int EPI, int TM>
__host__ __device__ constexpr int pair_threads() {
  return 64 + 32 * pair_epi_warps<EPI, TM>();
}

// Epilogues that write their tile through shared memory with TMA stores:
// each epilogue warp stages its 32 rows x 32 columns per output in an 8 KB
// buffer (64-byte swizzled bf16 boxes, 128-byte swizzled fp32 boxes) and one
// lane stores them as whole lines, instead of 32 rows x 16 bytes per store
// instruction from the threads.  The buffers take one operand stage.
constexpr int OUT_BUF = 8192;  // per epilogue warp

// With TMA stores the backward epilogues give each warp two slots: the next
// chunk's saved activations land in one while the other, once read, takes
// the current chunk's results for the store.  A slot holds a 32 x 32 block of
// a and one of g (4 KB, SwiGLU) or one of z (2 KB, GELU); the SwiGLU slots take
// two operand stages (five remain), the GELU slots one.
template <int EPI, int TM>
struct PairLayout {
  static constexpr bool AUX = aux_staged<EPI>();
  static constexpr bool TMA = TM != 0;
  static constexpr int STAGES = AUX ? ((TMA && EPI == EPI_SWIGLU_BWD) ? 5 : 6) : (TM == 2 ? 5 : (TMA ? 6 : 7));
  static constexpr int A_BYTES = BM * BK * 2;               // this CTA's 128 rows of A
  static constexpr int B_BYTES = (PAIR_BN / 2) * BK * 2;    // this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;     // 32 KB
  static constexpr int AUX_SLOT = EPI == EPI_SWIGLU_BWD ? 4096 : 2048;  // one slot
  static constexpr int SLOTS = AUX ? (TMA ? 2 : 1) : 0;     // slots per epilogue warp
  static constexpr int AUX_OFF = STAGES * STAGE_BYTES;
  static constexpr int AUX_BYTES = AUX ? epi_warps<EPI>() * SLOTS * AUX_SLOT : (TMA ? pair_epi_warps<EPI, TM>() * OUT_BUF : 0);
  static constexpr int BAR_OFF = AUX_OFF + AUX_BYTES;
  static constexpr int BAR_AREA = 512;  // barriers, then the TMEM address and the abort flag at 496, 500
  static constexpr int SMEM = BAR_OFF + BAR_AREA + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * PAIR_BN;
  // full/empty per stage, tfull/tempty x2, drain, the slot barriers
  static_assert((2 * STAGES + 5 + epi_warps<EPI>() * SLOTS) * 8 <= 496, "barrier area");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// Swizzled 16-byte chunk k of row r in a slot block of 64-byte rows (the
// 64-byte TMA swizzle: chunk bits 4..5 of the address XOR bits 7..8).
__device__ __forceinline__ uint32_t sw64(uint32_t base, int r, int k) {
  return base + static_cast<uint32_t>(r * 64) + (static_cast<uint32_t>(k ^ ((r >> 1) & 3)) << 4);
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Pair tile order (RASTER_*), over 256-row M blocks; the batch (shard) is
// the outermost coordinate in every order.
__host__ __device__ __forceinline__ void decode_pair_tile(const Params& p, int tile, int& b, int& mp, int& nb) {
  const int tiles_m2 = (p.tiles_m + 1) >> 1;
  const int tpb = tiles_m2 * p.tiles_n;
  b = tile / tpb;
  const int r = tile - b * tpb;
  if (p.raster == RASTER_M_FAST) {
    nb = r / tiles_m2;
    mp = r - nb * tiles_m2;
    return;
  }
  if (p.raster == RASTER_N_FAST) {
    mp = r / p.tiles_n;
    nb = r - mp * p.tiles_n;
    return;
  }
  // 8 pair-rows per raster group: about 8 x 9.5 tiles run at once, so each K
  // step fetches ~17.5 distinct operand blocks from DRAM (4 x 19: ~23).
  constexpr int GM = 8;
  const int group = r / (GM * p.tiles_n);
  const int first_m = group * GM;
  const int gm = tiles_m2 - first_m < GM ? tiles_m2 - first_m : GM;
  const int in_group = r - group * GM * p.tiles_n;
  mp = first_m + in_group % gm;
  nb = in_group / gm;
}

// Shared-memory address of 16-byte chunk k of row r in a staged box with
// 128-byte rows (128-byte TMA swizzle: chunk bits 4..6 XOR row bits 0..2).
__device__ __forceinline__ uint32_t sw128(uint32_t base, int r, int k) {
  return base + static_cast<uint32_t>(r * 128) + (static_cast<uint32_t>(k ^ (r & 7)) << 4);
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 q;
  q.x = pack_bf16x2(v[0], v[1]);
  q.y = pack_bf16x2(v[2], v[3]);
  q.z = pack_bf16x2(v[4], v[5]);
  q.w = pack_bf16x2(v[6], v[7]);
  return q;
}

// One tile's epilogue through TMA stores (pair kernel, one warp per TMEM lane
// quarter).  The warp's 32 rows start at row0; lane = its row within them.
// Rows past M and columns past n_store lie outside the output maps and are
// not written.  `k` counts this warp's staged chunks (buffer rotation).
template <int EPI, int NSPLIT>
__device__ __forceinline__ void epilogue_tile_tma(const Params& p, const CUtensorMap* tmO, const CUtensorMap* tmO2,
                                                  int b, int row0, int lane, int n0, int nb, uint32_t taddr,
                                                  uint8_t* sbuf, uint32_t& k, int part) {
  const uint32_t sb = smem_u32(sbuf);
  if constexpr (EPI == EPI_SWIGLU_FWD) {
    // chunk c: 32 hidden units -> h (2 KB box), a and g (2 KB boxes); one 6 KB buffer
#pragma unroll 1
    for (int c = part * (4 / NSPLIT); c < (part + 1) * (4 / NSPLIT); ++c) {
      uint32_t ra[32], rg[32];
      __syncwarp();
      tmem_ld32(taddr + c * 32, ra);
      tmem_ld32(taddr + 128 + c * 32, rg);
      tmem_wait_ld();
      if (lane == 0) bulk_wait_read<0>();  // the previous chunk's boxes have left the buffer
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float h[8], a[8], g[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          a[j] = __uint_as_float(ra[q * 8 + j]);
          g[j] = __uint_as_float(rg[q * 8 + j]);
          h[j] = a[j] * sigmoid_f(a[j]) * g[j];
        }
        sts128(sw64(sb, lane, q), pack8_bf16(h));
        if (p.out2) {
          sts128(sw64(sb + 2048, lane, q), pack8_bf16(a));
          sts128(sw64(sb + 4096, lane, q), pack8_bf16(g));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int hcol = nb * 128 + c * 32, acol = nb * 256 + c * 32;
        if (row0 >= p.M) {
          // every row of this warp lies past M: nothing to store (an empty
          // group keeps the buffer accounting)
        } else if (!p.o_swap) {
          tma_store_3d(tmO, sbuf, hcol, row0, b);
          if (p.out2) {
            tma_store_3d(tmO2, sbuf + 2048, acol, row0, b);
            tma_store_3d(tmO2, sbuf + 4096, acol + 128, row0, b);
          }
        } else {
          tma_store_3d(tmO, sbuf, hcol, b, row0);
          if (p.out2) {
            tma_store_3d(tmO2, sbuf + 2048, acol, b, row0);
            tma_store_3d(tmO2, sbuf + 4096, acol + 128, b, row0);
          }
        }
        bulk_commit();
      }
      ++k;
    }
    return;
  } else {
    // EPI_OUT / EPI_F32 / EPI_GELU_FWD: chunk c = 32 columns; two 4 KB buffers
    constexpr int NBUF = 2;
#pragma unroll 1
    for (int c = part * (PAIR_BN / 32 / NSPLIT); c < (part + 1) * (PAIR_BN / 32 / NSPLIT); ++c) {
      const int nc = n0 + c * 32;
      if (nc >= p.n_store) break;  // columns past n_store: nothing to store (n_store is a multiple of 8)
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(taddr + c * 32, r);
      tmem_wait_ld();
      float bv[32];
      if constexpr (EPI == EPI_OUT || EPI == EPI_GELU_FWD) {
        if (p.bias) {
          const __nv_bfloat16* bp = p.bias + b * p.bias_bs + nc;
          if (nc + 32 <= p.bias_len && (reinterpret_cast<uintptr_t>(bp) & 15) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) load_bf16x8(bp + q * 8, bv + q * 8);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) bv[j] = nc + j < p.bias_len ? __bfloat162float(bp[j]) : 0.f;
          }
        }
      }
      const uint32_t buf = sb + (k % NBUF) * 4096;
      if (lane == 0) bulk_wait_read<NBUF - 1>();  // this buffer's previous boxes have left it
      __syncwarp();
      if constexpr (EPI == EPI_F32) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          sts128(sw128(buf, lane, q), make_uint4(r[q * 4], r[q * 4 + 1], r[q * 4 + 2], r[q * 4 + 3]));
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[q * 8 + j]);
          if (p.bias) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] += bv[q * 8 + j];
          }
          if constexpr (EPI == EPI_OUT) {
            sts128(sw64(buf, lane, q), pack8_bf16(v));
          } else {  // EPI_GELU_FWD: h, and the saved z beside it
            if (p.out2) sts128(sw64(buf + 2048, lane, q), pack8_bf16(v));
            float h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = gelu_tanh_f(v[j]);
            sts128(sw64(buf, lane, q), pack8_bf16(h));
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const uint8_t* src = sbuf + (k % NBUF) * 4096;
        if (row0 >= p.M) {
          // every row of this warp lies past M: nothing to store (an empty
          // group keeps the buffer accounting)
        } else if (p.out_cs) {  // shards merged along N: column nc of shard nc / out_cs
          const int sb = nc / p.out_cs;
          tma_store_3d(tmO, src, nc - sb * p.out_cs, row0, sb);
        } else if (!p.o_swap) {
          tma_store_3d(tmO, src, nc, row0, b);
          if (EPI == EPI_GELU_FWD && p.out2) tma_store_3d(tmO2, src + 2048, nc, row0, b);
        } else {
          tma_store_3d(tmO, src, nc, b, row0);
          if (EPI == EPI_GELU_FWD && p.out2) tma_store_3d(tmO2, src + 2048, nc, b, row0);
        }
        bulk_commit();
      }
      ++k;
    }
  }
}

// Epilogue of a last-wave K part: the warp's 32 rows (tile row r_local on)
// of the tile's fp32 sum over its K part, stored as 32 x 32 boxes at (column
// within the tile, row within the tile, tb) of the {256, 256, parts x tail
// tiles} fp32 map.  Same staging buffers and bulk-group count as
// epilogue_tile_tma; after the SwiGLU epilogue, whose one 6 KB buffer spans
// both 4 KB buffers used here, each box waits for every earlier store to
// have read its source.
template <int EPI, int NSPLIT>
__device__ __forceinline__ void epilogue_tail_part(const Params& p, const CUtensorMap* tmT, int tb, int r_local,
                                                   int row0, int lane, uint32_t taddr, uint8_t* sbuf, uint32_t& k,
                                                   int part) {
  constexpr int NBUF = 2;
  constexpr int IN_FLIGHT = EPI == EPI_SWIGLU_FWD ? 0 : NBUF - 1;
  const uint32_t sb = smem_u32(sbuf);
#pragma unroll 1
  for (int c = part * (PAIR_BN / 32 / NSPLIT); c < (part + 1) * (PAIR_BN / 32 / NSPLIT); ++c) {
    // every chunk is stored (the map holds whole tiles); the fix-up skips
    // the columns past the output's
    uint32_t r[32];
    __syncwarp();
    tmem_ld32(taddr + c * 32, r);
    tmem_wait_ld();
    const uint32_t buf = sb + (k % NBUF) * 4096;
    if (lane == 0) bulk_wait_read<IN_FLIGHT>();  // this buffer's previous boxes have left it
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 8; ++q)
      sts128(sw128(buf, lane, q), make_uint4(r[q * 4], r[q * 4 + 1], r[q * 4 + 2], r[q * 4 + 3]));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (row0 < p.M) tma_store_3d(tmT, sbuf + (k % NBUF) * 4096, c * 32, r_local, tb);
      bulk_commit();
    }
    ++k;
  }
}

// Work unit of the pair kernel: tile `unit mod tiles` over K part
// `unit / tiles` of the (shard-major) K blocks, [kb0, kb0 + nkb).  Without a
// K split, one unit per tile over all K blocks.  With a last-wave split, the
// first tiles - tail_tiles units are whole tiles and unit whole + u is part
// u / tail_tiles of tail tile u mod tail_tiles; it returns -1 - u.
__device__ __forceinline__ int pair_unit(const Params& p, int unit, int num_tiles, int& tile, int& kb0, int& nkb) {
  if (p.tail_parts > 1) {
    const int whole = num_tiles - p.tail_tiles;
    const int kall = p.G * p.k_blocks;
    if (unit < whole) {
      tile = unit;
      kb0 = 0;
      nkb = kall;
      return 0;
    }
    // part j: K blocks [j kall / parts, (j + 1) kall / parts), none empty
    const int u = unit - whole, part = u / p.tail_tiles;
    tile = whole + (u - part * p.tail_tiles);
    kb0 = part * kall / p.tail_parts;
    nkb = (part + 1) * kall / p.tail_parts - kb0;
    return -1 - u;
  }
  const int kh = p.ksplit > 1 ? unit / num_tiles : 0;
  tile = unit - kh * num_tiles;
  const int kall = p.G * p.k_blocks;
  const int kbs = (kall + p.ksplit - 1) / p.ksplit;
  kb0 = kh * kbs;
  nkb = min(kall - kb0, kbs);
  return kh;
}

template <int EPI, bool AMN, bool BMN, int TM = 0>
__global__ void __launch_bounds__(pair_threads<EPI, TM>(), 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmO,
                        const __grid_constant__ CUtensorMap tmO2, const Params p) {
  using L = PairLayout<EPI, TM>;
  constexpr bool TMA = TM != 0;
  constexpr int EW = pair_epi_warps<EPI, TM>();
  constexpr int BN = PAIR_BN;
  constexpr int STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* xbar = drain + 1;  // saved-activation slots (backward epilogues)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + 496);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 500);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // leader: its own arrive + both CTAs' bytes
      mbar_init(&empty[s], 1);  // one multicast commit of the leader
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * EW);  // leader: the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    if constexpr (aux_staged<EPI>())
      for (int i = 0; i < epi_warps<EPI>() * L::SLOTS; ++i) mbar_init(&xbar[i], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if constexpr (aux_staged<EPI>()) prefetch_tmap(&tmX);
    if constexpr (TMA) {
      prefetch_tmap(&tmO);
      if (!aux_staged<EPI>() && p.out2) prefetch_tmap(&tmO2);
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // a programmatic dependent of the previous kernel: the set-up above
  // overlapped its tail; no global memory is touched before its results are
  // visible (dep_mode 2: nothing this GEMM reads or writes is touched by it)
  dep_prologue(p.dep_mode);

  const int tiles_m2 = (p.tiles_m + 1) >> 1;
  const int num_tiles = tiles_m2 * p.tiles_n * p.NB;
  // K parts of the split (fp32 partial) GEMMs, or of the last wave's tiles
  const int num_units =
      p.tail_parts > 1 ? num_tiles + p.tail_tiles * (p.tail_parts - 1) : num_tiles * p.ksplit;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_issue_phase[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) last_issue_phase[s] = -1;
      bool ok = true;
      const uint64_t pol_keep = l2_policy_evict_normal(), pol_stream = l2_policy_evict_first();
      for (int unit = cluster_id; unit < num_units && ok; unit += num_clusters) {
        int tile, kb0, nkb;
        pair_unit(p, unit, num_tiles, tile, kb0, nkb);
        int b, mp, nb;
        decode_pair_tile(p, tile, b, mp, nb);
        const int m0 = mp * 256 + static_cast<int>(rank) * 128;   // this CTA's A rows
        const int n0 = nb * BN + static_cast<int>(rank) * (BN / 2);  // this CTA's half of B
        for (int it = kb0; it < kb0 + nkb; ++it) {
          const int g = it / p.k_blocks;
          const int k0 = (it - g * p.k_blocks) * BK;
          {
            DBG_T0();
            const bool w_ok = wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p);
            DBG_ADD(3, _t0);
            if (!w_ok) {
              ok = false;
              break;
            }
          }
          const bool skip = p.debug_skip && unit == cluster_id && it == kb0;
          if (!skip) {
            uint8_t* sA = smem + stage * L::STAGE_BYTES;
            uint8_t* sB = sA + L::A_BYTES;
            // Only the leader arms its full barrier, for the bytes of both
            // CTAs; the peer's copies complete on it directly (its transaction
            // count may go below zero until the leader arms it).  A peer-side
            // arrive would need a cluster-scope release per stage, which
            // serialises the peer's copies.
            const uint32_t leader_full = map_to_rank(smem_u32(&full[stage]), 0);
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * L::STAGE_BYTES);
            const int ab = b * p.a_bsel + g * p.a_gsel;
            const int bb = b * p.b_bsel + g * p.b_gsel;
            if (p.keep_op) {
              // the per-batch operand streams through L2 with evict_first
              // priority, so that the operand all batches share stays there;
              // MN-major operands here always use the 4-D map (set on the host)
              const uint64_t pa = p.keep_op == 1 ? pol_keep : pol_stream;
              const uint64_t pb = p.keep_op == 1 ? pol_stream : pol_keep;
              if (!AMN) tma_load_3d_pair_hint(sA, &tmA, leader_full, k0, p.a_swap ? ab : m0, p.a_swap ? m0 : ab, pa);
              else tma_load_4d_pair_hint(sA, &tmA, leader_full, 0, k0, m0 / 64, ab, pa);
              if (!BMN) tma_load_3d_pair_hint(sB, &tmB, leader_full, k0, p.b_swap ? bb : n0, p.b_swap ? n0 : bb, pb);
              else tma_load_4d_pair_hint(sB, &tmB, leader_full, 0, k0, n0 / 64, bb, pb);
            } else {
              if (!AMN) {
                tma_load_3d_pair(sA, &tmA, leader_full, k0, p.a_swap ? ab : m0, p.a_swap ? m0 : ab);
              } else if (p.a_swap == 2) {
                tma_load_4d_pair(sA, &tmA, leader_full, 0, k0, m0 / 64, ab);
              } else {
#pragma unroll
                for (int i = 0; i < 2; ++i)
                  tma_load_3d_pair(sA + i * 8192, &tmA, leader_full, m0 + 64 * i, p.a_swap ? ab : k0,
                                   p.a_swap ? k0 : ab);
              }
              if (!BMN) {
                tma_load_3d_pair(sB, &tmB, leader_full, k0, p.b_swap ? bb : n0, p.b_swap ? n0 : bb);
              } else if (p.b_cs) {  // shards merged along N: B columns of shard n0 / b_cs
                const int sbb = n0 / p.b_cs;
                tma_load_4d_pair(sB, &tmB, leader_full, 0, k0, (n0 - sbb * p.b_cs) / 64, sbb);
              } else if (p.b_swap == 2) {
                tma_load_4d_pair(sB, &tmB, leader_full, 0, k0, n0 / 64, bb);
              } else {
#pragma unroll
                for (int i = 0; i < 2; ++i)
                  tma_load_3d_pair(sB + i * 8192, &tmB, leader_full, n0 + 64 * i, p.b_swap ? bb : k0,
                                   p.b_swap ? k0 : bb);
              }
            }
            last_issue_phase[stage] = static_cast<int>(phase);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain (leader): its full[] barriers count both CTAs' copies.
      if (leader) {
#pragma unroll 1
        for (int s = 0; s < STAGES; ++s)
          if (last_issue_phase[s] >= 0)
            wait_bounded(&full[s], static_cast<uint32_t>(last_issue_phase[s]), abort_flag, p, false);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader only)
    if (leader && lane == 0) {
      // M = 256 (two CTAs), N = 256
      constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(AMN) << 15) |
                                 (static_cast<uint32_t>(BMN) << 16) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                 (static_cast<uint32_t>(256 >> 4) << 24);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
#ifdef TPFFN_INSTRUMENT
      const long long t_start = clock64();
#endif
      for (int unit = cluster_id; unit < num_units && ok; unit += num_clusters, ++local) {
        int tile, kb0, nkb;
        pair_unit(p, unit, num_tiles, tile, kb0, nkb);
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        {
          DBG_T0();
          const bool w_ok = wait_bounded(&tempty[buf], (use & 1u) ^ 1u, abort_flag, p);
          DBG_ADD(1, _t0);
          if (!w_ok) break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int it = kb0; it < kb0 + nkb; ++it) {
          {
            DBG_T0();
            const bool w_ok = wait_bounded(&full[stage], phase, abort_flag, p);
            DBG_ADD(0, _t0);
            if (!w_ok) {
              ok = false;
              break;
            }
          }
#ifdef TPFFN_INSTRUMENT
          atomicAdd(&g_tpffn_dbg[p.dbg_slot & 7][blockIdx.x & 255][6], 1ull);
#endif
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * L::STAGE_BYTES);
          const uint32_t b_addr = a_addr + L::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16_pair(d_tmem, smem_desc<AMN>(a_addr, k), smem_desc<BMN>(b_addr, k), IDESC,
                           (it > kb0 || k > 0) ? 1u : 0u);
          umma_commit_pair(&empty[stage]);  // frees the stage in both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[buf]);  // accumulators of both CTAs ready
      }
      umma_commit_pair_local(drain);  // arrives once every MMA issued here has completed
      wait_bounded(drain, 0u, abort_flag, p, false);
#ifdef TPFFN_INSTRUMENT
      DBG_ADD(2, t_start);
#endif
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps 2..9 (both CTAs)
    const int quarter = warp & 3;
    const uint32_t leader_tempty0 = map_to_rank(smem_u32(&tempty[0]), 0);
    const uint32_t leader_tempty1 = map_to_rank(smem_u32(&tempty[1]), 0);
    int local = 0;
#ifdef TPFFN_INSTRUMENT
    const long long t_epi = clock64();
#endif
    if constexpr (aux_staged<EPI>() && TMA) {
      // Backward epilogue, TMA in and out: chunk k of this warp (its c-th
      // 32-column chunk of a tile) finds its saved activations in slot k & 1;
      // before waiting for them the warp sends the next chunk's copy into the
      // other slot (once the store that last read that slot has read it).  The
      // chunk's results replace the activations in slot k & 1 -- each lane
      // writes only its own row, which it has read -- and one lane stores
      // them.  The chunk after a tile's last is the next tile's first.
      constexpr int CPW = BN / 32 / 2;  // 32-column chunks per warp (two warps per lane quarter)
      constexpr uint32_t XBYTES = EPI == EPI_SWIGLU_BWD ? 4096u : 2048u;
      const int part = (warp - 2) >> 2;
      const int c0 = part * CPW;
      uint8_t* slots = smem + L::AUX_OFF + (warp - 2) * 2 * L::AUX_SLOT;
      uint64_t* xbw = &xbar[(warp - 2) * 2];
      uint32_t xph = 0, pendm = 0;  // per-slot phase and copy-in-flight bits
      uint32_t kc = 0;              // chunks done by this warp
      auto issue = [&](int t, int c, int sl) {  // lane 0
        int b, mp, nb;
        decode_pair_tile(p, t, b, mp, nb);
        const int row0 = mp * 256 + static_cast<int>(rank) * 128 + quarter * 32;
        const int n = nb * BN + c * 32;
        uint8_t* dst = slots + sl * L::AUX_SLOT;
        mbar_arrive_expect_tx(&xbw[sl], XBYTES);
        if constexpr (EPI == EPI_SWIGLU_BWD) {
          const int col = (n >> 7) * 256 + (n & 127);
          tma_load_3d(dst, &tmX, &xbw[sl], col, row0, b);
          tma_load_3d(dst + 2048, &tmX, &xbw[sl], col + 128, row0, b);
        } else {
          tma_load_3d(dst, &tmX, &xbw[sl], n, row0, b);
        }
      };
      if (cluster_id < num_tiles) {
        if (lane == 0) issue(cluster_id, c0, 0);
        pendm |= 1u;
      }
      bool ok = true;
      for (int tile = cluster_id; tile < num_tiles && ok; tile += num_clusters, ++local) {
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        ok = wait_bounded(&tfull[buf], use & 1u, abort_flag, p);
        if (!ok) break;
        tc_fence_after();
        int b, mp, nb;
        decode_pair_tile(p, tile, b, mp, nb);
        const int row0 = mp * 256 + static_cast<int>(rank) * 128 + quarter * 32;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(buf * BN);
#pragma unroll 1
        for (int c = c0; c < c0 + CPW; ++c, ++kc) {
          const int sl = static_cast<int>(kc & 1u);
          int nt = tile, ncc = c + 1;
          if (ncc == c0 + CPW) {
            nt = tile + num_clusters;
            ncc = c0;
          }
          if (nt < num_tiles) {
            if (lane == 0) {
              bulk_wait_read<0>();  // the store that last read the other slot is done with it
              issue(nt, ncc, sl ^ 1);
            }
            pendm |= 1u << (sl ^ 1);
          }
          if (!wait_bounded(&xbw[sl], (xph >> sl) & 1u, abort_flag, p)) {
            ok = false;
            break;
          }
          pendm &= ~(1u << sl);
          xph ^= 1u << sl;
          const uint32_t xs = smem_u32(slots + sl * L::AUX_SLOT);
          uint4 za[4], gg[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            za[k] = lds128(sw64(xs, lane, k));
            if constexpr (EPI == EPI_SWIGLU_BWD) gg[k] = lds128(sw64(xs + 2048, lane, k));
          }
          uint32_t r[32];
          __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
          tmem_ld32(taddr + c * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float v[8], a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[q * 8 + j]);
            unpack_bf16x8(za[q], a);
            if constexpr (EPI == EPI_GELU_BWD) {
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] *= gelu_tanh_grad_f(a[j]);
              sts128(sw64(xs, lane, q), pack8_bf16(v));
            } else {
              float g[8], da[8], dg[8];
              unpack_bf16x8(gg[q], g);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float sg = sigmoid_f(a[j]);
                dg[j] = v[j] * a[j] * sg;                                // dh * silu(a)
                da[j] = v[j] * g[j] * sg * (1.0f + a[j] * (1.0f - sg));  // dh * g * silu'(a)
              }
              sts128(sw64(xs, lane, q), pack8_bf16(da));
              sts128(sw64(xs + 2048, lane, q), pack8_bf16(dg));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int n = nb * BN + c * 32;
            if (row0 < p.M && n < p.n_store) {
              const uint8_t* src = slots + sl * L::AUX_SLOT;
              if constexpr (EPI == EPI_SWIGLU_BWD) {
                const int col = (n >> 7) * 256 + (n & 127);
                tma_store_3d(&tmO, src, col, row0, b);
                tma_store_3d(&tmO, src + 2048, col + 128, row0, b);
              } else {
                tma_store_3d(&tmO, src, n, row0, b);
              }
            }
            bulk_commit();  // (an empty group when nothing is stored)
          }
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(buf ? leader_tempty1 : leader_tempty0);
      }
      // copies still in flight into the slots, and the stores, complete
      // before the CTA exits
      for (int sl = 0; sl < 2; ++sl)
        if (pendm & (1u << sl)) wait_bounded(&xbw[sl], (xph >> sl) & 1u, abort_flag, p, false);
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    } else if constexpr (aux_staged<EPI>()) {
      // Backward epilogue with the saved activations staged by TMA: chunk c
      // of this warp's 32 rows lands in its slot while chunk c-1 is
      // computed; the chunk after the tile's last is the next tile's first.
      constexpr int CPW = BN / 32 / 2;  // 32-column chunks per warp (two warps per lane quarter)
      constexpr uint32_t XBYTES = EPI == EPI_SWIGLU_BWD ? 4096u : 2048u;
      const int part = (warp - 2) >> 2;
      const int c0 = part * CPW;
      uint8_t* xslot = smem + L::AUX_OFF + (warp - 2) * L::AUX_SLOT;
      const uint32_t xs = smem_u32(xslot);
      uint64_t* xb = &xbar[warp - 2];
      uint32_t xph = 0;
      bool pending = false;
      auto issue = [&](int t, int c) {  // lane 0
        int b, mp, nb;
        decode_pair_tile(p, t, b, mp, nb);
        const int row0 = mp * 256 + static_cast<int>(rank) * 128 + quarter * 32;
        const int n = nb * BN + c * 32;
        mbar_arrive_expect_tx(xb, XBYTES);
        if constexpr (EPI == EPI_SWIGLU_BWD) {
          // hidden unit n lives in 128-block n>>7 of the interleaved [a|g] rows
          const int col = (n >> 7) * 256 + (n & 127);
          tma_load_3d(xslot, &tmX, xb, col, row0, b);
          tma_load_3d(xslot + 2048, &tmX, xb, col + 128, row0, b);
        } else {
          tma_load_3d(xslot, &tmX, xb, n, row0, b);
        }
      };
      if (cluster_id < num_tiles) {
        if (lane == 0) issue(cluster_id, c0);
        pending = true;
      }
      bool ok = true;
      for (int tile = cluster_id; tile < num_tiles && ok; tile += num_clusters, ++local) {
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        {
          DBG_T0();
          ok = wait_bounded(&tfull[buf], use & 1u, abort_flag, p);
          if (warp == 2 && lane == 0) DBG_ADD(4, _t0);
        }
        if (!ok) break;
        tc_fence_after();
        int b, mp, nb;
        decode_pair_tile(p, tile, b, mp, nb);
        const int row = mp * 256 + static_cast<int>(rank) * 128 + quarter * 32 + lane;
        const bool row_ok = row < p.M;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(buf * BN);
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + b * p.out_bs + (long long)row * p.out_rs;
#pragma unroll 1
        for (int c = c0; c < c0 + CPW; ++c) {
          if (!wait_bounded(xb, xph, abort_flag, p)) {
            ok = false;
            break;
          }
          pending = false;
          xph ^= 1u;
          uint4 za[4], gg[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            za[k] = lds128(sw64(xs, lane, k));
            if constexpr (EPI == EPI_SWIGLU_BWD) gg[k] = lds128(sw64(xs + 2048, lane, k));
          }
          // the slot's reads are ordered before the next copy into it
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          int nt = tile, ncc = c + 1;
          if (ncc == c0 + CPW) {
            nt = tile + num_clusters;
            ncc = c0;
          }
          if (nt < num_tiles) {
            if (lane == 0) issue(nt, ncc);
            pending = true;
          }
          uint32_t r[32];
          __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
          tmem_ld32(taddr + c * 32, r);
          tmem_wait_ld();
          const int nc = nb * BN + c * 32;
          if (!row_ok || nc >= p.n_store) continue;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n = nc + q * 8;
            if (n >= p.n_store) break;  // n_store is a multiple of 8
            float v[8], a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[q * 8 + j]);
            unpack_bf16x8(za[q], a);
            if constexpr (EPI == EPI_GELU_BWD) {
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] *= gelu_tanh_grad_f(a[j]);
              store_bf16x8(out + n, v);
            } else {
              float g[8], da[8], dg[8];
              unpack_bf16x8(gg[q], g);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float sg = sigmoid_f(a[j]);
                dg[j] = v[j] * a[j] * sg;                                // dh * silu(a)
                da[j] = v[j] * g[j] * sg * (1.0f + a[j] * (1.0f - sg));  // dh * g * silu'(a)
              }
              const long long col = (long long)(n >> 7) * 256 + (n & 127);
              store_bf16x8(out + col, da);
              store_bf16x8(out + col + 128, dg);
            }
          }
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(buf ? leader_tempty1 : leader_tempty0);
      }
      // a copy still in flight into the slot completes before the CTA exits
      if (pending) wait_bounded(xb, xph, abort_flag, p, false);
    } else {
      uint32_t staged = 0;  // TMA-store epilogue: chunks this warp has staged
      for (int unit = cluster_id; unit < num_units; unit += num_clusters, ++local) {
        int tile, kb0, nkb;
        const int kh = pair_unit(p, unit, num_tiles, tile, kb0, nkb);
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        bool w_ok;
        {
          DBG_T0();
          w_ok = wait_bounded(&tfull[buf], use & 1u, abort_flag, p);
          if (warp == 2 && lane == 0) DBG_ADD(4, _t0);
        }
        if (!w_ok) break;
        tc_fence_after();
        int b, mp, nb;
        decode_pair_tile(p, tile, b, mp, nb);
        if (kh > 0) b += kh * p.NB;  // K part kh: fp32 batch kh * NB + b (EPI_F32 only)
        const int row0 = mp * 256 + static_cast<int>(rank) * 128 + quarter * 32;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(buf * BN);
        if constexpr (TMA) {
          if (kh < 0)  // a last-wave K part: fp32 boxes into batch -1 - kh of the tail map (in tmX)
            epilogue_tail_part<EPI, EW / 4>(p, &tmX, -1 - kh, row0 - mp * 256, row0, lane, taddr,
                                            smem + L::AUX_OFF + (warp - 2) * OUT_BUF, staged, (warp - 2) >> 2);
          else
            epilogue_tile_tma<EPI, EW / 4>(p, &tmO, &tmO2, b, row0, lane, nb * BN, nb, taddr,
                                           smem + L::AUX_OFF + (warp - 2) * OUT_BUF, staged, (warp - 2) >> 2);
        } else {
          const int row = row0 + lane;
          epilogue_tile<BN, EPI>(p, b, row, row < p.M, nb * BN, nb, taddr, (warp - 2) >> 2);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(buf ? leader_tempty1 : leader_tempty0);
      }
      // the stores this warp issued have completed before the CTA exits
      if (TMA && lane == 0) bulk_wait_all();
      __syncwarp();
    }
#ifdef TPFFN_INSTRUMENT
    if (warp == 2 && lane == 0) DBG_ADD(5, t_epi);
#endif
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's MMAs and copies into both CTAs have finished
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
  }
  dep_epilogue(p.dep_mode);
}

// ------------------------------------------------------------ host side
// TPFFN_MN4D=0 in the environment selects the 3-D maps (one request per
// 64-element group) for MN-major operands, for comparisons.
static bool getenv_flag_off(const char* name) {
  const char* v = getenv(name);
  return v && v[0] == '0';
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 3-D bf16 tensor map, 128-byte swizzle, zero fill out of bounds (declared
// in tc_ptx.cuh for the other tensor-core kernels of the library).
int encode_map_3d_bf16(CUtensorMap* m, const void* ptr, const uint64_t dims[3], const uint64_t strides_bytes[2],
                       const uint32_t box[3]) {
  if (reinterpret_cast<uintptr_t>(ptr) % 16 || strides_bytes[0] % 16 || strides_bytes[1] % 16) return TP_ERR_ALIGN;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return TP_ERR_CUDA;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]}, estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : TP_ERR_CUDA;
}

// 3-D bf16 tensor map of an operand.  Dimension order keeps strides
// increasing: {inner, rows, batch}, or {inner, batch, rows} ("swap") when the
// batch stride is the smaller one (e.g. heads inside a token row).
static int make_map(CUtensorMap* m, const Operand& op, int rows_box, int* swap) {
  const uint64_t es = 2;
  if (reinterpret_cast<uintptr_t>(op.ptr) % 16) return TP_ERR_ALIGN;
  if (op.inner < 1 || op.rows < 1 || op.batch < 1) return TP_ERR_INVALID;
  const int64_t bst = op.batch > 1 ? op.batch_stride : op.row_stride * op.rows;
  if ((op.row_stride * es) % 16 || (bst * es) % 16) return TP_ERR_ALIGN;
  const uint32_t rb = op.mn_major ? 64u : static_cast<uint32_t>(rows_box);
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  *swap = (op.batch > 1 && op.batch_stride < op.row_stride) ? 1 : 0;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return TP_ERR_CUDA;
  // MN-major operands whose M/N extent is whole 64-element groups: a 4-D view
  // {64 (M/N within a group), K rows, groups, batch} lets one request fetch
  // every group of the tile in the layout the MMA reads (group i at +8 KB i).
  if (op.mn_major && !*swap && op.inner % 64 == 0 && rows_box % 64 == 0 && !getenv_flag_off("TPFFN_MN4D")) {
    cuuint64_t d4[4] = {64, static_cast<cuuint64_t>(op.rows), static_cast<cuuint64_t>(op.inner / 64),
                        static_cast<cuuint64_t>(op.batch)};
    cuuint64_t s4[3] = {static_cast<cuuint64_t>(op.row_stride * es), 64 * es, static_cast<cuuint64_t>(bst * es)};
    cuuint32_t b4[4] = {64, 64, static_cast<cuuint32_t>(rows_box / 64), 1}, e4[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(op.ptr), d4, s4, b4, e4,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
      *swap = 2;
      return 0;
    }
    // otherwise the 3-D map below (one request per 64-element group)
  }
  dims[0] = static_cast<cuuint64_t>(op.inner);
  box[0] = 64;
  if (!*swap) {
    dims[1] = op.rows;
    dims[2] = op.batch;
    strides[0] = op.row_stride * es;
    strides[1] = bst * es;
    box[1] = rb;
    box[2] = 1;
  } else {
    dims[1] = op.batch;
    dims[2] = op.rows;
    strides[0] = op.batch_stride * es;
    strides[1] = op.row_stride * es;
    box[1] = 1;
    box[2] = rb;
  }
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(op.ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : TP_ERR_CUDA;
}

// TPFFN_PDL_OLD=1: the former dependent-launch order; TPFFN_NO_DEP_OVERLAP=1:
// GEMMs marked independent of their predecessor wait for it all the same
static int dep_mode_for(const GemmSpec& s) {
  static const bool old_order = getenv("TPFFN_PDL_OLD") != nullptr;
  static const bool no_overlap = getenv("TPFFN_NO_DEP_OVERLAP") != nullptr;
  if (old_order) return 0;
  return (s.no_dep_wait && !no_overlap) ? 2 : 1;
}

static bool l2_hint_enabled() {
  static const bool on = !getenv_flag_off("TPFFN_L2HINT");
  return on;
}

template <int BN, int STAGES, int EPI, bool AMN, bool BMN, int AR = BM>
static int launch_inst(const GemmSpec& s, LaunchCtx& ctx) {
  using L = Layout<BN, STAGES, AR>;
  if (AR < BM && s.M > AR) return TP_ERR_INVALID;
  CUtensorMap ta, tb;
  int sa = 0, sb = 0;
  int rc = make_map(&ta, s.A, AR, &sa);
  if (rc) return rc;
  rc = make_map(&tb, s.B, BN, &sb);
  if (rc) return rc;
  Params p{};
  p.M = static_cast<int>(s.M);
  p.N = static_cast<int>(s.N);
  p.K = static_cast<int>(s.K);
  p.NB = s.NB;
  p.G = s.G;
  p.tiles_m = static_cast<int>((s.M + BM - 1) / BM);
  p.tiles_n = static_cast<int>((s.N + BN - 1) / BN);
  p.k_blocks = static_cast<int>((s.K + BK - 1) / BK);
  p.a_bsel = s.A.bsel;
  p.a_gsel = s.A.gsel;
  p.b_bsel = s.B.bsel;
  p.b_gsel = s.B.gsel;
  p.a_swap = sa;
  p.b_swap = sb;
  p.out = s.out;
  p.out_bs = s.out_bs;
  p.out_rs = s.out_rs;
  p.out2 = s.out2;
  p.out2_bs = s.out2_bs;
  p.out2_rs = s.out2_rs;
  p.aux = s.aux;
  p.aux_bs = s.aux_bs;
  p.aux_rs = s.aux_rs;
  p.bias = static_cast<const __nv_bfloat16*>(s.bias);
  p.bias_bs = s.bias_bs;
  p.bias_len = s.bias_len;
  p.n_store = s.n_store;
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  p.debug_skip = ctx.debug_skip_load;
  ctx.debug_skip_load = 0;

  auto kern = tc_gemm_kernel<BN, STAGES, EPI, AMN, BMN, AR>;
  static std::atomic<uint32_t> attr_done{0};  // one bit per device
  int dev = 0;
  cudaGetDevice(&dev);
  const uint32_t bit = 1u << (dev & 31);
  if (!(attr_done.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) != cudaSuccess)
      return TP_ERR_CUDA;
    attr_done.fetch_or(bit);
  }
  p.ksplit = s.ksplit;
  if (s.ksplit < 1 || (s.ksplit > 1 && (EPI != EPI_F32 || s.G != 1 || p.k_blocks < 2 * s.ksplit)))
    return TP_ERR_INVALID;
  p.dep_mode = dep_mode_for(s);
  // Decode-sized GEMMs (32-row A tiles) stream their weights once: those
  // copies go through L2 with evict_first priority, so that the small fp32
  // parts and partials the next kernel reads stay there.
  p.keep_op = (AR < BM && !BMN && l2_hint_enabled()) ? 1 : 0;
  const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n * p.NB * s.ksplit;  // work units
  if (tiles <= 0 || p.k_blocks <= 0) return TP_ERR_INVALID;
  int grid = static_cast<int>(tiles < ctx.num_sms ? tiles : ctx.num_sms);
  // A single row of M tiles (decode-sized token counts) streams weights and
  // is HBM-bound: spread the tiles evenly -- every CTA gets the same number
  // of tiles -- rather than leaving a last wave on a fraction of the SMs.
  if (p.tiles_m == 1 && tiles > grid) {
    const long long waves = (tiles + grid - 1) / grid;
    grid = static_cast<int>((tiles + waves - 1) / waves);
  }
  if (ctx.before) ctx.before(ctx.user, s.name, ctx.stream);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(threads_for<EPI>());
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, p) != cudaSuccess) return TP_ERR_CUDA;
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

// Saved activations of a backward epilogue, {columns, rows, batch}: a
// 32 x 32 box per copy, 64-byte swizzle, zero fill past the rows / columns.
static int make_aux_map(CUtensorMap* m, const GemmSpec& s) {
  if (!s.aux || reinterpret_cast<uintptr_t>(s.aux) % 16) return TP_ERR_ALIGN;
  if ((s.aux_rs * 2) % 16 || (s.aux_bs * 2) % 16) return TP_ERR_ALIGN;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return TP_ERR_CUDA;
  const int64_t nb = s.NB > 1 ? s.NB : 1;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(s.aux_rs), static_cast<cuuint64_t>(s.M), static_cast<cuuint64_t>(nb)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(s.aux_rs * 2),
                           static_cast<cuuint64_t>(nb > 1 ? s.aux_bs * 2 : s.aux_rs * 2 * s.M)};
  cuuint32_t box[3] = {32, 32, 1}, estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(s.aux), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : TP_ERR_CUDA;
}

// TPFFN_RASTER=1 in the environment selects the shared-operand-fastest
// orders for the per-shard GEMMs (for comparisons).
static bool raster_by_sharing() {
  static const bool on = [] {
    const char* v = getenv("TPFFN_RASTER");
    return v && v[0] == '1';
  }();
  return on;
}

// Output tensor map of a TMA-store epilogue: {cols, rows, batch} (or
// {cols, batch, rows} when the batch stride is the smaller one), 32 x 32
// boxes, 64-byte swizzle for bf16 (64-byte box rows), 128-byte for fp32.
// Columns from `cols` and rows from `rows` on lie outside the map, so a store
// never writes them.  Returns 0 or a TP_ERR_* code.
static int make_out_map(CUtensorMap* m, const void* ptr, bool fp32, int64_t cols, int64_t rows, int64_t nb,
                        int64_t rs, int64_t bs, int* swap) {
  const uint64_t es = fp32 ? 4 : 2;
  if (!ptr || reinterpret_cast<uintptr_t>(ptr) % 16 || cols < 1 || rows < 1) return TP_ERR_ALIGN;
  nb = nb > 1 ? nb : 1;
  const int64_t bst = nb > 1 ? bs : rs * rows;
  if ((rs * es) % 16 || (bst * es) % 16 || bst <= 0) return TP_ERR_ALIGN;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return TP_ERR_CUDA;
  *swap = (nb > 1 && bs < rs) ? 1 : 0;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  dims[0] = static_cast<cuuint64_t>(cols);
  box[0] = 32;
  if (!*swap) {
    dims[1] = rows;
    dims[2] = nb;
    strides[0] = rs * es;
    strides[1] = bst * es;
    box[1] = 32;
    box[2] = 1;
  } else {
    dims[1] = nb;
    dims[2] = rows;
    strides[0] = bs * es;
    strides[1] = rs * es;
    box[1] = 1;
    box[2] = 32;
  }
  CUresult r = fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : TP_ERR_CUDA;
}

// K loops of at most this many 64-wide blocks count as short (store mode 2).
constexpr int kShortKBlocks = 24;

// TPFFN_TMA_STORE=0 in the environment makes the pair GEMMs' epilogues store
// from registers, as the backward epilogues do (for comparisons).
static bool tma_store_enabled() {
  static const bool on = !getenv_flag_off("TPFFN_TMA_STORE");
  return on;
}

// TPFFN_TAIL_SPLIT=0 in the environment turns the last-wave split off (for
// comparisons).
static bool tail_split_enabled() {
  static const bool on = !getenv_flag_off("TPFFN_TAIL_SPLIT");
  return on;
}

// Launch of one pair-kernel instance (its own attribute set-up and cluster
// occupancy query per device).
template <int EPI, bool AMN, bool BMN, int TM>
static int launch_pair_inst(const GemmSpec& s, LaunchCtx& ctx, const CUtensorMap& ta, const CUtensorMap& tb,
                            const CUtensorMap& tx, const CUtensorMap& to, const CUtensorMap& to2, const Params& p) {
  using L = PairLayout<EPI, TM>;
  auto kern = tc_gemm_pair_kernel<EPI, AMN, BMN, TM>;
  static std::atomic<uint32_t> attr_done{0};
  static std::atomic<int> max_clusters[32];
  int dev = 0;
  cudaGetDevice(&dev);
  const uint32_t bit = 1u << (dev & 31);
  if (!(attr_done.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) != cudaSuccess)
      return TP_ERR_CUDA;
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    attr_done.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(pair_threads<EPI, TM>(), 1, 1);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = ctx.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int mc = max_clusters[dev & 31].load();
  if (mc <= 0) {
    cfg.gridDim = dim3(2 * (ctx.num_sms / 2), 1, 1);
    int q = 0;
    cudaError_t qe = cudaOccupancyMaxActiveClusters(&q, kern, &cfg);
    mc = (qe == cudaSuccess && q > 0) ? q : ctx.num_sms / 2;
    if (getenv("TPFFN_VERBOSE"))
      fprintf(stderr, "tpffn: pair kernel: occupancy query rc=%d clusters=%d -> using %d clusters\n", (int)qe, q, mc);
    max_clusters[dev & 31].store(mc);
  }
  long long tiles = static_cast<long long>((p.tiles_m + 1) / 2) * p.tiles_n * p.NB * p.ksplit;  // units
  if (tiles <= 0 || p.k_blocks <= 0) return TP_ERR_INVALID;
  // Last-wave split: a last wave at most half full runs its tiles as K parts
  // (at least 8 K blocks each) spread over the SM pairs the wave leaves idle
  Params pl = p;
  CUtensorMap tt;
  TailTiles tail;
  if constexpr ((EPI == EPI_OUT || EPI == EPI_GELU_FWD || EPI == EPI_SWIGLU_FWD) && TM != 0) {
    if (s.tail_ws && (EPI != EPI_OUT || s.NB == 1) && s.ksplit == 1 && !s.out_cs && !p.o_swap &&
        tail_split_enabled()) {
      const int rem = static_cast<int>(tiles % mc);
      const int kall = p.G * p.k_blocks;
      int parts = rem > 0 ? mc / rem : 0;
      if (parts > kall / 8) parts = kall / 8;
      int sw = 0;
      if (rem > 0 && rem <= kMaxTailTiles && 2 * rem <= mc && parts >= 2 &&
          static_cast<size_t>(rem) * parts * 65536 * 4 <= s.tail_ws_bytes &&
          make_out_map(&tt, s.tail_ws, true, 256, 256, static_cast<int64_t>(rem) * parts, 256, 65536, &sw) == 0 &&
          sw == 0) {
        pl.tail_tiles = rem;
        pl.tail_parts = parts;
        tail.n = rem;
        tail.parts = parts;
        for (int i = 0; i < rem; ++i) {
          int b, mp, nb;
          decode_pair_tile(pl, static_cast<int>(tiles) - rem + i, b, mp, nb);
          tail.b[i] = b;
          tail.mp[i] = mp;
          tail.nb[i] = nb;
        }
        tiles += static_cast<long long>(rem) * (parts - 1);
      }
    }
  }
  const int clusters = static_cast<int>(tiles < mc ? tiles : mc);
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  if (ctx.before) ctx.before(ctx.user, s.name, ctx.stream);
  // the tail map travels in the aux-map slot, which these epilogues do not use
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, pl.tail_parts ? tt : tx, to, to2, pl);
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  if (e != cudaSuccess || cudaPeekAtLastError() != cudaSuccess) return TP_ERR_CUDA;
  if (pl.tail_parts) {
    TailOut o;
    o.out = s.out;
    o.out_bs = s.out_bs;
    o.out_rs = s.out_rs;
    o.out2 = EPI == EPI_OUT ? nullptr : s.out2;
    o.out2_bs = s.out2_bs;
    o.out2_rs = s.out2_rs;
    o.bias = s.bias;
    o.bias_bs = s.bias_bs;
    o.bias_len = s.bias_len;
    o.M = s.M;
    o.n_store = s.n_store;
    o.act = EPI == EPI_GELU_FWD ? 1 : (EPI == EPI_SWIGLU_FWD ? 2 : 0);
    return launch_tail_fixup(s.tail_ws, tail, o, ctx, "tail_fixup");
  }
  return 0;
}

template <int EPI, bool AMN, bool BMN>
static int launch_pair(const GemmSpec& s, LaunchCtx& ctx) {
  CUtensorMap ta, tb, tx, to, to2;
  int sa = 0, sb = 0;
  int rc = make_map(&ta, s.A, BM, &sa);
  if (rc) return rc;
  rc = make_map(&tb, s.B, PAIR_BN / 2, &sb);
  if (rc) return rc;
  memset(&tx, 0, sizeof(tx));
  memset(&to, 0, sizeof(to));
  memset(&to2, 0, sizeof(to2));
  if constexpr (aux_staged<EPI>()) {
    rc = make_aux_map(&tx, s);
    if (rc) return rc;
  }
  // a K split writes fp32 parts (EPI_F32) and needs at least one K block per part
  if (s.ksplit < 1 || (s.ksplit > 1 && (EPI != EPI_F32 || s.G * ((s.K + BK - 1) / BK) < 2 * s.ksplit)))
    return TP_ERR_INVALID;
  if (s.out_cs || s.b_cs) {
    // shards merged along N: plain output epilogues, one batch, TMA stores
    const bool ok = EPI == EPI_OUT && s.NB == 1 && s.G == 1 && s.ksplit == 1 && !s.bias && tma_store_enabled() &&
                    (s.out_cs == 0 || (s.out_cs % 128 == 0 && s.N % s.out_cs == 0 && s.n_store == s.N)) &&
                    (s.b_cs == 0 || (BMN && s.b_cs % 128 == 0));
    if (!ok) return TP_ERR_UNSUPPORTED;
  }
  Params p{};
  p.ksplit = s.ksplit;
  p.dep_mode = dep_mode_for(s);
  p.out_cs = static_cast<int>(s.out_cs);
  p.b_cs = static_cast<int>(s.b_cs);
  p.raster = RASTER_GROUPED;
  // Weight-gradient GEMMs (both operands MN-major, K = tokens): the
  // per-shard operand streams through L2 with evict_first priority, which
  // keeps the one all shards share (x or dy, 67 MB for Llama-3-8B shapes)
  // there across waves.  TPFFN_L2HINT=0 turns this off (for comparisons).
  p.keep_op = 0;
  if (AMN && BMN && s.NB > 1 && s.G == 1 && l2_hint_enabled()) {
    if (s.A.bsel == 0 && s.B.bsel != 0) p.keep_op = 1;
    if (s.B.bsel == 0 && s.A.bsel != 0) p.keep_op = 2;
  }
  if (s.NB > 1 && s.G == 1 && raster_by_sharing()) {
    if (s.A.bsel == 0 && s.B.bsel != 0) p.raster = RASTER_M_FAST;
    if (s.B.bsel == 0 && s.A.bsel != 0) p.raster = RASTER_N_FAST;
  }
  p.M = static_cast<int>(s.M);
  p.N = static_cast<int>(s.N);
  p.K = static_cast<int>(s.K);
  p.NB = s.NB;
  p.G = s.G;
  p.tiles_m = static_cast<int>((s.M + BM - 1) / BM);
  p.tiles_n = static_cast<int>((s.N + PAIR_BN - 1) / PAIR_BN);
  p.k_blocks = static_cast<int>((s.K + BK - 1) / BK);
  p.a_bsel = s.A.bsel;
  p.a_gsel = s.A.gsel;
  p.b_bsel = s.B.bsel;
  p.b_gsel = s.B.gsel;
  p.a_swap = sa;
  p.b_swap = sb;
  // the cache-hinted copies use the 4-D maps of MN-major operands
  if (p.keep_op && ((AMN && p.a_swap != 2) || (BMN && p.b_swap != 2))) p.keep_op = 0;
  if (p.b_cs && p.b_swap != 2) return TP_ERR_UNSUPPORTED;  // merged shards read B through its 4-D map
  p.out = s.out;
  p.out_bs = s.out_bs;
  p.out_rs = s.out_rs;
  p.out2 = s.out2;
  p.out2_bs = s.out2_bs;
  p.out2_rs = s.out2_rs;
  p.aux = s.aux;
  p.aux_bs = s.aux_bs;
  p.aux_rs = s.aux_rs;
  p.bias = static_cast<const __nv_bfloat16*>(s.bias);
  p.bias_bs = s.bias_bs;
  p.bias_len = s.bias_len;
  p.n_store = s.n_store;
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  p.debug_skip = ctx.debug_skip_load;
  ctx.debug_skip_load = 0;
#ifdef TPFFN_INSTRUMENT
  p.dbg_slot = g_dbg_launch++ & 7;
#endif
  if constexpr (EPI == EPI_SWIGLU_BWD) {
    if (tma_store_enabled()) {
      // the SwiGLU backward epilogue's output, the interleaved [da | dg] rows
      // (the GELU backward epilogue measured slower with TMA stores --
      // dgrad_h_gelu 0.431-0.435 -> 0.442-0.460 ms on the Megatron-8.3B
      // shapes -- and keeps its register stores)
      int sw = 0;
      if (make_out_map(&to, s.out, false, s.out_rs, s.M, s.NB > 1 ? s.NB : 1, s.out_rs, s.out_bs, &sw) == 0 &&
          sw == 0)
        return launch_pair_inst<EPI, AMN, BMN, 1>(s, ctx, ta, tb, tx, to, to2, p);
    }
  } else if constexpr (!aux_staged<EPI>()) {
    if (tma_store_enabled()) {
      // output maps: out (h for the forward epilogues; fp32 for EPI_F32) and
      // out2 (a|g rows, or z); any map that cannot be made keeps the register
      // stores of the plain epilogue
      const bool f32 = EPI == EPI_F32;
      int sw1 = 0, sw2 = 0;
      // the K parts, or the shards merged along N, are further batches
      const int64_t nb = s.out_cs ? s.N / s.out_cs : (s.NB > 1 ? s.NB : 1) * s.ksplit;
      const int64_t cols1 = EPI == EPI_SWIGLU_FWD ? s.out_rs : (s.out_cs ? s.out_cs : s.n_store);
      bool ok = make_out_map(&to, s.out, f32, cols1, s.M, nb, s.out_rs, s.out_bs, &sw1) == 0;
      if (ok && s.out2) {
        const int64_t cols2 = EPI == EPI_SWIGLU_FWD ? s.out2_rs : s.n_store;
        ok = make_out_map(&to2, s.out2, false, cols2, s.M, nb, s.out2_rs, s.out2_bs, &sw2) == 0 && sw2 == sw1;
      }
      if (ok && s.out_cs && sw1) ok = false;  // merged shards store {cols, rows, shard} boxes
      if (!ok && s.out_cs) return TP_ERR_UNSUPPORTED;
      if (ok) {
        p.o_swap = sw1;
        // forward epilogues of short K loops (GPT-2-sized widths): eight
        // epilogue warps, so that the epilogue keeps up with the products
        if constexpr (EPI == EPI_GELU_FWD || EPI == EPI_SWIGLU_FWD) {
          if (static_cast<int64_t>(p.G) * p.k_blocks <= kShortKBlocks)
            return launch_pair_inst<EPI, AMN, BMN, 2>(s, ctx, ta, tb, tx, to, to2, p);
        }
        return launch_pair_inst<EPI, AMN, BMN, 1>(s, ctx, ta, tb, tx, to, to2, p);
      }
    }
  }
  return launch_pair_inst<EPI, AMN, BMN, 0>(s, ctx, ta, tb, tx, to, to2, p);
}

}  // namespace tc

#ifdef TPFFN_INSTRUMENT
extern "C" __attribute__((visibility("default"))) int tpffn_debug_counters(unsigned long long* host, int clear) {
  if (clear) tc::g_dbg_launch = 0;  // the next pair GEMM records into slot 0
  if (cudaMemcpyFromSymbol(host, tc::g_tpffn_dbg, sizeof(tc::g_tpffn_dbg)) != cudaSuccess) return 1;
  if (clear) {
    static unsigned long long zeros[8][256][8];
    if (cudaMemcpyToSymbol(tc::g_tpffn_dbg, zeros, sizeof(zeros)) != cudaSuccess) return 1;
  }
  return 0;
}
#endif

// The two-SM kernel serves every GEMM with at least 256 rows; TPFFN_PAIR=0 in
// the environment selects the one-SM kernel everywhere (for comparisons).
static bool pair_path_enabled() {
  static const bool on = [] {
    const char* v = getenv("TPFFN_PAIR");
    return !(v && v[0] == '0');
  }();
  return on;
}

bool tc_pair_path(int64_t M) { return M >= 256 && pair_path_enabled(); }

int launch_tc_gemm(const GemmSpec& s, LaunchCtx& ctx) {
  using namespace tc;
  const bool amn = s.A.mn_major != 0, bmn = s.B.mn_major != 0;
  if (s.n_store % 8) return TP_ERR_UNSUPPORTED;
  if ((s.out_cs || s.b_cs) && !(s.M >= 256 && pair_path_enabled())) return TP_ERR_UNSUPPORTED;
  if (s.M >= 256 && pair_path_enabled()) {
    switch (s.epi) {
      case EPI_SWIGLU_FWD:
        if (!amn && !bmn) return launch_pair<EPI_SWIGLU_FWD, false, false>(s, ctx);
        break;
      case EPI_GELU_FWD:
        if (!amn && !bmn) return launch_pair<EPI_GELU_FWD, false, false>(s, ctx);
        break;
      case EPI_F32:
        if (!amn && !bmn) return launch_pair<EPI_F32, false, false>(s, ctx);
        if (!amn && bmn) return launch_pair<EPI_F32, false, true>(s, ctx);
        if (amn && bmn) return launch_pair<EPI_F32, true, true>(s, ctx);  // K-split weight gradients
        break;
      case EPI_OUT:
        if (!amn && !bmn) return launch_pair<EPI_OUT, false, false>(s, ctx);
        if (!amn && bmn) return launch_pair<EPI_OUT, false, true>(s, ctx);
        if (amn && bmn) return launch_pair<EPI_OUT, true, true>(s, ctx);
        break;
      case EPI_GELU_BWD:
        if (!amn && bmn) return launch_pair<EPI_GELU_BWD, false, true>(s, ctx);
        break;
      case EPI_SWIGLU_BWD:
        if (!amn && bmn) return launch_pair<EPI_SWIGLU_BWD, false, true>(s, ctx);
        break;
      default:
        break;
    }
  }
  if (s.M <= 32 && !amn && !bmn) {  // decode: weights stream from HBM
    if (s.epi == EPI_SWIGLU_FWD) return launch_inst<256, 6, EPI_SWIGLU_FWD, false, false, 32>(s, ctx);
    if (s.epi == EPI_F32) return launch_inst<256, 6, EPI_F32, false, false, 32>(s, ctx);
  }
  switch (s.epi) {
    case EPI_SWIGLU_FWD:
      if (!amn && !bmn) return launch_inst<256, 4, EPI_SWIGLU_FWD, false, false>(s, ctx);
      break;
    case EPI_GELU_FWD:
      if (!amn && !bmn) return launch_inst<256, 4, EPI_GELU_FWD, false, false>(s, ctx);
      break;
    case EPI_F32:
      if (!amn && !bmn) return launch_inst<256, 4, EPI_F32, false, false>(s, ctx);
      if (!amn && bmn) return launch_inst<256, 4, EPI_F32, false, true>(s, ctx);
      break;
    case EPI_OUT:
      if (!amn && !bmn) return launch_inst<256, 4, EPI_OUT, false, false>(s, ctx);
      if (!amn && bmn) return launch_inst<256, 4, EPI_OUT, false, true>(s, ctx);
      if (amn && bmn) return launch_inst<256, 4, EPI_OUT, true, true>(s, ctx);
      break;
    case EPI_GELU_BWD:
      if (!amn && bmn) return launch_inst<256, 4, EPI_GELU_BWD, false, true>(s, ctx);
      break;
    case EPI_SWIGLU_BWD:
      if (!amn && bmn) return launch_inst<256, 4, EPI_SWIGLU_BWD, false, true>(s, ctx);
      break;
    default:
      break;
  }
  return TP_ERR_UNSUPPORTED;
}

}  // namespace tpffn
