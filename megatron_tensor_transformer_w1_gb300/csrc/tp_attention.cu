// tp_attention.cu -- the attention core of the head-sharded attention sublayer.
//
// "7.9 Tensor and pipeline parallelism (TP, PP)", §2.2 "Attention, sharded":
// each shard owns H/T_p query heads and Hkv/T_p key/value heads (the GQA
// divisibility rule of "S17 Tensor & Pipeline Parallelism", "Attention shards
// by head, and GQA caps the degree"), and computes the scaled dot-product
// attention of its heads from its own Q/K/V columns -- no exchange happens
// before the row-sharded output projection.  Per head, with hd = 128:
//   s_ij = q_i . k_j / sqrt(hd)  (j <= i when causal),  p_i = softmax(s_i),
//   o_i = sum_j p_ij v_j;
// backward: dP_ij = dO_i . v_j, D_i = dO_i . o_i, dS_ij = p_ij (dP_ij - D_i),
//   dq = dS k / sqrt(hd), dk = dS^T q / sqrt(hd), dv = P^T dO.
//
// Blackwell design (sm_103a), three persistent kernels of 192 threads, one
// CTA per SM:  warp 0 issues TMA copies (128-byte swizzle, zero fill past the
// end of a sequence), one lane of warp 1 issues tcgen05.mma (bf16 in, fp32
// accumulators in tensor memory), warps 2..5 own one TMEM lane -- one row of
// the 128-row tile -- each, so every row reduction (max, sum) stays in one
// thread.  Probabilities and score gradients are written by those threads to
// shared memory in the swizzled K-major layout the MMA reads; nothing of size
// S x S ever reaches global memory.
//
//  * forward (per query head and 128-query block): S = Q K^T into one of two
//    TMEM buffers while the softmax threads work on the other; online softmax
//    in the log2 domain with a lazy rescale (the running maximum only moves
//    when it grew by more than 2^8, so the O accumulator in TMEM is rarely
//    read back); O += P V; output o / l in bf16 and the log-sum-exp.
//  * dq (per query head and 128-query block, 64-key blocks): S and dP into
//    double-buffered TMEM, p recomputed from the log-sum-exp, dS to shared
//    memory, dQ += dS K in TMEM.
//  * dk/dv (per key/value head and 128-key block, 64-query blocks of every
//    query head of its GQA group): S^T and dP^T, P^T and dS^T to shared
//    memory, dV += P^T dO and dK += dS^T Q in TMEM -- the whole group's sum
//    stays in fp32 and is rounded once.
// Outputs (o, dQ, dK, dV) leave through shared memory: each softmax warp
// stages its 32 rows, then either one TMA store writes them (the forward) or
// the warp stores whole row segments (dq, dk/dv) -- a row per lane stored
// directly touches 32 rows per store instruction.
// No atomics anywhere: the results are bit-identical run to run.
//
// Every mbarrier wait is bounded (device error word + CTA abort flag, then
// in-flight copies and MMAs are drained and tensor memory is freed).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "tc_ptx.cuh"
#include "tp_internal.h"
#include "tpffn.h"

namespace tpffn {
namespace attn {
using namespace tc;

constexpr int HD = 128;            // head width
constexpr int TILE = 128 * HD * 2; // [128 rows][128 cols] bf16: two 64-column boxes
constexpr int NT = 320;            // producer warp, MMA warp, 8 softmax warps
constexpr int NSM = 256;           // softmax threads: two warps per TMEM lane quarter,
                                   // each taking half of the tile's columns

// Column geometry of the packed q/k/v buffer (see AttnSpec).
struct Geo {
  int hq_per, hk_per, sq, sk, slice;
  __device__ __forceinline__ int qcol(int h) const { return (h / hq_per) * slice + (h % hq_per) * HD; }
  __device__ __forceinline__ int kcol(int hk) const { return (hk / hk_per) * slice + sq + (hk % hk_per) * HD; }
  __device__ __forceinline__ int vcol(int hk) const { return kcol(hk) + sk; }
};

struct Params {
  Geo g;
  int B, S, H, Hkv, G, causal;
  int n_qb;    // 128-row blocks per sequence
  int items;
  __nv_bfloat16* o;
  long long o_rs;
  const __nv_bfloat16* dO;
  long long do_rs;
  float* lse;
  long long s_pad;
  float* Dv;
  __nv_bfloat16* dqkv;
  long long dqkv_rs;      // row stride of qkv and dqkv
  const __nv_bfloat16* dqkv_src;  // the packed q/k/v (read by the dq kernel's Q copy)
  float scale_log2;  // log2(e) / sqrt(hd)
  float scale;       // 1 / sqrt(hd)
  int* err;
  unsigned long long timeout_ns;
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 2^x by the SFU instruction (ex2.approx, flush-to-zero): a few ulp, far
// below the bf16 rounding the probabilities get next; 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tcgen05.mma with the A operand in tensor memory: for kind::f16 each 32-bit
// TMEM cell of a lane holds two consecutive K elements of that row (the
// lower K index in the low half), so one K = 16 step spans 8 columns.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of a 128-byte-swizzled tile (version 1, SBO 1024).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// K-major operand: `rows` rows x 128 K-columns held as two 64-column boxes of
// rows*128 bytes; K step ks covers columns [16 ks, 16 ks + 16).
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int rows, int ks) {
  return sw128_desc(tile + static_cast<uint32_t>((ks >> 2) * rows * 128 + (ks & 3) * 32), 16);
}
// MN-major operand: `krows` rows along K, 128 M/N columns held as two boxes
// of krows*128 bytes; K step ks covers rows [16 ks, 16 ks + 16).
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int krows, int ks) {
  return sw128_desc(tile + static_cast<uint32_t>(ks * 2048), static_cast<uint32_t>(krows * 128));
}
// Instruction descriptor, kind::f16, M = 128, bf16 x bf16 -> fp32.
__host__ __device__ constexpr uint32_t idesc(int N, int amn, int bmn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(amn) << 15) |
         (static_cast<uint32_t>(bmn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (8u << 24);
}
// Address of 16-byte chunk col8 (= column / 8) of row r of a thread-written
// K-major swizzled tile of `rows` rows (the layout TMA's 128-byte swizzle
// gives: chunk index XOR row mod 8 inside each 1024-byte group of 8 rows).
__device__ __forceinline__ uint32_t sw_chunk(uint32_t tile, int rows, int r, int col8) {
  return tile + static_cast<uint32_t>((col8 >> 3) * rows * 128 + r * 128 + (((col8 & 7) ^ (r & 7)) << 4));
}

struct Waiter {
  volatile int* abort_flag;
  int* err;
  unsigned long long timeout_ns;
  __device__ __forceinline__ bool operator()(uint64_t* bar, uint32_t parity) const {
    return wait_bounded_raw(bar, parity, abort_flag, err, timeout_ns, true);
  }
  // drain wait: ignores the abort flag
  __device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) const {
    wait_bounded_raw(bar, parity, abort_flag, err, timeout_ns, false);
  }
  // warp-uniform wait of the softmax warps
  __device__ __forceinline__ bool warp(uint64_t* bar, uint32_t parity) const {
    const bool ok = wait_bounded_raw(bar, parity, abort_flag, err, timeout_ns, true);
    return __all_sync(0xffffffffu, ok) != 0;
  }
};

// Softmax-side hand-overs arrive once per warp (NSW arrivals complete a
// phase): every lane has finished its tensor-memory / shared-memory writes and
// the fence that publishes them, the warp reconverges, and lane 0 arrives.
// 256 per-thread arrivals on one barrier serialise on its shared-memory word.
constexpr int NSW = NSM / 32;
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

#ifdef TPFFN_INSTRUMENT
// Per-CTA cycle counters of the forward kernel, for performance work only
// (not in normal builds): see tpffn_attn_debug_counters.
__device__ unsigned long long g_attn_dbg[256][24];
__device__ unsigned long long g_attn_bwd_dbg[2][256][16];  // [dq, dk/dv][CTA][counter]
#define AT_T0(v) const long long v = clock64()
#define AT_ADD(slot, since) atomicAdd(&g_attn_dbg[blockIdx.x & 255][slot], (unsigned long long)(clock64() - (since)))
#define AT_CNT(slot) atomicAdd(&g_attn_dbg[blockIdx.x & 255][slot], 1ull)
#define BW_ADD(k, slot, since) \
  atomicAdd(&g_attn_bwd_dbg[k][blockIdx.x & 255][slot], (unsigned long long)(clock64() - (since)))
#define BW_CNT(k, slot) atomicAdd(&g_attn_bwd_dbg[k][blockIdx.x & 255][slot], 1ull)
#else
#define AT_T0(v)
#define AT_ADD(slot, since)
#define AT_CNT(slot)
#define BW_ADD(k, slot, since)
#define BW_CNT(k, slot)
#endif

// Query-major items, heaviest first under the causal mask: item ->
// (128-row block, sequence, head).
__device__ __forceinline__ void decode_item(const Params& p, int item, int heads, bool heavy_last_block, int& blk,
                                            int& b, int& h) {
  const int per = p.B * heads;
  const int r = item / per;
  blk = heavy_last_block ? p.n_qb - 1 - r : r;
  const int bh = item - r * per;
  b = bh / heads;
  h = bh - b * heads;
}

// The n-th work item of this CTA.  Items are numbered heaviest first, and the
// CTAs take them in rounds of gridDim.x, in alternating directions (CTA c
// takes item c of even rounds and item gridDim.x - 1 - c of odd ones), so
// every CTA's sum of item lengths is within one item of the mean: the
// causal mask makes the items' lengths fall off linearly, and plain
// round-robin left the most loaded CTA 10 % (8.3B block) and 7 % (Llama-3-8B)
// above it.  Per CTA the items increase with n.
__device__ __forceinline__ int item_of(uint32_t n) {
  const uint32_t G = gridDim.x, c = blockIdx.x;
  return static_cast<int>(n * G + ((n & 1u) ? G - 1u - c : c));
}

// Packs 32 fp32 values (times mul) into 16 bf16 pairs.
__device__ __forceinline__ void pack_row_bf16(uint32_t* dst, const uint32_t (&r)[32], float mul) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    dst[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
}

// A warp's 32 output rows (row r held by lane r as 16 NC bf16 pairs, NC
// 32-column chunks) go to global memory through the warp's own staging
// buffer of 32 x 64 NC bytes: each lane writes its row (stage_row_chunk, one
// 32-column chunk at a time), then the warp reads the rows back so that every
// store instruction covers whole 64 NC-byte row segments of 32 / (4 NC) rows
// (store_staged_rows), instead of 16 bytes of each of 32 rows (a row per
// lane, stored directly, costs one L1 wavefront per row and instruction).
// Row r goes to base + r * rs if r < valid_rows.  The staging rows are
// swizzled (16-byte chunk k of row r at k ^ (r & 7), or k ^ ((r >> 1) & 3)
// for 64-byte rows) so that both passes are free of bank conflicts.
template <int NC>
__device__ __forceinline__ int stage_swz(int k, int r) {
  return NC == 2 ? (k ^ (r & 7)) : (k ^ ((r >> 1) & 3));
}
template <int NC>
__device__ __forceinline__ void stage_row_chunk(uint32_t buf, int c, const uint32_t (&pk)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    st_shared_v4(buf + static_cast<uint32_t>(lane * 64 * NC + 16 * stage_swz<NC>(4 * c + k, lane)), pk[4 * k],
                 pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
}
template <int NC>
__device__ __forceinline__ void store_staged_rows(uint32_t buf, __nv_bfloat16* base, long long rs, int valid_rows) {
  constexpr int CH = 4 * NC;  // 16-byte chunks per row
  constexpr int RPI = 32 / CH;  // rows per store instruction
  const int lane = threadIdx.x & 31;
  __syncwarp();
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int r = i * RPI + lane / CH, k = lane % CH;
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(buf + static_cast<uint32_t>(r * 64 * NC + 16 * stage_swz<NC>(k, r))));
    if (r < valid_rows) *reinterpret_cast<uint4*>(base + r * rs + k * 8) = v;
  }
  __syncwarp();  // the buffer is rewritten only after every lane has read it
}

// ================================================================ forward
constexpr int F_Q = 0;                // 2 buffers: the next item's Q loads during this one
constexpr int F_K = F_Q + 2 * TILE;   // 2 stages
constexpr int F_V = F_K + 2 * TILE;   // 2 stages
constexpr int F_X = F_V + 2 * TILE;   // row max / sum exchange [2 halves][128 rows] fp32
constexpr int F_BAR = F_X + 1024;
constexpr int F_O = F_BAR + 1024;     // output staging, 4 KB per softmax warp (1024-byte aligned)
constexpr int F_SMEM = F_O + 8 * 4096 + 1024;

// P never leaves the chip: the softmax threads write it in bf16 over the S
// block it came from (two probabilities per 32-bit cell), and the PV product
// reads its A operand from tensor memory.  tcgen05 products of the CTA
// execute in issue order, so S_{j+2}, issued after PV_j, overwrites that
// buffer only after PV_j has read it.  The "PV done" barriers, indexed by the
// running count g of P blocks (g & 1), serve the lazy rescale of O and the
// final read of O.
// The two softmax warps of a row split each key block into halves, and each
// half is an independent online softmax: its own running maximum, row sum
// and O accumulator (O_0 at columns 256.., O_1 at 384..; its P over the
// first 32 of its own 64 S columns).  The halves meet once per work item,
// when O = (O_0 2^{m_0 - m} + O_1 2^{m_1 - m}) / l is written out, instead of
// exchanging their maxima for every block.
__global__ void __launch_bounds__(NT, 1) attn_fwd_kernel(const __grid_constant__ CUtensorMap tq,
                                                         const __grid_constant__ CUtensorMap to, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + F_BAR);
  uint64_t* q_full = bar + 29;  // [2] (placed after the others)
  uint64_t* q_empty = bar + 31; // [2]
  uint64_t* k_full = bar + 2;   // [2]
  // (bar + 4, 5 and 8, 9 unused: a K stage is free once the S product that read
  // it completes -- s_full of the same index, as K, V, S and PV all count the
  // same blocks -- and a V stage once its PV completes -- pv_done)
  uint64_t* v_full = bar + 6;   // [2]
  uint64_t* s_full = bar + 10;  // [2]
  // (bar + 12, 13 unused: an S buffer is rewritten only by an S product issued
  // after the PV product of the block it held, which waited for that block's P,
  // so the softmax warps have read it)
  // one "P written" barrier per S buffer: the softmax warps may run a block
  // ahead of the MMA thread's wait, and a single barrier would then advance
  // two phases before the wait sees the first
  uint64_t* p_full = bar + 14;  // [2]
  uint64_t* pv_done = bar + 16; // [2]
  uint64_t* o_empty = bar + 18;
  uint64_t* drain = bar + 19;
  uint64_t* pair_x = bar + 20;  // [4] both halves of a row wrote their value
  uint64_t* pair_r = bar + 24;  // [4] both halves read their partner's value
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 33);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 33) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&pv_done[i], 1);
      mbar_init(&p_full[i], NSW);
    }
    mbar_init(o_empty, NSW);
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&pair_x[i], 64);
      mbar_init(&pair_r[i], 64);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tq);
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S buffers at columns 0 and 128, O_0 at 256, O_1 at 384
  const Waiter W{abort_flag, p.err, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int q_last[2] = {-1, -1}, k_last[2] = {-1, -1}, v_last[2] = {-1, -1};
      uint32_t kv = 0, it = 0;
      bool ok = true;
      for (int item = item_of(0); item < p.items && ok; item = item_of(++it)) {
        int qb, b, h;
        decode_item(p, item, p.H, p.causal != 0, qb, b, h);
        const int nkb = p.causal ? qb + 1 : p.n_qb;
        const int qbuf = it & 1;
        const uint32_t qph = (it >> 1) & 1u;
        AT_T0(t16);
        if (!W(&q_empty[qbuf], qph ^ 1u)) break;
        AT_ADD(16, t16);
        mbar_arrive_expect_tx(&q_full[qbuf], TILE);
        const int qc = p.g.qcol(h);
        tma_load_3d(smem + F_Q + qbuf * TILE, &tq, &q_full[qbuf], qc, qb * 128, b);
        tma_load_3d(smem + F_Q + qbuf * TILE + TILE / 2, &tq, &q_full[qbuf], qc + 64, qb * 128, b);
        q_last[qbuf] = static_cast<int>(qph);
        const int hk = h / p.G, kc = p.g.kcol(hk), vc = p.g.vcol(hk);
        for (int j = 0; j < nkb; ++j, ++kv) {
          const int st = kv & 1;
          const uint32_t ph = (kv >> 1) & 1u;
          AT_T0(t17);
          if (!W(&s_full[st], ph ^ 1u)) { ok = false; break; }  // S of block kv-2 has read K
          AT_ADD(17, t17);
          uint8_t* kd = smem + F_K + st * TILE;
          mbar_arrive_expect_tx(&k_full[st], TILE);
          tma_load_3d(kd, &tq, &k_full[st], kc, j * 128, b);
          tma_load_3d(kd + TILE / 2, &tq, &k_full[st], kc + 64, j * 128, b);
          k_last[st] = static_cast<int>(ph);
          AT_T0(t18);
          if (!W(&pv_done[st], ph ^ 1u)) { ok = false; break; }  // PV of block kv-2 has read V
          AT_ADD(18, t18);
          uint8_t* vd = smem + F_V + st * TILE;
          mbar_arrive_expect_tx(&v_full[st], TILE);
          tma_load_3d(vd, &tq, &v_full[st], vc, j * 128, b);
          tma_load_3d(vd + TILE / 2, &tq, &v_full[st], vc + 64, j * 128, b);
          v_last[st] = static_cast<int>(ph);
        }
      }
      // every issued copy lands before the CTA may exit
      for (int s = 0; s < 2; ++s) {
        if (q_last[s] >= 0) W.drain(&q_full[s], static_cast<uint32_t>(q_last[s]));
        if (k_last[s] >= 0) W.drain(&k_full[s], static_cast<uint32_t>(k_last[s]));
        if (v_last[s] >= 0) W.drain(&v_full[s], static_cast<uint32_t>(v_last[s]));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc(128, 0, 0);   // S = Q K^T
      constexpr uint32_t ID_PV = idesc(128, 0, 1);  // O += P V (V: N = hd contiguous)
      uint32_t kv = 0, pg = 0, it = 0;
      bool ok = true;
      AT_T0(t_mma);
      // S = Q K^T of K/V block n (the n-th block of this CTA, all items in
      // turn) into S buffer n & 1; `last`: the item's last block, after which
      // its Q buffer is free
      auto issue_s = [&](uint32_t n, uint32_t qa, bool last, int qbuf) -> bool {
        const int st = n & 1;
        AT_T0(t0);
        if (!W(&k_full[st], (n >> 1) & 1u)) return false;
        AT_ADD(0, t0);
        tc_fence_after();
        const uint32_t ka = smem_u32(smem + F_K + st * TILE);
        AT_T0(t19);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tmem + (n & 1u) * 128, kdesc(qa, 128, ks), kdesc(ka, 128, ks), ID_S, ks > 0 ? 1u : 0u);
        AT_ADD(19, t19);
        AT_T0(t20);
        umma_commit(&s_full[n & 1u]);
        if (last) umma_commit(&q_empty[qbuf]);  // Q free once the item's last S is done
        AT_ADD(20, t20);
        return true;
      };
      auto q_addr = [&](int qbuf) { return smem_u32(smem + F_Q + qbuf * TILE); };
      bool s0_issued = false;  // this item's first S went out during the previous item
      for (int item = item_of(0); item < p.items && ok; item = item_of(++it)) {
        int qb, b, h;
        decode_item(p, item, p.H, p.causal != 0, qb, b, h);
        const int nkb = p.causal ? qb + 1 : p.n_qb;
        const int qbuf = it & 1;
        if (!s0_issued) {
          if (!W(&q_full[qbuf], (it >> 1) & 1u)) break;
          tc_fence_after();
          if (!issue_s(kv, q_addr(qbuf), nkb == 1, qbuf)) break;
        }
        s0_issued = false;
        const uint32_t qa = q_addr(qbuf);
        for (int j = 0; j < nkb; ++j) {
          if (j + 1 < nkb) {
            if (!issue_s(kv + j + 1, qa, j + 2 == nkb, qbuf)) { ok = false; break; }
          } else if (item_of(it + 1) < p.items) {
            // the next item's first S, ahead of this item's last PV: the
            // softmax warps take it before they read this item's O out
            int qb2, b2, h2;
            decode_item(p, item_of(it + 1), p.H, p.causal != 0, qb2, b2, h2);
            const int nkb2 = p.causal ? qb2 + 1 : p.n_qb;
            const int qbuf2 = (it + 1) & 1;
            if (!W(&q_full[qbuf2], ((it + 1) >> 1) & 1u)) { ok = false; break; }
            tc_fence_after();
            if (!issue_s(kv + nkb, q_addr(qbuf2), nkb2 == 1, qbuf2)) { ok = false; break; }
            s0_issued = true;
          }
          AT_T0(t2);
          if (!W(&p_full[pg & 1u], (pg >> 1) & 1u)) { ok = false; break; }
          AT_ADD(2, t2);
          AT_T0(t3);
          if (j == 0 && !W(o_empty, (it & 1u) ^ 1u)) { ok = false; break; }
          AT_ADD(3, t3);
          const uint32_t n = kv + j;
          const int st = n & 1;
          AT_T0(t4);
          if (!W(&v_full[st], (n >> 1) & 1u)) { ok = false; break; }
          AT_ADD(4, t4);
          AT_CNT(6);
          tc_fence_after();
          const uint32_t va = smem_u32(smem + F_V + st * TILE);
          // key half kh: its P over the first 32 of S columns [64 kh, 64 kh + 64), into O_kh
          const uint32_t pa = tmem + (n & 1u) * 128;
          AT_T0(t21);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ta(tmem + 256 + (ks >> 2) * 128, pa + (ks >> 2) * 64 + (ks & 3) * 8, mndesc(va, 128, ks),
                         ID_PV, (j > 0 || (ks & 3) > 0) ? 1u : 0u);
          AT_ADD(21, t21);
          AT_T0(t22);
          umma_commit(&pv_done[pg & 1u]);
          AT_ADD(22, t22);
          ++pg;
        }
        kv += nkb;
      }
      AT_ADD(5, t_mma);
      umma_commit(drain);  // all issued MMAs complete before tensor memory is released
      W.drain(drain, 0u);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps 2..9
    // warp w serves TMEM lanes 32 (w % 4) .. (rows of the tile) and the
    // columns [64 half, 64 half + 64) of the S and O accumulators
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* xs = reinterpret_cast<float*>(smem + F_X);
    uint32_t xe = 0;  // exchanges done with the partner warp
    // swap a per-row value with the partner half (bounded waits)
    auto exchange = [&](float mine, float& theirs) -> bool {
      if (xe > 0 && !W.warp(&pair_r[quarter], (xe - 1) & 1u)) return false;
      xs[half * 128 + row] = mine;
      mbar_arrive(&pair_x[quarter]);
      if (!W.warp(&pair_x[quarter], xe & 1u)) return false;
      theirs = xs[(1 - half) * 128 + row];
      mbar_arrive(&pair_r[quarter]);
      ++xe;
      return true;
    };
    uint32_t sc = 0, pg = 0;
#ifdef TPFFN_INSTRUMENT
    const bool rec = warp == 2 && lane == 0;
    const long long t_sm = clock64();
#endif
    // Each item's O is read out after the next item's block 0 (the MMA thread
    // issued that S ahead of the item's last PV), so that the tensor pipe
    // has the next P block during the read-out; a final pass without blocks
    // reads out the last item.
    bool pend = false;  // a read-out is pending
    float pf0 = 0.f, pf1 = 0.f, pinv = 1.f, plse = 0.f;
    int pb = 0, ph = 0, pqpos = 0;
    uint32_t pglast = 0;
    for (uint32_t n_item = 0;; ++n_item) {
      const int item = item_of(n_item);
      const bool has = item < p.items;
      int qb = 0, b = 0, h = 0;
      if (has) decode_item(p, item, p.H, p.causal != 0, qb, b, h);
      const int nkb = !has ? 1 : (p.causal ? qb + 1 : p.n_qb);
      const int qpos = qb * 128 + row;
      float m_used = -INFINITY, l = 0.f;  // this key half's running maximum (log2 units) and row sum
      bool ok = true;
      for (int j = 0; j < nkb; ++j) {
        if (has) {
          const uint32_t g = pg + j;
          const uint32_t buf = sc & 1u, use = sc >> 1;
          ++sc;
          AT_T0(t7);
          if (!W.warp(&s_full[buf], use & 1u)) { ok = false; break; }
#ifdef TPFFN_INSTRUMENT
          if (rec) AT_ADD(7, t7);
#endif
          AT_T0(t8);
          tc_fence_after();
          uint32_t r[64];
          tmem_ld32(tl + buf * 128 + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld32(tl + buf * 128 + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_wait_ld();
#ifdef TPFFN_INSTRUMENT
          if (rec) AT_ADD(8, t8);
#endif
          AT_T0(t9);
          const int kbase = j * 128 + half * 64;
          // only the diagonal block (causal) and a block past the end of the
          // sequence hold invisible keys; elsewhere every key is visible
          if ((p.causal && j * 128 + 127 > qb * 128) || j * 128 + 128 > p.S) {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const int key = kbase + c;
              const bool vis = key < p.S && (!p.causal || key <= qpos);
              r[c] = vis ? r[c] : __float_as_uint(-INFINITY);
            }
          }
          // this half's maximum of the raw scores: eight chains
          float m8[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) m8[c] = __uint_as_float(r[c]);
#pragma unroll
          for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(r[c]));
          const float mh = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
#ifdef TPFFN_INSTRUMENT
          if (rec) AT_ADD(9, t9);
#endif
          const float mx = mh * p.scale_log2;
          float alpha = 1.f;
          bool rescale = false;
          if (m_used == -INFINITY) {
            m_used = mx;  // first visible key of this half (O and l are still zero)
          } else if (mx > m_used + 8.f) {  // lazy rescale: p stays <= 2^8 otherwise
            alpha = ex2(m_used - mx);
            m_used = mx;
            rescale = true;
          }
          if (__any_sync(0xffffffffu, rescale)) {
            // O_half must hold PV g-1 before it is rescaled
            const uint32_t gp = g - 1;
            if (!W.warp(&pv_done[gp & 1u], (gp >> 1) & 1u)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              const uint32_t ta = tl + 256 + half * 128 + c * 32;
              tmem_ld32(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(ta, o);
            }
            tmem_wait_st();
          }
          // P (bf16 pairs) over the first 32 of this half's 64 S columns, which
          // this thread has already read
          AT_T0(t12);
          const float neg_m = m_used == -INFINITY ? 0.f : -m_used;  // no visible key yet: every p is 0
          float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float e0 = ex2(fmaf(__uint_as_float(r[2 * c]), p.scale_log2, neg_m));
            const float e1 = ex2(fmaf(__uint_as_float(r[2 * c + 1]), p.scale_log2, neg_m));
            l8[c & 7] += e0 + e1;
            pk[c] = pack_bf16x2(e0, e1);
          }
          tmem_st32(tl + buf * 128 + half * 64, pk);
          tmem_wait_st();
          l = l * alpha + (((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7])));
          tc_fence_before();
          warp_arrive(&p_full[g & 1u]);
#ifdef TPFFN_INSTRUMENT
          if (rec) {
            AT_ADD(12, t12);
            if (rescale) AT_CNT(13);
          }
#endif
        }
        if (j == 0 && pend) {
          AT_T0(t14);
          pend = false;
          if (!W.warp(&pv_done[pglast & 1u], (pglast >> 1) & 1u)) { ok = false; break; }
          tc_fence_after();
          const bool row_ok = pqpos < p.S;
          // this warp's 32 rows x 64 columns of o, staged in the 128-byte
          // swizzle of the output tensor map and written by one TMA store
          // (rows past the sequence are outside the map)
          uint8_t* obuf = smem + F_O + (warp - 2) * 4096;
          if (lane == 0) bulk_wait_read<0>();  // the previous item's store has read the buffer
          __syncwarp();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o0[32], o1[32], pk[16];
            tmem_ld32(tl + 256 + half * 64 + c * 32, o0);
            tmem_ld32(tl + 384 + half * 64 + c * 32, o1);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o0[i] = __float_as_uint(fmaf(__uint_as_float(o0[i]), pf0, __uint_as_float(o1[i]) * pf1));
            pack_row_bf16(pk, o0, pinv);
            stage_row_chunk<2>(smem_u32(obuf), c, pk);
          }
          // O has been read: the next item's PV products may start
          tc_fence_before();
          fence_proxy_async_smem();
          warp_arrive(o_empty);
          const int r0 = pqpos - lane;  // this warp's first row
          if (lane == 0) {
            if (r0 < p.S) tma_store_3d(&to, obuf, ph * HD + half * 64, r0, pb);
            bulk_commit();
          }
          // rows past the sequence get lse = +inf: the backward reads them as p = 0
          if (half == 0) p.lse[(static_cast<long long>(pb) * p.H + ph) * p.s_pad + pqpos] = row_ok ? plse : INFINITY;
#ifdef TPFFN_INSTRUMENT
          if (rec) AT_ADD(14, t14);
#endif
        }
      }
      if (!ok || !has) break;
      pglast = pg + nkb - 1;
      pg += nkb;
      // the two halves meet: m = max(m_0, m_1), l = sum of l_h 2^{m_h - m}
      float mo, lo;
      if (!exchange(m_used, mo) || !exchange(l, lo)) break;
      const float m = fmaxf(m_used, mo);  // finite: every row sees at least one key
      const float f_mine = ex2(m_used - m), f_other = ex2(mo - m);
      const float lsum = l * f_mine + lo * f_other;
      pf0 = half == 0 ? f_mine : f_other;
      pf1 = half == 0 ? f_other : f_mine;
      pinv = 1.f / lsum;
      plse = m + log2f(lsum);
      pb = b;
      ph = h;
      pqpos = qpos;
      pend = true;
    }
#ifdef TPFFN_INSTRUMENT
    if (rec) AT_ADD(15, t_sm);
#endif
    if (lane == 0) bulk_wait_all();  // the output stores are done before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================ D = rowsum(dO * o)
__global__ void attn_prep_kernel(const Params p) {
  // one thread per (sequence, head, padded position); positions past the
  // sequence get D = 0
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(p.B) * p.H * p.s_pad;
  if (idx >= total) return;
  const int i = static_cast<int>(idx % p.s_pad);
  const long long bh = idx / p.s_pad;
  const int h = static_cast<int>(bh % p.H), b = static_cast<int>(bh / p.H);
  float acc = 0.f;
  if (i < p.S) {
    const long long tok = static_cast<long long>(b) * p.S + i;
    const __nv_bfloat16* o = p.o + tok * p.o_rs + h * HD;
    const __nv_bfloat16* g = p.dO + tok * p.do_rs + h * HD;
#pragma unroll 4
    for (int c = 0; c < HD; c += 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(o + c);
      const uint4 d = *reinterpret_cast<const uint4*>(g + c);
      const __nv_bfloat162* ah = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* dh = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 af = __bfloat1622float2(ah[k]), df = __bfloat1622float2(dh[k]);
        acc = fmaf(af.x, df.x, acc);
        acc = fmaf(af.y, df.y, acc);
      }
    }
  }
  p.Dv[idx] = acc;
}

// ================================================================ dq
constexpr int DQ_KV = 3;               // key/value stages of 128 keys in shared memory
constexpr int Q_K = 0;
constexpr int Q_V = Q_K + DQ_KV * TILE;
constexpr int Q_DS = Q_V + DQ_KV * TILE;  // dS [128 q][128 keys] bf16, K-major
constexpr int Q_BAR = Q_DS + TILE;
constexpr int Q_SMEM = Q_BAR + 256 + 1024;
constexpr uint32_t DQ_S = 0, DQ_DP = 128, DQ_ACC = 256, DQ_QA = 384, DQ_DOA = 448;  // TMEM columns

// Blocks of 128 keys: S = Q K^T and dP = dO V^T are N = 128 products (an
// N = 64 tcgen05.mma costs as many cycles as ~90 % of an N = 128 one), with
// Q and dO, fixed for the item, as A operands in tensor memory (bf16 pairs,
// 64 columns each; the softmax warps copy them in at the start of each item,
// after the previous item's last S/dP has completed).  S and dP are freed as
// soon as the softmax warps have read them, so the next block's products run
// while they compute dS; dS goes to shared memory for dQ += dS K.
// This lane's row of 64 bf16 (zero when !ok) as 32 bf16 pairs.
__device__ __forceinline__ void load_row_pairs(const __nv_bfloat16* src, bool ok, uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 v = ok ? *reinterpret_cast<const uint4*>(src + c * 8) : make_uint4(0u, 0u, 0u, 0u);
    r[4 * c] = v.x;
    r[4 * c + 1] = v.y;
    r[4 * c + 2] = v.z;
    r[4 * c + 3] = v.w;
  }
}

// A warp's 32 rows of 64 bf16 (128 bytes each; row r at src + r * rs, zero
// from valid_rows on), lane r ending up with row r's 32 bf16 pairs.  Loaded
// coalesced -- load i brings row 8 g + i to lanes 8 g .. 8 g + 7, one 16-byte
// chunk each, so an instruction covers four whole rows instead of 16 bytes of
// each of 32 -- then transposed within each group of 8 lanes (chunk c of row
// 8 g + i, held by lane 8 g + c in slot i, moves to lane 8 g + i, slot c) by
// three butterfly stages of register shuffles.
__device__ __forceinline__ void load_rows_transposed(const __nv_bfloat16* src, long long rs, int valid_rows,
                                                     uint32_t (&r)[32]) {
  const int lane = threadIdx.x & 31, g = lane >> 3, c = lane & 7;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = 8 * g + i;
    v[i] = row < valid_rows ? *reinterpret_cast<const uint4*>(src + row * rs + c * 8) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int s = 1; s < 8; s <<= 1) {
    const bool hi = (c & s) != 0;
#pragma unroll
    for (int i0 = 0; i0 < 8; ++i0) {
      if (i0 & s) continue;
      const int i1 = i0 | s;
      // the lane with bit s clear gives slot i1 and takes the partner's slot
      // i0 there; its partner gives slot i0 and takes slot i1 there
      const uint4 send = hi ? v[i0] : v[i1];
      uint4 recv;
      recv.x = __shfl_xor_sync(0xffffffffu, send.x, s);
      recv.y = __shfl_xor_sync(0xffffffffu, send.y, s);
      recv.z = __shfl_xor_sync(0xffffffffu, send.z, s);
      recv.w = __shfl_xor_sync(0xffffffffu, send.w, s);
      if (hi) v[i0] = recv;
      else v[i1] = recv;
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    r[4 * k] = v[k].x;
    r[4 * k + 1] = v[k].y;
    r[4 * k + 2] = v[k].z;
    r[4 * k + 3] = v[k].w;
  }
}

// SHORT (sequences of at most 2048 tokens, so items of at most 16 key
// blocks): the next item's Q and dO rows are prefetched into L2 at the start
// of an item and loaded coalesced; long items keep the row-per-lane loads
// (measured: the short form gains 7 % on 1024-token sequences, and its code
// in the same kernel cost the 8192-token case 4 %).
template <bool SHORT>
__global__ void __launch_bounds__(NT, 1) attn_dq_kernel(const __grid_constant__ CUtensorMap tq128, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Q_BAR);
  uint64_t* qdo_ready = bar + 0;  // softmax warps wrote Q and dO of the item into TMEM
  uint64_t* qdo_free = bar + 1;   // the item's last S/dP has completed
  uint64_t* k_full = bar + 2;     // [DQ_KV]
  uint64_t* k_empty = bar + 5;    // [DQ_KV]
  uint64_t* v_full = bar + 8;     // [DQ_KV]
  uint64_t* v_empty = bar + 11;   // [DQ_KV]
  uint64_t* sdp_full = bar + 14;
  uint64_t* sdp_empty = bar + 15;
  uint64_t* ds_full = bar + 16;
  // (bar + 17 unused: the dS buffer is free once the previous block's dQ
  // product has read it, and that product's commit frees its K stage too)
  uint64_t* dq_full = bar + 18;
  uint64_t* dq_empty = bar + 19;
  uint64_t* drain = bar + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 21);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 21) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(qdo_ready, NSW);
    mbar_init(qdo_free, 1);
    for (int i = 0; i < DQ_KV; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(sdp_empty, NSW);
    mbar_init(ds_full, NSW);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, NSW);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tq128);
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{abort_flag, p.err, p.timeout_ns};

  auto nkb_of = [&](int qb) { return p.causal ? qb + 1 : p.n_qb; };

  if (warp == 0) {
    if (lane == 0) {
      int k_last[DQ_KV], v_last[DQ_KV];
      for (int i = 0; i < DQ_KV; ++i) k_last[i] = v_last[i] = -1;
      uint32_t kc = 0, it = 0;
      bool ok = true;
      for (int item = item_of(0); item < p.items && ok; item = item_of(++it)) {
        int qb, b, h;
        decode_item(p, item, p.H, p.causal != 0, qb, b, h);
        const int nkb = nkb_of(qb);
        const int hk = h / p.G, kcol = p.g.kcol(hk), vcol = p.g.vcol(hk);
        for (int j = 0; j < nkb; ++j, ++kc) {
          const int st = kc % DQ_KV;
          const uint32_t ph = (kc / DQ_KV) & 1u;
          if (!W(&k_empty[st], ph ^ 1u)) { ok = false; break; }
          uint8_t* kd = smem + Q_K + st * TILE;
          mbar_arrive_expect_tx(&k_full[st], TILE);
          tma_load_3d(kd, &tq128, &k_full[st], kcol, j * 128, b);
          tma_load_3d(kd + TILE / 2, &tq128, &k_full[st], kcol + 64, j * 128, b);
          k_last[st] = static_cast<int>(ph);
          if (!W(&v_empty[st], ph ^ 1u)) { ok = false; break; }
          uint8_t* vd = smem + Q_V + st * TILE;
          mbar_arrive_expect_tx(&v_full[st], TILE);
          tma_load_3d(vd, &tq128, &v_full[st], vcol, j * 128, b);
          tma_load_3d(vd + TILE / 2, &tq128, &v_full[st], vcol + 64, j * 128, b);
          v_last[st] = static_cast<int>(ph);
        }
      }
      for (int s2 = 0; s2 < DQ_KV; ++s2) {
        if (k_last[s2] >= 0) W.drain(&k_full[s2], static_cast<uint32_t>(k_last[s2]));
        if (v_last[s2] >= 0) W.drain(&v_full[s2], static_cast<uint32_t>(v_last[s2]));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc(128, 0, 0);   // S = Q K^T, dP = dO V^T (A in TMEM)
      constexpr uint32_t ID_DQ = idesc(128, 0, 1);  // dQ += dS K (K: N = hd contiguous)
      const uint32_t dsa = smem_u32(smem + Q_DS);
      uint32_t kc = 0, it = 0, blk = 0;
      bool ok = true;
      AT_T0(t_mma);
      for (int item = item_of(0); item < p.items && ok; item = item_of(++it)) {
        int qb, b, h;
        decode_item(p, item, p.H, p.causal != 0, qb, b, h);
        const int nkb = nkb_of(qb);
        if (!W(qdo_ready, it & 1u)) break;
        tc_fence_after();
        auto issue_sdp = [&](int j) -> bool {
          const uint32_t n = kc + j;
          const int st = n % DQ_KV;
          const uint32_t ph = (n / DQ_KV) & 1u;
          AT_T0(t0);
          if (!W(&k_full[st], ph) || !W(&v_full[st], ph)) return false;
          // S/dP buffer free once the softmax warps have read the previous block
          if (blk > 0 && !W(sdp_empty, (blk - 1) & 1u)) return false;
          BW_ADD(0, 0, t0);
          AT_T0(t1);
          tc_fence_after();
          const uint32_t ka = smem_u32(smem + Q_K + st * TILE), va = smem_u32(smem + Q_V + st * TILE);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ta(tmem + DQ_S, tmem + DQ_QA + ks * 8, kdesc(ka, 128, ks), ID_S, ks > 0 ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ta(tmem + DQ_DP, tmem + DQ_DOA + ks * 8, kdesc(va, 128, ks), ID_S, ks > 0 ? 1u : 0u);
          umma_commit(sdp_full);
          umma_commit(&v_empty[st]);
          if (j == nkb - 1) umma_commit(qdo_free);  // Q, dO of the item no longer read
          ++blk;
          BW_ADD(0, 1, t1);
          return true;
        };
        if (!issue_sdp(0)) break;
        for (int j = 0; j < nkb && ok; ++j) {
          if (j + 1 < nkb && !issue_sdp(j + 1)) { ok = false; break; }
          AT_T0(t2);
          if (!W(ds_full, (blk - (j + 1 < nkb ? 2 : 1)) & 1u)) { ok = false; break; }
          BW_ADD(0, 2, t2);
          AT_T0(t3);
          if (j == 0 && !W(dq_empty, (it & 1u) ^ 1u)) { ok = false; break; }
          BW_ADD(0, 3, t3);
          BW_CNT(0, 4);
          AT_T0(t5);
          tc_fence_after();
          const int st = (kc + j) % DQ_KV;
          const uint32_t ka = smem_u32(smem + Q_K + st * TILE);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16(tmem + DQ_ACC, kdesc(dsa, 128, ks), mndesc(ka, 128, ks), ID_DQ, (j > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&k_empty[st]);  // also tells the softmax warps the dS buffer is free
          BW_ADD(0, 5, t5);
        }
        if (!ok) break;
        umma_commit(dq_full);
        kc += nkb;
      }
      BW_ADD(0, 6, t_mma);
      umma_commit(drain);
      W.drain(drain, 0u);
    }
    __syncwarp();
  } else {
    // warp w: TMEM lanes 32 (w % 4) .., columns [64 half, 64 half + 64) of
    // the 128-key S and dP blocks and of dQ, and half of the row's Q and dO
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t dst = smem_u32(smem + Q_DS);
    // Q and dO of work item `item` (the it-th of this CTA) into tensor
    // memory, once the previous item's products no longer read them; done
    // for the next item before this one's dQ is written out, so the next
    // item's first S / dP products run during that write-out
    auto copy_qdo = [&](int item, uint32_t it) -> bool {
      int qb, b, h;
      decode_item(p, item, p.H, p.causal != 0, qb, b, h);
      const int qpos = qb * 128 + row;
      if (!W.warp(qdo_free, (it & 1u) ^ 1u)) return false;
      tc_fence_after();
      uint32_t r[32];
      if constexpr (SHORT) {
        const int r0 = qpos - lane;  // this warp's first row
        const long long tok0 = static_cast<long long>(b) * p.S + r0;
        load_rows_transposed(p.dqkv_src + tok0 * p.dqkv_rs + p.g.qcol(h) + half * 64, p.dqkv_rs, p.S - r0, r);
        tmem_st32(tl + DQ_QA + half * 32, r);
        load_rows_transposed(p.dO + tok0 * p.do_rs + h * HD + half * 64, p.do_rs, p.S - r0, r);
        tmem_st32(tl + DQ_DOA + half * 32, r);
      } else {
        const long long tok = static_cast<long long>(b) * p.S + qpos;
        load_row_pairs(p.dqkv_src + tok * p.dqkv_rs + p.g.qcol(h) + half * 64, qpos < p.S, r);
        tmem_st32(tl + DQ_QA + half * 32, r);
        load_row_pairs(p.dO + tok * p.do_rs + h * HD + half * 64, qpos < p.S, r);
        tmem_st32(tl + DQ_DOA + half * 32, r);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(qdo_ready);
      return true;
    };
    uint32_t it = 0, blk = 0;
    const bool started = item_of(0) >= p.items || copy_qdo(item_of(0), 0);
    for (int item = item_of(0); started && item < p.items; item = item_of(++it)) {
      int qb, b, h;
      decode_item(p, item, p.H, p.causal != 0, qb, b, h);
      const int nkb = nkb_of(qb);
      const int qpos = qb * 128 + row;
      const long long vrow = (static_cast<long long>(b) * p.H + h) * p.s_pad + qpos;
      // rows past the sequence read lse = +inf (written by the forward): p = 0
      const float lse_r = p.lse[vrow];
      const float ds_off = p.Dv[vrow] * p.scale;
      // short items: the next item's Q and dO rows start into L2 now, so
      // that their copy into tensor memory after this item's blocks finds
      // them there
      if (SHORT && item_of(it + 1) < p.items) {
        int qb2, b2, h2;
        decode_item(p, item_of(it + 1), p.H, p.causal != 0, qb2, b2, h2);
        const int qpos2 = qb2 * 128 + row;
        if (qpos2 < p.S) {
          const long long tok2 = static_cast<long long>(b2) * p.S + qpos2;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.dqkv_src + tok2 * p.dqkv_rs + p.g.qcol(h2) + half * 64));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.dO + tok2 * p.do_rs + h2 * HD + half * 64));
        }
      }
      bool ok = true;
      for (int j = 0; j < nkb; ++j, ++blk) {
        AT_T0(t7);
        if (!W.warp(sdp_full, blk & 1u)) { ok = false; break; }
#ifdef TPFFN_INSTRUMENT
        if (warp == 2 && lane == 0) BW_ADD(0, 7, t7);
#endif
        AT_T0(t8);
        tc_fence_after();
        // keys past the sequence need no mask here: their K rows are zero
        // filled, so they add nothing to dQ; only the causal diagonal does
        const bool diag = p.causal && j == qb;
        uint32_t pk[32];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t rs[32], rp[32];
          tmem_ld32(tl + DQ_S + half * 64 + c2 * 32, rs);
          tmem_ld32(tl + DQ_DP + half * 64 + c2 * 32, rp);
          tmem_wait_ld();
          const int kbase = j * 128 + half * 64 + c2 * 32;
          if (diag) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              rs[c] = (kbase + c <= qpos) ? rs[c] : __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float ds[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float pr = ex2(fmaf(__uint_as_float(rs[c + e]), p.scale_log2, -lse_r));
              ds[e] = pr * fmaf(__uint_as_float(rp[c + e]), p.scale, -ds_off);
            }
            pk[c2 * 16 + c / 2] = pack_bf16x2(ds[0], ds[1]);
          }
        }
        tc_fence_before();
        warp_arrive(sdp_empty);  // S and dP read: the next block's products may start
        // dS buffer free once the previous block's dQ has read it
        if (blk > 0 && !W.warp(&k_empty[(blk - 1) % DQ_KV], ((blk - 1) / DQ_KV) & 1u)) { ok = false; break; }
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          st_shared_v4(sw_chunk(dst, 128, row, half * 8 + c8), pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2],
                       pk[4 * c8 + 3]);
        fence_async_smem();
        tc_fence_before();
        warp_arrive(ds_full);
#ifdef TPFFN_INSTRUMENT
        if (warp == 2 && lane == 0) BW_ADD(0, 8, t8);
#endif
      }
      if (!ok) break;
      if (item_of(it + 1) < p.items && !copy_qdo(item_of(it + 1), it + 1)) break;
      if (!W.warp(dq_full, it & 1u)) break;
      tc_fence_after();
      // staged in this warp's own quarter of the dS tile, which the item's
      // last dQ product has read (dq_full) and which this warp rewrites next
      const uint32_t obuf = smem_u32(smem + Q_DS) + static_cast<uint32_t>(half * 16384 + quarter * 4096);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32], pk[16];
        tmem_ld32(tl + DQ_ACC + half * 64 + c * 32, o);
        tmem_wait_ld();
        pack_row_bf16(pk, o, 1.f);
        stage_row_chunk<2>(obuf, c, pk);
      }
      tc_fence_before();
      warp_arrive(dq_empty);
      const int r0 = qpos - lane;
      store_staged_rows<2>(obuf, p.dqkv + (static_cast<long long>(b) * p.S + r0) * p.dqkv_rs + p.g.qcol(h) + half * 64,
                           p.dqkv_rs, p.S - r0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================ dk, dv
// Blocks of 128 queries: S^T = K Q^T and dP^T = V dO^T are N = 128 products
// (full rate; N = 64 ones sit at the per-instruction floor), and dV += P^T dO,
// dK += dS^T Q contract over the block's 128 queries.  Tensor memory: S^T at
// columns 0..127, dP^T at 128..255, dV at 256..383, dK at 384..511 -- one
// S^T / dP^T stage, so a block's S^T / dP^T products follow the previous
// block's dV / dK products, which read the P^T / dS^T written over S^T / dP^T
// (tcgen05 products execute in issue order).  The softmax warps hand the block
// over in two halves (queries {0..31, 64..95}, then {32..63, 96..127}); the
// dV / dK products of the first half run while the second is computed.
constexpr int VST = 2;                    // query / dO stages of 128 rows
constexpr int V_K = 0;
constexpr int V_V = V_K + TILE;
constexpr int V_Q = V_V + TILE;           // VST stages of [128 q][128]
constexpr int V_DO = V_Q + VST * TILE;    // VST stages
constexpr int V_VEC = V_DO + VST * TILE;  // VST stages x (128 lse + 128 D) floats
constexpr int V_BAR = V_VEC + VST * 1024;
constexpr int V_O = V_BAR + 256;          // output staging, 2 KB per softmax warp
constexpr int V_SMEM = V_O + 8 * 2048 + 1024;

// The softmax warps keep P^T and dS^T in tensor memory: each thread writes
// its bf16 pairs (two per 32-bit cell, lower K in the low half) over the
// first half of its own fp32 columns of S^T / dP^T -- no other warp reads
// them -- and the dV / dK products read them as the A operand, one K = 16
// step (8 columns) at a time.  Tensor-memory column of K step ks within its
// S^T / dP^T block: the warps of half h own queries [64 h, 64 h + 64).
__device__ __forceinline__ uint32_t a_step128(uint32_t base, int ks) {
  return base + static_cast<uint32_t>((ks >> 2) * 64 + (ks & 3) * 8);
}

__global__ void __launch_bounds__(NT, 1) attn_dkdv_kernel(const __grid_constant__ CUtensorMap tq128,
                                                          const __grid_constant__ CUtensorMap tdo128,
                                                          const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + V_BAR);
  uint64_t* kv_full = bar + 0;
  uint64_t* kv_empty = bar + 1;
  uint64_t* qdo_full = bar + 2;              // [VST] Q, dO, lse and D of a block landed
  uint64_t* qdo_empty = qdo_full + VST;      // [VST] its dV / dK products completed
  uint64_t* sdp_full = qdo_empty + VST;
  uint64_t* pd_full = sdp_full + 1;          // [2] one per half-block hand-over
  uint64_t* dkv_full = pd_full + 2;
  uint64_t* dkv_empty = dkv_full + 1;
  uint64_t* drain = dkv_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(drain + 1) + 1;
  float* vec = reinterpret_cast<float*>(smem + V_VEC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int i = 0; i < VST; ++i) {
      mbar_init(&qdo_full[i], 1);
      mbar_init(&qdo_empty[i], 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(&pd_full[0], NSW);
    mbar_init(&pd_full[1], NSW);
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, NSW);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq128);
    prefetch_tmap(&tdo128);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{abort_flag, p.err, p.timeout_ns};

  // causal: key block kb sees the query blocks from kb on
  auto q0_of = [&](int kb) { return p.causal ? kb : 0; };

  if (warp == 0) {
    if (lane == 0) {
      int kv_last = -1, q_last[VST];
      for (int i = 0; i < VST; ++i) q_last[i] = -1;
      uint32_t qc = 0, it = 0;
      bool ok = true;
      for (int item = item_of(0); item < p.items && ok; item = item_of(++it)) {
        int kb, b, hk;
        decode_item(p, item, p.Hkv, false, kb, b, hk);
        if (!W(kv_empty, (it & 1u) ^ 1u)) break;
        mbar_arrive_expect_tx(kv_full, 2 * TILE);
        const int kcol = p.g.kcol(hk), vcol = p.g.vcol(hk);
        tma_load_3d(smem + V_K, &tq128, kv_full, kcol, kb * 128, b);
        tma_load_3d(smem + V_K + TILE / 2, &tq128, kv_full, kcol + 64, kb * 128, b);
        tma_load_3d(smem + V_V, &tq128, kv_full, vcol, kb * 128, b);
        tma_load_3d(smem + V_V + TILE / 2, &tq128, kv_full, vcol + 64, kb * 128, b);
        kv_last = static_cast<int>(it & 1u);
        const int i0 = q0_of(kb);
        for (int g = 0; g < p.G && ok; ++g) {
          const int h = hk * p.G + g;
          const int qcol = p.g.qcol(h);
          const float* lse_row = p.lse + (static_cast<long long>(b) * p.H + h) * p.s_pad;
          const float* d_row = p.Dv + (static_cast<long long>(b) * p.H + h) * p.s_pad;
          for (int i = i0; i < p.n_qb; ++i, ++qc) {
            const int st = qc % VST;
            const uint32_t ph = (qc / VST) & 1u;
            if (!W(&qdo_empty[st], ph ^ 1u)) { ok = false; break; }
            uint8_t* qd = smem + V_Q + st * TILE;
            uint8_t* dd = smem + V_DO + st * TILE;
            mbar_arrive_expect_tx(&qdo_full[st], 2 * TILE + 1024);
            tma_load_3d(qd, &tq128, &qdo_full[st], qcol, i * 128, b);
            tma_load_3d(qd + TILE / 2, &tq128, &qdo_full[st], qcol + 64, i * 128, b);
            bulk_g2s(vec + st * 256, lse_row + i * 128, 512, &qdo_full[st]);
            bulk_g2s(vec + st * 256 + 128, d_row + i * 128, 512, &qdo_full[st]);
            tma_load_3d(dd, &tdo128, &qdo_full[st], h * HD, i * 128, b);
            tma_load_3d(dd + TILE / 2, &tdo128, &qdo_full[st], h * HD + 64, i * 128, b);
            q_last[st] = static_cast<int>(ph);
          }
        }
      }
      if (kv_last >= 0) W.drain(kv_full, static_cast<uint32_t>(kv_last));
      for (int s2 = 0; s2 < VST; ++s2)
        if (q_last[s2] >= 0) W.drain(&qdo_full[s2], static_cast<uint32_t>(q_last[s2]));
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc(128, 0, 0);   // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t ID_G = idesc(128, 0, 1);   // dV += P^T dO, dK += dS^T Q (A in TMEM)
      const uint32_t ka = smem_u32(smem + V_K), va = smem_u32(smem + V_V);
      uint32_t qc = 0, sc = 0, it = 0;
      bool ok = true;
      AT_T0(t_mma);
      for (int item = item_of(0); item < p.items && ok; item = item_of(++it)) {
        int kb, b, hk;
        decode_item(p, item, p.Hkv, false, kb, b, hk);
        const int n_it = p.G * (p.n_qb - q0_of(kb));
        if (!W(kv_full, it & 1u)) break;
        tc_fence_after();
        for (int t = 0; t < n_it; ++t) {
          const uint32_t n = qc + t, g = sc + t;
          const int st = n % VST;
          const uint32_t ph = (n / VST) & 1u;
          AT_T0(t0);
          if (!W(&qdo_full[st], ph)) { ok = false; break; }
          BW_ADD(1, 0, t0);
          AT_T0(t1);
          tc_fence_after();
          const uint32_t qa = smem_u32(smem + V_Q + st * TILE), da = smem_u32(smem + V_DO + st * TILE);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16(tmem, kdesc(ka, 128, ks), kdesc(qa, 128, ks), ID_S, ks > 0 ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16(tmem + 128, kdesc(va, 128, ks), kdesc(da, 128, ks), ID_S, ks > 0 ? 1u : 0u);
          umma_commit(sdp_full);
          // K and V are read only by S^T / dP^T: the next item's copies may start
          if (t == n_it - 1) umma_commit(kv_empty);
          BW_ADD(1, 1, t1);
          AT_T0(t3);
          if (t == 0 && !W(dkv_empty, (it & 1u) ^ 1u)) { ok = false; break; }
          BW_ADD(1, 3, t3);
          BW_CNT(1, 4);
          for (int c = 0; c < 2; ++c) {
            AT_T0(t2);
            if (!W(&pd_full[c], g & 1u)) { ok = false; break; }
            BW_ADD(1, 2, t2);
            AT_T0(t5);
            tc_fence_after();
            // K steps of this half-block: queries 32c .. 32c + 31 and 64 + 32c .. 64 + 32c + 31
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int ks = (e >> 1) * 4 + 2 * c + (e & 1);
              umma_bf16_ta(tmem + 256, a_step128(tmem, ks), mndesc(da, 128, ks), ID_G,
                           (t > 0 || c > 0 || e > 0) ? 1u : 0u);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int ks = (e >> 1) * 4 + 2 * c + (e & 1);
              umma_bf16_ta(tmem + 384, a_step128(tmem + 128, ks), mndesc(qa, 128, ks), ID_G,
                           (t > 0 || c > 0 || e > 0) ? 1u : 0u);
            }
            BW_ADD(1, 5, t5);
          }
          if (!ok) break;
          umma_commit(&qdo_empty[st]);
        }
        if (!ok) break;
        umma_commit(dkv_full);
        qc += n_it;
        sc += n_it;
      }
      BW_ADD(1, 6, t_mma);
      umma_commit(drain);
      W.drain(drain, 0u);
    }
    __syncwarp();
  } else {
    // warp w: TMEM lanes 32 (w % 4) .. (keys of the tile), queries
    // [64 half, 64 half + 64) of each block (two 32-query pieces), and
    // columns [64 half, 64 half + 64) of dV and dK
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t qc = 0, sc = 0, it = 0;
    for (int item = item_of(0); item < p.items; item = item_of(++it)) {
      int kb, b, hk;
      decode_item(p, item, p.Hkv, false, kb, b, hk);
      const int i0 = q0_of(kb), nq = p.n_qb - i0;
      const int n_it = p.G * nq;
      const int kpos = kb * 128 + row;
      bool ok = true;
      for (int t = 0; t < n_it; ++t) {
        const int i = i0 + t % nq;
        const uint32_t n = qc + t, g = sc + t;
        const int st = n % VST;
        const uint32_t ph = (n / VST) & 1u;
        AT_T0(t7);
        if (!W.warp(sdp_full, g & 1u)) { ok = false; break; }
#ifdef TPFFN_INSTRUMENT
        if (warp == 2 && lane == 0) BW_ADD(1, 7, t7);
#endif
        AT_T0(t8);
        tc_fence_after();
        if (!W.warp(&qdo_full[st], ph)) { ok = false; break; }  // lse / D of this block landed
        for (int c = 0; c < 2; ++c) {
          const int col = half * 64 + c * 32;  // first query of this piece within the block
          uint32_t rs[32], rp[32];
          tmem_ld32(tl + col, rs);
          tmem_ld32(tl + 128 + col, rp);
          tmem_wait_ld();
          const float* lse_v = vec + st * 256 + col;
          const float* d_v = vec + st * 256 + 128 + col;
          // queries past the sequence read lse = +inf and D = 0 (p = 0); keys
          // past it are never stored; only the causal diagonal needs a mask
          const int qbase = i * 128 + col;
          if (p.causal && i == kb) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              rs[e] = (kpos <= qbase + e) ? rs[e] : __float_as_uint(-INFINITY);
          }
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 lv = *reinterpret_cast<const float4*>(lse_v + e);
            const float4 dv = *reinterpret_cast<const float4*>(d_v + e);
            const float l4[4] = {lv.x, lv.y, lv.z, lv.w}, d4[4] = {dv.x, dv.y, dv.z, dv.w};
            float pr[4], ds[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              pr[k] = ex2(fmaf(__uint_as_float(rs[e + k]), p.scale_log2, -l4[k]));
              ds[k] = pr[k] * ((__uint_as_float(rp[e + k]) - d4[k]) * p.scale);
            }
            pp[e / 2] = pack_bf16x2(pr[0], pr[1]);
            pp[e / 2 + 1] = pack_bf16x2(pr[2], pr[3]);
            pd[e / 2] = pack_bf16x2(ds[0], ds[1]);
            pd[e / 2 + 1] = pack_bf16x2(ds[2], ds[3]);
          }
          // P^T / dS^T of K steps 4 half + 2c, +1: columns 64 half + 16 c ..
          // +15, inside this thread's own (already read) S^T / dP^T columns
          tmem_st16(tl + half * 64 + c * 16, pp);
          tmem_st16(tl + 128 + half * 64 + c * 16, pd);
          tmem_wait_st();
          tc_fence_before();
          warp_arrive(&pd_full[c]);
        }
#ifdef TPFFN_INSTRUMENT
        if (warp == 2 && lane == 0) BW_ADD(1, 8, t8);
#endif
      }
      if (!ok) break;
      if (!W.warp(dkv_full, it & 1u)) break;
      tc_fence_after();
      // dV (columns 256..383) and dK (384..511) of this warp's rows, packed
      uint32_t pk[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tl + 256 + (c >> 1) * 128 + half * 64 + (c & 1) * 32, o);
        tmem_wait_ld();
        pack_row_bf16(pk[c], o, 1.f);
      }
      tc_fence_before();
      warp_arrive(dkv_empty);
      const int r0 = kpos - lane;
      __nv_bfloat16* out = p.dqkv + (static_cast<long long>(b) * p.S + r0) * p.dqkv_rs + half * 64;
      const int vcol = p.g.vcol(hk), kcol = p.g.kcol(hk);
      const uint32_t sbuf = smem_u32(smem + V_O) + static_cast<uint32_t>((warp - 2) * 2048);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        stage_row_chunk<1>(sbuf, 0, pk[c]);
        store_staged_rows<1>(sbuf, out + ((c >> 1) ? kcol : vcol) + (c & 1) * 32, p.dqkv_rs, p.S - r0);
      }
      qc += n_it;
      sc += n_it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================ packing
__global__ void pack_qkv_kernel(const __nv_bfloat16* Wq, const __nv_bfloat16* Wk, const __nv_bfloat16* Wv,
                                __nv_bfloat16* packed, int T, long long sq, long long sk, long long d, int unpack) {
  const long long slice = sq + 2 * sk;
  const long long rows = T * slice;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const long long t = r / slice, c = r - t * slice;
    const __nv_bfloat16* src;
    if (c < sq)
      src = Wq + (t * sq + c) * d;
    else if (c < sq + sk)
      src = Wk + (t * sk + c - sq) * d;
    else
      src = Wv + (t * sk + c - sq - sk) * d;
    __nv_bfloat16* dst = packed + r * d;
    const uint4* s4 = reinterpret_cast<const uint4*>(unpack ? dst : src);
    uint4* d4 = reinterpret_cast<uint4*>(unpack ? const_cast<__nv_bfloat16*>(src) : dst);
    for (long long k = threadIdx.x; k < d / 8; k += blockDim.x) d4[k] = s4[k];
  }
}

// barrier areas (mbarriers + TMEM slot + abort flag) fit their reserved bytes
static_assert(F_O - F_BAR >= 33 * 8 + 8 && F_O % 1024 == 0, "forward barrier area, staging alignment");
static_assert(Q_SMEM - Q_BAR - 1024 >= 21 * 8 + 8, "dq barrier area");
static_assert(V_SMEM - V_BAR - 1024 >= (8 + 2 * VST) * 8 + 8, "dk/dv barrier area");
static_assert(F_SMEM <= 232448 && Q_SMEM <= 232448 && V_SMEM <= 232448, "shared memory per CTA");

// ================================================================ host
Params make_params(const AttnSpec& a, const LaunchCtx& ctx) {
  Params p{};
  p.g.hq_per = a.H / a.T_p;
  p.g.hk_per = a.Hkv / a.T_p;
  p.g.sq = p.g.hq_per * HD;
  p.g.sk = p.g.hk_per * HD;
  p.g.slice = p.g.sq + 2 * p.g.sk;
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.causal = a.causal ? 1 : 0;
  p.n_qb = (a.S + 127) / 128;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.o_rs = a.o_rs;
  p.dO = static_cast<const __nv_bfloat16*>(a.dO);
  p.do_rs = a.do_rs;
  p.lse = a.lse;
  p.s_pad = a.s_pad;
  p.Dv = a.Dv;
  p.dqkv = static_cast<__nv_bfloat16*>(a.dqkv);
  p.dqkv_rs = a.qkv_rs;
  p.dqkv_src = static_cast<const __nv_bfloat16*>(a.qkv);
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(HD)));
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  p.err = ctx.err;
  p.timeout_ns = ctx.timeout_ns;
  return p;
}

int check_spec(const AttnSpec& a) {
  if (a.hd != HD) return TP_ERR_UNSUPPORTED;
  if (a.B < 1 || a.S < 1 || a.H < 1 || a.Hkv < 1 || a.T_p < 1) return TP_ERR_INVALID;
  if (a.H % a.T_p || a.Hkv % a.T_p || a.H % a.Hkv) return TP_ERR_INVALID;
  if (a.qkv_rs < static_cast<int64_t>(a.H + 2 * a.Hkv) * HD || a.qkv_rs % 8) return TP_ERR_INVALID;
  if (a.s_pad < (a.S + 127) / 128 * 128 || a.s_pad % 128) return TP_ERR_INVALID;
  if (a.o_rs < static_cast<int64_t>(a.H) * HD || a.o_rs % 8) return TP_ERR_INVALID;
  const long long blocks = static_cast<long long>((a.S + 127) / 128) * a.B * a.H;
  if (blocks > (1ll << 30) || static_cast<long long>(a.B) * a.S > (1ll << 30)) return TP_ERR_UNSUPPORTED;
  return TP_OK;
}

int map_rows(CUtensorMap* m, const void* ptr, int64_t rs, int S, int B, uint32_t box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(rs), static_cast<uint64_t>(S), static_cast<uint64_t>(B)};
  const uint64_t str[2] = {static_cast<uint64_t>(rs) * 2, static_cast<uint64_t>(rs) * 2 * static_cast<uint64_t>(S)};
  const uint32_t box[3] = {64, box_rows, 1};
  return encode_map_3d_bf16(m, ptr, dims, str, box);
}

template <typename K>
int set_smem_once(K kern, int bytes, std::atomic<uint32_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TP_ERR_CUDA;
  const uint32_t bit = 1u << (dev & 31);
  if (!(done.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return TP_ERR_CUDA;
    done.fetch_or(bit);
  }
  return TP_OK;
}

int grid_for(long long items, int sms) { return static_cast<int>(items < sms ? items : sms); }

}  // namespace attn

#ifdef TPFFN_INSTRUMENT
extern "C" __attribute__((visibility("default"))) int tpffn_attn_bwd_debug_counters(unsigned long long* host,
                                                                                   int clear) {
  if (cudaMemcpyFromSymbol(host, attn::g_attn_bwd_dbg, sizeof(attn::g_attn_bwd_dbg)) != cudaSuccess) return 1;
  if (clear) {
    static unsigned long long zeros[2][256][16];
    if (cudaMemcpyToSymbol(attn::g_attn_bwd_dbg, zeros, sizeof(zeros)) != cudaSuccess) return 1;
  }
  return 0;
}
extern "C" __attribute__((visibility("default"))) int tpffn_attn_debug_counters(unsigned long long* host, int clear) {
  if (cudaMemcpyFromSymbol(host, attn::g_attn_dbg, sizeof(attn::g_attn_dbg)) != cudaSuccess) return 1;
  if (clear) {
    static unsigned long long zeros[256][24];
    if (cudaMemcpyToSymbol(attn::g_attn_dbg, zeros, sizeof(zeros)) != cudaSuccess) return 1;
  }
  return 0;
}
#endif

int launch_attn_fwd(const AttnSpec& a, LaunchCtx& ctx) {
  using namespace attn;
  int rc = check_spec(a);
  if (rc) return rc;
  if (!a.qkv || !a.o || !a.lse) return TP_ERR_INVALID;
  CUtensorMap tq, to;
  if ((rc = map_rows(&tq, a.qkv, a.qkv_rs, a.S, a.B, 128))) return rc;
  if ((rc = map_rows(&to, a.o, a.o_rs, a.S, a.B, 32))) return rc;  // 32-row output boxes
  Params p = make_params(a, ctx);
  p.items = p.n_qb * a.B * a.H;
  static std::atomic<uint32_t> done{0};
  if ((rc = set_smem_once(attn_fwd_kernel, F_SMEM, done))) return rc;
  if (ctx.before) ctx.before(ctx.user, "attn_fwd", ctx.stream);
  attn_fwd_kernel<<<grid_for(p.items, ctx.num_sms), NT, F_SMEM, ctx.stream>>>(tq, to, p);
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

int launch_attn_bwd(const AttnSpec& a, LaunchCtx& ctx) {
  using namespace attn;
  int rc = check_spec(a);
  if (rc) return rc;
  if (!a.qkv || !a.o || !a.lse || !a.dO || !a.Dv || !a.dqkv) return TP_ERR_INVALID;
  if (a.do_rs < static_cast<int64_t>(a.H) * HD || a.do_rs % 8) return TP_ERR_INVALID;
  CUtensorMap tq128, tdo128;
  if ((rc = map_rows(&tq128, a.qkv, a.qkv_rs, a.S, a.B, 128))) return rc;
  if ((rc = map_rows(&tdo128, a.dO, a.do_rs, a.S, a.B, 128))) return rc;
  Params p = make_params(a, ctx);

  // D = rowsum(dO * o)
  {
    const long long total = static_cast<long long>(a.B) * a.H * a.s_pad;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    if (ctx.before) ctx.before(ctx.user, "attn_bwd_prep", ctx.stream);
    attn_prep_kernel<<<static_cast<unsigned>(blocks), threads, 0, ctx.stream>>>(p);
    if (ctx.after) ctx.after(ctx.user, ctx.stream);
    ctx.launches++;
  }
  {
    p.items = p.n_qb * a.B * a.H;
    static std::atomic<uint32_t> done_s{0}, done_l{0};
    const bool short_items = p.n_qb <= 16;
    if ((rc = short_items ? set_smem_once(attn_dq_kernel<true>, Q_SMEM, done_s)
                          : set_smem_once(attn_dq_kernel<false>, Q_SMEM, done_l)))
      return rc;
    if (ctx.before) ctx.before(ctx.user, "attn_bwd_dq", ctx.stream);
    if (short_items)
      attn_dq_kernel<true><<<grid_for(p.items, ctx.num_sms), NT, Q_SMEM, ctx.stream>>>(tq128, p);
    else
      attn_dq_kernel<false><<<grid_for(p.items, ctx.num_sms), NT, Q_SMEM, ctx.stream>>>(tq128, p);
    if (ctx.after) ctx.after(ctx.user, ctx.stream);
    ctx.launches++;
  }
  {
    p.items = p.n_qb * a.B * a.Hkv;
    static std::atomic<uint32_t> done{0};
    if ((rc = set_smem_once(attn_dkdv_kernel, V_SMEM, done))) return rc;
    if (ctx.before) ctx.before(ctx.user, "attn_bwd_dkdv", ctx.stream);
    attn_dkdv_kernel<<<grid_for(p.items, ctx.num_sms), NT, V_SMEM, ctx.stream>>>(tq128, tdo128, p);
    if (ctx.after) ctx.after(ctx.user, ctx.stream);
    ctx.launches++;
  }
  return cudaPeekAtLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

int launch_pack_qkv(const void* Wq, const void* Wk, const void* Wv, void* packed, int T_p, int64_t sq, int64_t sk,
                    int64_t d, int unpack, cudaStream_t st) {
  if (!Wq || !Wk || !Wv || !packed || d % 8) return TP_ERR_INVALID;
  const void* ptrs[] = {Wq, Wk, Wv, packed};
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) % 16) return TP_ERR_ALIGN;
  const long long rows = static_cast<long long>(T_p) * (sq + 2 * sk);
  const int grid = static_cast<int>(rows < 65535 ? rows : 65535);
  attn::pack_qkv_kernel<<<grid, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(Wq),
                                              static_cast<const __nv_bfloat16*>(Wk),
                                              static_cast<const __nv_bfloat16*>(Wv),
                                              static_cast<__nv_bfloat16*>(packed), T_p, sq, sk, d, unpack);
  return cudaPeekAtLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

}  // namespace tpffn
