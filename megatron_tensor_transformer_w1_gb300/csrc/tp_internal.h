// tp_internal.h -- declarations shared by the library's translation units.
//
// One GEMM description (GemmSpec) drives both compute back ends: the tcgen05
// tensor-core kernel (bf16 operands, fp32 accumulation in tensor memory) and
// the SIMT kernel (fp32 plans).  A GEMM here is
//
//   C_b[M, N] = sum_{g < G} A_{b,g}[M, K] * B_{b,g}[N, K]^T      (b < NB)
//
// where every operand is a strided 3-D view (inner, rows, batch) of a device
// buffer.  "K-major" operands keep K in the contiguous (inner) dimension and
// M (or N) in rows; "MN-major" operands keep M (or N) contiguous and K in
// rows.  The batch coordinate of operand X for (b, g) is b*X.bsel + g*X.gsel,
// which expresses the three uses of the shard index: per-shard GEMMs (bsel=1),
// a shared operand (0,0) and the shard loop of the fused shard-sum (gsel=1).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tpffn {

enum EpiKind : int {
  EPI_F32 = 0,         // out fp32 = acc                          (partials)
  EPI_OUT = 1,         // out (plan dtype) = acc + bias[n]        (y, dx, dW)
  EPI_GELU_FWD = 2,    // z = acc + b1; out2 = z (saved); out = gelu_tanh(z)
  EPI_SWIGLU_FWD = 3,  // acc = [a | g] per 256-col tile; out = silu(a)*g; out2 = a, g
  EPI_GELU_BWD = 4,    // out = acc * gelu_tanh'(aux)             (dz)
  EPI_SWIGLU_BWD = 5,  // acc = dh; aux = saved [a|g]; out = [da | dg]
};

struct Operand {
  const void* ptr = nullptr;
  int64_t inner = 0, rows = 0, batch = 1;   // extents (elements)
  int64_t row_stride = 0, batch_stride = 0; // element strides
  int mn_major = 0;
  int bsel = 0, gsel = 0;
};

struct GemmSpec {
  const char* name = "gemm";
  int64_t M = 0, N = 0, K = 0;
  int NB = 1, G = 1;
  Operand A, B;
  int epi = EPI_F32;
  void* out = nullptr;  int64_t out_bs = 0, out_rs = 0;
  void* out2 = nullptr; int64_t out2_bs = 0, out2_rs = 0;
  const void* aux = nullptr; int64_t aux_bs = 0, aux_rs = 0;
  const void* bias = nullptr; int64_t bias_bs = 0, bias_len = 0;
  int64_t n_store = 0;   // columns n < n_store of the output are written
  int out_bf16 = 1;      // plan dtype of out/out2 (EPI_F32 always fp32)
  // K split (EPI_F32 only): part k of the K blocks is accumulated on its own
  // and written as fp32 batch k * NB + b of `out` (one-SM kernel: G = 1)
  int ksplit = 1;
  // Shards merged along N (pair kernel, NB = 1, TMA-store epilogue only;
  // TP_ERR_UNSUPPORTED otherwise): out_cs > 0 writes output column n to
  // batch n / out_cs, column n % out_cs of `out` (out_bs apart); b_cs > 0
  // reads B's column n from batch n / b_cs, column n % b_cs of B's own batch
  // layout.  Both sizes are multiples of 128.
  int64_t out_cs = 0, b_cs = 0;
  // The GEMM neither reads nor writes any buffer that the kernel launched
  // before it on the stream writes (nor one that a no_dep_wait GEMM right
  // before it writes): it lets its successor launch and starts without
  // waiting (the kernel before it must have waited for its own
  // predecessor), and waits before exit.
  int no_dep_wait = 0;
  // Last-wave split (pair kernel with TMA stores; EPI_OUT with one batch, or
  // EPI_GELU_FWD): when the output tiles leave the last wave of SM pairs at
  // most half full, those tiles run as K parts that fill the idle pairs;
  // their fp32 sums go to tail_ws (tail_ws_bytes) and a fix-up kernel adds
  // them in part order, adds the bias (and applies GELU) and writes what the
  // epilogue would have.  nullptr: no split.
  float* tail_ws = nullptr;
  size_t tail_ws_bytes = 0;
};


// Launch context of one API call.
struct LaunchCtx {
  cudaStream_t stream = nullptr;
  int* err = nullptr;            // device error word (workspace header)
  int num_sms = 148;
  int debug_skip_load = 0;       // test hook (first tensor-core GEMM only)
  uint64_t timeout_ns = 2000000000ull;
  bool timing = false;
  int launches = 0;
  // timing records are appended by the caller through these hooks
  void (*before)(void* user, const char* name, cudaStream_t stream) = nullptr;
  void (*after)(void* user, cudaStream_t stream) = nullptr;
  void* user = nullptr;
};

// Row slices of a sequence-parallel caller: rank t's rows [t*rows, (t+1)*rows)
// of an [n][cols] tensor live in their own buffer ptr[t].
constexpr int kMaxSlices = 64;
struct RowSlices {
  void* ptr[kMaxSlices];
  int n = 0;
  int64_t rows = 0;
};

// Device error bits.
constexpr int DEV_ERR_TIMEOUT = 1;

// tensor-core GEMM (tp_gemm_tc.cu). Returns 0 or a TP_ERR_* code.
int launch_tc_gemm(const GemmSpec& s, LaunchCtx& ctx);
// True when a tensor-core GEMM of M rows runs on the two-SM pair kernel.
bool tc_pair_path(int64_t M);
// SIMT fp32 GEMM (tp_kernels.cu).
int launch_simt_gemm(const GemmSpec& s, LaunchCtx& ctx);

// Streaming kernels (tp_kernels.cu).  esz = element size of the plan dtype.
int launch_pack_columns(const void* W1, const void* W3, void* out, int T_p, int64_t s,
                        int64_t s_pad, int64_t d, int swiglu, int esz, int unpack,
                        cudaStream_t st);
int launch_pack_rows(const void* W2, void* out, int T_p, int64_t s, int64_t s_pad, int64_t d,
                     int esz, int unpack, cudaStream_t st);
// shard_stride: elements between consecutive shards' partials (0: rows*cols).
// Tiles of a last-wave split (256 x 256 output blocks of batch b at rows
// mp * 256 and columns nb * 256), each summed from `parts` fp32 K parts.
constexpr int kMaxTailTiles = 64;
struct TailTiles {
  int n = 0, parts = 0;
  int b[kMaxTailTiles], mp[kMaxTailTiles], nb[kMaxTailTiles];
};
// What the fix-up writes: the GEMM epilogue's output (bf16, + bias); for the
// GELU forward h = gelu(z) and, when out2 is given, z; for the SwiGLU forward
// (tiles of 128 a-columns then 128 g-columns) h = silu(a) g at the tile's 128
// hidden units and, when out2 is given, a and g (all bf16).
struct TailOut {
  void* out = nullptr;
  int64_t out_bs = 0, out_rs = 0;
  void* out2 = nullptr;
  int64_t out2_bs = 0, out2_rs = 0;
  const void* bias = nullptr;
  int64_t bias_bs = 0, bias_len = 0;
  int64_t M = 0, n_store = 0;
  int act = 0;  // 0 none, 1 GELU, 2 SwiGLU
};
int launch_tail_fixup(const float* parts, const TailTiles& t, const TailOut& o, LaunchCtx& ctx, const char* name);
// SwiGLU of the ksplit fp32 parts of a K-split up GEMM (see tp_kernels.cu).
int launch_swiglu_combine(const float* parts, int ksplit, int T_p, int64_t rows, int64_t s_pad, void* h,
                          void* saved, LaunchCtx& ctx, const char* name);
int launch_shard_sum(const float* partials, int T_p, int64_t rows, int64_t cols,
                     const void* bias, void* out, int out_bf16, LaunchCtx& ctx,
                     const char* name, int64_t shard_stride = 0);
// Sequence-parallel data movement (tp_kernels.cu): gather the slices into a
// contiguous [n][cols] buffer (all-gather), scatter a contiguous buffer into
// the slices, and the ordered shard-sum writing each row-slice into its own
// buffer (reduce-scatter).  esz = element size in bytes.
int launch_gather_rows(const RowSlices& src, void* dst, int64_t cols, int esz, LaunchCtx& ctx, const char* name);
int launch_scatter_rows(const void* src, int64_t n, int64_t cols, int esz, const RowSlices& dst, LaunchCtx& ctx,
                        const char* name);
int launch_shard_sum_scatter(const float* partials, int T_p, int64_t rows, int64_t cols, const void* bias,
                             const RowSlices& out, int out_bf16, LaunchCtx& ctx, const char* name);
// Column sums of a [batch][rows][cols] view (row stride rs, batch stride bs)
// into out[b*out_bs + col] for col < cols, deterministic two-pass order; the
// chunk sums go to `scratch` (colsum_scratch_floats floats).  Up to two such
// jobs share one pair of launches.
struct ColsumJob {
  const void* in = nullptr;
  void* out = nullptr;
  float* scratch = nullptr;
  long long rows = 0, cols = 0, rs = 0, bs = 0, out_bs = 0, chunk_rows = 64;
  int in_bf16 = 1, out_bf16 = 1, batch = 0;
  long long chunks = 0;       // set by launch_colsums
  int blocks1 = 0, blocks2 = 0;  // set by launch_colsums
};
struct ColsumJobs {
  ColsumJob j[2];
  int n = 0;
  // the inputs are written by nothing the kernel before it writes: pass 1
  // starts without waiting for that kernel and waits before exit (see the
  // GEMMs' no_dep_wait)
  int no_dep_wait = 0;
};
int launch_colsums(ColsumJobs jobs, LaunchCtx& ctx, const char* name);
// Clears the device error word at the start of a call (one tiny kernel).
int launch_reset_error_word(int* err, cudaStream_t stream);
int64_t colsum_scratch_floats(int64_t batch, int64_t rows, int64_t cols, int64_t chunk_rows);

// Attention core of the head-sharded attention sublayer (tp_attention.cu).
// Tokens of sequence b are rows b*S .. b*S+S-1.  The projected queries, keys
// and values live in one bf16 buffer `qkv` [B*S][qkv_rs] holding the T_p
// shard slices side by side; slice t (columns [t*slice, (t+1)*slice),
// slice = (H + 2*Hkv) / T_p * hd) is [query heads of shard t | key heads |
// value heads], each head hd columns wide.  `dqkv` has the same layout.
struct AttnSpec {
  int B = 0, S = 0, H = 0, Hkv = 0, T_p = 1, causal = 1;
  int64_t hd = 128;
  const void* qkv = nullptr; int64_t qkv_rs = 0;
  void* o = nullptr; int64_t o_rs = 0;          // head outputs [B*S][o_rs], head h at column h*hd
  float* lse = nullptr; int64_t s_pad = 0;      // log2-domain log-sum-exp [B*H][s_pad]
  const void* dO = nullptr; int64_t do_rs = 0;  // gradient of the head outputs
  float* Dv = nullptr;                          // rowsum(dO * o) [B*H][s_pad] (scratch)
  void* dqkv = nullptr;
};
int launch_attn_fwd(const AttnSpec& a, LaunchCtx& ctx);
int launch_attn_bwd(const AttnSpec& a, LaunchCtx& ctx);
// Pack Wq [H*hd][d], Wk, Wv [Hkv*hd][d] into shard slices [T_p][slice][d]
// (unpack = 1 reverses it).
int launch_pack_qkv(const void* Wq, const void* Wk, const void* Wv, void* packed, int T_p, int64_t sq, int64_t sk,
                    int64_t d, int unpack, cudaStream_t st);

}  // namespace tpffn
