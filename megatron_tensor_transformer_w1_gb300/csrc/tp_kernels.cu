// tp_kernels.cu -- the memory-bound kernels of the path and the fp32 GEMM.
//
//   pack / unpack  : shard_columns / shard_rows of "S17 Tensor & Pipeline
//                    Parallelism" (listing "the megatron pattern"), for all
//                    shards in one launch, into the layouts of tpffn.h
//   shard_sum      : the g-operator (forward) and f-operator (backward dx)
//                    all-reduce of "7.9 Tensor and pipeline parallelism
//                    (TP, PP)", §2.1, as an on-device sum of the fp32 shard
//                    partials in the fixed order t = 0..T_p-1 (+ bias once)
//   colsum         : bias gradients (sum over tokens), two fixed-order passes
//   simt_gemm      : fp32 GEMM with the same epilogues as the tensor-core
//                    kernel, for fp32 plans (TF32 would not meet fp32
//                    accuracy, so these use plain FMA)
#include <climits>
#include <cstdlib>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tp_act.cuh"
#include "tp_internal.h"
#include "tpffn.h"

namespace tpffn {

namespace {

__device__ __forceinline__ float to_f(const void* p, long long i, int bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]) : static_cast<const float*>(p)[i];
}
__device__ __forceinline__ void from_f(void* p, long long i, float v, int bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(p)[i] = v;
}

// ------------------------------------------------------------------ packing
// Copy `n` elements of `esz` bytes; 16-byte vectors when both ends allow.
__device__ __forceinline__ void copy_row(char* dst, const char* src, long long n, int esz) {
  const long long bytes = n * esz;
  if ((reinterpret_cast<uintptr_t>(dst) % 16) == 0 && (reinterpret_cast<uintptr_t>(src) % 16) == 0 &&
      bytes % 16 == 0) {
    for (long long i = threadIdx.x; i < bytes / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
  } else if (esz == 2) {
    for (long long i = threadIdx.x; i < n; i += blockDim.x)
      reinterpret_cast<uint16_t*>(dst)[i] = reinterpret_cast<const uint16_t*>(src)[i];
  } else {
    for (long long i = threadIdx.x; i < n; i += blockDim.x)
      reinterpret_cast<uint32_t*>(dst)[i] = reinterpret_cast<const uint32_t*>(src)[i];
  }
}
__device__ __forceinline__ void zero_row(char* dst, long long n, int esz) {
  const long long bytes = n * esz;
  if ((reinterpret_cast<uintptr_t>(dst) % 16) == 0 && bytes % 16 == 0) {
    for (long long i = threadIdx.x; i < bytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(dst)[i] = uint4{0, 0, 0, 0};
  } else {
    for (long long i = threadIdx.x; i < bytes; i += blockDim.x) dst[i] = 0;
  }
}

// One block per packed row (t, rr).  GELU: rr = hidden unit j.  SwiGLU: rows
// come in 256-row blocks, 128 of W1 then 128 of W3 for the same hidden units.
__global__ void pack_columns_kernel(const char* W1, const char* W3, char* out, long long s, long long s_pad,
                                    long long d, int swiglu, int esz, int unpack) {
  const long long rows_per_shard = swiglu ? 2 * s_pad : s_pad;
  const long long t = blockIdx.x / rows_per_shard;
  const long long rr = blockIdx.x - t * rows_per_shard;
  long long j = rr;
  int half = 0;
  if (swiglu) {
    half = static_cast<int>((rr >> 7) & 1);
    j = (rr >> 8) * 128 + (rr & 127);
  }
  char* prow = out + (t * rows_per_shard + rr) * d * esz;
  const bool valid = j < s;
  const char* base = half ? W3 : W1;
  if (!unpack) {
    if (valid)
      copy_row(prow, base + (t * s + j) * d * esz, d, esz);
    else
      zero_row(prow, d, esz);
  } else if (valid) {
    copy_row(const_cast<char*>(base) + (t * s + j) * d * esz, prow, d, esz);
  }
}

// One block per packed row (t, c): out[t][c][0:s] = W2[c][t*s : (t+1)*s].
__global__ void pack_rows_kernel(const char* W2, char* out, long long s, long long s_pad, long long d,
                                 int T_p, int esz, int unpack) {
  const long long t = blockIdx.x / d;
  const long long c = blockIdx.x - t * d;
  const long long d_ff = s * T_p;
  char* prow = out + (t * d + c) * s_pad * esz;
  const char* src = W2 + (c * d_ff + t * s) * esz;
  if (!unpack) {
    copy_row(prow, src, s, esz);
    if (s_pad > s) zero_row(prow + s * esz, s_pad - s, esz);
  } else {
    copy_row(const_cast<char*>(src), prow, s, esz);
  }
}

// ---------------------------------------------------------------- shard-sum
// y[i] = ((P_0[i] + P_1[i]) + ...) + P_{T-1}[i], then + bias[i % cols].
// 8 consecutive elements per thread, 16-byte streaming loads.
template <int OUT_BF16>
__global__ void __launch_bounds__(256) shard_sum_vec8_kernel(const float* __restrict__ P, int T, long long plane,
                                                             long long cols, const __nv_bfloat16* bias_bf,
                                                             const float* bias_f, void* out, long long stride) {
  // a programmatic dependent of the GEMM that wrote the partials; once they
  // are visible, the next kernel may launch
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long n8 = plane / 8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4* p0 = reinterpret_cast<const float4*>(P) + 2 * i;
    float4 a = __ldcs(p0), b = __ldcs(p0 + 1);
    for (int t = 1; t < T; ++t) {
      const float4* pt = reinterpret_cast<const float4*>(P + t * stride) + 2 * i;
      const float4 c = __ldcs(pt), e = __ldcs(pt + 1);
      a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
      b.x += e.x; b.y += e.y; b.z += e.z; b.w += e.w;
    }
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const long long col = (i * 8) % cols;
    if (bias_bf) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] += __bfloat162float(bias_bf[col + j]);
    } else if (bias_f) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] += bias_f[col + j];
    }
    if (OUT_BF16) {
      uint4 q;
      __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(v[4], v[5]), h3 = __floats2bfloat162_rn(v[6], v[7]);
      q.x = *reinterpret_cast<uint32_t*>(&h0);
      q.y = *reinterpret_cast<uint32_t*>(&h1);
      q.z = *reinterpret_cast<uint32_t*>(&h2);
      q.w = *reinterpret_cast<uint32_t*>(&h3);
      reinterpret_cast<uint4*>(out)[i] = q;
    } else {
      float4* o = reinterpret_cast<float4*>(out) + 2 * i;
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

__global__ void shard_sum_scalar_kernel(const float* P, int T, long long plane, long long cols, const void* bias,
                                        int bias_bf16, void* out, int out_bf16, long long stride) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < plane; i += (long long)gridDim.x * blockDim.x) {
    float acc = P[i];
    for (int t = 1; t < T; ++t) acc += P[t * stride + i];
    if (bias) acc += to_f(bias, i % cols, bias_bf16);
    from_f(out, i, acc, out_bf16);
  }
}

// ------------------------------------------------------- sequence parallel
struct SliceTable {
  char* p[kMaxSlices];
};

// Copy between T contiguous [rows][row_bytes] slices and one [T*rows] buffer.
// to_slices = 0: gather (slices -> buffer); 1: scatter (buffer -> slices).
__global__ void slice_copy_kernel(SliceTable tab, char* buf, long long slice_bytes, long long total_bytes,
                                  int to_slices) {
  const long long n16 = total_bytes / 16;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n16; i += (long long)gridDim.x * blockDim.x) {
    const long long o = i * 16;
    const long long t = o / slice_bytes;
    uint4* sl = reinterpret_cast<uint4*>(tab.p[t] + (o - t * slice_bytes));
    uint4* bf = reinterpret_cast<uint4*>(buf + o);
    if (to_slices)
      *sl = *bf;
    else
      *bf = *sl;
  }
}
__global__ void slice_copy_bytes_kernel(SliceTable tab, char* buf, long long slice_bytes, long long total_bytes,
                                        int to_slices) {
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total_bytes;
       o += (long long)gridDim.x * blockDim.x) {
    const long long t = o / slice_bytes;
    char* sl = tab.p[t] + (o - t * slice_bytes);
    if (to_slices)
      *sl = buf[o];
    else
      buf[o] = *sl;
  }
}

// Ordered shard-sum whose output row r goes to slice r / rows_per_slice.
template <int OUT_BF16>
__global__ void __launch_bounds__(256) shard_sum_scatter_kernel(const float* __restrict__ P, int T, long long plane,
                                                                long long cols, const void* bias, SliceTable out,
                                                                long long rows_per_slice) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < plane; i += (long long)gridDim.x * blockDim.x) {
    float acc = P[i];
    for (int t = 1; t < T; ++t) acc += P[t * plane + i];
    const long long row = i / cols, col = i - row * cols;
    if (bias) acc += to_f(bias, col, OUT_BF16);
    const long long sl = row / rows_per_slice;
    from_f(out.p[sl], (row - sl * rows_per_slice) * cols + col, acc, OUT_BF16);
  }
}
template <int OUT_BF16>
__global__ void __launch_bounds__(256) shard_sum_scatter_vec8_kernel(const float* __restrict__ P, int T,
                                                                     long long plane, long long cols,
                                                                     const void* bias, SliceTable out,
                                                                     long long rows_per_slice) {
  const long long n8 = plane / 8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4* p0 = reinterpret_cast<const float4*>(P) + 2 * i;
    float4 a = __ldcs(p0), b = __ldcs(p0 + 1);
    for (int t = 1; t < T; ++t) {
      const float4* pt = reinterpret_cast<const float4*>(P + t * plane) + 2 * i;
      const float4 c = __ldcs(pt), e = __ldcs(pt + 1);
      a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
      b.x += e.x; b.y += e.y; b.z += e.z; b.w += e.w;
    }
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const long long e0 = i * 8, row = e0 / cols, col = e0 - row * cols;
    if (bias) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] += to_f(bias, col + j, OUT_BF16);
    }
    const long long sl = row / rows_per_slice;
    const long long o = (row - sl * rows_per_slice) * cols + col;
    if (OUT_BF16) {
      uint4 q;
      __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(v[4], v[5]), h3 = __floats2bfloat162_rn(v[6], v[7]);
      q.x = *reinterpret_cast<uint32_t*>(&h0);
      q.y = *reinterpret_cast<uint32_t*>(&h1);
      q.z = *reinterpret_cast<uint32_t*>(&h2);
      q.w = *reinterpret_cast<uint32_t*>(&h3);
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out.p[sl]) + o) = q;
    } else {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out.p[sl]) + o);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

// ------------------------------------------------------------------ colsum
// Column sums over the rows of up to two [batch][rows][cols] inputs (the
// bias gradients db1 and db2 of one backward call) in two launches, each
// block taking its job and coordinates from its linear index.
// Pass 1: a block covers 256 columns of one chunk of rows: 32 column groups
// of 8 (16-byte loads of bf16 rows where the layout allows) times 8 row
// lanes, lane l taking rows l, l+8, ...; the lanes' partial sums are then
// added in lane order.  Pass 2: a block covers 32 columns: 8 lanes, lane l
// adding chunks l, l+8, ... in order, then the lane sums in lane order.  The
// result is fixed for a given chunking.
__device__ __forceinline__ int colsum_pick(const ColsumJobs& J, int& local, bool pass2) {
  const int b0 = pass2 ? J.j[0].blocks2 : J.j[0].blocks1;
  if (J.n > 1 && local >= b0) {
    local -= b0;
    return 1;
  }
  return 0;
}

__global__ void __launch_bounds__(256) colsum_pass1_kernel(const ColsumJobs J) {
  __shared__ float part[8][256 + 4];
  // a programmatic dependent of the kernel that wrote the inputs (or, with
  // no_dep_wait, of one that wrote none of them: it waits before exit)
  if (!J.no_dep_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int local = static_cast<int>(blockIdx.x);
  const ColsumJob& q = J.j[colsum_pick(J, local, false)];
  const int cbs = static_cast<int>((q.cols + 255) / 256);
  const long long cb = local % cbs;
  const long long chunk = (local / cbs) % q.chunks;
  const long long b = (local / cbs) / q.chunks;
  const int cg = threadIdx.x & 31, lane = threadIdx.x >> 5;
  const long long c0 = cb * 256 + cg * 8;
  const long long r0 = chunk * q.chunk_rows;
  const long long r1 = min(q.rows, r0 + q.chunk_rows);
  const bool vec = q.in_bf16 && q.rs % 8 == 0 && q.bs % 8 == 0 && (reinterpret_cast<uintptr_t>(q.in) & 15) == 0 &&
                   c0 + 8 <= q.cols;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (long long r = r0 + lane; r < r1; r += 8) {
    const long long base = b * q.bs + r * q.rs + c0;
    if (vec) {
      const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(q.in) + base);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        acc[2 * k] += f.x;
        acc[2 * k + 1] += f.y;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < q.cols) acc[j] += to_f(q.in, base + j, q.in_bf16);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[lane][cg * 8 + j] = acc[j];
  __syncthreads();
  if (J.no_dep_wait && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long col = cb * 256 + threadIdx.x;
  if (col >= q.cols) return;
  float sum = 0.f;
#pragma unroll
  for (int l = 0; l < 8; ++l) sum += part[l][threadIdx.x];
  q.scratch[(b * q.chunks + chunk) * q.cols + col] = sum;
}

__global__ void __launch_bounds__(256) colsum_pass2_kernel(const ColsumJobs J) {
  __shared__ float part[8][32 + 1];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // pass 1's chunk sums are visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int local = static_cast<int>(blockIdx.x);
  const ColsumJob& q = J.j[colsum_pick(J, local, true)];
  const int cbs = static_cast<int>((q.cols + 31) / 32);
  const long long b = local / cbs;
  const long long col = (local % cbs) * 32LL + (threadIdx.x & 31);
  const int lane = threadIdx.x >> 5;
  float acc = 0.f;
  if (col < q.cols)
    for (long long c = lane; c < q.chunks; c += 8) acc += q.scratch[(b * q.chunks + c) * q.cols + col];
  part[lane][threadIdx.x & 31] = acc;
  __syncthreads();
  if (threadIdx.x >= 32 || col >= q.cols) return;
  float sum = 0.f;
#pragma unroll
  for (int l = 0; l < 8; ++l) sum += part[l][threadIdx.x];
  from_f(q.out, b * q.out_bs + col, sum, q.out_bf16);
}

// ---------------------------------------------------------------- SIMT GEMM
struct SimtOp {
  const float* p;
  long long inner, rows, rs, bs;
  int mn, bsel, gsel;
};
struct SimtParams {
  SimtOp A, B;
  long long M, N, K;
  int NB, G, epi;
  float* out;
  long long out_bs, out_rs;
  float* out2;
  long long out2_bs, out2_rs;
  const float* aux;
  long long aux_bs, aux_rs;
  const float* bias;
  long long bias_bs, bias_len, n_store;
};

// Element (mn, k) of operand X for batch coordinate bc; zero outside the
// operand's extents (the same rule as the tensor-core path's zero fill).
__device__ __forceinline__ float op_at(const SimtOp& X, long long bc, long long mn, long long k) {
  if (!X.mn) {
    if (mn >= X.rows || k >= X.inner) return 0.f;
    return X.p[bc * X.bs + mn * X.rs + k];
  }
  if (mn >= X.inner || k >= X.rows) return 0.f;
  return X.p[bc * X.bs + k * X.rs + mn];
}

__device__ __forceinline__ float dot_gk(const SimtParams& p, long long b, long long m, long long n) {
  float acc = 0.f;
  for (int g = 0; g < p.G; ++g) {
    const long long ab = b * p.A.bsel + g * p.A.gsel, bb = b * p.B.bsel + g * p.B.gsel;
    for (long long k = 0; k < p.K; ++k) acc = fmaf(op_at(p.A, ab, m, k), op_at(p.B, bb, n, k), acc);
  }
  return acc;
}

__global__ void simt_gemm_kernel(const SimtParams p) {
  const long long ncols = (p.epi == EPI_SWIGLU_FWD) ? p.N / 2 : p.N;
  const long long total = (long long)p.NB * p.M * ncols;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long n = idx % ncols;
    const long long m = (idx / ncols) % p.M;
    const long long b = idx / (ncols * p.M);
    if (p.epi == EPI_SWIGLU_FWD) {
      // hidden unit n: rows (n>>7)*256 + (n&127) (a) and +128 (g) of B
      const long long ra = (n >> 7) * 256 + (n & 127);
      const float a = dot_gk(p, b, m, ra), g = dot_gk(p, b, m, ra + 128);
      p.out[b * p.out_bs + m * p.out_rs + n] = a * sigmoid_f(a) * g;
      if (p.out2) {
        p.out2[b * p.out2_bs + m * p.out2_rs + ra] = a;
        p.out2[b * p.out2_bs + m * p.out2_rs + ra + 128] = g;
      }
      continue;
    }
    if (n >= p.n_store) continue;
    float v = dot_gk(p, b, m, n);
    switch (p.epi) {
      case EPI_F32:
        p.out[b * p.out_bs + m * p.out_rs + n] = v;
        break;
      case EPI_OUT:
        if (p.bias && n < p.bias_len) v += p.bias[b * p.bias_bs + n];
        p.out[b * p.out_bs + m * p.out_rs + n] = v;
        break;
      case EPI_GELU_FWD:
        if (p.bias && n < p.bias_len) v += p.bias[b * p.bias_bs + n];
        if (p.out2) p.out2[b * p.out2_bs + m * p.out2_rs + n] = v;
        p.out[b * p.out_bs + m * p.out_rs + n] = gelu_tanh_f(v);
        break;
      case EPI_GELU_BWD:
        p.out[b * p.out_bs + m * p.out_rs + n] = v * gelu_tanh_grad_f(p.aux[b * p.aux_bs + m * p.aux_rs + n]);
        break;
      case EPI_SWIGLU_BWD: {
        const long long col = (n >> 7) * 256 + (n & 127);
        const float a = p.aux[b * p.aux_bs + m * p.aux_rs + col];
        const float g = p.aux[b * p.aux_bs + m * p.aux_rs + col + 128];
        const float sg = sigmoid_f(a);
        p.out[b * p.out_bs + m * p.out_rs + col] = v * g * sg * (1.0f + a * (1.0f - sg));
        p.out[b * p.out_bs + m * p.out_rs + col + 128] = v * a * sg;
        break;
      }
      default:
        break;
    }
  }
}

SimtOp to_simt(const Operand& o) {
  SimtOp s;
  s.p = static_cast<const float*>(o.ptr);
  s.inner = o.inner;
  s.rows = o.rows;
  s.rs = o.row_stride;
  s.bs = o.batch_stride;
  s.mn = o.mn_major;
  s.bsel = o.bsel;
  s.gsel = o.gsel;
  return s;
}

int grid_for(long long work, int per_block, int num_sms) {
  long long g = (work + per_block - 1) / per_block;
  const long long cap = (long long)num_sms * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

int launch_simt_gemm(const GemmSpec& s, LaunchCtx& ctx) {
  SimtParams p{};
  p.A = to_simt(s.A);
  p.B = to_simt(s.B);
  p.M = s.M;
  p.N = s.N;
  p.K = s.K;
  p.NB = s.NB;
  p.G = s.G;
  p.epi = s.epi;
  p.out = static_cast<float*>(s.out);
  p.out_bs = s.out_bs;
  p.out_rs = s.out_rs;
  p.out2 = static_cast<float*>(s.out2);
  p.out2_bs = s.out2_bs;
  p.out2_rs = s.out2_rs;
  p.aux = static_cast<const float*>(s.aux);
  p.aux_bs = s.aux_bs;
  p.aux_rs = s.aux_rs;
  p.bias = static_cast<const float*>(s.bias);
  p.bias_bs = s.bias_bs;
  p.bias_len = s.bias_len;
  p.n_store = s.n_store;
  const long long cols = (s.epi == EPI_SWIGLU_FWD) ? s.N / 2 : s.N;
  const long long total = (long long)s.NB * s.M * cols;
  if (total <= 0) return 0;
  if (ctx.before) ctx.before(ctx.user, s.name, ctx.stream);
  simt_gemm_kernel<<<grid_for(total, 256, ctx.num_sms), 256, 0, ctx.stream>>>(p);
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

int launch_pack_columns(const void* W1, const void* W3, void* out, int T_p, int64_t s, int64_t s_pad, int64_t d,
                        int swiglu, int esz, int unpack, cudaStream_t st) {
  const long long blocks = (long long)T_p * (swiglu ? 2 * s_pad : s_pad);
  if (blocks <= 0) return 0;
  pack_columns_kernel<<<static_cast<unsigned>(blocks), 128, 0, st>>>(
      static_cast<const char*>(W1), static_cast<const char*>(W3), static_cast<char*>(out), s, s_pad, d, swiglu, esz,
      unpack);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

int launch_pack_rows(const void* W2, void* out, int T_p, int64_t s, int64_t s_pad, int64_t d, int esz, int unpack,
                     cudaStream_t st) {
  const long long blocks = (long long)T_p * d;
  if (blocks <= 0) return 0;
  pack_rows_kernel<<<static_cast<unsigned>(blocks), 128, 0, st>>>(static_cast<const char*>(W2),
                                                                  static_cast<char*>(out), s, s_pad, d, T_p, esz,
                                                                  unpack);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

// Launch as a programmatic dependent of the stream's previous kernel (the
// kernel waits for its results with griddepcontrol.wait).
template <typename... KArgs, typename... Args>
static void launch_pdl(void (*kern)(KArgs...), dim3 grid, int block, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

int launch_shard_sum(const float* partials, int T_p, int64_t rows, int64_t cols, const void* bias, void* out,
                     int out_bf16, LaunchCtx& ctx, const char* name, int64_t shard_stride) {
  const long long plane = (long long)rows * cols;
  if (plane <= 0) return 0;
  const long long stride = shard_stride > 0 ? shard_stride : plane;
  if (ctx.before) ctx.before(ctx.user, name, ctx.stream);
  const bool vec = (cols % 8 == 0) && (reinterpret_cast<uintptr_t>(partials) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  if (vec) {
    const int grid = grid_for(plane / 8, 256, ctx.num_sms);
    if (out_bf16)
      launch_pdl(shard_sum_vec8_kernel<1>, dim3(grid), 256, ctx.stream, partials, T_p, plane, cols,
                 static_cast<const __nv_bfloat16*>(bias), static_cast<const float*>(nullptr), out, stride);
    else
      launch_pdl(shard_sum_vec8_kernel<0>, dim3(grid), 256, ctx.stream, partials, T_p, plane, cols,
                 static_cast<const __nv_bfloat16*>(nullptr), static_cast<const float*>(bias), out, stride);
  } else {
    shard_sum_scalar_kernel<<<grid_for(plane, 256, ctx.num_sms), 256, 0, ctx.stream>>>(
        partials, T_p, plane, cols, bias, out_bf16, out, out_bf16, stride);
  }
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

// SwiGLU of a K-split up GEMM (decode-sized token counts): the fp32 parts
// P[k][t][m][c] (k < ksplit, t < T, m < rows, c < W = 2 s_pad, hidden unit u
// of shard t at column (u / 128) 256 + u % 128 for a and + 128 for g) are
// summed in the order k = 0, 1, ..; then h = silu(a) g, as the GEMM's own
// SwiGLU epilogue forms it, in bf16 at h[t][m][u], and, when `saved` is
// given, a and g in bf16 at saved[t][m][c].  One thread per 8 hidden units.
__global__ void __launch_bounds__(256) swiglu_combine_kernel(const float* __restrict__ P, int ksplit, long long part,
                                                             int T, long long rows, long long s_pad,
                                                             __nv_bfloat16* h, __nv_bfloat16* saved) {
  // a programmatic dependent of the GEMM that wrote the parts
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long W = 2 * s_pad;
  const long long u8 = s_pad / 8;
  const long long total = (long long)T * rows * u8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long tm = i / u8;  // t * rows + m
    const long long u = (i - tm * u8) * 8;
    const long long ca = (u >> 7) * 256 + (u & 127);
    const float* pa = P + tm * W + ca;
    float a[8], g[8];
    {
      const float4 a0 = reinterpret_cast<const float4*>(pa)[0], a1 = reinterpret_cast<const float4*>(pa)[1];
      const float4 g0 = reinterpret_cast<const float4*>(pa + 128)[0], g1 = reinterpret_cast<const float4*>(pa + 128)[1];
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w; g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
    }
    for (int k = 1; k < ksplit; ++k) {
      const float* q = pa + k * part;
      const float4 a0 = reinterpret_cast<const float4*>(q)[0], a1 = reinterpret_cast<const float4*>(q)[1];
      const float4 g0 = reinterpret_cast<const float4*>(q + 128)[0], g1 = reinterpret_cast<const float4*>(q + 128)[1];
      a[0] += a0.x; a[1] += a0.y; a[2] += a0.z; a[3] += a0.w; a[4] += a1.x; a[5] += a1.y; a[6] += a1.z; a[7] += a1.w;
      g[0] += g0.x; g[1] += g0.y; g[2] += g0.z; g[3] += g0.w; g[4] += g1.x; g[5] += g1.y; g[6] += g1.z; g[7] += g1.w;
    }
    float hv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) hv[j] = a[j] * sigmoid_f(a[j]) * g[j];
    auto pack8 = [](const float* v) {
      uint4 q;
      __nv_bfloat162 x0 = __floats2bfloat162_rn(v[0], v[1]), x1 = __floats2bfloat162_rn(v[2], v[3]);
      __nv_bfloat162 x2 = __floats2bfloat162_rn(v[4], v[5]), x3 = __floats2bfloat162_rn(v[6], v[7]);
      q.x = *reinterpret_cast<uint32_t*>(&x0);
      q.y = *reinterpret_cast<uint32_t*>(&x1);
      q.z = *reinterpret_cast<uint32_t*>(&x2);
      q.w = *reinterpret_cast<uint32_t*>(&x3);
      return q;
    };
    *reinterpret_cast<uint4*>(h + tm * s_pad + u) = pack8(hv);
    if (saved) {
      *reinterpret_cast<uint4*>(saved + tm * W + ca) = pack8(a);
      *reinterpret_cast<uint4*>(saved + tm * W + ca + 128) = pack8(g);
    }
  }
}

int launch_swiglu_combine(const float* parts, int ksplit, int T_p, int64_t rows, int64_t s_pad, void* h,
                          void* saved, LaunchCtx& ctx, const char* name) {
  const long long total = (long long)T_p * rows * (s_pad / 8);
  if (total <= 0) return 0;
  if (s_pad % 128 || reinterpret_cast<uintptr_t>(parts) % 16 || reinterpret_cast<uintptr_t>(h) % 16 ||
      reinterpret_cast<uintptr_t>(saved) % 16)
    return TP_ERR_ALIGN;
  if (ctx.before) ctx.before(ctx.user, name, ctx.stream);
  launch_pdl(swiglu_combine_kernel, dim3(grid_for(total, 256, ctx.num_sms)), 256, ctx.stream, parts, ksplit,
             (long long)T_p * rows * 2 * s_pad, T_p, rows, s_pad, static_cast<__nv_bfloat16*>(h),
             static_cast<__nv_bfloat16*>(saved));
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

// Fix-up of a pair GEMM's last-wave split: tail tile i (the 256 x 256 output
// block of batch b[i] at rows mp[i] * 256, columns nb[i] * 256) was
// accumulated as t.parts K parts, part k's fp32 block at
// P + (k * t.n + i) * 65536 (row-major, 256 columns).  The parts are added in
// the order k = 0, 1, .., then the bias, and the result written as the GEMM's
// own epilogue would have: v in bf16 (GEMM output), or h = gelu(v) and, with
// out2, z = v (GELU forward), or, for the SwiGLU forward, h = silu(a) g and,
// with out2, a and g.  Rows >= M and columns >= n_store (hidden units for
// SwiGLU) are not written.  One thread per 4 columns (4 hidden units, SwiGLU);
// the parts are read four at a time with independent loads (the sum order
// stays k = 0, 1, ..).
__device__ __forceinline__ float4 tail_part_sum(const float4* q, long long stride, int parts) {
  float4 acc = q[0];
  int k = 1;
  for (; k + 3 < parts; k += 4) {
    const float4 a = q[k * stride], b = q[(k + 1) * stride], e = q[(k + 2) * stride], f = q[(k + 3) * stride];
    acc.x = (((acc.x + a.x) + b.x) + e.x) + f.x;
    acc.y = (((acc.y + a.y) + b.y) + e.y) + f.y;
    acc.z = (((acc.z + a.z) + b.z) + e.z) + f.z;
    acc.w = (((acc.w + a.w) + b.w) + e.w) + f.w;
  }
  for (; k < parts; ++k) {
    const float4 a = q[k * stride];
    acc.x += a.x;
    acc.y += a.y;
    acc.z += a.z;
    acc.w += a.w;
  }
  return acc;
}
__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, const float* v) {
  __nv_bfloat162 h[2] = {__floats2bfloat162_rn(v[0], v[1]), __floats2bfloat162_rn(v[2], v[3])};
  *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(h);
}
__global__ void __launch_bounds__(256) tail_fixup_kernel(const float* __restrict__ P, TailTiles t, TailOut o) {
  // a programmatic dependent of the GEMM that wrote the parts
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long stride = static_cast<long long>(t.n) * (65536 / 4);  // float4s between parts
  if (o.act == 2) {
    // SwiGLU: a at the tile's columns [0, 128), g at [128, 256)
    const long long total = static_cast<long long>(t.n) * 256 * 32;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
      const int ti = static_cast<int>(i >> 13);
      const int r = static_cast<int>((i >> 5) & 255), u = static_cast<int>(i & 31) * 4;
      const long long row = static_cast<long long>(t.mp[ti]) * 256 + r;
      const long long hcol = static_cast<long long>(t.nb[ti]) * 128 + u;
      if (row >= o.M || hcol >= o.n_store) continue;
      const float4* q = reinterpret_cast<const float4*>(P) + ti * (65536 / 4) + r * 64 + u / 4;
      const float4 a4 = tail_part_sum(q, stride, t.parts), g4 = tail_part_sum(q + 32, stride, t.parts);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w}, g[4] = {g4.x, g4.y, g4.z, g4.w};
      float h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = a[j] * sigmoid_f(a[j]) * g[j];
      const long long bt = t.b[ti];
      store_bf16x4(static_cast<__nv_bfloat16*>(o.out) + bt * o.out_bs + row * o.out_rs + hcol, h);
      if (o.out2) {
        __nv_bfloat16* sv = static_cast<__nv_bfloat16*>(o.out2) + bt * o.out2_bs + row * o.out2_rs +
                            static_cast<long long>(t.nb[ti]) * 256 + u;
        store_bf16x4(sv, a);
        store_bf16x4(sv + 128, g);
      }
    }
    return;
  }
  const long long total = static_cast<long long>(t.n) * 256 * 64;
  const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(o.bias);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ti = static_cast<int>(i >> 14);
    const int r = static_cast<int>((i >> 6) & 255), c = static_cast<int>(i & 63) * 4;
    const long long row = static_cast<long long>(t.mp[ti]) * 256 + r, col = static_cast<long long>(t.nb[ti]) * 256 + c;
    if (row >= o.M || col >= o.n_store) continue;  // n_store is a multiple of 8: the 4 columns are all in or all out
    const float4 acc = tail_part_sum(reinterpret_cast<const float4*>(P) + ti * (65536 / 4) + r * 64 + c / 4, stride,
                                     t.parts);
    float v[4] = {acc.x, acc.y, acc.z, acc.w};
    const long long bt = t.b[ti];
    if (bias) {
      const __nv_bfloat16* bp = bias + bt * o.bias_bs;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (col + j < o.bias_len) v[j] += __bfloat162float(bp[col + j]);
    }
    if (o.act == 1) {
      if (o.out2) store_bf16x4(static_cast<__nv_bfloat16*>(o.out2) + bt * o.out2_bs + row * o.out2_rs + col, v);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = gelu_tanh_f(v[j]);
    }
    store_bf16x4(static_cast<__nv_bfloat16*>(o.out) + bt * o.out_bs + row * o.out_rs + col, v);
  }
}

int launch_tail_fixup(const float* parts, const TailTiles& t, const TailOut& o, LaunchCtx& ctx, const char* name) {
  if (t.n < 1 || t.n > kMaxTailTiles || t.parts < 2) return TP_ERR_INVALID;
  const auto a16 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
  if (!a16(parts) || !a16(o.out) || (o.out2 && !a16(o.out2)) || o.out_rs % 8 || o.out_bs % 8 || o.out2_rs % 8 ||
      o.out2_bs % 8 || o.n_store % 8)
    return TP_ERR_ALIGN;
  const long long total = static_cast<long long>(t.n) * 256 * (o.act == 2 ? 32 : 64);
  if (ctx.before) ctx.before(ctx.user, name, ctx.stream);
  launch_pdl(tail_fixup_kernel, dim3(grid_for(total, 256, ctx.num_sms)), 256, ctx.stream, parts, t, o);
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

static SliceTable to_table(const RowSlices& r) {
  SliceTable t{};
  for (int i = 0; i < r.n && i < kMaxSlices; ++i) t.p[i] = static_cast<char*>(r.ptr[i]);
  return t;
}

static bool all_aligned16(const RowSlices& r) {
  for (int i = 0; i < r.n; ++i)
    if (reinterpret_cast<uintptr_t>(r.ptr[i]) % 16) return false;
  return true;
}

static int slice_copy(const RowSlices& r, void* buf, int64_t cols, int esz, int to_slices, LaunchCtx& ctx,
                      const char* name) {
  const long long slice_bytes = r.rows * cols * esz;
  const long long total = slice_bytes * r.n;
  if (total <= 0) return 0;
  if (ctx.before) ctx.before(ctx.user, name, ctx.stream);
  if (slice_bytes % 16 == 0 && all_aligned16(r) && reinterpret_cast<uintptr_t>(buf) % 16 == 0)
    slice_copy_kernel<<<grid_for(total / 16, 256, ctx.num_sms), 256, 0, ctx.stream>>>(
        to_table(r), static_cast<char*>(buf), slice_bytes, total, to_slices);
  else
    slice_copy_bytes_kernel<<<grid_for(total, 256, ctx.num_sms), 256, 0, ctx.stream>>>(
        to_table(r), static_cast<char*>(buf), slice_bytes, total, to_slices);
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

int launch_gather_rows(const RowSlices& src, void* dst, int64_t cols, int esz, LaunchCtx& ctx, const char* name) {
  return slice_copy(src, dst, cols, esz, 0, ctx, name);
}

int launch_scatter_rows(const void* src, int64_t n, int64_t cols, int esz, const RowSlices& dst, LaunchCtx& ctx,
                        const char* name) {
  (void)n;
  return slice_copy(dst, const_cast<void*>(src), cols, esz, 1, ctx, name);
}

int launch_shard_sum_scatter(const float* partials, int T_p, int64_t rows, int64_t cols, const void* bias,
                             const RowSlices& out, int out_bf16, LaunchCtx& ctx, const char* name) {
  const long long plane = (long long)rows * cols;
  if (plane <= 0) return 0;
  if (ctx.before) ctx.before(ctx.user, name, ctx.stream);
  const bool vec = cols % 8 == 0 && reinterpret_cast<uintptr_t>(partials) % 16 == 0 && all_aligned16(out);
  const SliceTable tab = to_table(out);
  if (vec) {
    const int grid = grid_for(plane / 8, 256, ctx.num_sms);
    if (out_bf16)
      shard_sum_scatter_vec8_kernel<1><<<grid, 256, 0, ctx.stream>>>(partials, T_p, plane, cols, bias, tab, out.rows);
    else
      shard_sum_scatter_vec8_kernel<0><<<grid, 256, 0, ctx.stream>>>(partials, T_p, plane, cols, bias, tab, out.rows);
  } else {
    const int grid = grid_for(plane, 256, ctx.num_sms);
    if (out_bf16)
      shard_sum_scatter_kernel<1><<<grid, 256, 0, ctx.stream>>>(partials, T_p, plane, cols, bias, tab, out.rows);
    else
      shard_sum_scatter_kernel<0><<<grid, 256, 0, ctx.stream>>>(partials, T_p, plane, cols, bias, tab, out.rows);
  }
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  ctx.launches++;
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

int64_t colsum_scratch_floats(int64_t batch, int64_t rows, int64_t cols, int64_t chunk_rows) {
  const int64_t chunks = (rows + chunk_rows - 1) / chunk_rows;
  return batch * (chunks > 0 ? chunks : 1) * cols;
}

// The call's device error word cleared at its start, as a programmatic
// dependent: the call's first kernel may launch at once (its set-up overlaps
// the previous kernel on the stream), and the word is written only after
// every kernel before this one has completed.
__global__ void reset_error_word_kernel(int* err) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) *err = 0;
}

int launch_reset_error_word(int* err, cudaStream_t stream) {
  launch_pdl(reset_error_word_kernel, dim3(1), 32, stream, err);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

int launch_colsums(ColsumJobs J, LaunchCtx& ctx, const char* name) {
  static const bool no_overlap = getenv("TPFFN_NO_DEP_OVERLAP") != nullptr;  // for comparisons
  if (no_overlap) J.no_dep_wait = 0;
  long long g1 = 0, g2 = 0;
  int kept = 0;
  for (int i = 0; i < J.n; ++i) {
    ColsumJob& q = J.j[i];
    if (q.batch <= 0 || q.cols <= 0) continue;
    q.chunks = q.rows > 0 ? (q.rows + q.chunk_rows - 1) / q.chunk_rows : 0;
    const long long b1 = (q.cols + 255) / 256 * q.chunks * q.batch, b2 = (q.cols + 31) / 32 * q.batch;
    if (b1 > INT_MAX || b2 > INT_MAX) return TP_ERR_UNSUPPORTED;
    q.blocks1 = static_cast<int>(b1);
    q.blocks2 = static_cast<int>(b2);
    g1 += b1;
    g2 += b2;
    J.j[kept++] = q;
  }
  J.n = kept;
  if (kept == 0) return 0;
  if (g1 > INT_MAX || g2 > INT_MAX) return TP_ERR_UNSUPPORTED;
  if (ctx.before) ctx.before(ctx.user, name, ctx.stream);
  if (g1 > 0) {  // no rows: pass 2 writes zeros
    launch_pdl(colsum_pass1_kernel, dim3(static_cast<unsigned>(g1)), 256, ctx.stream, J);
    ctx.launches++;
  }
  launch_pdl(colsum_pass2_kernel, dim3(static_cast<unsigned>(g2)), 256, ctx.stream, J);
  ctx.launches++;
  if (ctx.after) ctx.after(ctx.user, ctx.stream);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : TP_ERR_CUDA;
}

}  // namespace tpffn
