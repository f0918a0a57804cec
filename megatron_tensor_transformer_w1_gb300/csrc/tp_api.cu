// tp_api.cu -- the C ABI of include/tpffn.h: plans, buffer sizes, packing,
// and the forward/backward orchestration of the shard computations.
//
// Forward ("7.9 Tensor and pipeline parallelism (TP, PP)", §2.1 "The FFN,
// sharded"; SwiGLU per "S17 Tensor & Pipeline Parallelism", listing "the
// megatron pattern"):
//   1. up GEMM, all shards in one launch: h^(t) = sigma(x W1^(t)T [+ b1^(t)])
//      (SwiGLU: a and g from one interleaved tile, h = silu(a) * g)
//   2. down GEMM: y^(t) = h^(t) W2^(t)T as fp32 partials, then the ordered
//      shard-sum y = sum_t y^(t) (+ b2)   [standalone], or one GEMM whose
//      K loop walks shard 0..T_p-1 into the same accumulator    [fused]
// Backward (g is the identity, f sums dx):
//   3. dh^(t) = dy W2^(t) with the activation derivative fused (dz, or da|dg)
//   4. dx = sum_t dz^(t) W1^(t) (+ dg^(t) W3^(t))   [fused or standalone]
//   5. dW2^(t) = dy^T h^(t);  dW1^(t) (|dW3^(t)) = dz^(t)T x  -- per shard
//   6. db1 = sum_n dz, db2 = sum_n dy (ordered two-pass column sums)
// The attention output projection (§2.2 "Attention, sharded") is steps 2, 3
// and 5 with the concatenated head outputs as h and no activation.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "tp_internal.h"
#include "tpffn.h"

using namespace tpffn;

struct TimingRec {
  const char* name;
  cudaEvent_t start, stop;
};

struct tp_ffn_plan {
  int64_t d = 0, d_ff = 0, s = 0, s_pad = 0;
  int T_p = 1, act = TP_ACT_GELU_TANH, dtype = TP_BF16;
  int n_heads = 0, n_kv_heads = 0;
  int64_t head_dim = 0;
  // diagnostics (host side; not thread-safe when TP_FLAG_TIMING is used)
  mutable std::vector<TimingRec> events;
  mutable int n_events = 0;
  mutable int last_launches = 0;
  mutable cudaStream_t timing_stream = nullptr;
  // second stream and events of the overlapped shard-sum (host handles,
  // created on first use on a device; not thread-safe)
  mutable int ov_device = -1;
  mutable cudaStream_t ov_stream = nullptr;
  mutable std::vector<cudaEvent_t> ov_events;
  mutable cudaEvent_t ov_join = nullptr;
};

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline int esz(const tp_ffn_plan* p) { return p->dtype == TP_BF16 ? 2 : 4; }
inline int64_t hidden_width(const tp_ffn_plan* p) {  // columns per shard of the up GEMM / of dz
  return p->act == TP_ACT_SWIGLU ? 2 * p->s_pad : p->s_pad;
}
inline bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

int num_sms_current() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) return 148;
  int v = cache[dev].load();
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    cache[dev].store(v);
  }
  return v;
}

// Rows per block of the first column-sum pass: 64 (enough blocks to spread
// a short token axis over the SMs), more for very long token
// counts so that the chunk count stays within the grid's y limit.
int64_t colsum_chunk(int64_t rows) {
  int64_t c = 64;
  while ((rows + c - 1) / c > 4096) c *= 2;
  return c;
}

ColsumJob colsum_job(const void* in, int in_bf16, int64_t batch, int64_t rows, int64_t cols, int64_t rs, int64_t bs,
                     void* out, int out_bf16, int64_t out_bs, float* scratch, int64_t n) {
  ColsumJob q;
  q.in = in;
  q.in_bf16 = in_bf16;
  q.batch = static_cast<int>(batch);
  q.rows = rows;
  q.cols = cols;
  q.rs = rs;
  q.bs = bs;
  q.out = out;
  q.out_bf16 = out_bf16;
  q.out_bs = out_bs;
  q.scratch = scratch;
  q.chunk_rows = colsum_chunk(n);
  return q;
}

struct WsLayout {
  size_t h = 0, part = 0, D = 0, cs = 0, ks = 0, wk = 0, tail = 0, tail_bytes = 0, total = 0;
  bool has_part = false, has_ks = false, has_wk = false, has_tail = false;
};

// Decode-sized SwiGLU forwards (at most 32 tokens: one 32-row A tile) may
// split the up GEMM's K: its T_p x ceil(W / 256) weight tiles are too few to
// give every SM the same number, and two K parts per tile fill the GPU
// evenly; the fp32 parts are summed, in order, by the SwiGLU combine kernel.
constexpr int kMaxKsplit = 2;
bool ksplit_shape(const tp_ffn_plan* p, int64_t n) {
  return p->act == TP_ACT_SWIGLU && p->dtype == TP_BF16 && n >= 1 && n <= 32;
}
int choose_ksplit(const tp_ffn_plan* p, int64_t n, int num_sms) {
  static const bool off = [] {
    const char* v = getenv("TPFFN_KSPLIT");
    return v && v[0] == '0';
  }();
  if (off || !ksplit_shape(p, n) || num_sms < 1) return 1;
  const int64_t k_blocks = (p->d + 63) / 64;
  const int64_t tiles = p->T_p * ((hidden_width(p) + 255) / 256);
  auto eff = [&](int64_t units) {  // share of the SM-unit slots the busiest wave count leaves in use
    const int64_t waves = (units + num_sms - 1) / num_sms;
    return static_cast<double>(units) / static_cast<double>(waves * num_sms);
  };
  int best = 1;
  for (int k = 2; k <= kMaxKsplit; ++k)
    if (k_blocks >= 16 * k && eff(tiles * k) > eff(tiles * best) + 0.05) best = k;
  return best;
}

// Weight-gradient GEMMs (K = the token axis) with fewer 256 x 256 output
// tile pairs than the GPU has SM pairs leave most SMs idle for their whole K
// loop -- GPT-2-small-shaped shards have 3 x 3 tiles x 4 shards for 76 SM
// pairs.  Splitting K into parts gives each SM pair a part of a tile; the
// pair kernel writes each part in fp32 and the shard-sum kernel adds them in
// part order (deterministic).  The split is taken where it shortens the
// busiest SM pair's K loop (waves of units x K blocks per unit) by more than
// a tenth, each part keeping at least 16 K blocks of 64 tokens.
constexpr int kMaxWgradKsplit = 4;
// TPFFN_MERGE_SHARDS=0: the W_O backward GEMMs run per shard (for comparisons)
bool merge_shards_enabled() {
  static const bool on = [] {
    const char* v = getenv("TPFFN_MERGE_SHARDS");
    return !(v && v[0] == '0');
  }();
  return on;
}
int wgrad_ksplit(const tp_ffn_plan* p, int64_t n, int64_t M, int64_t N, int num_sms) {
  static const bool off = [] {
    const char* v = getenv("TPFFN_WGRAD_KSPLIT");
    return v && v[0] == '0';
  }();
  if (off || p->dtype != TP_BF16 || p->act == TP_ACT_NONE || !tc_pair_path(M) || num_sms < 2) return 1;
  const int64_t pairs = num_sms / 2;
  const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256) * p->T_p;
  const int64_t k_blocks = (n + 63) / 64;
  auto busiest = [&](int64_t k) { return ((tiles * k + pairs - 1) / pairs) * ((k_blocks + k - 1) / k); };
  int best = 1;
  for (int k = 2; k <= kMaxWgradKsplit; ++k)
    if (k_blocks >= 16 * k && 10 * busiest(k) < 9 * busiest(best)) best = k;
  return best;
}
// fp32 bytes of the K parts of the two weight-gradient GEMMs (0: no split)
size_t wgrad_parts_bytes(const tp_ffn_plan* p, int64_t n, int num_sms) {
  const size_t T = static_cast<size_t>(p->T_p), d = static_cast<size_t>(p->d), sp = static_cast<size_t>(p->s_pad);
  const size_t W = static_cast<size_t>(hidden_width(p));
  const int ka = wgrad_ksplit(p, n, p->d, p->s_pad, num_sms), kb = wgrad_ksplit(p, n, W, p->d, num_sms);
  const size_t a = ka > 1 ? ka * T * d * sp : 0, b = kb > 1 ? kb * T * W * d : 0;
  return 4 * (a > b ? a : b);
}

WsLayout ws_layout(const tp_ffn_plan* p, int64_t n, int flags) {
  WsLayout L;
  size_t off = kAlign;  // error word + header
  const size_t e = esz(p);
  if (p->act != TP_ACT_NONE) {
    L.h = off;
    off += align_up(static_cast<size_t>(p->T_p) * n * p->s_pad * e);
    L.D = off;
    off += align_up(static_cast<size_t>(p->T_p) * n * hidden_width(p) * e);
  }
  if (!(flags & TP_SUM_FUSED)) {
    L.has_part = true;
    L.part = off;
    off += align_up(static_cast<size_t>(p->T_p) * n * p->d * 4);
  }
  if (ksplit_shape(p, n)) {
    L.has_ks = true;
    L.ks = off;
    off += align_up(static_cast<size_t>(kMaxKsplit) * p->T_p * n * hidden_width(p) * 4);
  }
  if (p->act != TP_ACT_NONE) {
    const size_t wk = wgrad_parts_bytes(p, n, num_sms_current());
    if (wk) {
      L.has_wk = true;
      L.wk = off;
      off += align_up(wk);
    }
  }
  if (((flags & TP_SUM_FUSED) || p->act != TP_ACT_NONE) && p->dtype == TP_BF16 && tc_pair_path(n)) {
    // fp32 K parts of the last-wave tiles of a fused-sum GEMM or of the up
    // GEMM: at most one 256 x 256 block per SM pair
    L.has_tail = true;
    L.tail = off;
    L.tail_bytes = static_cast<size_t>(num_sms_current() / 2) * 256 * 256 * 4;
    off += align_up(L.tail_bytes);
  }
  L.cs = off;
  const int64_t cs1 = colsum_scratch_floats(p->T_p, n, p->s_pad, colsum_chunk(n));
  const int64_t cs2 = colsum_scratch_floats(1, n, p->d, colsum_chunk(n));
  // db1 (GELU plans only) and db2 sum in the same launches, side by side
  off += align_up(static_cast<size_t>(p->act == TP_ACT_GELU_TANH ? cs1 + cs2 : (cs1 > cs2 ? cs1 : cs2)) * 4);
  L.total = off;
  return L;
}

struct SavedLayout {
  size_t act = 0, h = 0, total = 0;
};
SavedLayout saved_layout(const tp_ffn_plan* p, int64_t n) {
  SavedLayout S;
  if (p->act == TP_ACT_NONE) return S;
  const size_t e = esz(p);
  S.act = 0;
  S.h = align_up(static_cast<size_t>(p->T_p) * n * hidden_width(p) * e);
  S.total = S.h + align_up(static_cast<size_t>(p->T_p) * n * p->s_pad * e);
  return S;
}

// Timing hooks: an event pair per launch, kept in the plan.
void timing_before(void* user, const char* name, cudaStream_t stream) {
  const tp_ffn_plan* p = static_cast<const tp_ffn_plan*>(user);
  if (p->n_events >= static_cast<int>(p->events.size())) {
    TimingRec r{name, nullptr, nullptr};
    cudaEventCreate(&r.start);
    cudaEventCreate(&r.stop);
    p->events.push_back(r);
  }
  TimingRec& r = p->events[p->n_events];
  r.name = name;
  cudaEventRecord(r.start, stream);
}
void timing_after(void* user, cudaStream_t stream) {
  const tp_ffn_plan* p = static_cast<const tp_ffn_plan*>(user);
  cudaEventRecord(p->events[p->n_events].stop, stream);
  p->n_events++;
}

int make_ctx(const tp_ffn_plan* p, void* workspace, int flags, cudaStream_t stream, LaunchCtx& ctx) {
  ctx.stream = stream;
  ctx.err = static_cast<int*>(workspace);
  ctx.num_sms = num_sms_current();
  ctx.debug_skip_load = (flags & TP_FLAG_DEBUG_SKIP_LOAD) ? 1 : 0;
  ctx.timing = (flags & TP_FLAG_TIMING) != 0;
  if (ctx.timing) {
    p->timing_stream = stream;
    ctx.before = timing_before;
    ctx.after = timing_after;
    ctx.user = const_cast<tp_ffn_plan*>(p);
  }
  static const bool memset_reset = getenv("TPFFN_MEMSET") != nullptr;  // for comparisons
  if (memset_reset) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess) return TP_ERR_CUDA;
  } else {
    if (launch_reset_error_word(ctx.err, stream)) return TP_ERR_CUDA;
    ctx.launches++;
  }
  return TP_OK;
}

int finish_call(const tp_ffn_plan* p, LaunchCtx& ctx, int rc, int flags, void* workspace) {
  p->last_launches = ctx.launches;
  if (rc != TP_OK) return rc;
  if (cudaPeekAtLastError() != cudaSuccess) return TP_ERR_CUDA;
  if (flags & TP_FLAG_SYNC) return tp_ffn_last_device_error(p, workspace, ctx.stream);
  return TP_OK;
}

int run_gemm(const tp_ffn_plan* p, const GemmSpec& g, LaunchCtx& ctx) {
  return p->dtype == TP_BF16 ? launch_tc_gemm(g, ctx) : launch_simt_gemm(g, ctx);
}

// Token chunks of the overlapped sum.  Measured on GB300 (Llama-3-8B step):
// 1, 2 and 4 chunks all lose to the plain standalone path, because the
// persistent GEMM already holds every SM and the sum is HBM-bound either way.
constexpr int kOverlapChunks = 4;

void release_overlap(const tp_ffn_plan* p) {
  for (cudaEvent_t e : p->ov_events) cudaEventDestroy(e);
  p->ov_events.clear();
  if (p->ov_join) cudaEventDestroy(p->ov_join);
  if (p->ov_stream) cudaStreamDestroy(p->ov_stream);
  p->ov_join = nullptr;
  p->ov_stream = nullptr;
  p->ov_device = -1;
}

int ensure_overlap(const tp_ffn_plan* p) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TP_ERR_CUDA;
  if (p->ov_device == dev && p->ov_stream) return TP_OK;
  release_overlap(p);
  if (cudaStreamCreateWithFlags(&p->ov_stream, cudaStreamNonBlocking) != cudaSuccess) return TP_ERR_CUDA;
  for (int i = 0; i < kOverlapChunks; ++i) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return TP_ERR_CUDA;
    p->ov_events.push_back(e);
  }
  if (cudaEventCreateWithFlags(&p->ov_join, cudaEventDisableTiming) != cudaSuccess) return TP_ERR_CUDA;
  p->ov_device = dev;
  return TP_OK;
}

// Row-sharded GEMM into fp32 partials followed by the ordered shard-sum,
// split into token chunks: the sum of chunk i runs on the plan's second
// stream while the GEMM of chunk i+1 runs on the call's stream.  `g` is the
// whole-problem spec (NB = T_p, EPI_F32, out = partials [T_p][n][d]) whose A
// operand has the tokens as rows; chunk results are bit-identical to the
// unchunked path (same per-element arithmetic).
int gemm_sum_overlapped(const tp_ffn_plan* p, const GemmSpec& g, LaunchCtx& ctx, float* part, int64_t n,
                        int64_t d, const void* bias, void* out, int out_bf16, const char* sum_name) {
  int rc = ensure_overlap(p);
  if (rc) return rc;
  const size_t esz_in = p->dtype == TP_BF16 ? 2 : 4;
  const int64_t per = ((n + kOverlapChunks - 1) / kOverlapChunks + 255) / 256 * 256;
  int i = 0;
  for (int64_t r0 = 0; r0 < n; r0 += per, ++i) {
    const int64_t rows = (n - r0) < per ? (n - r0) : per;
    GemmSpec c = g;
    c.M = rows;
    c.A.rows = rows;
    c.A.ptr = static_cast<const char*>(g.A.ptr) + static_cast<size_t>(r0) * g.A.row_stride * esz_in;
    c.out = part + r0 * d;
    rc = run_gemm(p, c, ctx);
    if (rc) return rc;
    if (cudaEventRecord(p->ov_events[i], ctx.stream) != cudaSuccess ||
        cudaStreamWaitEvent(p->ov_stream, p->ov_events[i], 0) != cudaSuccess)
      return TP_ERR_CUDA;
    LaunchCtx actx = ctx;
    actx.stream = p->ov_stream;
    actx.launches = 0;
    rc = launch_shard_sum(part + r0 * d, p->T_p, rows, d, bias,
                          static_cast<char*>(out) + static_cast<size_t>(r0) * d * (out_bf16 ? 2 : 4), out_bf16,
                          actx, sum_name, n * d);
    ctx.launches += actx.launches;
    if (rc) return rc;
  }
  if (cudaEventRecord(p->ov_join, p->ov_stream) != cudaSuccess ||
      cudaStreamWaitEvent(ctx.stream, p->ov_join, 0) != cudaSuccess)
    return TP_ERR_CUDA;
  return TP_OK;
}

Operand kmajor(const void* ptr, int64_t inner, int64_t rows, int64_t batch, int64_t rs, int64_t bs, int bsel,
               int gsel) {
  Operand o;
  o.ptr = ptr;
  o.inner = inner;
  o.rows = rows;
  o.batch = batch;
  o.row_stride = rs;
  o.batch_stride = bs;
  o.mn_major = 0;
  o.bsel = bsel;
  o.gsel = gsel;
  return o;
}
Operand mnmajor(const void* ptr, int64_t inner, int64_t rows, int64_t batch, int64_t rs, int64_t bs, int bsel,
                int gsel) {
  Operand o = kmajor(ptr, inner, rows, batch, rs, bs, bsel, gsel);
  o.mn_major = 1;
  return o;
}

}  // namespace

// ======================================================================= ABI
extern "C" {

const char* tp_ffn_status_string(int status) {
  switch (status) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID: return "TP_ERR_INVALID: invalid argument";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED: not supported by this build";
    case TP_ERR_CUDA: return "TP_ERR_CUDA: CUDA call or kernel launch failed";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT: a device-side bounded wait expired";
    case TP_ERR_ALIGN: return "TP_ERR_ALIGN: pointer or stride not 16-byte aligned";
    default: return "unknown status";
  }
}

int tp_ffn_plan_create(tp_ffn_plan** out, int64_t d, int64_t d_ff, int T_p, int act, int dtype) {
  if (!out) return TP_ERR_INVALID;
  *out = nullptr;
  if (d < 1 || d_ff < 1 || T_p < 1 || d_ff % T_p != 0) return TP_ERR_INVALID;
  if (act != TP_ACT_NONE && act != TP_ACT_GELU_TANH && act != TP_ACT_SWIGLU) return TP_ERR_INVALID;
  if (dtype != TP_BF16 && dtype != TP_F32) return TP_ERR_INVALID;
  const int64_t s = d_ff / T_p;
  if (dtype == TP_BF16) {
    if (d % 8 != 0) return TP_ERR_UNSUPPORTED;
    if (act == TP_ACT_NONE && s % 8 != 0) return TP_ERR_UNSUPPORTED;
  }
  if (d > (int64_t(1) << 30) || d_ff > (int64_t(1) << 30)) return TP_ERR_UNSUPPORTED;
  tp_ffn_plan* p = new (std::nothrow) tp_ffn_plan();
  if (!p) return TP_ERR_INVALID;
  p->d = d;
  p->d_ff = d_ff;
  p->T_p = T_p;
  p->act = act;
  p->dtype = dtype;
  p->s = s;
  if (act == TP_ACT_SWIGLU)
    p->s_pad = (s + 127) / 128 * 128;
  else if (act == TP_ACT_NONE)
    p->s_pad = s;
  else
    p->s_pad = (s + 7) / 8 * 8;
  *out = p;
  return TP_OK;
}

int tp_attn_out_plan_create(tp_ffn_plan** out, int64_t d_model, int n_heads, int n_kv_heads, int64_t head_dim,
                            int T_p, int dtype) {
  if (!out) return TP_ERR_INVALID;
  *out = nullptr;
  if (n_heads < 1 || n_kv_heads < 1 || head_dim < 1 || T_p < 1) return TP_ERR_INVALID;
  if (n_heads % T_p != 0 || n_kv_heads % T_p != 0) return TP_ERR_INVALID;
  if (n_heads % n_kv_heads != 0) return TP_ERR_INVALID;
  int rc = tp_ffn_plan_create(out, d_model, static_cast<int64_t>(n_heads) * head_dim, T_p, TP_ACT_NONE, dtype);
  if (rc == TP_OK) {
    (*out)->n_heads = n_heads;
    (*out)->n_kv_heads = n_kv_heads;
    (*out)->head_dim = head_dim;
  }
  return rc;
}

void tp_ffn_plan_destroy(tp_ffn_plan* plan) {
  if (!plan) return;
  release_overlap(plan);
  for (auto& r : plan->events) {
    if (r.start) cudaEventDestroy(r.start);
    if (r.stop) cudaEventDestroy(r.stop);
  }
  delete plan;
}

int tp_ffn_plan_info(const tp_ffn_plan* p, int64_t* d, int64_t* d_ff, int* T_p, int* act, int* dtype, int64_t* s,
                     int64_t* s_pad) {
  if (!p) return TP_ERR_INVALID;
  if (d) *d = p->d;
  if (d_ff) *d_ff = p->d_ff;
  if (T_p) *T_p = p->T_p;
  if (act) *act = p->act;
  if (dtype) *dtype = p->dtype;
  if (s) *s = p->s;
  if (s_pad) *s_pad = p->s_pad;
  return TP_OK;
}

size_t tp_ffn_packed_bytes(const tp_ffn_plan* p, int which) {
  if (!p) return 0;
  const size_t e = esz(p);
  if (which == TP_PACK_COLUMNS)
    return p->act == TP_ACT_NONE ? 0 : static_cast<size_t>(p->T_p) * hidden_width(p) * p->d * e;
  if (which == TP_PACK_ROWS) return static_cast<size_t>(p->T_p) * p->d * p->s_pad * e;
  return 0;
}

size_t tp_ffn_saved_bytes(const tp_ffn_plan* p, int64_t n) {
  if (!p || n < 0) return 0;
  return saved_layout(p, n).total;
}

size_t tp_ffn_workspace_bytes(const tp_ffn_plan* p, int64_t n, int flags) {
  if (!p || n < 0) return 0;
  return ws_layout(p, n, flags).total;
}

int tp_ffn_shard_columns(const tp_ffn_plan* p, const void* W1, const void* W3, void* packed, tp_stream_t stream) {
  if (!p || !W1 || !packed || p->act == TP_ACT_NONE) return TP_ERR_INVALID;
  if (p->act == TP_ACT_SWIGLU && !W3) return TP_ERR_INVALID;
  return launch_pack_columns(W1, W3, packed, p->T_p, p->s, p->s_pad, p->d, p->act == TP_ACT_SWIGLU, esz(p), 0,
                             stream);
}

int tp_ffn_shard_rows(const tp_ffn_plan* p, const void* W2, void* packed, tp_stream_t stream) {
  if (!p || !W2 || !packed) return TP_ERR_INVALID;
  return launch_pack_rows(W2, packed, p->T_p, p->s, p->s_pad, p->d, esz(p), 0, stream);
}

int tp_ffn_unshard_columns(const tp_ffn_plan* p, const void* packed, void* W1, void* W3, tp_stream_t stream) {
  if (!p || !W1 || !packed || p->act == TP_ACT_NONE) return TP_ERR_INVALID;
  if (p->act == TP_ACT_SWIGLU && !W3) return TP_ERR_INVALID;
  return launch_pack_columns(W1, W3, const_cast<void*>(packed), p->T_p, p->s, p->s_pad, p->d,
                             p->act == TP_ACT_SWIGLU, esz(p), 1, stream);
}

int tp_ffn_unshard_rows(const tp_ffn_plan* p, const void* packed, void* W2, tp_stream_t stream) {
  if (!p || !W2 || !packed) return TP_ERR_INVALID;
  return launch_pack_rows(W2, const_cast<void*>(packed), p->T_p, p->s, p->s_pad, p->d, esz(p), 1, stream);
}

static int validate_fwd(const tp_ffn_plan* p, int64_t n, const void* x, const void* w13p, const void* w2p,
                        const void* b1, const void* b2, const void* y, const float* partials, const void* saved,
                        const void* workspace, size_t workspace_bytes, int flags) {
  const bool none = p->act == TP_ACT_NONE;
  const bool fused = (flags & TP_SUM_FUSED) != 0;
  if (!x || !w2p || !y || !workspace) return TP_ERR_INVALID;
  if (!none && !w13p) return TP_ERR_INVALID;
  if (fused && partials) return TP_ERR_INVALID;
  if (fused && (flags & TP_SUM_OVERLAP)) return TP_ERR_INVALID;
  if (b1 && p->act != TP_ACT_GELU_TANH) return TP_ERR_UNSUPPORTED;
  if (n > (int64_t(1) << 30)) return TP_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(p, n, flags);
  if (workspace_bytes < L.total) return TP_ERR_INVALID;
  const void* ptrs[] = {x, w13p, w2p, b1, b2, y, partials, saved, workspace};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return TP_ERR_ALIGN;
  return TP_OK;
}

// Forward on an initialised launch context.  With `sc`, the result rows go to
// the T_p slice buffers of a sequence-parallel caller: the standalone sum
// writes each row-slice straight into its buffer (reduce-scatter), the fused
// GEMM writes `y` (a workspace buffer) and a copy scatters it.
static int fwd_impl(const tp_ffn_plan* p, int64_t n, const void* x, const void* w13p, const void* w2p,
                    const void* b1, const void* b2, void* y, float* partials, void* saved, void* workspace,
                    int flags, LaunchCtx& ctx, const RowSlices* sc) {
  const bool none = p->act == TP_ACT_NONE;
  const bool fused = (flags & TP_SUM_FUSED) != 0;
  const WsLayout L = ws_layout(p, n, flags);
  int rc = TP_OK;
  char* ws = static_cast<char*>(workspace);
  const SavedLayout S = saved_layout(p, n);
  const int64_t T = p->T_p, d = p->d, sp = p->s_pad, W = hidden_width(p);
  const int out_bf16 = p->dtype == TP_BF16;

  // ---- 1. up GEMM (column-sharded W1 / W3) + activation
  const void* hbuf = x;  // NONE: the head outputs are the hidden activations
  if (!none) {
    void* h = saved ? static_cast<char*>(saved) + S.h : ws + L.h;
    GemmSpec g;
    g.name = p->act == TP_ACT_SWIGLU ? "up_swiglu" : "up_gelu";
    g.M = n;
    g.N = W;
    g.K = d;
    g.NB = static_cast<int>(T);
    g.G = 1;
    g.A = kmajor(x, d, n, 1, d, n * d, 0, 0);
    g.B = kmajor(w13p, d, W, T, d, W * d, 1, 0);
    g.epi = p->act == TP_ACT_SWIGLU ? EPI_SWIGLU_FWD : EPI_GELU_FWD;
    g.out = h;
    g.out_bs = n * sp;
    g.out_rs = sp;
    if (saved) {
      g.out2 = static_cast<char*>(saved) + S.act;
      g.out2_bs = n * W;
      g.out2_rs = W;
    }
    g.bias = b1;
    g.bias_bs = p->s;
    g.bias_len = p->s;
    g.n_store = sp;
    g.out_bf16 = out_bf16;
    if (L.has_tail) {
      g.tail_ws = reinterpret_cast<float*>(ws + L.tail);
      g.tail_ws_bytes = L.tail_bytes;
    }
    const int ks = L.has_ks ? choose_ksplit(p, n, ctx.num_sms) : 1;
    if (ks > 1) {
      // fp32 parts of a and g, then the SwiGLU combine
      float* parts = reinterpret_cast<float*>(ws + L.ks);
      g.epi = EPI_F32;
      g.ksplit = ks;
      g.out = parts;
      g.out_bs = n * W;
      g.out_rs = W;
      g.out2 = nullptr;
      g.n_store = W;
      rc = run_gemm(p, g, ctx);
      if (!rc)
        rc = launch_swiglu_combine(parts, ks, static_cast<int>(T), n, sp, h,
                                   saved ? static_cast<char*>(saved) + S.act : nullptr, ctx, "swiglu_combine");
    } else {
      rc = run_gemm(p, g, ctx);
    }
    if (rc) return rc;
    hbuf = h;
  }

  // ---- 2. down GEMM (row-sharded W2) + g-operator shard-sum
  GemmSpec g;
  g.M = n;
  g.N = d;
  g.K = sp;
  if (none)
    g.A = kmajor(hbuf, p->s, n, T, p->d_ff, p->s, 0, 0);  // heads of shard t: columns [t*s, (t+1)*s)
  else
    g.A = kmajor(hbuf, sp, n, T, sp, n * sp, 0, 0);
  g.B = kmajor(w2p, sp, d, T, sp, d * sp, 0, 0);
  g.n_store = d;
  g.out_bf16 = out_bf16;
  if (fused) {
    g.name = "down_fused_sum";
    g.NB = 1;
    g.G = static_cast<int>(T);
    g.A.gsel = 1;
    g.B.gsel = 1;
    g.epi = EPI_OUT;
    g.out = y;
    g.out_bs = 0;
    g.out_rs = d;
    g.bias = b2;
    g.bias_bs = 0;
    g.bias_len = d;
    if (L.has_tail) {
      g.tail_ws = reinterpret_cast<float*>(ws + L.tail);
      g.tail_ws_bytes = L.tail_bytes;
    }
    rc = run_gemm(p, g, ctx);
    if (!rc && sc) rc = launch_scatter_rows(y, n, d, out_bf16 ? 2 : 4, *sc, ctx, "scatter_y");
  } else {
    float* part = partials ? partials : reinterpret_cast<float*>(ws + L.part);
    g.name = "down_partials";
    g.NB = static_cast<int>(T);
    g.G = 1;
    g.A.bsel = 1;
    g.B.bsel = 1;
    g.epi = EPI_F32;
    g.out = part;
    g.out_bs = n * d;
    g.out_rs = d;
    if (flags & TP_SUM_OVERLAP) {
      rc = gemm_sum_overlapped(p, g, ctx, part, n, d, b2, y, out_bf16, "shard_sum_y");
    } else {
      rc = run_gemm(p, g, ctx);
      if (!rc && sc)
        rc = launch_shard_sum_scatter(part, static_cast<int>(T), n, d, b2, *sc, out_bf16, ctx, "reduce_scatter_y");
      else if (!rc)
        rc = launch_shard_sum(part, static_cast<int>(T), n, d, b2, y, out_bf16, ctx, "shard_sum_y");
    }
  }
  return rc;
}

int tp_ffn_fwd(const tp_ffn_plan* p, int64_t n, const void* x, const void* w13p, const void* w2p, const void* b1,
               const void* b2, void* y, float* partials, void* saved, void* workspace, size_t workspace_bytes,
               int flags, tp_stream_t stream) {
  if (!p || n < 0) return TP_ERR_INVALID;
  if (n == 0) {
    p->last_launches = 0;
    return TP_OK;
  }
  int rc = validate_fwd(p, n, x, w13p, w2p, b1, b2, y, partials, saved, workspace, workspace_bytes, flags);
  if (rc) return rc;
  LaunchCtx ctx;
  rc = make_ctx(p, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  if (!rc) rc = fwd_impl(p, n, x, w13p, w2p, b1, b2, y, partials, saved, workspace, flags, ctx, nullptr);
  return finish_call(p, ctx, rc, flags, workspace);
}

static int validate_bwd(const tp_ffn_plan* p, int64_t n, const void* x, const void* w13p, const void* w2p,
                        const void* saved, const void* dy, const void* dx, const float* dx_partials,
                        const void* dw13p, const void* dw2p, const void* db1, const void* db2,
                        const void* workspace, size_t workspace_bytes, int flags) {
  const bool none = p->act == TP_ACT_NONE;
  const bool fused = (flags & TP_SUM_FUSED) != 0;
  if (!x || !w2p || !dy || !dx || !dw2p || !workspace) return TP_ERR_INVALID;
  if (!none && (!w13p || !saved || !dw13p)) return TP_ERR_INVALID;
  if ((fused || none) && dx_partials) return TP_ERR_INVALID;
  if (fused && (flags & TP_SUM_OVERLAP)) return TP_ERR_INVALID;
  if (db1 && p->act != TP_ACT_GELU_TANH) return TP_ERR_UNSUPPORTED;
  if (n > (int64_t(1) << 30)) return TP_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(p, n, flags);
  if (workspace_bytes < L.total) return TP_ERR_INVALID;
  const void* ptrs[] = {x, w13p, w2p, saved, dy, dx, dx_partials, dw13p, dw2p, db1, db2, workspace};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return TP_ERR_ALIGN;
  return TP_OK;
}

// The backward GEMMs of the row-sharded projection without activation (W_O)
// have N = s per shard; with s = 384 (the 8.3B block's three heads) each
// shard's second 256-column tile is half empty.  Run as one GEMM over all
// shards' columns (N = T_p s) where the tensor-core pair kernel takes it:
// dc = dy W_O reads shard n / s's B columns (dgrad, `b_side`), dW_O writes
// shard n / s's packed block (wgrad).  Otherwise, or when the kernel
// declines, the per-shard GEMM g runs.  Measured on GB300: dW_O merged is
// faster for s = 384 and 512 (8.3B 932 -> 1451, Llama-3-8B 1258 -> 1357
// TFLOP/s); dc merged only where it removes half-empty tiles (s = 384: 1196
// -> 1235; s = 512: 1606 -> 1457, so s a multiple of 256 stays per shard).
static int run_merged_or_sharded(const tp_ffn_plan* p, const GemmSpec& g, LaunchCtx& ctx, bool b_side) {
  const int64_t T = p->T_p, s = p->s;
  if (p->dtype == TP_BF16 && T > 1 && s % 128 == 0 && (!b_side || s % 256 != 0) && p->d_ff == T * s &&
      merge_shards_enabled()) {
    GemmSpec m = g;
    m.N = T * s;
    m.NB = 1;
    m.n_store = T * s;
    if (b_side) {  // dgrad: B = the packed W_O shards, output columns already global
      m.B.bsel = 0;
      m.b_cs = s;
      m.out_bs = 0;
    } else {  // wgrad: B = all heads' columns of c, output to the packed shards
      m.B = g.B;
      m.B.inner = T * s;
      m.B.batch = 1;
      m.B.batch_stride = g.B.row_stride * g.B.rows;
      m.B.bsel = 0;
      m.out_cs = s;
    }
    const int rc = run_gemm(p, m, ctx);
    if (rc != TP_ERR_UNSUPPORTED) return rc;
  }
  return run_gemm(p, g, ctx);
}

// A weight-gradient GEMM g (bf16 out, dense [NB][M][N] planes): as it stands,
// or split along K into fp32 parts in the workspace and summed in part order.
static int run_wgrad(const tp_ffn_plan* p, const GemmSpec& g, int64_t n, const WsLayout& L, char* ws,
                     LaunchCtx& ctx, const char* sum_name) {
  const int ks = L.has_wk ? wgrad_ksplit(p, n, g.M, g.N, ctx.num_sms) : 1;
  const int64_t plane = g.NB * g.M * g.N;
  if (ks == 1 || g.out_rs != g.N || g.out_bs != g.M * g.N || g.n_store != g.N ||
      static_cast<size_t>(ks) * plane * 4 > wgrad_parts_bytes(p, n, ctx.num_sms))
    return run_gemm(p, g, ctx);
  float* parts = reinterpret_cast<float*>(ws + L.wk);
  GemmSpec k = g;
  k.epi = EPI_F32;
  k.ksplit = ks;
  k.no_dep_wait = 0;  // small problems: starting in the previous kernel's tail measured slower
  k.out = parts;
  k.out_bs = g.M * g.N;
  k.out_rs = g.N;
  int rc = run_gemm(p, k, ctx);
  if (!rc) rc = launch_shard_sum(parts, ks, g.NB * g.M, g.N, nullptr, g.out, g.out_bf16, ctx, sum_name, plane);
  return rc;
}

// Backward on an initialised launch context; `sc` as in fwd_impl, for dx.
static int bwd_impl(const tp_ffn_plan* p, int64_t n, const void* x, const void* w13p, const void* w2p,
                    const void* saved, const void* dy, void* dx, float* dx_partials, void* dw13p, void* dw2p,
                    void* db1, void* db2, void* workspace, int flags, LaunchCtx& ctx, const RowSlices* sc) {
  const bool none = p->act == TP_ACT_NONE;
  const bool fused = (flags & TP_SUM_FUSED) != 0;
  const WsLayout L = ws_layout(p, n, flags);
  int rc = TP_OK;
  char* ws = static_cast<char*>(workspace);
  const SavedLayout S = saved_layout(p, n);
  const int64_t T = p->T_p, d = p->d, sp = p->s_pad, W = hidden_width(p), s = p->s;
  const int out_bf16 = p->dtype == TP_BF16;
  float* cs_scratch = reinterpret_cast<float*>(ws + L.cs);

  if (none) {
    // dc^(t) = dy W_O^(t): each shard writes its own head columns of dx.
    GemmSpec g;
    g.name = "dgrad_heads";
    g.M = n;
    g.N = s;
    g.K = d;
    g.NB = static_cast<int>(T);
    g.A = kmajor(dy, d, n, 1, d, n * d, 0, 0);
    g.B = mnmajor(w2p, sp, d, T, sp, d * sp, 1, 0);
    g.epi = EPI_OUT;
    g.out = dx;
    g.out_bs = s;
    g.out_rs = p->d_ff;
    g.n_store = s;
    g.out_bf16 = out_bf16;
    rc = run_merged_or_sharded(p, g, ctx, true);
    if (!rc && sc) rc = launch_scatter_rows(dx, n, p->d_ff, out_bf16 ? 2 : 4, *sc, ctx, "scatter_dx");
    if (rc) return rc;
    // dW_O^(t) = dy^T c^(t)
    GemmSpec w;
    w.name = "wgrad_rows";
    w.M = d;
    w.N = s;
    w.K = n;
    w.NB = static_cast<int>(T);
    w.A = mnmajor(dy, d, n, 1, d, n * d, 0, 0);
    w.B = mnmajor(x, s, n, T, p->d_ff, s, 1, 0);
    w.epi = EPI_OUT;
    w.out = dw2p;
    w.out_bs = d * sp;
    w.out_rs = sp;
    w.n_store = s;
    w.out_bf16 = out_bf16;
    w.no_dep_wait = 1;  // reads dy and c, writes dW_O: nothing the dc GEMM before it touches
    rc = run_merged_or_sharded(p, w, ctx, false);
    if (!rc && db2) {
      ColsumJobs J;
      J.j[J.n++] = colsum_job(dy, out_bf16, 1, n, d, d, n * d, db2, out_bf16, 0, cs_scratch, n);
      J.no_dep_wait = 1;  // dy: nothing the dW_O GEMM before it writes
      rc = launch_colsums(J, ctx, "colsum_db2");
    }
    return rc;
  }

  void* D = ws + L.D;
  const void* hsaved = static_cast<const char*>(saved) + S.h;
  const void* asaved = static_cast<const char*>(saved) + S.act;

  // ---- 3. dh^(t) = dy W2^(t), activation derivative fused
  {
    GemmSpec g;
    g.name = p->act == TP_ACT_SWIGLU ? "dgrad_h_swiglu" : "dgrad_h_gelu";
    g.M = n;
    g.N = sp;
    g.K = d;
    g.NB = static_cast<int>(T);
    g.A = kmajor(dy, d, n, 1, d, n * d, 0, 0);
    g.B = mnmajor(w2p, sp, d, T, sp, d * sp, 1, 0);
    g.epi = p->act == TP_ACT_SWIGLU ? EPI_SWIGLU_BWD : EPI_GELU_BWD;
    g.out = D;
    g.out_bs = n * W;
    g.out_rs = W;
    g.aux = asaved;
    g.aux_bs = n * W;
    g.aux_rs = W;
    g.n_store = sp;
    g.out_bf16 = out_bf16;
    rc = run_gemm(p, g, ctx);
    if (rc) return rc;
  }
  // ---- 4. dx = sum_t D^(t) W13^(t)   (f operator)
  {
    GemmSpec g;
    g.M = n;
    g.N = d;
    g.K = W;
    g.A = kmajor(D, W, n, T, W, n * W, 0, 0);
    g.B = mnmajor(w13p, d, W, T, d, W * d, 0, 0);
    g.n_store = d;
    g.out_bf16 = out_bf16;
    if (fused) {
      g.name = "dgrad_x_fused_sum";
      g.NB = 1;
      g.G = static_cast<int>(T);
      g.A.gsel = 1;
      g.B.gsel = 1;
      g.epi = EPI_OUT;
      g.out = dx;
      g.out_bs = 0;
      g.out_rs = d;
      rc = run_gemm(p, g, ctx);
      if (!rc && sc) rc = launch_scatter_rows(dx, n, d, out_bf16 ? 2 : 4, *sc, ctx, "scatter_dx");
    } else {
      float* part = dx_partials ? dx_partials : reinterpret_cast<float*>(ws + L.part);
      g.name = "dgrad_x_partials";
      g.NB = static_cast<int>(T);
      g.A.bsel = 1;
      g.B.bsel = 1;
      g.epi = EPI_F32;
      g.out = part;
      g.out_bs = n * d;
      g.out_rs = d;
      if (flags & TP_SUM_OVERLAP) {
        rc = gemm_sum_overlapped(p, g, ctx, part, n, d, nullptr, dx, out_bf16, "shard_sum_dx");
      } else {
        rc = run_gemm(p, g, ctx);
        if (!rc && sc)
          rc = launch_shard_sum_scatter(part, static_cast<int>(T), n, d, nullptr, *sc, out_bf16, ctx,
                                        "reduce_scatter_dx");
        else if (!rc)
          rc = launch_shard_sum(part, static_cast<int>(T), n, d, nullptr, dx, out_bf16, ctx, "shard_sum_dx");
      }
    }
    if (rc) return rc;
  }
  // ---- 5. weight gradients, per shard
  {
    GemmSpec g;
    g.name = "wgrad_w2";
    g.M = d;
    g.N = sp;
    g.K = n;
    g.NB = static_cast<int>(T);
    // reads dy and the saved h, writes dW2 (or its K parts): nothing the dx
    // GEMM or sum before it touches, so it starts in that kernel's tail
    g.no_dep_wait = 1;
    g.A = mnmajor(dy, d, n, 1, d, n * d, 0, 0);
    g.B = mnmajor(hsaved, sp, n, T, sp, n * sp, 1, 0);
    g.epi = EPI_OUT;
    g.out = dw2p;
    g.out_bs = d * sp;
    g.out_rs = sp;
    g.n_store = sp;
    g.out_bf16 = out_bf16;
    rc = run_wgrad(p, g, n, L, ws, ctx, "wgrad_w2_ksum");
    if (rc) return rc;
  }
  {
    GemmSpec g;
    g.name = p->act == TP_ACT_SWIGLU ? "wgrad_w13" : "wgrad_w1";
    // reads D (written before the dx GEMM) and x, writes dW1|dW3: nothing
    // dW2's GEMM or its part sum writes; starts in their tail
    g.no_dep_wait = 1;
    g.M = W;
    g.N = d;
    g.K = n;
    g.NB = static_cast<int>(T);
    g.A = mnmajor(D, W, n, T, W, n * W, 1, 0);
    g.B = mnmajor(x, d, n, 1, d, n * d, 0, 0);
    g.epi = EPI_OUT;
    g.out = dw13p;
    g.out_bs = W * d;
    g.out_rs = d;
    g.n_store = d;
    g.out_bf16 = out_bf16;
    rc = run_wgrad(p, g, n, L, ws, ctx, p->act == TP_ACT_SWIGLU ? "wgrad_w13_ksum" : "wgrad_w1_ksum");
    if (rc) return rc;
  }
  // ---- 6. bias gradients (both column sums in one pair of launches)
  ColsumJobs J;
  if (db1) J.j[J.n++] = colsum_job(D, out_bf16, T, n, s, W, n * W, db1, out_bf16, s, cs_scratch, n);
  if (db2)
    J.j[J.n++] = colsum_job(dy, out_bf16, 1, n, d, d, n * d, db2, out_bf16, 0,
                            cs_scratch + (db1 ? colsum_scratch_floats(T, n, sp, colsum_chunk(n)) : 0), n);
  J.no_dep_wait = 1;  // D and dy: nothing the weight-gradient kernels before it write
  if (J.n) rc = launch_colsums(J, ctx, db1 && db2 ? "colsum_db" : db1 ? "colsum_db1" : "colsum_db2");
  return rc;
}

int tp_ffn_bwd(const tp_ffn_plan* p, int64_t n, const void* x, const void* w13p, const void* w2p, const void* saved,
               const void* dy, void* dx, float* dx_partials, void* dw13p, void* dw2p, void* db1, void* db2,
               void* workspace, size_t workspace_bytes, int flags, tp_stream_t stream) {
  if (!p || n < 0) return TP_ERR_INVALID;
  if (n == 0) {
    p->last_launches = 0;
    return TP_OK;
  }
  int rc = validate_bwd(p, n, x, w13p, w2p, saved, dy, dx, dx_partials, dw13p, dw2p, db1, db2, workspace,
                        workspace_bytes, flags);
  if (rc) return rc;
  LaunchCtx ctx;
  rc = make_ctx(p, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  if (!rc)
    rc = bwd_impl(p, n, x, w13p, w2p, saved, dy, dx, dx_partials, dw13p, dw2p, db1, db2, workspace, flags, ctx,
                  nullptr);
  return finish_call(p, ctx, rc, flags, workspace);
}

// ------------------------------------------------------ sequence parallel
static size_t sp_extra_region(const tp_ffn_plan* p, int64_t n) {
  const int64_t w = p->d > p->d_ff ? p->d : p->d_ff;
  return align_up(static_cast<size_t>(n) * w * esz(p));
}

size_t tp_ffn_seq_parallel_workspace_bytes(const tp_ffn_plan* p, int64_t n, int flags) {
  if (!p || n < 0) return 0;
  return ws_layout(p, n, flags).total + 3 * sp_extra_region(p, n);
}

static int sp_slices(const tp_ffn_plan* p, int64_t n, const void* const* ptrs, RowSlices* out) {
  if (!ptrs || p->T_p > kMaxSlices || n % p->T_p != 0) return TP_ERR_INVALID;
  out->n = p->T_p;
  out->rows = n / p->T_p;
  for (int t = 0; t < p->T_p; ++t) {
    if (!ptrs[t]) return TP_ERR_INVALID;
    if (!aligned16(ptrs[t])) return TP_ERR_ALIGN;
    out->ptr[t] = const_cast<void*>(ptrs[t]);
  }
  return TP_OK;
}

int tp_ffn_fwd_seq_parallel(const tp_ffn_plan* p, int64_t n, const void* const* x_slices, const void* w13p,
                            const void* w2p, const void* b1, const void* b2, void* const* y_slices, void* saved,
                            void* workspace, size_t workspace_bytes, int flags, tp_stream_t stream) {
  if (!p || n < 0) return TP_ERR_INVALID;
  if (n == 0) {
    p->last_launches = 0;
    return TP_OK;
  }
  if (flags & TP_SUM_OVERLAP) return TP_ERR_INVALID;
  RowSlices xs, ys;
  int rc = sp_slices(p, n, x_slices, &xs);
  if (!rc) rc = sp_slices(p, n, y_slices, &ys);
  if (rc) return rc;
  if (!workspace || workspace_bytes < tp_ffn_seq_parallel_workspace_bytes(p, n, flags)) return TP_ERR_INVALID;
  const size_t base = ws_layout(p, n, flags).total, extra = sp_extra_region(p, n);
  char* x_full = static_cast<char*>(workspace) + base;
  char* y_full = x_full + extra;
  rc = validate_fwd(p, n, x_full, w13p, w2p, b1, b2, y_full, nullptr, saved, workspace, base, flags);
  if (rc) return rc;
  LaunchCtx ctx;
  rc = make_ctx(p, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  const int64_t d_in = p->act == TP_ACT_NONE ? p->d_ff : p->d;
  if (!rc) rc = launch_gather_rows(xs, x_full, d_in, esz(p), ctx, "all_gather_x");
  if (!rc) rc = fwd_impl(p, n, x_full, w13p, w2p, b1, b2, y_full, nullptr, saved, workspace, flags, ctx, &ys);
  return finish_call(p, ctx, rc, flags, workspace);
}

int tp_ffn_bwd_seq_parallel(const tp_ffn_plan* p, int64_t n, const void* const* x_slices, const void* w13p,
                            const void* w2p, const void* saved, const void* const* dy_slices, void* const* dx_slices,
                            void* dw13p, void* dw2p, void* db1, void* db2, void* workspace, size_t workspace_bytes,
                            int flags, tp_stream_t stream) {
  if (!p || n < 0) return TP_ERR_INVALID;
  if (n == 0) {
    p->last_launches = 0;
    return TP_OK;
  }
  if (flags & TP_SUM_OVERLAP) return TP_ERR_INVALID;
  RowSlices xs, dys, dxs;
  int rc = sp_slices(p, n, x_slices, &xs);
  if (!rc) rc = sp_slices(p, n, dy_slices, &dys);
  if (!rc) rc = sp_slices(p, n, dx_slices, &dxs);
  if (rc) return rc;
  if (!workspace || workspace_bytes < tp_ffn_seq_parallel_workspace_bytes(p, n, flags)) return TP_ERR_INVALID;
  const size_t base = ws_layout(p, n, flags).total, extra = sp_extra_region(p, n);
  char* x_full = static_cast<char*>(workspace) + base;
  char* dy_full = x_full + extra;
  char* dx_full = dy_full + extra;
  rc = validate_bwd(p, n, x_full, w13p, w2p, saved, dy_full, dx_full, nullptr, dw13p, dw2p, db1, db2, workspace,
                    base, flags);
  if (rc) return rc;
  LaunchCtx ctx;
  rc = make_ctx(p, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  const int64_t d_in = p->act == TP_ACT_NONE ? p->d_ff : p->d;
  if (!rc) rc = launch_gather_rows(xs, x_full, d_in, esz(p), ctx, "all_gather_x");
  if (!rc) rc = launch_gather_rows(dys, dy_full, p->d, esz(p), ctx, "all_gather_dy");
  if (!rc)
    rc = bwd_impl(p, n, x_full, w13p, w2p, saved, dy_full, dx_full, nullptr, dw13p, dw2p, db1, db2, workspace, flags,
                  ctx, &dxs);
  return finish_call(p, ctx, rc, flags, workspace);
}

int tp_ffn_last_device_error(const tp_ffn_plan* p, const void* workspace, tp_stream_t stream) {
  if (!p || !workspace) return TP_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return TP_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TP_ERR_CUDA;
  if (word & DEV_ERR_TIMEOUT) return TP_ERR_TIMEOUT;
  return word ? TP_ERR_CUDA : TP_OK;
}

int tp_ffn_kernel_times(const tp_ffn_plan* p, int max, const char** names, float* ms) {
  if (!p) return -1;
  for (int i = 0; i < p->n_events && i < max; ++i) {
    const TimingRec& r = p->events[i];
    cudaEventSynchronize(r.stop);
    float t = 0.f;
    cudaEventElapsedTime(&t, r.start, r.stop);
    if (names) names[i] = r.name;
    if (ms) ms[i] = t;
  }
  const int n = p->n_events;
  p->n_events = 0;  // read and clear: the next timed call starts a new list
  return n;
}

int tp_ffn_last_launch_count(const tp_ffn_plan* p) { return p ? p->last_launches : -1; }

// ------------------------------------------------------ attention sublayer
// "7.9 Tensor and pipeline parallelism (TP, PP)", §2.2 "Attention, sharded".
// Forward: qkv = x wqkv^T (one GEMM over all shards' column slices), the
// attention core, then the row-sharded output projection of the inner
// act-NONE plan with its ordered shard-sum.  Backward: that projection's
// backward (dc per shard, dW_O), the attention-core backward (dqkv), dx =
// sum_t dqkv^(t) wqkv^(t) in shard order (fused K loop or partials + sum), and
// dwqkv = dqkv^T x (one GEMM: the packed weight is shard-major).
struct tp_attn_plan {
  tp_ffn_plan* wo = nullptr;  // output projection (act NONE, d_ff = H * hd)
  int64_t d = 0, hd = 0;
  int H = 0, Hkv = 0, T_p = 1, causal = 1;
  int64_t sq = 0, sk = 0, slice = 0, W = 0;
};

namespace {
int64_t seq_pad(int64_t S) { return (S + 127) / 128 * 128; }

struct AttnSaved {
  size_t qkv = 0, c = 0, lse = 0, total = 0;
};
AttnSaved attn_saved(const tp_attn_plan* a, int64_t B, int64_t S) {
  AttnSaved L;
  const size_t n = static_cast<size_t>(B) * S;
  L.qkv = 0;
  L.c = align_up(n * a->W * 2);
  L.lse = L.c + align_up(n * a->H * a->hd * 2);
  L.total = L.lse + align_up(static_cast<size_t>(B) * a->H * seq_pad(S) * 4);
  return L;
}

struct AttnWs {
  size_t wo = 0, wo_bytes = 0, dc = 0, dqkv = 0, Dv = 0, total = 0;
};
AttnWs attn_ws(const tp_attn_plan* a, int64_t B, int64_t S, int flags) {
  AttnWs L;
  const size_t n = static_cast<size_t>(B) * S;
  size_t off = kAlign;  // error word
  L.wo = off;
  L.wo_bytes = ws_layout(a->wo, static_cast<int64_t>(n), flags).total;
  off += align_up(L.wo_bytes);
  L.dc = off;
  off += align_up(n * a->H * a->hd * 2);
  L.dqkv = off;
  off += align_up(n * a->W * 2);
  L.Dv = off;
  off += align_up(static_cast<size_t>(B) * a->H * seq_pad(S) * 4);
  L.total = off;
  return L;
}

AttnSpec attn_spec(const tp_attn_plan* a, int64_t B, int64_t S) {
  AttnSpec sp;
  sp.B = static_cast<int>(B);
  sp.S = static_cast<int>(S);
  sp.H = a->H;
  sp.Hkv = a->Hkv;
  sp.T_p = a->T_p;
  sp.causal = a->causal;
  sp.hd = a->hd;
  sp.qkv_rs = a->W;
  sp.o_rs = a->H * a->hd;
  sp.do_rs = a->H * a->hd;
  sp.s_pad = seq_pad(S);
  return sp;
}

int attn_check(const tp_attn_plan* a, int64_t B, int64_t S, size_t ws_bytes, const void* workspace, int flags,
               std::initializer_list<const void*> ptrs) {
  if (!a || B < 0 || S < 0 || !workspace) return TP_ERR_INVALID;
  if (B > (int64_t(1) << 24) || S > (int64_t(1) << 24) || B * S > (int64_t(1) << 30)) return TP_ERR_UNSUPPORTED;
  if ((flags & TP_SUM_FUSED) && (flags & TP_SUM_OVERLAP)) return TP_ERR_INVALID;
  if (ws_bytes < attn_ws(a, B, S, flags).total) return TP_ERR_INVALID;
  for (const void* q : ptrs) {
    if (!q) return TP_ERR_INVALID;
    if (!aligned16(q)) return TP_ERR_ALIGN;
  }
  if (!aligned16(workspace)) return TP_ERR_ALIGN;
  return TP_OK;
}
}  // namespace

int tp_attn_plan_create(tp_attn_plan** out, int64_t d_model, int n_heads, int n_kv_heads, int64_t head_dim, int T_p,
                        int causal, int dtype) {
  if (!out) return TP_ERR_INVALID;
  *out = nullptr;
  if (d_model < 1 || n_heads < 1 || n_kv_heads < 1 || head_dim < 1 || T_p < 1) return TP_ERR_INVALID;
  if (n_heads % T_p || n_kv_heads % T_p || n_heads % n_kv_heads) return TP_ERR_INVALID;
  if (dtype != TP_BF16 && dtype != TP_F32) return TP_ERR_INVALID;
  if (dtype != TP_BF16 || head_dim != 128 || d_model % 8) return TP_ERR_UNSUPPORTED;
  tp_attn_plan* a = new (std::nothrow) tp_attn_plan();
  if (!a) return TP_ERR_INVALID;
  int rc = tp_attn_out_plan_create(&a->wo, d_model, n_heads, n_kv_heads, head_dim, T_p, dtype);
  if (rc) {
    delete a;
    return rc;
  }
  a->d = d_model;
  a->hd = head_dim;
  a->H = n_heads;
  a->Hkv = n_kv_heads;
  a->T_p = T_p;
  a->causal = causal ? 1 : 0;
  a->sq = static_cast<int64_t>(n_heads / T_p) * head_dim;
  a->sk = static_cast<int64_t>(n_kv_heads / T_p) * head_dim;
  a->slice = a->sq + 2 * a->sk;
  a->W = a->slice * T_p;
  *out = a;
  return TP_OK;
}

void tp_attn_plan_destroy(tp_attn_plan* a) {
  if (!a) return;
  tp_ffn_plan_destroy(a->wo);
  delete a;
}

int tp_attn_plan_info(const tp_attn_plan* a, int64_t* qkv_width, int64_t* slice, int64_t* sq, int64_t* sk) {
  if (!a) return TP_ERR_INVALID;
  if (qkv_width) *qkv_width = a->W;
  if (slice) *slice = a->slice;
  if (sq) *sq = a->sq;
  if (sk) *sk = a->sk;
  return TP_OK;
}

size_t tp_attn_packed_bytes(const tp_attn_plan* a, int which) {
  if (!a) return 0;
  if (which == TP_PACK_COLUMNS) return static_cast<size_t>(a->W) * a->d * 2;
  if (which == TP_PACK_ROWS) return tp_ffn_packed_bytes(a->wo, TP_PACK_ROWS);
  return 0;
}

int tp_attn_shard_weights(const tp_attn_plan* a, const void* Wq, const void* Wk, const void* Wv, const void* Wo,
                          void* wqkv, void* wo_packed, tp_stream_t stream) {
  if (!a || !Wo || !wo_packed) return TP_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc = launch_pack_qkv(Wq, Wk, Wv, wqkv, a->T_p, a->sq, a->sk, a->d, 0, st);
  return rc ? rc : tp_ffn_shard_rows(a->wo, Wo, wo_packed, stream);
}

int tp_attn_unshard_weights(const tp_attn_plan* a, const void* wqkv, const void* wo_packed, void* Wq, void* Wk,
                            void* Wv, void* Wo, tp_stream_t stream) {
  if (!a || !Wo || !wo_packed) return TP_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc = launch_pack_qkv(Wq, Wk, Wv, const_cast<void*>(wqkv), a->T_p, a->sq, a->sk, a->d, 1, st);
  return rc ? rc : tp_ffn_unshard_rows(a->wo, wo_packed, Wo, stream);
}

size_t tp_attn_saved_bytes(const tp_attn_plan* a, int64_t B, int64_t S) {
  if (!a || B < 0 || S < 0) return 0;
  return attn_saved(a, B, S).total;
}

int tp_attn_saved_offsets(const tp_attn_plan* a, int64_t B, int64_t S, size_t* qkv_off, size_t* c_off,
                          size_t* lse_off) {
  if (!a || B < 0 || S < 0) return TP_ERR_INVALID;
  const AttnSaved L = attn_saved(a, B, S);
  if (qkv_off) *qkv_off = L.qkv;
  if (c_off) *c_off = L.c;
  if (lse_off) *lse_off = L.lse;
  return TP_OK;
}

size_t tp_attn_workspace_bytes(const tp_attn_plan* a, int64_t B, int64_t S, int flags) {
  if (!a || B < 0 || S < 0) return 0;
  return attn_ws(a, B, S, flags).total;
}

int tp_attn_fwd(const tp_attn_plan* a, int64_t B, int64_t S, const void* x, const void* wqkv, const void* wo_packed,
                void* y, void* saved, void* workspace, size_t workspace_bytes, int flags, tp_stream_t stream) {
  int rc = attn_check(a, B, S, workspace_bytes, workspace, flags, {x, wqkv, wo_packed, y, saved});
  if (rc) return rc;
  const int64_t n = B * S;
  if (n == 0) {
    a->wo->last_launches = 0;
    return TP_OK;
  }
  LaunchCtx ctx;
  rc = make_ctx(a->wo, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  if (rc) return rc;
  const AttnSaved SV = attn_saved(a, B, S);
  const AttnWs L = attn_ws(a, B, S, flags);
  char* sv = static_cast<char*>(saved);
  char* ws = static_cast<char*>(workspace);
  // q, k, v of every shard: one GEMM over the shard-major packed weight
  GemmSpec g;
  g.name = "qkv_proj";
  g.M = n;
  g.N = a->W;
  g.K = a->d;
  g.A = kmajor(x, a->d, n, 1, a->d, n * a->d, 0, 0);
  g.B = kmajor(wqkv, a->d, a->W, 1, a->d, a->W * a->d, 0, 0);
  g.epi = EPI_OUT;
  g.out = sv + SV.qkv;
  g.out_rs = a->W;
  g.n_store = a->W;
  g.out_bf16 = 1;
  {
    // the W_O forward's last-wave region is free until that GEMM runs
    const WsLayout WL = ws_layout(a->wo, n, flags);
    if (WL.has_tail) {
      g.tail_ws = reinterpret_cast<float*>(ws + L.wo + WL.tail);
      g.tail_ws_bytes = WL.tail_bytes;
    }
  }
  rc = run_gemm(a->wo, g, ctx);
  if (!rc) {
    AttnSpec sp = attn_spec(a, B, S);
    sp.qkv = sv + SV.qkv;
    sp.o = sv + SV.c;
    sp.lse = reinterpret_cast<float*>(sv + SV.lse);
    rc = launch_attn_fwd(sp, ctx);
  }
  if (!rc)
    rc = fwd_impl(a->wo, n, sv + SV.c, nullptr, wo_packed, nullptr, nullptr, y, nullptr, nullptr, ws + L.wo, flags,
                  ctx, nullptr);
  return finish_call(a->wo, ctx, rc, flags, workspace);
}

int tp_attn_bwd(const tp_attn_plan* a, int64_t B, int64_t S, const void* x, const void* wqkv, const void* wo_packed,
                const void* saved, const void* dy, void* dx, void* dwqkv, void* dwo_packed, void* workspace,
                size_t workspace_bytes, int flags, tp_stream_t stream) {
  int rc = attn_check(a, B, S, workspace_bytes, workspace, flags,
                      {x, wqkv, wo_packed, saved, dy, dx, dwqkv, dwo_packed});
  if (rc) return rc;
  const int64_t n = B * S;
  if (n == 0) {
    a->wo->last_launches = 0;
    return TP_OK;
  }
  LaunchCtx ctx;
  rc = make_ctx(a->wo, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  if (rc) return rc;
  const AttnSaved SV = attn_saved(a, B, S);
  const AttnWs L = attn_ws(a, B, S, flags);
  const char* sv = static_cast<const char*>(saved);
  char* ws = static_cast<char*>(workspace);
  const bool fused = (flags & TP_SUM_FUSED) != 0;
  const int64_t T = a->T_p, d = a->d, W = a->W, sl = a->slice;
  // 1. output projection backward: dc per shard (no sum), dW_O
  rc = bwd_impl(a->wo, n, sv + SV.c, nullptr, wo_packed, nullptr, dy, ws + L.dc, nullptr, nullptr, dwo_packed,
                nullptr, nullptr, ws + L.wo, flags, ctx, nullptr);
  // 2. attention core backward -> dqkv
  if (!rc) {
    AttnSpec sp = attn_spec(a, B, S);
    sp.qkv = sv + SV.qkv;
    sp.o = const_cast<char*>(sv + SV.c);
    sp.lse = reinterpret_cast<float*>(const_cast<char*>(sv + SV.lse));
    sp.dO = ws + L.dc;
    sp.Dv = reinterpret_cast<float*>(ws + L.Dv);
    sp.dqkv = ws + L.dqkv;
    rc = launch_attn_bwd(sp, ctx);
  }
  // 3. dx = sum_t dqkv^(t) wqkv^(t)   (f operator, shard order)
  if (!rc) {
    const void* dq = ws + L.dqkv;
    GemmSpec g;
    g.M = n;
    g.N = d;
    g.K = sl;
    g.A = kmajor(dq, sl, n, T, W, sl, 0, 0);
    g.B = mnmajor(wqkv, d, sl, T, d, sl * d, 0, 0);
    g.n_store = d;
    g.out_bf16 = 1;
    if (fused) {
      g.name = "attn_dgrad_x_fused_sum";
      g.NB = 1;
      g.G = static_cast<int>(T);
      g.A.gsel = 1;
      g.B.gsel = 1;
      g.epi = EPI_OUT;
      g.out = dx;
      g.out_rs = d;
      rc = run_gemm(a->wo, g, ctx);
    } else {
      // the output projection's partial buffer is free again: reuse it
      float* part = reinterpret_cast<float*>(ws + L.wo + ws_layout(a->wo, n, flags).part);
      g.name = "attn_dgrad_x_partials";
      g.NB = static_cast<int>(T);
      g.A.bsel = 1;
      g.B.bsel = 1;
      g.epi = EPI_F32;
      g.out = part;
      g.out_bs = n * d;
      g.out_rs = d;
      if (flags & TP_SUM_OVERLAP) {
        rc = gemm_sum_overlapped(a->wo, g, ctx, part, n, d, nullptr, dx, 1, "attn_shard_sum_dx");
      } else {
        rc = run_gemm(a->wo, g, ctx);
        if (!rc) rc = launch_shard_sum(part, static_cast<int>(T), n, d, nullptr, dx, 1, ctx, "attn_shard_sum_dx");
      }
    }
  }
  // 4. dwqkv = dqkv^T x, every shard's slice in one GEMM
  if (!rc) {
    GemmSpec g;
    g.name = "attn_wgrad_qkv";
    g.M = W;
    g.N = d;
    g.K = n;
    // reads dqkv (written before the dx GEMM) and x, writes dWqkv: nothing
    // the dx GEMM or sum before it writes; starts in its tail
    g.no_dep_wait = 1;
    g.A = mnmajor(ws + L.dqkv, W, n, 1, W, n * W, 0, 0);
    g.B = mnmajor(x, d, n, 1, d, n * d, 0, 0);
    g.epi = EPI_OUT;
    g.out = dwqkv;
    g.out_rs = d;
    g.n_store = d;
    g.out_bf16 = 1;
    rc = run_gemm(a->wo, g, ctx);
  }
  return finish_call(a->wo, ctx, rc, flags, workspace);
}

int tp_attn_core_fwd(const tp_attn_plan* a, int64_t B, int64_t S, const void* qkv, void* o, float* lse,
                     void* workspace, size_t workspace_bytes, int flags, tp_stream_t stream) {
  int rc = attn_check(a, B, S, workspace_bytes, workspace, flags, {qkv, o, lse});
  if (rc) return rc;
  if (B * S == 0) {
    a->wo->last_launches = 0;
    return TP_OK;
  }
  LaunchCtx ctx;
  rc = make_ctx(a->wo, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  if (rc) return rc;
  AttnSpec sp = attn_spec(a, B, S);
  sp.qkv = qkv;
  sp.o = o;
  sp.lse = lse;
  rc = launch_attn_fwd(sp, ctx);
  return finish_call(a->wo, ctx, rc, flags, workspace);
}

int tp_attn_core_bwd(const tp_attn_plan* a, int64_t B, int64_t S, const void* qkv, const void* o, const float* lse,
                     const void* dO, void* dqkv, void* workspace, size_t workspace_bytes, int flags,
                     tp_stream_t stream) {
  int rc = attn_check(a, B, S, workspace_bytes, workspace, flags, {qkv, o, lse, dO, dqkv});
  if (rc) return rc;
  if (B * S == 0) {
    a->wo->last_launches = 0;
    return TP_OK;
  }
  LaunchCtx ctx;
  rc = make_ctx(a->wo, workspace, flags, reinterpret_cast<cudaStream_t>(stream), ctx);
  if (rc) return rc;
  const AttnWs L = attn_ws(a, B, S, flags);
  AttnSpec sp = attn_spec(a, B, S);
  sp.qkv = qkv;
  sp.o = const_cast<void*>(o);
  sp.lse = const_cast<float*>(lse);
  sp.dO = dO;
  sp.Dv = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.Dv);
  sp.dqkv = dqkv;
  rc = launch_attn_bwd(sp, ctx);
  return finish_call(a->wo, ctx, rc, flags, workspace);
}

int tp_attn_kernel_times(const tp_attn_plan* a, int max, const char** names, float* ms) {
  return a ? tp_ffn_kernel_times(a->wo, max, names, ms) : -1;
}

int tp_attn_last_launch_count(const tp_attn_plan* a) { return a ? a->wo->last_launches : -1; }

}  // extern "C"
