// api.cu - the extern "C" entry points of libmoe: argument validation, workspace carving, tensor-map
// encoding and the launch sequence of each call.  See include/moe.h for the contract of every function.
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace moe {

static thread_local int g_last_cuda_error = 0;
static std::atomic<uint64_t> g_launches{0};

int record_cuda_error(cudaError_t err) {
  g_last_cuda_error = static_cast<int>(err);
  return MOE_ERR_CUDA;
}

int record_cu_error(CUresult res) {
  g_last_cuda_error = static_cast<int>(res);
  return MOE_ERR_CUDA;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
struct ProfRec {
  const char *name;
  cudaEvent_t start, stop;
};
struct ProfState {
  std::mutex mu;
  bool enabled = false;
  std::vector<ProfRec> recs;       // recorded this session, in launch order
  std::vector<cudaEvent_t> pool;   // events reused across sessions
  size_t pool_used = 0;
  struct Agg {
    std::string name;
    int launches;
    double total_ms;
  };
  std::vector<Agg> summary;
};
ProfState &prof() {
  static ProfState p;
  return p;
}
cudaEvent_t prof_event(ProfState &p) {
  if (p.pool_used == p.pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    p.pool.push_back(e);
  }
  return p.pool[p.pool_used++];
}
}  // namespace

void prof_begin(const char *name, cudaStream_t s) {
  ProfState &p = prof();
  if (!p.enabled) return;
  std::lock_guard<std::mutex> lk(p.mu);
  ProfRec r{name, prof_event(p), prof_event(p)};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, s);
  p.recs.push_back(r);
}

void prof_end(cudaStream_t s) {
  ProfState &p = prof();
  if (!p.enabled) return;
  std::lock_guard<std::mutex> lk(p.mu);
  if (!p.recs.empty()) cudaEventRecord(p.recs.back().stop, s);
}

// While per-kernel timing is on, side-stream work stays on the caller's stream, so that each kernel's events
// bracket that kernel alone rather than the time it spends beside another one.
static bool prof_serial() { return prof().enabled; }

int num_sms() {
  static DeviceCache cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  return cache.get(dev, [&]() {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  });
}

// MOE_OK on a compute capability 10.3 device, else MOE_ERR_DEVICE (or MOE_ERR_CUDA when no device is current).
int check_device() {
  static DeviceCache cache;  // 1 = supported, 2 = not supported
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return record_cuda_error(err);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
  const int v = cache.get(dev, [&]() {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return (major == 10 && minor == 3) ? 1 : 2;
  });
  return v == 1 ? MOE_OK : MOE_ERR_DEVICE;
}

// Memory-bound steps that do not feed the next GEMM (zeroing an fp32 accumulator, the final cast of dX)
// run on a library-owned side stream of the current device, so that they overlap the operand-feed-bound
// GEMMs.  A Fork makes the side stream wait for the caller's stream; join() makes the caller's stream
// wait for the side stream, and the destructor joins whatever is still open, so every call returns with
// all of its work ordered before whatever the caller enqueues next on its own stream.  The per-device
// mutex is held for the whole call: the two events are reused, and cudaStreamWaitEvent takes the latest
// record at the time it is enqueued.
namespace {
struct SideStream {
  std::mutex mu;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];

class Fork {
 public:
  Fork() = default;
  Fork(const Fork &) = delete;
  Fork &operator=(const Fork &) = delete;
  ~Fork() {
    if (open_) join();
  }
  // side waits for the work enqueued on s so far
  int open(cudaStream_t s) {
    if (prof_serial()) {
      serial_ = true;
      s_ = s;
      return MOE_OK;
    }
    if (!sd_) {
      int dev = 0;
      cudaError_t err = cudaGetDevice(&dev);
      if (err != cudaSuccess) return record_cuda_error(err);
      if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
      sd_ = &g_side[dev];
      lk_ = std::unique_lock<std::mutex>(sd_->mu);
      if (!sd_->stream) {
        err = cudaStreamCreateWithFlags(&sd_->stream, cudaStreamNonBlocking);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&sd_->fork, cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&sd_->join, cudaEventDisableTiming);
        if (err != cudaSuccess) {
          sd_->stream = nullptr;  // retried on the next call; a partial creation leaks at most two handles
          sd_ = nullptr;
          lk_.unlock();
          return record_cuda_error(err);
        }
      }
    }
    s_ = s;
    cudaError_t err = cudaEventRecord(sd_->fork, s);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(sd_->stream, sd_->fork, 0);
    if (err != cudaSuccess) return record_cuda_error(err);
    open_ = true;
    return MOE_OK;
  }
  // s waits for the work enqueued on the side stream so far
  int join() {
    open_ = false;
    if (serial_ || !sd_) return MOE_OK;
    cudaError_t err = cudaEventRecord(sd_->join, sd_->stream);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(s_, sd_->join, 0);
    return err == cudaSuccess ? MOE_OK : record_cuda_error(err);
  }
  cudaStream_t side() const { return serial_ ? s_ : sd_->stream; }

 private:
  bool serial_ = false;  // per-kernel timing: the "side" stream is the caller's
  SideStream *sd_ = nullptr;
  std::unique_lock<std::mutex> lk_;
  cudaStream_t s_ = nullptr;
  bool open_ = false;
};
}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn lookup_encode_fn() {
  void *p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<EncodeTiledFn>(p);
  return nullptr;
}

static EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = lookup_encode_fn();  // initialised once, thread-safe
  return fn;
}

int make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return record_cuda_error(cudaErrorNotSupported);
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : record_cu_error(r);
}

int make_tmap_bf16_epi(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return record_cuda_error(cudaErrorNotSupported);
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : record_cu_error(r);
}

static int encode_bf16(CUtensorMap *tm, const void *base, cuuint32_t rank, const cuuint64_t *dims,
                       const cuuint64_t *strides, const cuuint32_t *box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return record_cuda_error(cudaErrorNotSupported);
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : record_cu_error(r);
}

int make_tmap_bf16_chunks(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                          uint32_t chunks) {
  if (inner % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  const cuuint64_t dims[3] = {64, rows, inner / 64};
  const cuuint64_t strides[2] = {inner * 2, 128};  // row pitch; the next 64-column chunk is 128 bytes on
  const cuuint32_t box[3] = {64, box_rows, chunks};
  return encode_bf16(tm, base, 3, dims, strides, box);
}

int make_tmap_bf16_halves(CUtensorMap *tm, const void *base, uint64_t n, uint64_t rows) {
  if (n % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  const cuuint64_t dims[4] = {64, rows, n / 64, 2};
  const cuuint64_t strides[3] = {4 * n, 128, 2 * n};  // row pitch (2n bf16), next chunk, the up half n columns on
  const cuuint32_t box[4] = {64, 64, 2, 2};
  return encode_bf16(tm, base, 4, dims, strides, box);
}

static void fill_unused(TensorMaps &tm) { tm.h = tm.dh = tm.sa = tm.b; }

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static int check_route_shape(int T, int E, int K, int mode) {
  if (T <= 0 || E <= 0 || K <= 0 || K > E) return MOE_ERR_INVALID_ARG;
  if (mode < MOE_ROUTE_TC || mode > MOE_ROUTE_EC) return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts || K > kMaxTopK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (route_selects(mode) && T > kMaxTrTokens) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)T * K > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

static int check_layer_shape(int T, int d, int n, int E, int K, size_t p_cap) {
  if (T <= 0 || d <= 0 || n <= 0 || E <= 0 || K <= 0 || K > E) return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts || K > kMaxTopK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d % 256 != 0 || n % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (p_cap < (size_t)T * K || p_cap >= ((size_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if ((uint64_t)E * d * 2 * n >= ((uint64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

static bool routing_ok(const moe_routing *r) {
  return r && r->topk_idx && r->topk_score && r->tc_counts && r->counts && r->offsets && r->tile_offsets &&
         r->row_token && r->row_slot && r->row_score && r->status;
}

static bool det_flag(unsigned flags) { return (flags & MOE_FLAG_DETERMINISTIC) != 0u; }
static bool a_from_h_flag(unsigned flags) { return (flags & MOE_FLAG_A_FROM_H) != 0u; }
constexpr unsigned kForwardFlags = MOE_FLAG_DETERMINISTIC | MOE_FLAG_A_FROM_H;

// Column tile of the dH GEMM (n = 256 * k uses 256-wide tiles, else 128).
static int dh_bn(int n) { return (n % 256 == 0) ? 256 : 128; }

// A [P_cap, n] bf16 (not with MOE_FLAG_A_FROM_H), then the accumulator of O: fp32, or 64-bit fixed point when
// deterministic.
static size_t fwd_ws_bytes(int T, int d, int n, size_t p_cap, unsigned flags) {
  return (a_from_h_flag(flags) ? 0 : align256(p_cap * n * 2)) + align256((size_t)T * d * (det_flag(flags) ? 8 : 4));
}

// dH [P_cap, 2n], s*A [P_cap, n], the accumulator of dX (fp32 or fixed point); deterministic mode adds the
// per-column-tile dS partials [P_cap, n / BN].
static size_t bwd_ws_bytes(int T, int d, int n, size_t p_cap, unsigned flags) {
  const bool det = det_flag(flags);
  return align256(p_cap * 2 * n * 2) + align256(p_cap * n * 2) + align256((size_t)T * d * (det ? 8 : 4)) +
         (det ? align256(p_cap * (n / dh_bn(n)) * 4) : 0);
}

// Column tiles (of 256) per pass of a scatter-add GEMM: the largest divisor of d/256 whose fp32 slab
// T x (256 * group) stays within 80 MiB (about two thirds of L2), so A is re-read d / (256 * group) times.
static int scatter_nt_group(int T, int d) {
  const int n_tiles = d / 256;
  int best = 1;
  for (int g = 1; g <= n_tiles; ++g)
    if (n_tiles % g == 0 && (size_t)T * 256 * g * 4 <= ((size_t)80 << 20)) best = g;
  return best;
}

static GemmArgs base_args(const moe_routing *r, int T, int d, int n, int E, size_t p_cap) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.offsets = r->offsets;
  a.tile_offsets = r->tile_offsets;
  a.row_token = r->row_token;
  a.row_score = r->row_score;
  a.status = r->status;
  a.T = T;
  a.d = d;
  a.n = n;
  a.E = E;
  a.p_cap = static_cast<int>(p_cap);
  a.nt_group = scatter_nt_group(T, d);
  a.wide_m = 0;
  return a;
}

int route_call(const float *logits, const float *uniforms, int T, int E, int K, int mode, const moe_routing *r,
               void *ws, size_t ws_bytes, int32_t *P_host, void *stream, bool em_keys) {
  int rc = check_route_shape(T, E, K, mode);
  if (rc != MOE_OK) return rc;
  if (!logits || !routing_ok(r)) return MOE_ERR_INVALID_ARG;
  if (mode == MOE_ROUTE_TR_STOCHASTIC && !uniforms) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < route_workspace_bytes(T, E, K, mode, em_keys)) return MOE_ERR_WORKSPACE;
  rc = check_device();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_route(logits, uniforms, T, E, K, mode, r, ws, s, em_keys);
  if (rc != MOE_OK) return rc;
  if (P_host) {
    cudaError_t err = cudaMemcpyAsync(P_host, r->status + 1, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess) return record_cuda_error(err);
  }
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_route_capacity(int T, int E, int K, int mode, size_t *p_cap) {
  if (!p_cap) return MOE_ERR_INVALID_ARG;
  const int rc = check_route_shape(T, E, K, mode);
  if (rc != MOE_OK) return rc;
  // padding adds fewer than M_tile/2 rows per expert under the nearest rule, fewer than M_tile under up and
  // stochastic rounding; token choice, rounding down and expert choice (E * floor(T*K/E) rows) stay within T*K
  size_t pad = 0;
  if (mode == MOE_ROUTE_TR) pad = (size_t)E * (MOE_M_TILE / 2);
  if (mode == MOE_ROUTE_TR_UP || mode == MOE_ROUTE_TR_STOCHASTIC) pad = (size_t)E * (MOE_M_TILE - 1);
  *p_cap = (size_t)T * K + pad;
  return MOE_OK;
}

int moe_route_workspace_size(int T, int E, int K, int mode, size_t *bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const int rc = check_route_shape(T, E, K, mode);
  if (rc != MOE_OK) return rc;
  *bytes = route_workspace_bytes(T, E, K, mode);
  return MOE_OK;
}

int moe_route(const float *logits, int T, int E, int K, int mode, const moe_routing *r, void *ws, size_t ws_bytes,
              int32_t *P_host, void *stream) {
  return moe::route_call(logits, nullptr, T, E, K, mode, r, ws, ws_bytes, P_host, stream, true);
}

int moe_route_ex(const float *logits, const float *uniforms, int T, int E, int K, int mode, const moe_routing *r,
                 void *ws, size_t ws_bytes, int32_t *P_host, void *stream) {
  return moe::route_call(logits, uniforms, T, E, K, mode, r, ws, ws_bytes, P_host, stream, true);
}


int moe_forward_workspace_size_ex(int T, int d, int n, int E, int K, size_t p_cap, unsigned flags, size_t *bytes) {
  if (!bytes || (flags & ~kForwardFlags)) return MOE_ERR_INVALID_ARG;
  const int rc = check_layer_shape(T, d, n, E, K, p_cap);
  if (rc != MOE_OK) return rc;
  *bytes = fwd_ws_bytes(T, d, n, p_cap, flags);
  return MOE_OK;
}

int moe_forward_workspace_size(int T, int d, int n, int E, int K, size_t p_cap, size_t *bytes) {
  return moe_forward_workspace_size_ex(T, d, n, E, K, p_cap, 0u, bytes);
}

int moe_forward_ex(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2, const moe_routing *r, int T, int d,
                   int n, int E, int K, size_t p_cap, moe_bf16 *O, moe_bf16 *H, void *ws, size_t ws_bytes,
                   unsigned flags, void *stream) {
  int rc = check_layer_shape(T, d, n, E, K, p_cap);
  if (rc != MOE_OK) return rc;
  if (!X || !W1 || !W2 || !O || !H || !routing_ok(r) || (flags & ~kForwardFlags)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < fwd_ws_bytes(T, d, n, p_cap, flags)) return MOE_ERR_WORKSPACE;
  rc = check_device();
  if (rc != MOE_OK) return rc;
  const bool det = det_flag(flags);
  const bool a_from_h = a_from_h_flag(flags);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *p = static_cast<char *>(ws);
  moe_bf16 *A = a_from_h ? nullptr : reinterpret_cast<moe_bf16 *>(p);
  if (!a_from_h) p += align256(p_cap * n * 2);
  void *Oacc = p;  // fp32, or 64-bit fixed point when deterministic

  Fork side;
  if ((rc = side.open(s)) != MOE_OK) return rc;
  cudaError_t err = cudaMemsetAsync(Oacc, 0, (size_t)T * d * (det ? 8 : 4), side.side());
  if (err != cudaSuccess) return record_cuda_error(err);

  GemmArgs a = base_args(r, T, d, n, E, p_cap);
  TensorMaps tm;
  // up-projection: H = X[tok] W1_e (N = 2n, K = d); X rows are gathered with cp.async
  if ((rc = make_tmap_bf16_halves(&tm.b, W1, n, (uint64_t)E * d)) != MOE_OK) return rc;
  tm.a = tm.b;  // unused by this GEMM
  a.gsrc = X;
  a.gld = d;
  a.Ndim = 2 * n;
  a.Kdim = d;
  a.out0 = H;
  a.out1 = A;
  fill_unused(tm);
  // the epilogue stores H (and A) as 32 x 32 boxes from shared memory
  if ((rc = make_tmap_bf16_epi(&tm.dh, H, 2 * (uint64_t)n, p_cap)) != MOE_OK) return rc;
  if (!a_from_h && (rc = make_tmap_bf16_epi(&tm.sa, A, n, p_cap)) != MOE_OK) return rc;
  if ((rc = launch_up(a, tm, s)) != MOE_OK) return rc;
  // down-projection + aggregation: O32[tok] += s * A W2_e (N = d, K = n), A read from the workspace or
  // recomputed from H inside the kernel
  if (a_from_h) tm.a = tm.b;  // unused
  else if ((rc = make_tmap_bf16(&tm.a, A, n, p_cap, 128)) != MOE_OK) return rc;
  // W2_e tiles: a CTA of a pair loads half of the 256 columns, a lone CTA all of them
  const bool down_pairs = !a_from_h && use_cta_pairs(n);
  if ((rc = make_tmap_bf16_chunks(&tm.b, W2, d, (uint64_t)E * n, 64, down_pairs ? 2 : 4)) != MOE_OK) return rc;
  a.Ndim = d;
  a.Kdim = n;
  a.out0 = nullptr;
  a.out1 = nullptr;
  a.gsrc = nullptr;
  a.Hin = H;
  a.out_f32 = det ? nullptr : static_cast<float *>(Oacc);
  a.out_i64 = det ? static_cast<long long *>(Oacc) : nullptr;
  if ((rc = side.join()) != MOE_OK) return rc;
  fill_unused(tm);
  if (a_from_h) {
    if ((rc = launch_down_h(a, tm, s, det)) != MOE_OK) return rc;
  } else if (!det && d % 512 == 0 && (int64_t)T * d >= ((int64_t)48 << 20)) {
    // Two launches over the column halves: the first half of O is final once the first launch ends, so its cast
    // runs on the side stream beside the second launch and only the second half's cast stays on this stream.
    // The second launch costs a prologue and a tail of its own, so this pays only where the cast is large
    // (measured: T*d = 67 M gains about 1.5-2.5% of the step; T*d = 38 M loses 0.4%).
    const int half = d / 2;
    float *O32 = static_cast<float *>(Oacc);
    a.Ndim = half;
    a.nt_group = scatter_nt_group(T, half);
    a.n_off = 0;
    if ((rc = launch_down(a, tm, s, false)) != MOE_OK) return rc;
    if ((rc = side.open(s)) != MOE_OK) return rc;
    if ((rc = launch_f32_to_bf16_cols(O32, O, T, d, 0, half, side.side())) != MOE_OK) return rc;
    a.n_off = half;
    if ((rc = launch_down(a, tm, s, false)) != MOE_OK) return rc;
    if ((rc = launch_f32_to_bf16_cols(O32, O, T, d, half, half, s)) != MOE_OK) return rc;
    return side.join();
  } else if ((rc = launch_down(a, tm, s, det)) != MOE_OK) {
    return rc;
  }
  if (det) return launch_fixed_to_bf16(static_cast<long long *>(Oacc), O, (size_t)T * d, s);
  return launch_f32_to_bf16(static_cast<float *>(Oacc), O, T, d, s);
}

int moe_forward(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2, const moe_routing *r, int T, int d, int n,
                int E, int K, size_t p_cap, moe_bf16 *O, moe_bf16 *H, void *ws, size_t ws_bytes, void *stream) {
  return moe_forward_ex(X, W1, W2, r, T, d, n, E, K, p_cap, O, H, ws, ws_bytes, 0u, stream);
}

int moe_backward_workspace_size_ex(int T, int d, int n, int E, int K, size_t p_cap, unsigned flags, size_t *bytes) {
  if (!bytes || (flags & ~MOE_FLAG_DETERMINISTIC)) return MOE_ERR_INVALID_ARG;
  const int rc = check_layer_shape(T, d, n, E, K, p_cap);
  if (rc != MOE_OK) return rc;
  *bytes = bwd_ws_bytes(T, d, n, p_cap, flags);
  return MOE_OK;
}

int moe_backward_workspace_size(int T, int d, int n, int E, int K, size_t p_cap, size_t *bytes) {
  return moe_backward_workspace_size_ex(T, d, n, E, K, p_cap, 0u, bytes);
}

int moe_backward_ex(const moe_bf16 *dO, const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2, const moe_bf16 *H,
                    const moe_routing *r, int T, int d, int n, int E, int K, size_t p_cap, moe_bf16 *dX, moe_bf16 *dW1,
                    moe_bf16 *dW2, float *dS, void *ws, size_t ws_bytes, unsigned flags, void *stream) {
  int rc = check_layer_shape(T, d, n, E, K, p_cap);
  if (rc != MOE_OK) return rc;
  if (!dO || !X || !W1 || !W2 || !H || !dX || !dW1 || !dW2 || !dS || !routing_ok(r) ||
      (flags & ~MOE_FLAG_DETERMINISTIC))
    return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < bwd_ws_bytes(T, d, n, p_cap, flags)) return MOE_ERR_WORKSPACE;
  rc = check_device();
  if (rc != MOE_OK) return rc;
  const bool det = det_flag(flags);
  const int bn = dh_bn(n);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *p = static_cast<char *>(ws);
  moe_bf16 *dH = reinterpret_cast<moe_bf16 *>(p);
  p += align256(p_cap * 2 * n * 2);
  moe_bf16 *sA = reinterpret_cast<moe_bf16 *>(p);
  p += align256(p_cap * n * 2);
  void *dXacc = p;  // fp32, or 64-bit fixed point when deterministic
  p += align256((size_t)T * d * (det ? 8 : 4));
  float *dS_part = det ? reinterpret_cast<float *>(p) : nullptr;

  Fork side;
  if ((rc = side.open(s)) != MOE_OK) return rc;
  cudaError_t err = cudaMemsetAsync(dXacc, 0, (size_t)T * d * (det ? 8 : 4), side.side());
  if (err == cudaSuccess) err = cudaMemsetAsync(dS, 0, p_cap * 4, s);
  if (err != cudaSuccess) return record_cuda_error(err);

  GemmArgs a = base_args(r, T, d, n, E, p_cap);
  TensorMaps tm;
  // dH: dA' = dO[tok] W2_e^T (N = n, K = d); epilogue dSwiGLU, dS, s*A
  if ((rc = make_tmap_bf16(&tm.b, W2, d, (uint64_t)E * n, bn)) != MOE_OK) return rc;  // all BN rows of W2_e
  tm.a = tm.b;  // unused: dO rows are gathered with cp.async
  a.gsrc = dO;
  a.gld = d;
  a.Ndim = n;
  a.Kdim = d;
  a.out0 = dH;
  a.out1 = sA;
  a.dS = dS;
  a.dS_part = dS_part;
  a.Hin = H;
  if ((rc = make_tmap_bf16_epi(&tm.h, H, 2 * (uint64_t)n, p_cap)) != MOE_OK) return rc;
  if ((rc = make_tmap_bf16_epi(&tm.dh, dH, 2 * (uint64_t)n, p_cap)) != MOE_OK) return rc;
  if ((rc = make_tmap_bf16_epi(&tm.sa, sA, n, p_cap)) != MOE_OK) return rc;
  if ((rc = launch_dh(a, tm, s, bn, det)) != MOE_OK) return rc;
  if (det && (rc = launch_ds_sum(dS_part, n / bn, r->offsets, E, dS, s)) != MOE_OK) return rc;
  // dX~: dX32[tok] += dH W1_e^T (N = d, K = 2n)
  if ((rc = make_tmap_bf16(&tm.a, dH, 2 * (uint64_t)n, p_cap, 128)) != MOE_OK) return rc;
  // W1_e rows: half of the 256-row tile per CTA of a pair, all of it for a lone CTA
  const uint32_t dx_rows = use_cta_pairs(2 * n) ? 128 : 256;
  if ((rc = make_tmap_bf16(&tm.b, W1, 2 * (uint64_t)n, (uint64_t)E * d, dx_rows)) != MOE_OK) return rc;
  GemmArgs ax = base_args(r, T, d, n, E, p_cap);
  ax.Ndim = d;
  ax.Kdim = 2 * n;
  ax.out_f32 = det ? nullptr : static_cast<float *>(dXacc);
  ax.out_i64 = det ? static_cast<long long *>(dXacc) : nullptr;
  if ((rc = side.join()) != MOE_OK) return rc;
  if ((rc = (fill_unused(tm), launch_dx(ax, tm, s, det))) != MOE_OK) return rc;
  // the cast of dX overlaps the weight-gradient GEMMs, which read neither the accumulator nor dX
  if ((rc = side.open(s)) != MOE_OK) return rc;
  rc = det ? launch_fixed_to_bf16(static_cast<long long *>(dXacc), dX, (size_t)T * d, side.side())
           : launch_f32_to_bf16(static_cast<float *>(dXacc), dX, T, d, side.side());
  if (rc != MOE_OK) return rc;
  GemmArgs aw = base_args(r, T, d, n, E, p_cap);
  // 256-row blocks (one accumulator, B shared by two M blocks) once experts average >= 256 rows (>= 4 k-blocks per
  // tile): measured faster than double-buffered 128-row blocks there (high-sparsity layer, 256 rows on average:
  // dW1 + dW2 239 -> 198 us)
  aw.wide_m = (int64_t)T * K >= (int64_t)256 * E;
  if (aw.wide_m && d % 256 == 0 && n % 256 == 0) {
    // both weight gradients in one launch: dW1 tiles gather X into A and load dH as B, dW2 tiles load s*A
    // as A and gather dO into B (one wave quantisation instead of two)
    if ((rc = make_tmap_bf16_chunks(&tm.b, dH, 2 * (uint64_t)n, p_cap, 64, 4)) != MOE_OK) return rc;
    if ((rc = make_tmap_bf16_chunks(&tm.a, sA, n, p_cap, 64, 4)) != MOE_OK) return rc;
    aw.out0 = dW1;
    aw.out1 = dW2;
    aw.gsrc = X;
    aw.gsrc2 = dO;
    aw.gld = d;
    fill_unused(tm);
    if ((rc = make_tmap_bf16_epi(&tm.dh, dW1, 2 * (uint64_t)n, (uint64_t)E * d)) != MOE_OK) return rc;
    if ((rc = make_tmap_bf16_epi(&tm.sa, dW2, d, (uint64_t)E * n)) != MOE_OK) return rc;
    if ((rc = launch_dw12(aw, tm, s)) != MOE_OK) return rc;
    return side.join();
  }
  // dW1_e = X[tok]^T dH_e (M = d, N = 2n, K = rows of e); X rows gathered with cp.async
  if ((rc = make_tmap_bf16_chunks(&tm.b, dH, 2 * (uint64_t)n, p_cap, 64, 4)) != MOE_OK) return rc;  // BN = 256
  tm.a = tm.b;
  aw.Mdim = d;
  aw.Ndim = 2 * n;
  aw.out0 = dW1;
  aw.gsrc = X;
  aw.gld = d;
  fill_unused(tm);
  if ((rc = make_tmap_bf16_epi(&tm.dh, dW1, 2 * (uint64_t)n, (uint64_t)E * d)) != MOE_OK) return rc;
  if ((rc = launch_dw1(aw, tm, s)) != MOE_OK) return rc;
  // dW2_e = (s*A)_e^T dO[tok] (M = n, N = d, K = rows of e); dO rows gathered with cp.async
  // the s*A tile spans the M block: 256 columns (four chunks) in 256-row blocks, else 128 (two)
  const uint32_t sa_chunks = (aw.wide_m && n % 256 == 0) ? 4 : 2;
  if ((rc = make_tmap_bf16_chunks(&tm.a, sA, n, p_cap, 64, sa_chunks)) != MOE_OK) return rc;
  tm.b = tm.a;
  aw.Mdim = n;
  aw.Ndim = d;
  aw.out0 = dW2;
  aw.gsrc = dO;
  aw.gld = d;
  fill_unused(tm);
  if ((rc = make_tmap_bf16_epi(&tm.dh, dW2, d, (uint64_t)E * n)) != MOE_OK) return rc;
  if ((rc = launch_dw2(aw, tm, s)) != MOE_OK) return rc;
  return side.join();
}

int moe_backward(const moe_bf16 *dO, const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2, const moe_bf16 *H,
                 const moe_routing *r, int T, int d, int n, int E, int K, size_t p_cap, moe_bf16 *dX, moe_bf16 *dW1,
                 moe_bf16 *dW2, float *dS, void *ws, size_t ws_bytes, void *stream) {
  return moe_backward_ex(dO, X, W1, W2, H, r, T, d, n, E, K, p_cap, dX, dW1, dW2, dS, ws, ws_bytes, 0u, stream);
}

int moe_get_status(const moe_routing *r, int32_t *code, int32_t *P, void *stream) {
  if (!r || !r->status) return MOE_ERR_INVALID_ARG;
  int32_t words[MOE_STATUS_WORDS];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(words, r->status, sizeof(words), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return record_cuda_error(err);
  if (code) *code = words[0];
  if (P) *P = words[1];
  return MOE_OK;
}

const char *moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_NONFINITE_LOGITS: return "non-finite router logit";
    case MOE_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case MOE_ERR_BAD_METADATA: return "routing metadata out of range";
    case MOE_ERR_DEVICE: return "device is not compute capability 10.3";
    case MOE_ERR_RANGE: return "value beyond the deterministic accumulator's range";
    default: return "unknown status";
  }
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_profile_enable(int on) {
  ProfState &p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  if (on) {
    p.recs.clear();
    p.summary.clear();
    p.pool_used = 0;
    p.enabled = true;
    return MOE_OK;
  }
  p.enabled = false;
  // aggregate the session: per kernel name, launches and summed event time
  p.summary.clear();
  for (const ProfRec &r : p.recs) {
    cudaError_t err = cudaEventSynchronize(r.stop);
    if (err != cudaSuccess) return record_cuda_error(err);
    float ms = 0.f;
    err = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (err != cudaSuccess) return record_cuda_error(err);
    size_t i = 0;
    while (i < p.summary.size() && p.summary[i].name != r.name) ++i;
    if (i == p.summary.size()) p.summary.push_back({r.name, 0, 0.0});
    p.summary[i].launches += 1;
    p.summary[i].total_ms += ms;
  }
  p.recs.clear();
  p.pool_used = 0;
  return MOE_OK;
}

int moe_profile_count(void) {
  ProfState &p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  return static_cast<int>(p.summary.size());
}

int moe_profile_entry(int i, char *name, size_t name_len, int *launches, double *total_ms) {
  ProfState &p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  if (i < 0 || static_cast<size_t>(i) >= p.summary.size() || !name || name_len == 0) return MOE_ERR_INVALID_ARG;
  std::strncpy(name, p.summary[i].name.c_str(), name_len - 1);
  name[name_len - 1] = 0;
  if (launches) *launches = p.summary[i].launches;
  if (total_ms) *total_ms = p.summary[i].total_ms;
  return MOE_OK;
}

}  // extern "C"
