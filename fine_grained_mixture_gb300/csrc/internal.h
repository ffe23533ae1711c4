// internal.h - declarations shared by the library's translation units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "moe.h"

namespace moe {

constexpr int kMaxTrTokens = 49152;  // token rounding keeps one expert's keys for all T tokens in shared memory
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxDevices = 64;

// One positive int per device (a grid size, or 1 for "attributes set"), computed once by the first call on
// that device and safe to read from several host threads at once.  `init` runs under the lock; a result <= 0
// (a failure code) is returned but not kept, so the next call tries again.
struct DeviceCache {
  std::atomic<int> value[kMaxDevices];
  std::mutex mu;
  template <class F>
  int get(int dev, F &&init) {
    int v = value[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
    std::lock_guard<std::mutex> lk(mu);
    v = value[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    v = init();
    if (v > 0) value[dev].store(v, std::memory_order_release);
    return v;
  }
};

// Remembers `err` as this thread's last CUDA error and returns MOE_ERR_CUDA.
int record_cuda_error(cudaError_t err);
int record_cu_error(CUresult res);
void count_launch();

// Optional per-kernel CUDA-event timing (off unless moe_profile_enable(1)): brackets one kernel launch.
void prof_begin(const char *name, cudaStream_t s);
void prof_end(cudaStream_t s);

// Launches `kernel` with programmatic stream serialization, so that it may start while the previous kernel
// in the stream drains; the kernel calls griddep_wait() before reading that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// routing (route.cu)
// Every mode but token choice selects each expert's rows from a per-expert ranking of all tokens.
inline bool route_selects(int mode) { return mode != MOE_ROUTE_TC; }
// Routing scratch.  em_keys: the selection modes keep an expert-major copy of the logit order keys (4*T*E bytes)
// so that the per-expert selection reads them coalesced; without it the selection reads the logits in place.
size_t route_workspace_bytes(int T, int E, int K, int mode, bool em_keys = true);
// uniforms: per-expert draws of stochastic rounding (device fp32 [E]); unused by the other modes.
int launch_route(const float *logits, const float *uniforms, int T, int E, int K, int mode, const moe_routing *r,
                 void *ws, cudaStream_t stream, bool em_keys = true);
// moe_route_ex with the scratch layout chosen by the caller (moe_route_noalloc drops the expert-major keys when
// they would not fit its static array).
int route_call(const float *logits, const float *uniforms, int T, int E, int K, int mode, const moe_routing *r,
               void *ws, size_t ws_bytes, int32_t *P_host, void *stream, bool em_keys);

// grouped GEMMs (gemm_fwd.cu, gemm_bwd.cu)
struct GemmArgs {
  const int32_t *offsets;
  const int32_t *tile_offsets;
  const int32_t *row_token;
  const float *row_score;
  int32_t *status;
  int T, d, n, E;
  int p_cap;
  int Mdim;  // varlen-K: output rows of one expert's weight gradient
  int Ndim;  // output columns
  int Kdim;  // varlen-M: reduction length
  int nt_group;  // scatter-add GEMMs: column tiles per pass over all m-tiles (the fp32 slab kept in L2)
  int n_off;     // varlen-M GEMMs: first output column of this launch (a launch may cover a column range)
  int wide_m;    // weight-gradient GEMMs: 256-row blocks (experts average >= 1024 rows) instead of 128
  void *out0;        // up: H;  dH: dH;  dW1/dW2: the weight gradient (both in one launch: dW1)
  void *out1;        // up: A;  dH: s*A;  both weight gradients in one launch: dW2
  float *out_f32;    // down: fp32 O;  dX~: fp32 dX
  long long *out_i64;  // deterministic down / dX~: the fixed-point accumulator of O or dX
  float *dS;         // dH: per-row dS
  float *dS_part;    // deterministic dH: per-row, per-column-tile partial dS [p_cap][n / BN]
  const void *Hin;   // dH: cached H
  const void *gsrc;  // the operand gathered by token id: X (up, dW1) or dO (dH, dW2), bf16 rows
  const void *gsrc2; // both weight gradients in one launch: dO (gsrc is X)
  int gld;           // row length of the gathered operands in elements
};

// Tensor maps of one GEMM launch: a/b are the operands; h, dh, sa are the dH epilogue's cached-H input and
// dH / s*A outputs (32 x 32 boxes, 64-byte swizzle).  Unused maps are copies of `b`.
struct TensorMaps {
  CUtensorMap a, b, h, dh, sa;
};

// Encodes a 2D bf16 tensor map over [rows, inner] (row-major) with a {64, box_rows} box, 128-byte swizzle.
int make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows);
// Same with a {32, 32} box and 64-byte swizzle (the dH epilogue's per-warp tiles).
int make_tmap_bf16_epi(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t rows);
// 3D view (64 columns, rows, inner / 64 column chunks) of a row-major bf16 [rows, inner] matrix (inner a multiple of
// 64) with a {64, box_rows, chunks} box: one load lands `chunks` consecutive 128-byte-swizzled [box_rows x 64]
// tiles, column chunk c at c * box_rows * 128 bytes.
int make_tmap_bf16_chunks(CUtensorMap *tm, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                          uint32_t chunks);
// 4D view of W1 [rows, 2n] as (64 columns, rows, n / 64 chunks of one half, the gate and up halves) with a
// {64, 64, 2, 2} box: the two 64-column chunks of the gate half and the same two of the up half in one load.
int make_tmap_bf16_halves(CUtensorMap *tm, const void *base, uint64_t n, uint64_t rows);

// The scatter-add GEMMs (down-projection, dX~) run on CTA pairs when their K loop is at least this long: measured
// at K = 768 and above (coarse, skew layers: the step 4-7% faster); at K = 256 and 512 (fine7b, sparse) the pair's
// coupled epilogues and its half-empty last tiles cost more than the operand traffic saved (step 2% slower).
constexpr int kPairMinK = 768;
inline bool use_cta_pairs(int Kdim) { return Kdim >= kPairMinK; }

int num_sms();
// MOE_OK when the current device is compute capability 10.3 (the only target of this library), else
// MOE_ERR_DEVICE, or MOE_ERR_CUDA when no device can be made current.
int check_device();

// det: deterministic aggregation (fixed-point accumulators, dS partials per column tile)
int launch_up(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s);
int launch_down(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, bool det);
// The down-projection with A = SwiGLU(H) recomputed from the cached H (a.Hin) inside the kernel.
int launch_down_h(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, bool det);
int launch_dh(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, int bn, bool det);
int launch_dx(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, bool det);
int launch_dw1(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s);
int launch_dw2(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s);
// Both weight gradients in one launch (256-row blocks; d and n multiples of 256).
int launch_dw12(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s);

// elementwise (elementwise.cu)
// fp32 [rows, ld] -> bf16 (ld a multiple of 256); the fp32 lines are discarded from L2, not written back.
int launch_f32_to_bf16(const float *src, void *dst, int rows, int ld, cudaStream_t s);
// Same for columns [c0, c0 + w) (c0 and w multiples of 256).
int launch_f32_to_bf16_cols(const float *src, void *dst, int rows, int ld, int c0, int w, cudaStream_t s);
// The fixed-point accumulator of the deterministic aggregation (32 fractional bits) to bf16.
int launch_fixed_to_bf16(const long long *src, void *dst, size_t count, cudaStream_t s);
// dS[r] = sum over the column tiles, in tile order, of the deterministic dH epilogue's partials [p_cap][tiles].
int launch_ds_sum(const float *part, int tiles, const int32_t *offsets, int E, float *dS, cudaStream_t s);
}  // namespace moe
