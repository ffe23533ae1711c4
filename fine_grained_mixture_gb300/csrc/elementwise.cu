// elementwise.cu - the fp32 -> bf16 cast that finishes the fused aggregations (O and dX are accumulated
// in fp32 by the down-projection and dX~ epilogues, then rounded once to bf16), its fixed-point counterpart and
// the ordered dS sum of the deterministic mode, and the bounded-wait self-test.
#include "common.cuh"
#include "internal.h"

namespace moe {

// Columns [c0, c0 + w) of rows [0, rows) of an fp32 accumulator (row length ld) to bf16; CTA b takes rows
// [b*rows/grid, (b+1)*rows/grid).  The accumulator is dead once cast, so its lines are dropped from L2 rather
// than written back.
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float *__restrict__ src, uint16_t *__restrict__ dst,
                                                          int rows, int ld, int c0, int w) {
  griddep_wait();
  griddep_launch_dependents();
  const int r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * rows / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * rows / gridDim.x);
  cast_rows_discard<4>(src, dst, ld, r0, r1, c0, w, threadIdx.x, blockDim.x);
}

int launch_f32_to_bf16_cols(const float *src, void *dst, int rows, int ld, int c0, int w, cudaStream_t s) {
  const int blocks = num_sms() * 4;
  prof_begin("cast_f32_bf16", s);
  cudaError_t err = launch_pdl(f32_to_bf16_kernel, dim3(blocks), dim3(256), 0, s, src, static_cast<uint16_t *>(dst),
                               rows, ld, c0, w);
  prof_end(s);
  count_launch();
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : record_cuda_error(err);
}

int launch_f32_to_bf16(const float *src, void *dst, int rows, int ld, cudaStream_t s) {
  return launch_f32_to_bf16_cols(src, dst, rows, ld, 0, ld, s);
}

// Fixed-point accumulator (32 fractional bits) of the deterministic aggregation -> bf16, four elements per step.
__global__ void __launch_bounds__(256) fixed_to_bf16_kernel(const longlong2 *__restrict__ src, uint2 *__restrict__ dst,
                                                            size_t n4) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr float kInv = 2.3283064365386962890625e-10f;  // 2^-32
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const longlong2 a = __ldcs(src + 2 * i), b = __ldcs(src + 2 * i + 1);
    uint2 o;
    o.x = pack_bf16x2(__ll2float_rn(a.x) * kInv, __ll2float_rn(a.y) * kInv);
    o.y = pack_bf16x2(__ll2float_rn(b.x) * kInv, __ll2float_rn(b.y) * kInv);
    __stcs(dst + i, o);
  }
}

int launch_fixed_to_bf16(const long long *src, void *dst, size_t count, cudaStream_t s) {
  const size_t n4 = count / 4;  // count is a multiple of 256 (d % 256 == 0)
  const int blocks = num_sms() * 8;
  prof_begin("cast_fixed_bf16", s);
  cudaError_t err = launch_pdl(fixed_to_bf16_kernel, dim3(blocks), dim3(256), 0, s,
                               reinterpret_cast<const longlong2 *>(src), reinterpret_cast<uint2 *>(dst), n4);
  prof_end(s);
  count_launch();
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : record_cuda_error(err);
}

// dS[r] for r < P: the deterministic dH epilogue's per-column-tile partials added in tile order.
__global__ void __launch_bounds__(256) ds_sum_kernel(const float *__restrict__ part, int tiles,
                                                     const int32_t *__restrict__ offsets, int E,
                                                     float *__restrict__ dS) {
  griddep_wait();
  griddep_launch_dependents();
  const size_t P = static_cast<size_t>(offsets[E]);
  for (size_t r = blockIdx.x * (size_t)blockDim.x + threadIdx.x; r < P; r += (size_t)gridDim.x * blockDim.x) {
    float v = 0.f;
    for (int j = 0; j < tiles; ++j) v += part[r * tiles + j];
    dS[r] = v;
  }
}

int launch_ds_sum(const float *part, int tiles, const int32_t *offsets, int E, float *dS, cudaStream_t s) {
  prof_begin("ds_sum", s);
  cudaError_t err = launch_pdl(ds_sum_kernel, dim3(num_sms() * 2), dim3(256), 0, s, part, tiles, offsets, E, dS);
  prof_end(s);
  count_launch();
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : record_cuda_error(err);
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait ends it with a status code.
__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait(b, 0)) set_status(status, MOE_ERR_DEVICE_TIMEOUT);
}

}  // namespace moe

extern "C" int moe_selftest_bounded_wait(int32_t *status, void *stream) {
  if (!status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe::wait_selftest_kernel<<<1, 32, 0, s>>>(status);
  moe::count_launch();
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : moe::record_cuda_error(err);
}
