// router.cu - the router on either side of the MoE layer.
//
// "SonicMoE: Accelerating MoE with IO and Tile-aware Optimizations" (ICLR 2026 reading note), "Method details /
// overall framework": router scoring of the input tokens feeds the routing step.  The router is z = X W_r
// (X [T, d] bf16, W_r [d, E] bf16, z [T, E] fp32).  Its backward holds the routing fixed (top-K selection and
// token rounding are piecewise constant in z) and differentiates the gates: a row r = (t, e) has
//     s_r = exp(z_te) / sum_{j in N(t)} exp(z_tj)
// with N(t) the token's K token-choice experts (token choice and every token-rounding rule) or all E experts
// (expert choice), so for L = sum_r dS_r s_r
//     dz_tj = sum_{r of t} dS_r s_r [j = e_r]  -  [j in N(t)] s_tj G_t,     G_t = sum_{r of t} dS_r s_r,
// then dX += dz W_r^T and dW_r = X^T dz.
//
// Kernels:
//   router_gemm_kernel<kRLogits>  z = X W_r            M = T, N = E (128-column tiles), K = d
//   router_dz_rows_kernel         one thread per routed row: dS_r s_r into dz[t, e] (each pair is unique)
//   router_dz_tokens_kernel       one warp per token: G_t as the sum of its dz row (fixed order), the normaliser
//                                 term, dz in fp32 (output) and bf16
//   router_gemm_kernel<kRDX>      dX (bf16, read-modify-write) += dz W_r^T   M = T, N = d (256), K = E
//   router_gemm_kernel<kRDW>      one partial of X^T dz per token split       M = d, N = E (128), K = T split
//   router_dw_sum_kernel          dW_r = the partials added in split order (reproducible bit for bit)
// The GEMMs are dense contractions on tcgen05: operands arrive by TMA (128-byte swizzle, K-major or MN-major),
// one thread issues the MMAs into TMEM, four warps drain it.  One output tile per CTA; two CTAs share an SM, so
// one CTA's epilogue overlaps the other's main loop.  Epilogue staging reuses the drained pipeline stages.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

enum RouterGemm : int { kRLogits = 0, kRDX = 1, kRDW = 2 };

struct RouterArgs {
  int T, d, E;
  int n_tiles;       // output column tiles
  int kb_total;      // 64-wide k-blocks of the whole reduction
  int kb_per_split;  // k-blocks per CTA (the dW_r reduction over tokens is split across CTAs)
  float *out;        // logits [T, E], or the dW_r partials [splits][d][E] (split s at out + s * d * E)
  int32_t *status;   // device error word (may be null)
};

struct RouterMaps {
  CUtensorMap a, b, c;  // c: dX as 32 x 32 bf16 boxes (kRDX); unused otherwise
};

template <int MODE>
struct RTraits {
  static constexpr int BN = MODE == kRDX ? 256 : 128;
  static constexpr int STAGES = MODE == kRDX ? 2 : 3;
  static constexpr bool a_mn = MODE == kRDW;   // A = X^T: MN-major
  static constexpr bool b_mn = MODE != kRDX;   // B = W_r (logits) or dz (dW_r): MN-major; W_r^T (dX): K-major
  static constexpr int kA = 128 * 64 * 2;
  static constexpr int kB = BN * 64 * 2;
  static constexpr int kStage = kA + kB;
  static constexpr int kBarOff = STAGES * kStage;
  static constexpr int kSmem = kBarOff + 256 + 1024;  // + barriers + alignment slack
};

constexpr int kRThreads = 192;     // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int kRStgRow = 144;      // bytes of one thread's fp32 staging row (32 fp32 + 16 bytes against conflicts)

template <int MODE>
__global__ void __launch_bounds__(kRThreads) router_gemm_kernel(const __grid_constant__ RouterMaps tm,
                                                                const RouterArgs a) {
  using TR = RTraits<MODE>;
  constexpr int BN = TR::BN, STAGES = TR::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t bar = base + TR::kBarOff;
  auto full_bar = [&](int s) { return bar + 8u * s; };
  auto empty_bar = [&](int s) { return bar + 8u * (STAGES + s); };
  const uint32_t tfull_bar = bar + 8u * (2 * STAGES);
  const uint32_t drain_bar = bar + 8u * (2 * STAGES + 1);
  auto rmw_bar = [&](int w, int b) { return bar + 8u * (2 * STAGES + 2 + 2 * w + b); };  // kRDX epilogue
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + TR::kBarOff + 8 * (2 * STAGES + 10));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + TR::kBarOff + 8 * (2 * STAGES + 10) + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile of this CTA: column tile fastest, then the reduction split (dW_r only), then the row tile
  const int nt = blockIdx.x % a.n_tiles;
  const int rest = blockIdx.x / a.n_tiles;
  const int splits = MODE == kRDW ? (a.kb_total + a.kb_per_split - 1) / a.kb_per_split : 1;
  const int split = rest % splits;
  const int mt = rest / splits;
  const int m0 = mt * 128, n0 = nt * BN;
  const int kb0 = split * a.kb_per_split;
  const int kb1 = min(a.kb_total, kb0 + a.kb_per_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    for (int i = 0; i < 8; ++i) mbar_init(rmw_bar(i >> 1, i & 1), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm.a);
    tma_prefetch_desc(&tm.b);
    if (MODE == kRDX) tma_prefetch_desc(&tm.c);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // the previous kernel's outputs (dz) are read only after this
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool aborted = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(empty_bar(s), ph ^ 1u) || *abort_flag) {
          set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
          *abort_flag = 1;
          aborted = true;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), TR::kStage);
        const uint32_t sa = base + s * TR::kStage, sb = sa + TR::kA, fb = full_bar(s);
        if (MODE == kRLogits) {
          tma_load_2d(sa, &tm.a, kb * 64, m0, fb, pol);                     // X rows m0.., K columns
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + c * 8192, &tm.b, n0 + c * 64, kb * 64, fb, pol);
        } else if (MODE == kRDX) {
          tma_load_2d(sa, &tm.a, kb * 64, m0, fb, pol);                     // dz rows m0.., expert columns
#pragma unroll
          for (int h = 0; h < 2; ++h) tma_load_2d(sb + h * 16384, &tm.b, kb * 64, n0 + h * 128, fb, pol);
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) tma_load_2d(sa + c * 8192, &tm.a, m0 + c * 64, kb * 64, fb, pol);  // X^T
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + c * 8192, &tm.b, n0 + c * 64, kb * 64, fb, pol);
        }
        ++issued;
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (aborted) {
        for (int st = 0; st < STAGES && st < issued; ++st) {
          const int last = st + ((issued - 1 - st) / STAGES) * STAGES;
          mbar_wait(full_bar(st), static_cast<uint32_t>((last / STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN, TR::a_mn, TR::b_mn);
      int s = 0;
      uint32_t ph = 0;
      bool aborted = false;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(full_bar(s), ph) || *abort_flag) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t sa = base + s * TR::kStage, sb = sa + TR::kA;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = TR::a_mn ? smem_desc_sw128(sa + k * 2048, 8192, 1024) : smem_desc_sw128(sa + k * 32, 16, 1024);
          const uint64_t bd = TR::b_mn ? smem_desc_sw128(sb + k * 2048, 8192, 1024) : smem_desc_sw128(sb + k * 32, 16, 1024);
          umma_bf16(tmem_base, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        }
        umma_commit(empty_bar(s));
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (aborted) {
        set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      } else {
        umma_commit(tfull_bar);
      }
    }
  } else {
    // ---------------------------------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int row = q * 32 + lane;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(tfull_bar, 0) && !*abort_flag;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    } else {
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      if (MODE == kRDX) {
        // dX tile rows m0 + 32q.., columns n0..n0+256: load each 32 x 32 bf16 box, add, store it back.  Two 2 KB
        // buffers per warp in the drained stage memory, each refilled once its store has read it.
        const uint32_t wb = base + q * 4096;
        const int sw = (lane >> 1) & 3;  // 64-byte swizzle: piece p of row `lane` at piece p ^ sw
        const int r0 = m0 + q * 32;
        auto issue = [&](int c) {
          const uint32_t hb = rmw_bar(q, c & 1);
          mbar_arrive_expect_tx(hb, 2048);
          tma_load_2d(wb + (c & 1) * 2048, &tm.c, n0 + c * 32, r0, hb, policy_evict_first());
        };
        const int n_chunks = r0 < a.T ? BN / 32 : 0;  // a warp whose 32 rows all lie past T has nothing to do
        if (lane == 0 && n_chunks > 0) {
          issue(0);
          issue(1);
        }
        uint32_t par = 0u;
#pragma unroll 1
        for (int c = 0; c < n_chunks; ++c) {
          const int b = c & 1;
          uint32_t v[32];
          tmem_ld32(tacc + c * 32, v);
          const bool got = mbar_wait(rmw_bar(q, b), (par >> b) & 1u);
          par ^= 1u << b;
          if (!got) {
            set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
          }
          tmem_ld_wait();
          const uint32_t buf = wb + b * 2048;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const uint32_t o = buf + lane * 64 + ((p ^ sw) << 4);
            const float4 x4 = ld_shared_v4(o);
            const uint32_t xw[4] = {__float_as_uint(x4.x), __float_as_uint(x4.y), __float_as_uint(x4.z),
                                    __float_as_uint(x4.w)};
            uint32_t yw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float lo = bf16_lo(xw[i]) + __uint_as_float(v[8 * p + 2 * i]);
              const float hi = bf16_hi(xw[i]) + __uint_as_float(v[8 * p + 2 * i + 1]);
              yw[i] = pack_bf16x2(lo, hi);
            }
            st_shared_v4(o, __uint_as_float(yw[0]), __uint_as_float(yw[1]), __uint_as_float(yw[2]),
                         __uint_as_float(yw[3]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tm.c, buf, n0 + c * 32, r0, policy_evict_first());
            bulk_commit();
            if (c + 2 < n_chunks) {
              bulk_wait_read<0>();  // the store has read the buffer: refill it
              issue(c + 2);
            }
          }
          __syncwarp();
        }
      } else {
        // fp32 rows of the tile leave as per-row bulk copies (logits) or bulk reduce-adds (dW_r) of up to 128
        // bytes from this thread's staging row; columns past E are not written
        const uint32_t stg = base + (q * 32 + lane) * kRStgRow;
        const int grow = m0 + row;
        const bool live = MODE == kRLogits ? grow < a.T : grow < a.d;
        float *out_row = a.out + (MODE == kRDW ? (size_t)split * a.d * a.E : 0) + (size_t)(live ? grow : 0) * a.E;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int col = n0 + c * 32;
          if (col >= a.E) break;
          uint32_t v[32];
          tmem_ld32(tacc + c * 32, v);
          tmem_ld_wait();
          bulk_wait_read<0>();  // the previous copy has read the staging row
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_v4(stg + i * 16, __uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                         __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          fence_proxy_async_smem();
          const uint32_t bytes = static_cast<uint32_t>(min(32, a.E - col)) * 4u;
          if (live) bulk_store(out_row + col, stg, bytes);
          bulk_commit();
        }
      }
      bulk_wait<0>();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag && lane == 0) {
      umma_commit(drain_bar);  // every MMA this CTA issued is complete once this arrives
      mbar_wait(drain_bar, 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, BN);
  }
}

// One thread per routed row r = (t, e): dS_r s_r goes to dz[t, e] (the pair is unique, so a plain store into the
// zeroed dz).  The row's expert is found by a binary search over the offsets, which each CTA keeps in shared memory.
constexpr int kDzRowsThreads = 256;
__global__ void __launch_bounds__(kDzRowsThreads) router_dz_rows_kernel(const float *__restrict__ dS,
                                                                        const int32_t *__restrict__ offsets,
                                                                        const int32_t *__restrict__ row_token,
                                                                        const float *__restrict__ row_score, int T,
                                                                        int E, int p_cap, float *__restrict__ dz,
                                                                        int32_t *__restrict__ status) {
  __shared__ int s_off[kMaxExperts + 1];
  griddep_wait();
  griddep_launch_dependents();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = offsets[e];
  __syncthreads();
  const int P = s_off[E];
  if (P < 0 || P > p_cap) {
    if (threadIdx.x == 0) set_status(status, MOE_ERR_BAD_METADATA);
    return;
  }
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= P) return;
  int lo = 0, hi = E;  // largest e with s_off[e] <= r
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= r) lo = mid;
    else hi = mid;
  }
  const int t = row_token[r];
  if (t < 0 || t >= T) {
    set_status(status, MOE_ERR_BAD_METADATA);
    return;
  }
  dz[(size_t)t * E + lo] = dS[r] * row_score[r];
}

// One warp per token: the row dz[t, :] holds exactly the token's dS_r s_r at their experts, so G_t is its sum,
// taken in a fixed order (each lane its own columns, then a butterfly), which keeps dz reproducible.  Then
// dz[t, j] -= s_tj G_t over the token's normaliser set, and the row is written in fp32 (the caller's dlogits) and
// bf16 (the operand of the two backward GEMMs).  Token choice and token rounding take s_tj from topk_score (the
// token-choice gates); expert choice recomputes the softmax over all E logits.
template <int NV>
__global__ void __launch_bounds__(256) router_dz_tokens_kernel(const float *__restrict__ logits,
                                                               const int32_t *__restrict__ topk_idx,
                                                               const float *__restrict__ topk_score, int T, int E,
                                                               int K, int ec, float *__restrict__ dz,
                                                               uint16_t *__restrict__ dz16) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? dz[(size_t)t * E + e] : 0.f;
  }
  float g = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) g += v[j];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
  if (ec) {
    float z[NV], m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int e = lane + 32 * j;
      z[j] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
      m = fmaxf(m, z[j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    double den = 0.0;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      z[j] = (lane + 32 * j) < E ? expf(z[j] - m) : 0.f;
      den += static_cast<double>(z[j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    const float inv = static_cast<float>(1.0 / den);
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] -= (z[j] * inv) * g;
  } else {
    for (int k = 0; k < K; ++k) {
      const int idx = topk_idx[(size_t)t * K + k];
      const float s = topk_score[(size_t)t * K + k];
#pragma unroll
      for (int j = 0; j < NV; ++j)
        if (idx == lane + 32 * j) v[j] -= s * g;
    }
  }
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      dz[(size_t)t * E + e] = v[j];
      dz16[(size_t)t * E + e] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
    }
  }
}

// dW_r[i] = sum over the token splits, in split order, of the partials [splits][d][E]; four elements a step.
__global__ void __launch_bounds__(256) router_dw_sum_kernel(const float4 *__restrict__ part, int splits, size_t n4,
                                                            float4 *__restrict__ dWr) {
  griddep_wait();
  griddep_launch_dependents();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    float4 acc = __ldcs(part + i);
    for (int sp = 1; sp < splits; ++sp) {
      const float4 v = __ldcs(part + (size_t)sp * n4 + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    dWr[i] = acc;
  }
}

// ------------------------------------------------------------------------------------------------ host

namespace {

template <int MODE>
int launch_router_gemm(const RouterMaps &tm, const RouterArgs &a, int grid, cudaStream_t s, const char *name) {
  static DeviceCache attrs;  // the shared-memory attribute, set once per device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return record_cuda_error(err);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
  const int attr_rc = attrs.get(dev, [&]() -> int {
    const cudaError_t e = cudaFuncSetAttribute(router_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               RTraits<MODE>::kSmem);
    return e == cudaSuccess ? 1 : -static_cast<int>(e);
  });
  if (attr_rc <= 0) return record_cuda_error(static_cast<cudaError_t>(-attr_rc));
  prof_begin(name, s);
  err = launch_pdl(router_gemm_kernel<MODE>, dim3(grid), dim3(kRThreads), RTraits<MODE>::kSmem, s, tm, a);
  prof_end(s);
  count_launch();
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : record_cuda_error(err);
}

int check_router_shape(int T, int d, int E) {
  if (T <= 0 || d <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (E % 8 != 0 || E > kMaxExperts || d % 256 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)T * E >= ((int64_t)1 << 31) || (int64_t)T * d >= ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The token splits of dW_r (each a [d, E] fp32 partial); the count follows the SM count but never exceeds this,
// so the workspace size does not depend on the device.
constexpr int kRMaxSplits = 32;

// dz in bf16 [T, E], then the dW_r partials [kRMaxSplits][d][E].
size_t router_bwd_ws_bytes(int T, int d, int E) {
  return align256((size_t)T * E * 2) + align256((size_t)kRMaxSplits * d * E * 4);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_router_forward(const moe_bf16 *X, const moe_bf16 *Wr, int T, int d, int E, float *logits, int32_t *status,
                       void *stream) {
  int rc = check_router_shape(T, d, E);
  if (rc != MOE_OK) return rc;
  if (!X || !Wr || !logits) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RouterMaps tm;
  if ((rc = make_tmap_bf16(&tm.a, X, d, T, 128)) != MOE_OK) return rc;   // X: K-major A, 128-row boxes
  if ((rc = make_tmap_bf16(&tm.b, Wr, E, d, 64)) != MOE_OK) return rc;   // W_r [d, E]: MN-major B
  tm.c = tm.b;
  RouterArgs a{};
  a.T = T;
  a.d = d;
  a.E = E;
  a.n_tiles = (E + 127) / 128;
  a.kb_total = d / 64;
  a.kb_per_split = a.kb_total;
  a.out = logits;
  a.status = status;
  const int grid = ((T + 127) / 128) * a.n_tiles;
  return launch_router_gemm<kRLogits>(tm, a, grid, s, "router_logits");
}

int moe_router_backward_workspace_size(int T, int d, int E, size_t *bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const int rc = check_router_shape(T, d, E);
  if (rc != MOE_OK) return rc;
  *bytes = router_bwd_ws_bytes(T, d, E);
  return MOE_OK;
}

int moe_router_backward(const float *dS, const moe_routing *r, const float *logits, const moe_bf16 *X,
                        const moe_bf16 *Wr, int T, int d, int E, int K, int mode, size_t p_cap, float *dlogits,
                        moe_bf16 *dX, float *dWr, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_router_shape(T, d, E);
  if (rc != MOE_OK) return rc;
  if (K <= 0 || K > E || K > kMaxTopK || mode < MOE_ROUTE_TC || mode > MOE_ROUTE_EC) return MOE_ERR_INVALID_ARG;
  if (!dS || !r || !r->topk_idx || !r->topk_score || !r->offsets || !r->row_token || !r->row_score || !r->status ||
      !logits || !X || !Wr || !dlogits || !dX || !dWr)
    return MOE_ERR_INVALID_ARG;
  if (p_cap < (size_t)T * K || p_cap >= ((size_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < router_bwd_ws_bytes(T, d, E)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t *dz16 = static_cast<uint16_t *>(ws);
  float *part = reinterpret_cast<float *>(static_cast<char *>(ws) + align256((size_t)T * E * 2));

  cudaError_t err = cudaMemsetAsync(dlogits, 0, (size_t)T * E * 4, s);
  if (err != cudaSuccess) return record_cuda_error(err);

  prof_begin("router_dz_rows", s);
  // one thread per row of the capacity (rows at and past P return at once)
  err = launch_pdl(router_dz_rows_kernel, dim3(static_cast<unsigned>((p_cap + kDzRowsThreads - 1) / kDzRowsThreads)),
                   dim3(kDzRowsThreads), 0, s, dS, r->offsets, r->row_token, r->row_score, T, E,
                   static_cast<int>(p_cap), dlogits, r->status);
  prof_end(s);
  count_launch();
  if (err != cudaSuccess) return record_cuda_error(err);

  const int ec = mode == MOE_ROUTE_EC ? 1 : 0;
  const int nv = (E + 31) / 32;
  const dim3 tgrid((T + 7) / 8);
  prof_begin("router_dz_tokens", s);
#define MOE_DZ_LAUNCH(NV)                                                                                           \
  err = launch_pdl(router_dz_tokens_kernel<NV>, tgrid, dim3(256), 0, s, logits, r->topk_idx, r->topk_score, T, E, K, \
                   ec, dlogits, dz16)
  if (nv <= 1) MOE_DZ_LAUNCH(1);
  else if (nv <= 2) MOE_DZ_LAUNCH(2);
  else if (nv <= 4) MOE_DZ_LAUNCH(4);
  else if (nv <= 8) MOE_DZ_LAUNCH(8);
  else if (nv <= 16) MOE_DZ_LAUNCH(16);
  else MOE_DZ_LAUNCH(32);
#undef MOE_DZ_LAUNCH
  prof_end(s);
  count_launch();
  if (err != cudaSuccess) return record_cuda_error(err);

  // dX += dz W_r^T  (M = T, N = d, K = E)
  RouterMaps tm;
  if ((rc = make_tmap_bf16(&tm.a, dz16, E, T, 128)) != MOE_OK) return rc;   // dz: K-major A
  if ((rc = make_tmap_bf16(&tm.b, Wr, E, d, 128)) != MOE_OK) return rc;     // W_r rows (d) with K = E inner
  if ((rc = make_tmap_bf16_epi(&tm.c, dX, d, T)) != MOE_OK) return rc;
  RouterArgs a{};
  a.T = T;
  a.d = d;
  a.E = E;
  a.n_tiles = d / 256;
  a.kb_total = (E + 63) / 64;
  a.kb_per_split = a.kb_total;
  a.status = r->status;
  if ((rc = launch_router_gemm<kRDX>(tm, a, ((T + 127) / 128) * a.n_tiles, s, "router_dx")) != MOE_OK) return rc;

  // dW_r = X^T dz  (M = d, N = E, K = T split into chunks across CTAs, one fp32 partial per split)
  if ((rc = make_tmap_bf16(&tm.a, X, d, T, 64)) != MOE_OK) return rc;       // X^T: MN-major A
  if ((rc = make_tmap_bf16(&tm.b, dz16, E, T, 64)) != MOE_OK) return rc;    // dz: MN-major B
  tm.c = tm.b;
  a.n_tiles = (E + 127) / 128;
  a.kb_total = (T + 63) / 64;
  const int tiles = (d / 128) * a.n_tiles;
  const int want_splits = std::min(kRMaxSplits, std::max(1, (2 * num_sms() + tiles - 1) / tiles));  // ~2 CTAs/SM
  a.kb_per_split = std::max(4, (a.kb_total + want_splits - 1) / want_splits);
  const int splits = (a.kb_total + a.kb_per_split - 1) / a.kb_per_split;  // <= want_splits <= kRMaxSplits
  a.out = part;
  if ((rc = launch_router_gemm<kRDW>(tm, a, tiles * splits, s, "router_dw")) != MOE_OK) return rc;
  const size_t n4 = (size_t)d * E / 4;  // d % 256 == 0
  prof_begin("router_dw_sum", s);
  err = launch_pdl(router_dw_sum_kernel, dim3(num_sms() * 4), dim3(256), 0, s, reinterpret_cast<const float4 *>(part),
                   splits, n4, reinterpret_cast<float4 *>(dWr));
  prof_end(s);
  count_launch();
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : record_cuda_error(err);
}

}  // extern "C"
