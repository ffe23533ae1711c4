// route.cu - routing metadata kernels: token-choice top-K, per-expert counts and offsets, and token
// rounding.  Integer/compare work plus one fp32 softmax per token; every output is deterministic.
//
// Method: "SonicMoE: Accelerating MoE with IO and Tile-aware Optimizations" (ICLR 2026 reading note),
// "Key design 1: Token Rounding routing": token choice first; per expert, an expert-choice ordering of the
// tokens with the token-choice tokens ahead of expert-choice candidates; round_and_sparsify pads an
// expert with expert-choice tokens when the distance up to the next multiple of M_tile is strictly
// smaller than the distance down, and drops its weakest token-choice tokens otherwise.
//
// The rounding subroutine is a free choice ("Loss function / training strategy": token rounding is robust to
// it): nearest (the default above), always up, always down, or stochastic (up with probability
// (f - floor)/M_tile, from one caller-drawn uniform per expert).  Expert choice (the "EC" rows of the ablation
// table) reuses the same per-expert selection: every token is a candidate and each expert keeps C of them.
//
// Pipeline (one stream, no host synchronisation):
//   route_topk_kernel   one warp per token (32 tokens per CTA): top-K by (logit desc, expert asc), softmax over the K,
//                       the CTA's expert histogram; selection modes (all but TC): the CTA's word of the membership
//                       bitmap and its 32 columns of the expert-major key matrix, both written whole (no zero fill)
//   route_scan_kernel   one CTA per expert: per-chunk (256 tokens) bases, counts (f_e, rounded r_e, or C)
//   route_fill_tc       one CTA per 256-token chunk: rows in ascending token order via bitmap ranks
//   route_fill_tr       one CTA per expert: radix selection of the kept set, rows in token order
//                       (each fill CTA scans the E counts into offsets; CTA 0 publishes them)
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kChunk = 256;  // tokens per routing chunk

// Total order on fp32 logits used everywhere: larger value first; -0.0 equals +0.0.
__device__ __forceinline__ uint32_t order_key(float z) {
  uint32_t b = __float_as_uint(z);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

constexpr int kTopkThreads = 256;                    // 8 warps, 4 tokens each: 32 tokens per CTA
constexpr int kTokensPerWarp = 4;
constexpr int kTopkTokens = (kTopkThreads / 32) * kTokensPerWarp;
static_assert(kTopkTokens == 32, "a top-K CTA covers exactly one 32-token word of the membership bitmap");
constexpr int kCtasPerChunk = kChunk / kTopkTokens;  // top-K histograms summed into one routing chunk

// Inverse of order_key.
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int kKeyStride = 33;  // words per expert row of the TR key tile (odd: conflict-free transpose)

// Dynamic shared memory of route_topk_kernel: the CTA histogram, plus for TR the membership words and the
// [E][32] key tile.
size_t route_topk_smem_bytes(int E, int mode) {
  return (size_t)E * 4 + (route_selects(mode) ? (size_t)E * 4 + (size_t)E * kKeyStride * 4 : 0);
}

template <int NV, bool TR>  // NV = logits held per lane = ceil(E / 32)
__global__ void __launch_bounds__(kTopkThreads) route_topk_kernel(const float *__restrict__ logits, int T, int E, int K,
                                                         int32_t *__restrict__ topk_idx,
                                                         float *__restrict__ topk_score, float *__restrict__ tok_max,
                                                         float *__restrict__ tok_den, int32_t *__restrict__ cta_hist,
                                                         uint32_t *__restrict__ member, int member_words,
                                                         uint32_t *__restrict__ keys_em, int32_t *__restrict__ status,
                                                         int den_all) {
  // den_all (expert choice): tok_den holds the softmax denominator over all E logits instead of the K selected
  extern __shared__ int32_t hist[];                                      // [E]
  uint32_t *mbits = reinterpret_cast<uint32_t *>(hist + E);             // [E]     TR: bit i = token t_first + i chose e
  uint32_t *ktile = mbits + E;                                           // [E][33] TR: order keys of the 32 tokens
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    hist[e] = 0;
    if (TR) mbits[e] = 0u;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int t_first = blockIdx.x * kTopkTokens;
  // the warp's logit rows are loaded up front so that their latencies overlap (only while they fit in
  // registers); rows past T read as -inf and are skipped
  constexpr int kPre = NV <= 8 ? kTokensPerWarp : 1;
  float vpre[kPre][NV];
  if (kPre > 1) {
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const int t = t_first + warp * kTokensPerWarp + i;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int e = lane + 32 * j;
        vpre[i][j] = (t < T && e < E) ? __ldcs(&logits[(size_t)t * E + e]) : -INFINITY;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kTokensPerWarp; ++i) {
    const int tl = warp * kTokensPerWarp + i;  // token within the CTA
    const int t = t_first + tl;
    if (t >= T) break;
    float v[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int e = lane + 32 * j;
      if (kPre > 1) v[j] = vpre[kPre > 1 ? i : 0][j];
      else v[j] = (e < E) ? __ldcs(&logits[(size_t)t * E + e]) : -INFINITY;
    }
    bool bad = false;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int e = lane + 32 * j;
      if (TR && e < E) ktile[e * kKeyStride + tl] = order_key(v[j]);
      if (e < E && !isfinite(v[j])) bad = true;
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) set_status(status, MOE_ERR_NONFINITE_LOGITS);
#pragma unroll
      for (int j = 0; j < NV; ++j)
        if (!isfinite(v[j])) v[j] = -INFINITY;
    }
    int my_e = -1;  // lane k keeps the k-th selection
    float my_z = 0.f, z0 = 0.f;
    if (NV <= 8) {
      // each lane sorts its NV logits once (key descending; equal keys keep the lower expert first), then
      // every round is two warp reductions: the largest key, then the lowest expert holding it
      uint32_t key[NV];
      int ex[NV];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int e = lane + 32 * j;
        key[j] = (e < E) ? order_key(v[j]) : 0u;
        ex[j] = (e < E) ? e : 0x7fffffff;
      }
#pragma unroll
      for (int i = 1; i < NV; ++i)
#pragma unroll
        for (int j = i; j > 0; --j)
          if (key[j] > key[j - 1]) {
            const uint32_t tk = key[j];
            key[j] = key[j - 1];
            key[j - 1] = tk;
            const int te = ex[j];
            ex[j] = ex[j - 1];
            ex[j - 1] = te;
          }
      for (int k = 0; k < K; ++k) {
        const uint32_t mx = __reduce_max_sync(0xffffffffu, key[0]);
        const uint32_t we = __reduce_min_sync(0xffffffffu, key[0] == mx ? static_cast<uint32_t>(ex[0]) : 0xffffffffu);
        if (static_cast<uint32_t>(ex[0]) == we) {
#pragma unroll
          for (int j = 0; j + 1 < NV; ++j) {
            key[j] = key[j + 1];
            ex[j] = ex[j + 1];
          }
          key[NV - 1] = 0u;
          ex[NV - 1] = 0x7fffffff;
        }
        const float z = key_to_float(mx);
        if (k == 0) z0 = z;
        if (lane == k) {
          my_e = static_cast<int>(we);
          my_z = z;
        }
      }
    } else {
      uint32_t taken = 0;  // bit j: v[j] already selected
      for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          const int e = lane + 32 * j;
          if (e < E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < be) || be == 0x7fffffff)) {
            bv = v[j];
            be = e;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          const int oe = __shfl_xor_sync(0xffffffffu, be, off);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (k == 0) z0 = bv;
        if (lane == k) {
          my_e = be;
          my_z = bv;
        }
      }
    }
    // softmax over the K selected logits, in selection order
    const float w = (lane < K) ? expf(my_z - z0) : 0.f;
    float den = 0.f;
    for (int k = 0; k < K; ++k) den += __shfl_sync(0xffffffffu, w, k);
    // expert choice: sum over all E of exp(z - z0), accumulated in fp64 so that up to 1024 terms round once
    double den_e = 0.0;
    if (den_all) {
#pragma unroll
      for (int j = 0; j < NV; ++j)
        if (lane + 32 * j < E) den_e += static_cast<double>(expf(v[j] - z0));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den_e += __shfl_xor_sync(0xffffffffu, den_e, off);
    }
    if (lane < K) {
      topk_idx[(size_t)t * K + lane] = my_e;
      topk_score[(size_t)t * K + lane] = w / den;
      atomicAdd(&hist[my_e], 1);
      if (TR) atomicOr(&mbits[my_e], 1u << tl);
    }
    if (lane == 0) {
      tok_max[t] = z0;
      tok_den[t] = den_all ? static_cast<float>(den_e) : den;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    cta_hist[(size_t)blockIdx.x * E + e] = hist[e];
    if (TR) member[(size_t)e * member_words + blockIdx.x] = mbits[e];  // a CTA covers one 32-token word
  }
  if (TR && keys_em) {
    // expert-major keys: each warp writes whole 32-token rows (128 bytes) of experts warp, warp + 8, ...
    const int t = t_first + lane;
    for (int e = warp; e < E; e += kTopkThreads / 32)
      if (t < T) keys_em[(size_t)e * T + t] = ktile[e * kKeyStride + lane];
  }
}

// Exclusive scan of one value per thread across the block (blockDim.x a multiple of 32); returns the
// exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch /*[32]*/, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    scratch[lane] = s;  // inclusive per-warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? scratch[warp - 1] : 0);
  *total = scratch[nwarps - 1];
  __syncthreads();
  return before + x - v;
}


// Row offsets and m-tile offsets of every expert (exclusive scans of counts[0..E) and of their tile counts)
// into shared memory, entries 0..E.  Thread i takes a contiguous run of experts.
__device__ void expert_offsets(const int32_t *__restrict__ counts, int E, int m_tile, int *s_off, int *s_toff,
                               int *scratch) {
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int c = 0, tl = 0;
  for (int e = e0; e < e1; ++e) {
    const int v = counts[e];
    c += v;
    tl += (v + m_tile - 1) / m_tile;
  }
  int P, tiles;
  int o = block_exclusive_scan(c, scratch, &P);
  int to = block_exclusive_scan(tl, scratch, &tiles);
  for (int e = e0; e < e1; ++e) {
    const int v = counts[e];
    s_off[e] = o;
    s_toff[e] = to;
    o += v;
    to += (v + m_tile - 1) / m_tile;
  }
  if (threadIdx.x == 0) {
    s_off[E] = P;
    s_toff[E] = tiles;
  }
  __syncthreads();
}

// CTA 0 of a fill kernel publishes the offsets (read by the GEMMs once the fill kernel has finished).
__device__ void publish_offsets(int E, const int *s_off, const int *s_toff, int32_t *__restrict__ offsets,
                                int32_t *__restrict__ tile_offsets, int32_t *__restrict__ status) {
  if (blockIdx.x != 0) return;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    offsets[e] = s_off[e];
    tile_offsets[e] = s_toff[e];
  }
  if (threadIdx.x == 0) {
    status[1] = s_off[E];
    status[2] = s_toff[E];
  }
}

// One CTA per expert: the expert's count in every 256-token chunk (the sum of its top-K CTAs' histograms),
// their exclusive prefix (chunk_base), the token-choice count f_e and the routed count (f_e, or r_e after
// rounding).  Thread i takes a contiguous run of chunks.
constexpr int kScanThreads = 256;
__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(int T, int E, int nctas, int mode, int m_tile,
                                                                  const float *__restrict__ uniforms, int ec_cap,
                                                                  const int32_t *__restrict__ cta_hist,
                                                                  int32_t *__restrict__ chunk_base,
                                                                  int32_t *__restrict__ tc_counts,
                                                                  int32_t *__restrict__ counts) {
  __shared__ int scratch[32];
  griddep_wait();
  griddep_launch_dependents();
  const int e = blockIdx.x;
  const int nchunks = (nctas + kCtasPerChunk - 1) / kCtasPerChunk;
  const int per = (nchunks + kScanThreads - 1) / kScanThreads;
  const int c0 = threadIdx.x * per, c1 = min(nchunks, c0 + per);
  auto chunk_sum = [&](int c) {
    int v = 0;
#pragma unroll
    for (int i = 0; i < kCtasPerChunk; ++i) {
      const int b = c * kCtasPerChunk + i;
      if (b < nctas) v += cta_hist[(size_t)b * E + e];
    }
    return v;
  };
  int run = 0;
  for (int c = c0; c < c1; ++c) run += chunk_sum(c);
  int f;
  int base = block_exclusive_scan(run, scratch, &f);
  for (int c = c0; c < c1; ++c) {
    chunk_base[(size_t)c * E + e] = base;
    base += chunk_sum(c);
  }
  if (threadIdx.x == 0) {
    int cnt = f;
    if (mode == MOE_ROUTE_EC) {
      cnt = ec_cap;
    } else if (mode != MOE_ROUTE_TC) {
      const int lo = (f / m_tile) * m_tile;
      const int hi = ((f + m_tile - 1) / m_tile) * m_tile;
      bool up;
      if (mode == MOE_ROUTE_TR) up = (hi - f) < (f - lo);  // nearest; a tie takes the floor
      else if (mode == MOE_ROUTE_TR_UP) up = hi > f;
      else if (mode == MOE_ROUTE_TR_DOWN) up = false;
      else up = uniforms[e] * static_cast<float>(m_tile) < static_cast<float>(f - lo);  // both sides exact in fp32
      cnt = (up && hi <= T) ? hi : lo;  // no padding beyond the T tokens there are
    }
    tc_counts[e] = f;
    counts[e] = cnt;
  }
}

__global__ void __launch_bounds__(kChunk) route_fill_tc_kernel(int T, int E, int K, int m_tile,
                                                               const int32_t *__restrict__ topk_idx,
                                                               const float *__restrict__ topk_score,
                                                               const int32_t *__restrict__ chunk_base,
                                                               const int32_t *__restrict__ counts,
                                                               int32_t *__restrict__ offsets,
                                                               int32_t *__restrict__ tile_offsets,
                                                               int32_t *__restrict__ status,
                                                               int32_t *__restrict__ row_token, int32_t *__restrict__ row_slot,
                                                               float *__restrict__ row_score) {
  extern __shared__ uint32_t bm[];  // [E][8]: bit i of word w = token chunk*256 + 32w + i chose the expert
  __shared__ int s_off[kMaxExperts + 1], s_toff[kMaxExperts + 1], scratch[32];
  const int chunk = blockIdx.x;
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) bm[i] = 0u;
  griddep_wait();
  griddep_launch_dependents();
  expert_offsets(counts, E, m_tile, s_off, s_toff, scratch);
  publish_offsets(E, s_off, s_toff, offsets, tile_offsets, status);
  const int tl = threadIdx.x;
  const int t = chunk * kChunk + tl;
  const bool live = t < T;
  if (live)
    for (int k = 0; k < K; ++k) atomicOr(&bm[topk_idx[(size_t)t * K + k] * 8 + (tl >> 5)], 1u << (tl & 31));
  __syncthreads();
  if (!live) return;
  for (int k = 0; k < K; ++k) {
    const int e = topk_idx[(size_t)t * K + k];
    const uint32_t *w = &bm[e * 8];
    int rank = __popc(w[tl >> 5] & ((1u << (tl & 31)) - 1u));
    for (int j = 0; j < (tl >> 5); ++j) rank += __popc(w[j]);
    const int row = s_off[e] + chunk_base[(size_t)chunk * E + e] + rank;
    row_token[row] = t;
    row_slot[row] = k;
    row_score[row] = topk_score[(size_t)t * K + k];
  }
}

// Token rounding and expert choice: the kept rows of each expert.  A cluster of C CTAs (C = 1 .. 8) takes one
// expert; CTA c takes the token words [c * Wc, (c + 1) * Wc) (Wc = ceil(ceil(T / 32) / C)) and keeps that slice's
// keys in shared memory.  The CTAs of a cluster combine their results through distributed shared memory (plain
// loads of each other's shared memory; nothing is multicast):
//   selection: a 4-pass radix select (8 bits per pass, most significant first) over the candidates finds the key
//              of the R-th best.  Each CTA fills a 256-bin histogram of its slice (lanes in one bin add once) and
//              every CTA sums the cluster's histograms in the same order, so all of them take the same boundary.
//              After the first pass (or from the start when dropping) each CTA lists its candidates, so the later
//              passes skip the rest of its tokens.
//   ties:      candidates equal to the boundary key are kept lowest token first: a CTA's ties rank after the ties
//              of the CTAs before it.
//   output:    a CTA's kept rows follow those of the CTAs before it, in ascending token order.
constexpr int kTrThreads = 512;
constexpr int kTrWarps = kTrThreads / 32;
constexpr int kTrHists = 4;  // histogram copies, one per four warps
constexpr int kTrMaxCluster = 8;

__device__ __forceinline__ int warp_scan_exclusive(int v, int *total) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

__global__ void __launch_bounds__(kTrThreads, 4) route_fill_tr_kernel(
    const uint32_t *__restrict__ keys_em, const float *__restrict__ logits, int T, int E, int K,
    const int32_t *__restrict__ topk_idx,
    const float *__restrict__ topk_score, const float *__restrict__ tok_max, const float *__restrict__ tok_den,
    const uint32_t *__restrict__ member, int member_words, int m_tile, const int32_t *__restrict__ tc_counts,
    const int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ tile_offsets,
    int32_t *__restrict__ status, int32_t *__restrict__ row_token, int32_t *__restrict__ row_slot,
    float *__restrict__ row_score, int slice_words, int list_cap, int ec) {
  // ec (expert choice): every token is a candidate (as if all had chosen the expert) and a row's gate is the
  // token's softmax over all E logits (tok_den holds that denominator)
  extern __shared__ uint32_t sm[];
  uint32_t *key = sm;                                          // [32 * slice_words]: key of token t0 + i at i
  uint32_t *mem = key + 32 * slice_words;                      // [slice_words] token-choice membership
  uint32_t *keep_bits = mem + slice_words;                     // [slice_words]
  uint32_t *tie = keep_bits + slice_words;                     // [slice_words] ties, then kept rows before a word
  int *hist = reinterpret_cast<int *>(tie + slice_words);      // [2][kTrHists][256], alternate passes
  int *list = hist + 2 * kTrHists * 256;                       // [list_cap] candidate (local) token indices
  __shared__ int list_n;
  __shared__ int sel_state[2];
  __shared__ int xch[2];     // shown to the cluster: this CTA's boundary ties, its kept rows
  __shared__ int before[2];  // the same, summed over the CTAs before this one
  __shared__ int s_off[kMaxExperts + 1], s_toff[kMaxExperts + 1], scratch[32];
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = static_cast<int>(cluster_nctarank()), c = static_cast<int>(cluster_ctarank());
  const int e = static_cast<int>(blockIdx.x) / C;
  expert_offsets(counts, E, m_tile, s_off, s_toff, scratch);
  publish_offsets(E, s_off, s_toff, offsets, tile_offsets, status);
  const int f = ec ? T : tc_counts[e], r = counts[e], base = s_off[e];
  if (r == 0) return;  // the same in every CTA of the cluster: none of them touches another's shared memory
  const int w0 = c * slice_words, w1 = min(member_words, w0 + slice_words);
  const int nw = max(0, w1 - w0);                  // words of this CTA's slice
  const int t0 = 32 * w0;
  const int nloc = max(0, min(T, 32 * w1) - t0);   // tokens of this CTA's slice
  for (int w = threadIdx.x; w < nw; w += blockDim.x) mem[w] = member[(size_t)e * member_words + w0 + w];
  if (keys_em && (T & 3) == 0) {
    // the slice of the expert's row of keys, 16 bytes a load and four loads in flight per thread before any store
    const uint4 *src = reinterpret_cast<const uint4 *>(keys_em + (size_t)e * T + t0);
    uint4 *dst = reinterpret_cast<uint4 *>(key);
    const int n4 = nloc >> 2;
    for (int i0 = threadIdx.x; i0 < n4; i0 += 4 * kTrThreads) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * kTrThreads < n4) v[u] = __ldcs(src + i0 + u * kTrThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * kTrThreads < n4) dst[i0 + u * kTrThreads] = v[u];
    }
  } else if (keys_em) {
    for (int i = threadIdx.x; i < nloc; i += blockDim.x) key[i] = __ldcs(&keys_em[(size_t)e * T + t0 + i]);
  } else {  // compact scratch: the expert's column of the logits, one strided word per token
    for (int i = threadIdx.x; i < nloc; i += blockDim.x) key[i] = order_key(logits[(size_t)(t0 + i) * E + e]);
  }
  __syncthreads();
  // candidates: token-choice tokens when dropping, the other tokens when padding
  const bool drop = r < f;
  const int R = drop ? r : r - f;  // how many candidates the cluster keeps
  uint32_t prefix = 0u, mask = 0u;
  int remaining = R;
  const uint32_t lt = (1u << lane) - 1u;
  // This slice's tokens satisfying `pred`, in no particular order, into list[]; -1 when more than list_cap.
  auto build_list = [&](auto pred) -> int {
    if (threadIdx.x == 0) list_n = 0;
    __syncthreads();
    for (int i0 = 0; i0 < nloc; i0 += blockDim.x) {
      const int i = i0 + threadIdx.x;
      const bool p = i < nloc && pred(i);
      const uint32_t b = __ballot_sync(0xffffffffu, p);
      int at = 0;
      if (lane == 0 && b) at = atomicAdd(&list_n, __popc(b));
      at = __shfl_sync(0xffffffffu, at, 0) + __popc(b & lt);
      if (p && at < list_cap) list[at] = i;
    }
    __syncthreads();
    return list_n <= list_cap ? list_n : -1;
  };
  auto is_tc = [&](int i) { return ((mem[i >> 5] >> (i & 31)) & 1u) != 0u; };
  auto first = [&](int i) { return ec || is_tc(i); };  // ranked ahead of the other tokens
  int nlist = -1;  // this slice's candidates listed in list[] (-1: not listed)
  if (r != f) {
    // Candidates are few next to T: the expert's token-choice tokens when dropping, and when padding the other
    // tokens in the top-byte bin of the boundary.  Once they are listed, the remaining radix passes walk the list
    // instead of all the slice's tokens (all of them when the list would overflow its space, or under expert
    // choice, where every token is a candidate).
    nlist = (drop && !ec) ? build_list(is_tc) : -1;
    for (int pass = 0, shift = 24; shift >= 0; ++pass, shift -= 8) {
      // the two buffers alternate: a CTA zeroes this pass's buffer only after the whole cluster has passed the
      // barrier of the previous pass, by which time every CTA has read the buffer's previous contents
      int *hb = hist + (pass & 1) * kTrHists * 256;
      for (int i = threadIdx.x; i < kTrHists * 256; i += blockDim.x) hb[i] = 0;
      __syncthreads();
      int *my_hist = hb + (warp >> 2) * 256;
      const int n_iter = nlist >= 0 ? nlist : nloc;
      for (int i0 = 0; i0 < n_iter; i0 += blockDim.x) {
        const int i = i0 + threadIdx.x;
        uint32_t bin = 256u;
        if (i < n_iter) {
          const int t = nlist >= 0 ? list[i] : i;
          const uint32_t k = key[t];
          if ((nlist >= 0 || first(t) == drop) && (k & mask) == prefix) bin = (k >> shift) & 255u;
        }
        // lanes that fall in the same bin add once (many keys share their leading bits)
        const uint32_t same = __match_any_sync(0xffffffffu, bin);
        if (bin < 256u && lane == __ffs(same) - 1) atomicAdd(&my_hist[bin], __popc(same));
      }
      __syncthreads();
      for (int b = threadIdx.x; b < 256; b += blockDim.x) {
        int v = 0;
#pragma unroll
        for (int g = 1; g < kTrHists; ++g) v += hb[g * 256 + b];
        hb[b] += v;
      }
      cluster_sync();  // every CTA's histogram of this pass is complete in its copy 0
      if (warp == 0) {
        // lane l owns bins 255 - 8l - i (i = 0..7), i.e. lane 0 the highest bins, summed over the cluster
        int cnt[8], lane_sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int b = 255 - (lane * 8 + i);
          int v = 0;
          for (int q = 0; q < C; ++q) v += static_cast<int>(ld_dsmem_u32(hb + b, static_cast<uint32_t>(q)));
          cnt[i] = v;
          lane_sum += v;
        }
        int tot;
        const int bef = warp_scan_exclusive(lane_sum, &tot);
        if (bef < remaining && remaining <= bef + lane_sum) {
          int acc = bef;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (acc + cnt[i] >= remaining) {
              sel_state[0] = 255 - (lane * 8 + i);
              sel_state[1] = remaining - acc;
              break;
            }
            acc += cnt[i];
          }
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(sel_state[0]) << shift;
      mask |= 255u << shift;
      remaining = sel_state[1];
      if (shift == 24 && (!drop || nlist < 0)) {
        // the slice's candidates whose top byte is at or above the boundary's: every candidate that can still be
        // kept (when padding, or when the first list would not fit or was not built, as under expert choice)
        const uint32_t top = prefix;
        nlist = build_list([&](int i) { return first(i) == drop && (key[i] & 0xff000000u) >= top; });
      }
    }
  }
  // prefix = key of the R-th best candidate of the expert; `remaining` candidates equal to it are kept, lowest
  // token first.  Keep masks word by word; each thread owns a contiguous run of the slice's words.
  const int per = (nw + kTrThreads - 1) / kTrThreads;
  const int wa = min(nw, static_cast<int>(threadIdx.x) * per), wb = min(nw, wa + per);
  for (int w = wa; w < wb; ++w) {
    uint32_t m = 0u;
    if (r == f || !drop) {
      const int gw = w0 + w;  // the word's index over all T tokens
      if (ec) m = (32 * gw + 32 <= T) ? 0xffffffffu : ((1u << (T - 32 * gw)) - 1u);
      else m = mem[w];
    }
    keep_bits[w] = m;
    tie[w] = 0u;
  }
  __syncthreads();
  if (r != f) {
    const int n_iter = nlist >= 0 ? nlist : nloc;
    for (int i = threadIdx.x; i < n_iter; i += blockDim.x) {
      const int t = nlist >= 0 ? list[i] : i;
      if (nlist < 0 && first(t) != drop) continue;
      const uint32_t k = key[t];
      if (k > prefix) atomicOr(&keep_bits[t >> 5], 1u << (t & 31));
      else if (k == prefix) atomicOr(&tie[t >> 5], 1u << (t & 31));
    }
    __syncthreads();
    int ties = 0, total;
    for (int w = wa; w < wb; ++w) ties += __popc(tie[w]);
    int rank = block_exclusive_scan(ties, scratch, &total);
    if (threadIdx.x == 0) xch[0] = total;
    cluster_sync();  // the ties of every slice are counted
    if (threadIdx.x == 0) {
      int sum = 0;
      for (int q = 0; q < c; ++q) sum += static_cast<int>(ld_dsmem_u32(&xch[0], static_cast<uint32_t>(q)));
      before[0] = sum;
    }
    __syncthreads();
    rank += before[0];
    for (int w = wa; w < wb; ++w) {
      uint32_t m = tie[w];
      while (m) {
        const uint32_t bit = m & (0u - m);
        if (rank < remaining) keep_bits[w] |= bit;
        ++rank;
        m ^= bit;
      }
    }
    __syncthreads();
  }
  // rows: this thread's words start after the kept rows of the earlier threads and of the earlier slices
  int kept = 0, ktotal;
  for (int w = wa; w < wb; ++w) kept += __popc(keep_bits[w]);
  int kbase = block_exclusive_scan(kept, scratch, &ktotal);
  if (threadIdx.x == 0) xch[1] = ktotal;
  cluster_sync();  // the kept rows of every slice are counted
  if (threadIdx.x == 0) {
    int sum = 0;
    for (int q = 0; q < c; ++q) sum += static_cast<int>(ld_dsmem_u32(&xch[1], static_cast<uint32_t>(q)));
    before[1] = sum;
  }
  for (int w = wa; w < wb; ++w) {  // kept rows of the slice before each word
    tie[w] = static_cast<uint32_t>(kbase);
    kbase += __popc(keep_bits[w]);
  }
  __syncthreads();
  const int row0 = base + before[1];
  // the row of kept token t0 + i at position pos: its token-choice slot (if any) and its gate
  auto write_row = [&](int pos, int i) {
    const int t = t0 + i;
    int slot = -1;
    if (is_tc(i)) {
      for (int k = 0; k < K; ++k)
        if (topk_idx[(size_t)t * K + k] == e) slot = k;
    }
    const float sc = (slot >= 0 && !ec) ? topk_score[(size_t)t * K + slot]
                                        : expf(key_to_float(key[i]) - tok_max[t]) / tok_den[t];
    row_token[pos] = t;
    row_slot[pos] = slot;
    row_score[pos] = sc;
  };
  if (ktotal <= list_cap) {
    // the kept tokens compacted in token order into the (free again) candidate list, then one thread per row, so
    // the rows' global loads (slot, gate) are all in flight at once
    for (int w = wa; w < wb; ++w) {
      uint32_t m = keep_bits[w];
      int at = static_cast<int>(tie[w]);
      while (m) {
        const int b = __ffs(m) - 1;
        list[at++] = 32 * w + b;
        m &= m - 1u;
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < ktotal; i += blockDim.x) write_row(row0 + i, list[i]);
  } else {
    // more rows than the list holds: one word per warp at a time, one lane per token
    for (int w = warp; w < nw; w += kTrWarps) {
      const uint32_t m = keep_bits[w];
      if ((m >> lane) & 1u) write_row(row0 + static_cast<int>(tie[w]) + __popc(m & lt), 32 * w + lane);
    }
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

// ------------------------------------------------------------------------------------------- host

struct RouteWs {
  int32_t *cta_hist, *chunk_base;
  uint32_t *member, *keys_em;
  float *tok_max, *tok_den;
  int nctas, nchunks, member_words;
};

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// cta_hist [nctas][E] | chunk_base [nchunks][E] | TR: member [E][words], keys_em [E][T] | tok_max [T] | tok_den [T]
size_t route_workspace_bytes(int T, int E, int K, int mode, bool em_keys) {
  (void)K;
  const size_t nctas = (T + kTopkTokens - 1) / kTopkTokens;
  const size_t nchunks = (T + kChunk - 1) / kChunk;
  const size_t words = (T + 31) / 32;
  size_t b = align256(nctas * E * 4) + align256(nchunks * E * 4);
  if (route_selects(mode)) b += align256(words * E * 4) + (em_keys ? align256((size_t)T * E * 4) : 0);
  b += align256((size_t)T * 4) * 2;
  return b;
}

static RouteWs carve(void *ws, int T, int E, int mode, bool em_keys) {
  RouteWs w{};
  w.nctas = (T + kTopkTokens - 1) / kTopkTokens;
  w.nchunks = (T + kChunk - 1) / kChunk;
  w.member_words = (T + 31) / 32;
  char *p = static_cast<char *>(ws);
  w.cta_hist = reinterpret_cast<int32_t *>(p);
  p += align256((size_t)w.nctas * E * 4);
  w.chunk_base = reinterpret_cast<int32_t *>(p);
  p += align256((size_t)w.nchunks * E * 4);
  if (route_selects(mode)) {
    w.member = reinterpret_cast<uint32_t *>(p);
    p += align256((size_t)w.member_words * E * 4);
    if (em_keys) {
      w.keys_em = reinterpret_cast<uint32_t *>(p);
      p += align256((size_t)T * E * 4);
    }
  }
  w.tok_max = reinterpret_cast<float *>(p);
  p += align256((size_t)T * 4);
  w.tok_den = reinterpret_cast<float *>(p);
  return w;
}

// The token-rounding fill's launch: C CTAs per expert, each with slice_words words of tokens.  C doubles (up to 8)
// while E*C CTAs stay within about four per SM (so one cluster per expert still runs in a single wave), and no
// slice is empty.
struct TrLaunch {
  int C, slice_words, list_cap;
  size_t smem;
};

// Dynamic shared memory of one CTA: the slice's keys, three word arrays, two sets of histograms.
static size_t route_tr_fixed_bytes(int slice_words) {
  return (size_t)slice_words * 32 * 4 + (size_t)slice_words * 4 * 3 + 2 * kTrHists * 256 * 4;
}

constexpr size_t kTrDynSmemMax = 218 * 1024;  // + about 8.3 KB of static shared memory stays under 227 KB
static TrLaunch route_tr_launch(int T, int E) {
  TrLaunch l;
  const int words = (T + 31) / 32;
  l.C = 1;
  while (l.C < kTrMaxCluster && (int64_t)E * l.C * 2 <= 4 * (int64_t)num_sms() && l.C * 2 <= words) l.C *= 2;
  l.slice_words = (words + l.C - 1) / l.C;
  // candidate-list entries beside the fixed part: up to 4096, and with several CTAs per expert no more than keeps
  // a CTA (with its 8.4 KB of static shared memory) to a quarter of the SM's 228 KB: four CTAs of 512 threads
  const size_t fixed = route_tr_fixed_bytes(l.slice_words);
  const size_t cap_bytes = l.C > 1 ? std::max<size_t>(fixed + 4096, 46 * 1024) : kTrDynSmemMax;
  const size_t room = fixed < cap_bytes ? (cap_bytes - fixed) / 4 : 0;
  l.list_cap = static_cast<int>(room < 4096 ? room : 4096);
  l.smem = fixed + (size_t)l.list_cap * 4;
  return l;
}

int launch_route(const float *logits, const float *uniforms, int T, int E, int K, int mode, const moe_routing *r,
                 void *ws, cudaStream_t stream, bool em_keys) {
  RouteWs w = carve(ws, T, E, mode, em_keys);
  cudaError_t err = cudaMemsetAsync(r->status, 0, MOE_STATUS_WORDS * sizeof(int32_t), stream);
  if (err != cudaSuccess) return record_cuda_error(err);
  const bool tr = route_selects(mode);
  const int den_all = mode == MOE_ROUTE_EC ? 1 : 0;
  const size_t topk_smem = route_topk_smem_bytes(E, mode);
  const int nv = (E + 31) / 32;
  // the key tile of E = 1024 needs more than the default 48 KB of dynamic shared memory (set once per device)
  static DeviceCache attrs;
  int dev = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return record_cuda_error(err);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
#define MOE_TOPK_KERNEL(NV, TRB) route_topk_kernel<NV, TRB>
#define MOE_TOPK_EACH(F)                                                                                          \
  F(1, false) F(2, false) F(4, false) F(8, false) F(16, false) F(32, false) F(1, true) F(2, true) F(4, true)      \
      F(8, true) F(16, true) F(32, true)
  const int attr_rc = attrs.get(dev, [&]() -> int {
    cudaError_t e = cudaSuccess;
#define MOE_TOPK_ATTR(NV, TRB)                                                                                    \
  if (e == cudaSuccess)                                                                                           \
    e = cudaFuncSetAttribute(MOE_TOPK_KERNEL(NV, TRB), cudaFuncAttributeMaxDynamicSharedMemorySize,               \
                             static_cast<int>(route_topk_smem_bytes(1024, TRB ? MOE_ROUTE_TR : MOE_ROUTE_TC)));
    MOE_TOPK_EACH(MOE_TOPK_ATTR)
#undef MOE_TOPK_ATTR
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(route_fill_tr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kTrDynSmemMax));
    return e == cudaSuccess ? 1 : -static_cast<int>(e);
  });
  if (attr_rc <= 0) return record_cuda_error(static_cast<cudaError_t>(-attr_rc));
#undef MOE_TOPK_EACH
#define MOE_TOPK_LAUNCH(NV)                                                                                       \
  do {                                                                                                            \
    auto kern = tr ? MOE_TOPK_KERNEL(NV, true) : MOE_TOPK_KERNEL(NV, false);                                      \
    kern<<<w.nctas, kTopkThreads, topk_smem, stream>>>(logits, T, E, K, r->topk_idx, r->topk_score, w.tok_max,    \
                                                       w.tok_den, w.cta_hist, w.member, w.member_words, w.keys_em, \
                                                       r->status, den_all);                                       \
  } while (0)
  prof_begin("route_topk", stream);
  if (nv <= 1) MOE_TOPK_LAUNCH(1);
  else if (nv <= 2) MOE_TOPK_LAUNCH(2);
  else if (nv <= 4) MOE_TOPK_LAUNCH(4);
  else if (nv <= 8) MOE_TOPK_LAUNCH(8);
  else if (nv <= 16) MOE_TOPK_LAUNCH(16);
  else MOE_TOPK_LAUNCH(32);
#undef MOE_TOPK_LAUNCH
#undef MOE_TOPK_KERNEL
  prof_end(stream);
  count_launch();
  prof_begin("route_scan", stream);
  const int ec_cap = static_cast<int>(std::min<int64_t>(T, (int64_t)T * K / E));
  err = launch_pdl(route_scan_kernel, dim3(E), dim3(kScanThreads), 0, stream, T, E, w.nctas, mode, MOE_M_TILE,
                   uniforms, ec_cap, w.cta_hist, w.chunk_base, r->tc_counts, r->counts);
  if (err != cudaSuccess) return record_cuda_error(err);
  prof_end(stream);
  count_launch();
  if (mode == MOE_ROUTE_TC) {
    prof_begin("route_fill_tc", stream);
    err = launch_pdl(route_fill_tc_kernel, dim3(w.nchunks), dim3(kChunk), (size_t)E * 8 * 4, stream, T, E, K,
                     MOE_M_TILE, r->topk_idx, r->topk_score, w.chunk_base, r->counts, r->offsets, r->tile_offsets,
                     r->status, r->row_token, r->row_slot, r->row_score);
    if (err != cudaSuccess) return record_cuda_error(err);
  } else {
    const TrLaunch tl = route_tr_launch(T, E);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;  // one cluster of C CTAs per expert
    attr[0].val.clusterDim.x = tl.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(E * tl.C);
    cfg.blockDim = dim3(kTrThreads);
    cfg.dynamicSmemBytes = tl.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    prof_begin("route_fill_tr", stream);
    err = cudaLaunchKernelEx(&cfg, route_fill_tr_kernel, static_cast<const uint32_t *>(w.keys_em), logits, T, E, K,
                             static_cast<const int32_t *>(r->topk_idx), static_cast<const float *>(r->topk_score),
                             static_cast<const float *>(w.tok_max), static_cast<const float *>(w.tok_den),
                             static_cast<const uint32_t *>(w.member), w.member_words, static_cast<int>(MOE_M_TILE),
                             static_cast<const int32_t *>(r->tc_counts), static_cast<const int32_t *>(r->counts),
                             r->offsets, r->tile_offsets, r->status, r->row_token, r->row_slot, r->row_score,
                             tl.slice_words, tl.list_cap, den_all);
    if (err != cudaSuccess) return record_cuda_error(err);
  }
  prof_end(stream);
  count_launch();
  err = cudaGetLastError();
  if (err != cudaSuccess) return record_cuda_error(err);
  return MOE_OK;
}

}  // namespace moe
