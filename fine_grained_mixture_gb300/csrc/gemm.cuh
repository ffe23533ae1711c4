// gemm.cuh - the grouped-GEMM kernel family of the MoE layer on tcgen05 / TMEM / TMA (sm_103a).
//
// "SonicMoE: Accelerating MoE with IO and Tile-aware Optimizations" (ICLR 2026 reading note) splits the
// layer into varlen-M grouped GEMMs (rows of one expert are a variable-length M range) and varlen-K
// grouped GEMMs (the weight gradients reduce over an expert's rows), with the token gather fused into the
// operand load and elementwise work fused into the epilogue ("Key design 2: IO-aware fused kernels"), and
// on Blackwell a two-stage TMEM accumulator so one tile's epilogue overlaps the next tile's MMAs.
//
// One persistent kernel template serves the GEMMs of the layer:
//   kUp   H = X[tok] W1_e, epilogue SwiGLU -> H (bf16, cached) and A (bf16)        M=rows  N=2n  K=d
//   kDown O32[tok] += s * (A W2_e)  (Y never stored)                              M=rows  N=d   K=n
//   kDH   dA' = dO[tok] W2_e^T, epilogue: A'=SwiGLU(H), dS=<dA',A'>, dH, s*A'      M=rows  N=n   K=d
//   kDX   dX32[tok] += dH W1_e^T                                                    M=rows  N=d   K=2n
//   kDW1  dW1_e = X[tok]^T dH   (reduction over the expert's rows)                  M=d     N=2n  K=rows
//   kDW2  dW2_e = (sA)^T dO[tok]                                                    M=n     N=d   K=rows
//   kDW   both weight gradients in one launch: the dW1 pairs of every expert, then the dW2 pairs (256-row blocks)
//   kDownH  as kDown, with the A operand recomputed from the cached H (A = SiLU(H_gate) * H_up) by producer
//           warps straight into shared memory, so A [P, n] is never written to or read from HBM
//
// CTA = 6 or 10 warps: warp 0 issues TMA tiled loads of the dense operands, warp 1 owns TMEM and one
// elected lane issues tcgen05.mma, warps 2..5 (2..9 in the scatter-add GEMMs) drain TMEM in the epilogue,
// and in the GEMMs that read rows by token id warps 6..9 gather those rows with 16-byte cp.async into the
// 128-byte-swizzled layout (a TMA gather costs one request per 128-byte row, which starves the tensor cores
// here; the LSU path moves the same rows at a fraction of the issue cost).  Epilogue outputs leave through
// TMA stores (or bulk reduce-adds) from shared-memory staging: per-row stores from registers would crowd
// the gather out of L1.
// Tiles: 128 x BN x 64 (256-row blocks in the weight gradients), STAGES-deep shared-memory ring, two TMEM
// accumulators of BN fp32 columns.  Each CTA decodes its tiles once into shared memory.
// CTAs 2i and 2i+1 take neighbouring tiles (consecutive m-tiles of one expert, or neighbouring tiles of one
// weight gradient), so the operand they share is read from L2 by the second CTA; every CTA loads its whole
// tiles itself and releases its own stages.
// CTA pairs (CG = 2; the scatter-add GEMMs with K loops of 768 and more): CTAs 2i and 2i+1 form a two-CTA
// cluster and share one M = 256 tcgen05.mma.cta_group::2 issued by the even CTA.  Each loads its own 128 rows
// of A and half of B's columns; both CTAs' TMA loads complete on the leader's barrier, and the leader commits
// each stage and accumulator to both CTAs' barriers (no multicast form).  Work items are 256-row pair tiles of
// one expert.
// Every wait is bounded; on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT, drains its own copies and
// MMAs, frees TMEM and returns.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

enum GemmMode : int { kUp = 0, kDown = 1, kDH = 2, kDX = 3, kDW1 = 4, kDW2 = 5, kDW = 6, kDownH = 7 };

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB per stage

template <int MODE>
struct Traits {
  static constexpr bool varlen_k = (MODE == kDW1 || MODE == kDW2 || MODE == kDW);
  static constexpr bool gather_a_k = (MODE == kUp || MODE == kDH);  // A: token rows, K-major
  static constexpr bool gather_a_mn = (MODE == kDW1);                // A: token rows along K, MN-major
  static constexpr bool gather_b_mn = (MODE == kDW2);                // B: token rows along K, MN-major
  static constexpr bool gather = gather_a_k || gather_a_mn || gather_b_mn || MODE == kDW;  // kDW: A or B per tile
  static constexpr bool transform_a = (MODE == kDownH);  // A computed from H by warps 6..9
  static constexpr bool producers = gather || transform_a;  // warps 6..9 fill the A (or B) stages
  static constexpr bool nt_outer_ = (MODE == kDown || MODE == kDX || MODE == kDownH);
  // the scatter-add GEMMs drain TMEM with eight warps (two per TMEM lane quarter, half the columns each)
  static constexpr int epi_warps = nt_outer_ ? 8 : 4;
  static constexpr bool a_mn = varlen_k;  // A operand MN-major in shared memory
  static constexpr bool b_mn = (MODE == kUp || MODE == kDown || MODE == kDownH || varlen_k);
  static constexpr bool nt_outer = nt_outer_;  // keep one fp32 column slab hot in L2
  // the scatter-add GEMMs with TMA-loaded operands may run on CTA pairs (M = 256 across two SMs, each holding its
  // 128 rows of A and half of B's columns): a third fewer operand bytes per FLOP on each SM.  (The gather GEMMs
  // would need the peer's gathered rows forwarded to the leader's barrier: measured 2x slower, not built.)
  static constexpr bool pairable = (MODE == kDown || MODE == kDX);
};

constexpr int kGatherThreads = 128;

// Scatter-add epilogues: every thread stages 64 fp32 of its row (256 B, padded to 272 B against bank
// conflicts) and hands it to the TMA engine as one bulk reduce-add into the fp32 accumulator row of its
// token.  256-byte bulk adds reach about 1.6x the L2 reduction rate of per-lane red.v4.
constexpr int kStgRowBytes = 272;
constexpr int kStgBytes = 256 * kStgRowBytes;  // eight epilogue warps x 32 threads

// dH epilogue, per warp: one 4 KB buffer of cached H (gate | up, 32 rows x 32 columns each), refilled by TMA as
// soon as the warp has read the current chunk, and a 4 KB staging tile (dH gate | dH up) drained by TMA stores;
// 64-byte swizzle.  s*A leaves from registers.  This keeps the epilogue to 32 KB, so the mainloop gets four stages.
constexpr int kDhWarpBytes = 4096 + 4096;

// MB = 128-row M blocks per CTA.  The weight-gradient GEMMs (long K loop, light epilogue) use MB = 2: two
// M=128 MMAs per k-step share the B tile, halving shared-memory bytes per FLOP so the same shared memory
// covers twice the load latency; both accumulators fill TMEM (512 columns), so there is one buffer.
template <int BN, int STAGES, int EPI_BYTES, int MB = 1, int CACHE_BYTES = 0, int CG = 1>
struct Smem {
  static constexpr int kABytesMB = MB * kABytes;
  static constexpr int kBBytes = (BN / CG) * kBK * 2;  // a CTA pair holds half of B in each CTA
  static constexpr int kStageBytes = kABytesMB + kBBytes;
  static constexpr int kStgOff = STAGES * kStageBytes;
  static constexpr int kBarOff = kStgOff + EPI_BYTES;
  static constexpr int kCacheOff = kBarOff + 256;  // barriers/flags, then the tile cache
  static constexpr int kPairOff = kCacheOff + CACHE_BYTES;  // CTA pairs: per-expert prefix of 256-row pair tiles
  static constexpr int kBytes = kPairOff + (CG == 2 ? 4 * (kMaxExperts + 1 + 32) : 0) + 1024;  // + alignment slack
};

// Up-projection epilogue, per warp: one 6 KB staging tile (H gate | H up | A, 32 rows x 32 columns each,
// 64-byte swizzle) drained by TMA stores.  Per-row stores from registers would send three uncoalesced 64-byte
// pieces per lane and chunk through L1, twice the requests of the cp.async gather they compete with.
constexpr int kUpWarpBytes = 6144;

// Weight-gradient epilogue, per warp: two 2 KB staging tiles (32 rows x 32 columns of dW, 64-byte swizzle)
// drained by TMA stores, one box in flight while the next is written.
constexpr int kDwWarpBytes = 2 * 2048;

// Epilogue warps: the weight-gradient GEMMs with 256-row blocks drain their single (unoverlapped) 256 x 256
// accumulator with eight warps, one 128-row block per group of four (warps 2..5 and 10..13).
template <int MODE, int MB>
__host__ __device__ constexpr int epi_warps() {
  return (Traits<MODE>::varlen_k && MB == 2) ? 8 : Traits<MODE>::epi_warps;
}

template <int MODE, int MB>
__host__ __device__ constexpr int cta_threads() {
  return Traits<MODE>::producers ? 192 + 32 * epi_warps<MODE, MB>() : 64 + 32 * epi_warps<MODE, MB>();
}

template <int MODE, int MB = 1>
__host__ __device__ constexpr int epi_bytes() {
  return Traits<MODE>::nt_outer ? kStgBytes
         : MODE == kDH          ? 4 * kDhWarpBytes
         : MODE == kUp          ? 4 * kUpWarpBytes
         : Traits<MODE>::varlen_k ? epi_warps<MODE, MB>() * kDwWarpBytes
                                  : 0;
}

struct Tile {
  int e, m0, n0, row0, row_end, kblocks;
  bool w2;  // weight gradients: a dW2 tile (gathered B, TMA-loaded A) rather than a dW1 tile
};

// Pairs of one expert's weight-gradient tiles: dW1 pairs along M (they share the dH tile), dW2 pairs along N
// (they share the s*A tile).
template <int BN, int MB>
__device__ __forceinline__ int dw_pairs(int Mdim, int Ndim, bool w2) {
  const int m_tiles = Mdim / (kBM * MB), n_tiles = Ndim / BN;
  return w2 ? m_tiles * ((n_tiles + 1) / 2) : ((m_tiles + 1) / 2) * n_tiles;
}

// Largest e in [0, E) with tile_offsets[e] <= mt.
__device__ __forceinline__ int find_expert(const int32_t *__restrict__ tile_offsets, int E, int mt) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(&tile_offsets[mid]) <= mt) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Number of work items (pairs of tiles; CTA 2i + rank takes tile `rank` of pair i, i + grid/2, ...).
template <int MODE, int BN, int MB>
__device__ __forceinline__ int total_pairs(const GemmArgs &a, int total_m) {
  const int n_tiles = a.Ndim / BN;
  const int m_tiles = a.Mdim / (kBM * MB);
  if (MODE == kDW1) return a.E * ((m_tiles + 1) / 2) * n_tiles;  // pairs along M
  if (MODE == kDW2) return a.E * m_tiles * ((n_tiles + 1) / 2);  // pairs along N
  if (MODE == kDW) return a.E * (dw_pairs<BN, MB>(a.d, 2 * a.n, false) + dw_pairs<BN, MB>(a.n, a.d, true));
  return ((total_m + 1) / 2) * n_tiles;                           // pairs of consecutive m-tiles
}

// poff: CTA pairs only, the per-expert prefix of 256-row pair tiles (shared memory), else null.
template <int MODE, int BN, int MB>
__device__ __forceinline__ Tile decode_tile(const GemmArgs &a, int pair, int rank, int total_m,
                                            const int32_t *poff = nullptr) {
  Tile t;
  const int n_tiles = a.Ndim / BN;
  t.w2 = false;
  if (Traits<MODE>::varlen_k) {
    bool w2 = MODE == kDW2;
    int Md = a.Mdim, Nd = a.Ndim, rem;
    if (MODE == kDW) {
      // all dW1 pairs (expert by expert), then all dW2 pairs: the gathered rows in flight come from X, then
      // from dO, rather than from both at once
      const int p1 = dw_pairs<BN, MB>(a.d, 2 * a.n, false);
      w2 = pair >= a.E * p1;
      if (w2) {
        const int p2 = dw_pairs<BN, MB>(a.n, a.d, true);
        const int q = pair - a.E * p1;
        t.e = q / p2;
        rem = q - t.e * p2;
        Md = a.n;
        Nd = a.d;
      } else {
        t.e = pair / p1;
        rem = pair - t.e * p1;
        Md = a.d;
        Nd = 2 * a.n;
      }
    } else {
      const int per_e = dw_pairs<BN, MB>(Md, Nd, w2);
      t.e = pair / per_e;
      rem = pair - t.e * per_e;
    }
    t.w2 = w2;
    const int m_tiles = Md / (kBM * MB), nt_count = Nd / BN;
    int mt, nt;
    if (!w2) {
      mt = min(2 * (rem / nt_count) + rank, m_tiles - 1);  // an odd last row pair computes its tile twice
      nt = rem % nt_count;
    } else {
      const int np = (nt_count + 1) / 2;
      mt = rem / np;
      nt = min(2 * (rem % np) + rank, nt_count - 1);  // an odd last column pair computes its tile twice
    }
    t.m0 = mt * kBM * MB;
    t.n0 = nt * BN;
    t.row0 = __ldg(&a.offsets[t.e]);
    t.row_end = __ldg(&a.offsets[t.e + 1]);
    if (t.row0 < 0 || t.row_end < t.row0 || t.row_end > a.p_cap) {
      set_status(a.status, MOE_ERR_BAD_METADATA);
      t.row_end = t.row0 = 0;
    }
    t.kblocks = (t.row_end - t.row0 + kBK - 1) / kBK;
  } else if (Traits<MODE>::pairable && poff != nullptr) {
    // CTA pairs: a work item is (256-row pair tile of one expert, column tile), passes of nt_group column tiles
    // as below.  CTA `rank` takes m-tile 2*lp + rank of the expert's pair tile lp; when the expert has an odd
    // number of m-tiles the last pair's second m-tile lies past its rows: that CTA loads whatever is there (zeros
    // past P_cap) for the pair's MMA and writes nothing.
    const int per_pass = poff[a.E] * a.nt_group;
    const int g = pair / per_pass;
    const int rem = pair - g * per_pass;
    const int mp = rem / a.nt_group;
    const int nt = g * a.nt_group + (rem - mp * a.nt_group);
    int lo = 0, hi = a.E;  // largest e with poff[e] <= mp
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (poff[mid] <= mp) lo = mid;
      else hi = mid;
    }
    t.e = lo;
    const int mt_local = 2 * (mp - poff[lo]) + rank;
    const int mt_e = __ldg(&a.tile_offsets[lo + 1]) - __ldg(&a.tile_offsets[lo]);
    t.m0 = 0;
    t.n0 = a.n_off + nt * BN;
    t.row0 = __ldg(&a.offsets[lo]) + mt_local * kBM;
    t.row_end = __ldg(&a.offsets[lo + 1]);
    t.kblocks = a.Kdim / kBK;
    if (mt_local < mt_e && (t.row0 < 0 || t.row_end > a.p_cap || t.row0 >= t.row_end)) {
      set_status(a.status, MOE_ERR_BAD_METADATA);
      t.row_end = t.row0;  // nothing is written
    }
  } else {
    const int n_pairs_m = (total_m + 1) / 2;
    int mp, nt;
    if (Traits<MODE>::nt_outer) {
      // passes over all m-tile pairs, nt_group column tiles per pass (neighbours share the A tile in L2)
      const int per_pass = n_pairs_m * a.nt_group;
      const int g = pair / per_pass;
      const int rem = pair - g * per_pass;
      mp = rem / a.nt_group;
      nt = g * a.nt_group + (rem - mp * a.nt_group);
    } else {
      mp = pair / n_tiles;
      nt = pair - mp * n_tiles;
    }
    const int mt = 2 * mp + rank;
    t.e = find_expert(a.tile_offsets, a.E, mt);
    t.m0 = 0;
    t.n0 = a.n_off + nt * BN;  // n_off: first output column of this launch
    // a missing last tile (odd tile count) runs on rows past the last expert: zero operands, no output
    t.row0 = __ldg(&a.offsets[t.e]) + (mt - __ldg(&a.tile_offsets[t.e])) * kBM;
    t.row_end = __ldg(&a.offsets[t.e + 1]);
    t.kblocks = a.Kdim / kBK;  // every tile runs the full k-loop so both CTAs stay in step
    if (mt < total_m && (t.row0 < 0 || t.row_end > a.p_cap || t.row0 >= t.row_end)) {
      set_status(a.status, MOE_ERR_BAD_METADATA);
      t.row_end = t.row0;  // nothing is written
    }
  }
  return t;
}

// The tiles of one CTA, decoded once after the grid-dependency wait: finding a tile's expert and rows is a chain
// of dependent loads (a search over the tile offsets, or the expert's row offsets), and done per tile in every
// role it stalls the MMA issuer at each tile start (about 0.5 us, more than a k-block of MMA).
constexpr int kTileCache = 128;  // tiles per CTA kept in shared memory; later tiles are decoded on the fly
struct TileRec {
  int row0, row_end;
  uint32_t code;  // expert (bits 0-10) | n-tile (bits 11-18) | m-tile (bits 19-30) | dW2 tile (bit 31)
};
template <int MODE>
__host__ __device__ constexpr int tile_cache_bytes() {
  return kTileCache * static_cast<int>(sizeof(TileRec));
}

// The packing above holds every tile of a launch when its column tiles number at most 256 (and hence its
// m-tiles at most 4096); E <= 1024 always fits.
template <int BN>
__device__ __forceinline__ bool tiles_cacheable(const GemmArgs &a) {
  return max(a.d, 2 * a.n) / BN < 256;
}

template <int BN, int MB>
__device__ __forceinline__ TileRec pack_tile(const Tile &t) {
  return TileRec{t.row0, t.row_end,
                 static_cast<uint32_t>(t.e) | (static_cast<uint32_t>(t.n0 / BN) << 11) |
                     (static_cast<uint32_t>(t.m0 / (kBM * MB)) << 19) | (t.w2 ? 0x80000000u : 0u)};
}

// Tile i of this CTA (pair = first_pair + i * pair_step): from the cache when it holds it.
template <int MODE, int BN, int MB>
__device__ __forceinline__ Tile tile_at(const GemmArgs &a, const TileRec *cache, bool cached, int i, int pair,
                                        int rank, int total_m, const int32_t *poff) {
  if (!cached || i >= kTileCache) return decode_tile<MODE, BN, MB>(a, pair, rank, total_m, poff);
  const TileRec r = cache[i];
  Tile t;
  t.e = static_cast<int>(r.code & 0x7ffu);
  t.n0 = static_cast<int>((r.code >> 11) & 0xffu) * BN;
  t.m0 = static_cast<int>((r.code >> 19) & 0xfffu) * (kBM * MB);
  t.w2 = (r.code >> 31) != 0u;
  t.row0 = r.row0;
  t.row_end = r.row_end;
  t.kblocks = Traits<MODE>::varlen_k ? (t.row_end - t.row0 + kBK - 1) / kBK : a.Kdim / kBK;
  return t;
}

// Token id of row r, or an out-of-range row (zero fill) when r is past the expert or the id is invalid.
__device__ __forceinline__ int token_or_oob(const GemmArgs &a, int r, int row_end) {
  if (r >= row_end) return a.T;
  const int t = __ldg(&a.row_token[r]);
  return (t >= 0 && t < a.T) ? t : a.T;
}

// Deterministic aggregation: a row's contribution enters the accumulator as a 64-bit fixed-point integer with
// 32 fractional bits, so the sum is the same whatever order the reduce-adds land in.  One contribution may not
// exceed 2^21 in magnitude (a token has at most 1024 rows, so no sum leaves the +-2^31 range).
constexpr float kFixScale = 4294967296.0f;  // 2^32
constexpr float kFixLimit = 2097152.0f;     // 2^21

__device__ __forceinline__ long long to_fixed(float x, bool &range_ok) {
  if (!(fabsf(x) < kFixLimit)) {  // also catches NaN
    range_ok = false;
    return 0;
  }
  return __float2ll_rn(x * kFixScale);
}

// CG: CTAs per MMA (2: this CTA and its cluster peer; see the CTA-pair helpers in common.cuh).
template <int MODE, int BN, int STAGES, int MB, bool DET, int CG>
__global__ void __launch_bounds__(cta_threads<MODE, MB>(), 1)
    moe_gemm_kernel(const __grid_constant__ TensorMaps tm, const GemmArgs a) {
  const CUtensorMap &tmA = tm.a;
  const CUtensorMap &tmB = tm.b;
  using TR = Traits<MODE>;
  using SM = Smem<BN, STAGES, epi_bytes<MODE, MB>(), MB, tile_cache_bytes<MODE>(), CG>;
  static_assert(MODE != kDW || MB == 2, "merged weight gradients: 256-row blocks");
  static_assert(CG == 1 || (CG == 2 && Traits<MODE>::pairable && MB == 1), "CTA pairs: the TMA-fed scatter-add GEMMs");
  constexpr int kEpiWarps = epi_warps<MODE, MB>();
  static_assert(cta_threads<MODE, MB>() <= 448, "one CTA per SM at up to 146 registers a thread");
  // TMEM accumulator buffers: two (one tile's epilogue overlaps the next tile's MMAs) whenever two fit in the
  // 512 columns; 256-row blocks of 256 columns fill TMEM with one
  constexpr int kBufs = MB * BN * 2 <= 512 ? 2 : 1;
  constexpr uint32_t kBufCols = MB * BN;  // columns of one accumulator (M block mb at columns mb * BN)
  constexpr uint32_t kTmemCols = kBufCols * kBufs < 32 ? 32 : kBufCols * kBufs;
  static_assert(kBufCols * kBufs <= 512, "the accumulators fit TMEM");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + STAGES * SM::kABytesMB;
  const uint32_t bar = base + SM::kBarOff;
  auto full_bar = [&](int s) { return bar + 8u * s; };
  auto empty_bar = [&](int s) { return bar + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar + 8u * (2 * STAGES + 4);
  auto hin_bar = [&](int w, int b) { return bar + 8u * (2 * STAGES + 6 + 2 * w + b); };  // dH epilogue
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + SM::kBarOff + 8 * (2 * STAGES + 5));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + SM::kBarOff + 8 * (2 * STAGES + 5) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), TR::producers ? 1 + kGatherThreads : 1);
      mbar_init(empty_bar(s), 1);  // released by this CTA's MMA issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), CG * kEpiWarps);  // a pair's leader counts both CTAs' epilogue warps
    }
    mbar_init(drain_bar, 1);
    if (MODE == kDH)
      for (int i = 0; i < 8; ++i) mbar_init(hin_bar(i >> 1, i & 1), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (MODE == kDH || MODE == kUp || TR::varlen_k) {
      if (MODE == kDH) tma_prefetch_desc(&tm.h);
      tma_prefetch_desc(&tm.dh);
      tma_prefetch_desc(&tm.sa);
    }
  }
  if (warp == 1) {
    if (CG == 2) {  // collective over the pair: the same columns in both CTAs
      tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();  // barriers initialised and the TMEM address published before any role starts
  if (CG == 2) cluster_sync();  // the peer's barriers too: its loads and arrivals may target the leader's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything above overlaps the previous kernel's tail; its outputs are read only after this wait
  griddep_wait();
  griddep_launch_dependents();

  const int rank = static_cast<int>(blockIdx.x & 1u);
  const int first_pair = static_cast<int>(blockIdx.x >> 1);
  const int pair_step = static_cast<int>(gridDim.x >> 1);  // the grid is even
  const int total_m = TR::varlen_k ? 0 : __ldg(&a.tile_offsets[a.E]);
  const int32_t *poff = nullptr;
  if (CG == 2) {
    // per-expert prefix of 256-row pair tiles, ceil(m-tiles / 2) per expert: each thread scans a run of experts,
    // then the runs are offset by a block-wide exclusive scan of their sums
    int32_t *ps = reinterpret_cast<int32_t *>(gbase + SM::kPairOff);
    int32_t *wsum = ps + kMaxExperts + 1;  // one total per warp
    const int per = (a.E + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
    const int e0 = min(a.E, static_cast<int>(threadIdx.x) * per), e1 = min(a.E, e0 + per);
    auto pairs_of = [&](int e) { return (__ldg(&a.tile_offsets[e + 1]) - __ldg(&a.tile_offsets[e]) + 1) >> 1; };
    int sum = 0;
    for (int e = e0; e < e1; ++e) sum += pairs_of(e);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int nw = static_cast<int>(blockDim.x) >> 5;
      const int v = lane < nw ? wsum[lane] : 0;
      int inc2 = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc2, o);
        if (lane >= o) inc2 += u;
      }
      if (lane < nw) wsum[lane] = inc2 - v;
    }
    __syncthreads();
    int run = wsum[warp] + incl - sum;
    for (int e = e0; e < e1; ++e) {
      ps[e] = run;
      run += pairs_of(e);
    }
    if (e0 < e1 && e1 == a.E) ps[a.E] = run;
    __syncthreads();
    poff = ps;
  }
  const int total = CG == 2 ? poff[a.E] * (a.Ndim / BN) : total_pairs<MODE, BN, MB>(a, total_m);
  TileRec *tile_cache = reinterpret_cast<TileRec *>(gbase + SM::kCacheOff);
  const bool cached = tiles_cacheable<BN>(a);
  if (cached) {
    const int mine = first_pair < total ? (total - first_pair + pair_step - 1) / pair_step : 0;
    for (int i = threadIdx.x; i < min(mine, kTileCache); i += blockDim.x)
      tile_cache[i] = pack_tile<BN, MB>(decode_tile<MODE, BN, MB>(a, first_pair + i * pair_step, rank, total_m, poff));
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------------------------ TMA producer
    // weights: reused by the m-tiles of one expert, which run close together -> normal priority;
    // the dense activation operand of the scatter-add GEMMs streams through once per column slab -> first
    const uint64_t pol_w = TR::gather ? policy_evict_first() : policy_evict_normal();
    const uint64_t pol_x = TR::nt_outer ? policy_evict_first() : policy_evict_normal();
    constexpr uint32_t kTmaBytes = MODE == kUp ? SM::kBBytes
                                   : MODE == kDH ? SM::kBBytes
                                   : MODE == kDW1 ? SM::kBBytes
                                   : MODE == kDW2 ? SM::kABytesMB
                                   : MODE == kDW ? SM::kBBytes
                                   : MODE == kDownH ? SM::kBBytes
                                                  : SM::kStageBytes;
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    bool aborted = false;
    if (lane == 0) {
      for (int pair = first_pair, ti = 0; pair < total && !aborted; pair += pair_step, ++ti) {
        const Tile t = tile_at<MODE, BN, MB>(a, tile_cache, cached, ti, pair, rank, total_m, poff);
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u) || *abort_flag) {
            set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            aborted = true;
            break;
          }
          // merged weight gradients: a dW2 tile loads its A (s*A, 256 rows) by TMA, a dW1 tile its B (dH).
          // CTA pairs: both CTAs' loads complete on the leader's barrier, which expects both
          if (CG == 1 || rank == 0)
            mbar_arrive_expect_tx(full_bar(s),
                                  (MODE == kDW && t.w2) ? static_cast<uint32_t>(SM::kABytesMB) : CG * kTmaBytes);
          const uint32_t a_dst = sA + s * SM::kABytesMB;
          const uint32_t b_dst = sB + s * SM::kBBytes;
          const uint32_t fb = full_bar(s);
          // one request per operand: the tensor maps' boxes span the whole stage tile
          if (CG == 2) {
            // this CTA's 128 rows of A and its half of the BN columns of B
            const uint32_t lead = mapa_shared(fb, 0);
            tma_load_2d_pair(a_dst, &tmA, kb * kBK, t.row0, lead, pol_x);
            if (MODE == kDown)  // W2_e rows [kb*64, +64), columns [n0 + rank*BN/2, +BN/2): BN/128 chunks
              tma_load_3d_pair(b_dst, &tmB, 0, t.e * a.n + kb * kBK, t.n0 / 64 + rank * (BN / 128), lead, pol_w);
            else  // a {64, BN/2} box of W1_e rows
              tma_load_2d_pair(b_dst, &tmB, kb * kBK, t.e * a.d + t.n0 + rank * (BN / 2), lead, pol_w);
          } else if (MODE == kUp) {
            // W1_e rows [kb*64, +64): gate columns [n0/2, +128) and up columns [n + n0/2, +128), as the
            // chunks (gate 0, gate 1, up 0, up 1) of a {64, 64, 2, 2} box
            const int wrow = t.e * a.d + kb * kBK;
            tma_load_4d(b_dst, &tmB, 0, wrow, t.n0 / 128, 0, fb, pol_w);
          } else if (MODE == kDH) {
            // K-major W2_e: N index = rows n0..n0+BN of W2_e (a {64, BN} box), K-elements [kb*64, +64)
            tma_load_2d(b_dst, &tmB, kb * kBK, t.e * a.n + t.n0, fb, pol_w);
          } else if (MODE == kDown || MODE == kDownH) {
            if (MODE == kDown) tma_load_2d(a_dst, &tmA, kb * kBK, t.row0, fb, pol_x);
            // W2_e rows [kb*64, +64), columns [n0, +BN) as BN/64 chunks of a {64, 64, BN/64} box
            tma_load_3d(b_dst, &tmB, 0, t.e * a.n + kb * kBK, t.n0 / 64, fb, pol_w);
          } else if (MODE == kDX) {
            tma_load_2d(a_dst, &tmA, kb * kBK, t.row0, fb, pol_x);
            tma_load_2d(b_dst, &tmB, kb * kBK, t.e * a.d + t.n0, fb, pol_w);  // a {64, 256} box of W1_e rows
          } else if (MODE == kDW1 || (MODE == kDW && !t.w2)) {
            // B = dH rows [rb, rb+64) (MN-major), columns [n0, +BN); rows past the expert meet zero A rows
            tma_load_3d(b_dst, &tmB, 0, t.row0 + kb * kBK, t.n0 / 64, fb, pol_w);
          } else {
            // kDW2: A = (s*A) rows [rb, rb+64) (MN-major), columns [m0, +MB*128); rows past the expert meet
            // zero B rows
            tma_load_3d(a_dst, &tmA, 0, t.row0 + kb * kBK, t.m0 / 64, fb, pol_w);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (CG == 2 && !aborted) {
        // the leader's last releases of this CTA's stages are arrivals from another SM: they land before the
        // CTA may exit
        for (int st = 0; st < STAGES && st < issued; ++st) {
          const int last = st + ((issued - 1 - st) / STAGES) * STAGES;
          mbar_wait(empty_bar(st), static_cast<uint32_t>((last / STAGES) & 1));
        }
      }
      if (aborted && (CG == 1 || rank == 0)) {
        // let every copy this CTA issued land before the CTA's shared memory is released (a pair's copies land
        // on the leader's barriers: the leader drains both, and the pair's closing cluster barrier holds the peer)
        for (int st = 0; st < STAGES && st < issued; ++st) {
          const int last = st + ((issued - 1 - st) / STAGES) * STAGES;
          mbar_wait(full_bar(st), static_cast<uint32_t>((last / STAGES) & 1));
        }
      }
    }
  } else if (TR::gather && warp >= 6 && warp < 10) {
    // --------------------------------------------------------------- cp.async token-row gatherers
    const int gt = threadIdx.x - 192;  // 0..127
    const int j = gt & 7;              // 16-byte piece of a 128-byte row segment
    const int rsub = gt >> 3;          // 0..15
    const uint32_t swz = static_cast<uint32_t>((j ^ (rsub & 7)) << 4);
    const uint8_t *src_a = static_cast<const uint8_t *>(a.gsrc);
    const uint8_t *src_b = static_cast<const uint8_t *>(MODE == kDW ? a.gsrc2 : a.gsrc);
    const size_t ld_bytes = static_cast<size_t>(a.gld) * 2;
    // token rows (X or dO) are gathered about K times each: keep them in L2 ahead of the streamed weights
    const uint64_t pol_rows = policy_evict_last();
    int s = 0;
    uint32_t ph = 0;
    bool aborted = false;
    // token ids of the next tile are fetched while the current tile's rows are copied
    int tok_next[8];
    auto fetch_tokens = [&](const Tile &tt) {
#pragma unroll
      for (int q = 0; q < 8; ++q) tok_next[q] = token_or_oob(a, tt.row0 + rsub + 16 * q, tt.row_end);
    };
    Tile t_next;
    if (TR::gather_a_k && first_pair < total) {
      t_next = tile_at<MODE, BN, MB>(a, tile_cache, cached, 0, first_pair, rank, total_m, poff);
      fetch_tokens(t_next);
    }
    for (int pair = first_pair, ti = 0; pair < total && !aborted; pair += pair_step, ++ti) {
      const Tile t = TR::gather_a_k ? t_next : tile_at<MODE, BN, MB>(a, tile_cache, cached, ti, pair, rank, total_m, poff);
      if (t.kblocks == 0) continue;
      const uint8_t *rowp[8];
      uint32_t rown[8];
      if (TR::gather_a_k) {
        // this thread copies piece j of rows rsub + 16q (q = 0..7) of the 128-row tile at every k-block
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int tok = tok_next[q];
          rown[q] = tok < a.T ? 16u : 0u;
          rowp[q] = src_a + (tok < a.T ? tok : 0) * ld_bytes + j * 16;
        }
        if (pair + pair_step < total) {
          t_next = tile_at<MODE, BN, MB>(a, tile_cache, cached, ti + 1, pair + pair_step, rank, total_m, poff);
          fetch_tokens(t_next);
        }
      }
      // weight gradients: dW1 tiles gather X into A, dW2 tiles gather dO into B
      const bool into_a = TR::gather_a_mn || (MODE == kDW && !t.w2);
      const uint8_t *src_base = (MODE == kDW && t.w2) ? src_b : src_a;
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!TR::gather_a_k) {
          // varlen-K: rows rb + rsub + 16q (q = 0..3) of this k-block, by token id
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int tok = token_or_oob(a, t.row0 + kb * kBK + rsub + 16 * q, t.row_end);
            rown[q] = tok < a.T ? 16u : 0u;
            rowp[q] = src_base + (tok < a.T ? tok : 0) * ld_bytes + j * 16;
          }
          // the next k-block's ids (256 bytes: at most three lines) into L1 while this one's copies are issued;
          // loading them into registers one k-block ahead measured slower (fine7b dW 373 -> 595 us before the
          // stage wait, 362 -> 381 us after the copies), this prefetch faster (362 -> 357 us)
          if (gt < 3 && kb + 1 < t.kblocks)
            prefetch_l1(a.row_token + min(t.row0 + (kb + 1) * kBK + gt * 31, t.row_end - 1));
        }
        if (!mbar_wait(empty_bar(s), ph ^ 1u) || *abort_flag) {
          set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
          *abort_flag = 1;
          aborted = true;
          break;
        }
        if (TR::gather_a_k) {
          const uint32_t dst = sA + s * SM::kABytesMB + rsub * 128 + swz;
          const size_t koff = static_cast<size_t>(kb) * kBK * 2;
#pragma unroll
          for (int q = 0; q < 8; ++q) cp_async_16_hint(dst + q * 2048, rowp[q] + koff, rown[q], pol_rows);
        } else {
          // MN-major: K-row k = rsub + 16q at byte k*128 of each 64-column chunk c (8 KB apart)
          constexpr int kChunksA = MB * kBM / 64, kChunksB = BN / 64;
          constexpr int kChunks = TR::gather_a_mn ? kChunksA : TR::gather_b_mn ? kChunksB
                                                                : (kChunksA > kChunksB ? kChunksA : kChunksB);
          const int nchunks = into_a ? kChunksA : kChunksB;  // kDW: the gathered operand of this tile
          const uint32_t base_dst = (into_a ? sA + s * SM::kABytesMB : sB + s * SM::kBBytes) + rsub * 128 + swz;
          const int mn0 = into_a ? t.m0 : t.n0;
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              if (c < nchunks)
                cp_async_16_hint(base_dst + q * 2048 + c * 8192, rowp[q] + static_cast<size_t>(mn0 + c * 64) * 2,
                                 rown[q], pol_rows);
        }
        // the stage's barrier counts this thread's arrival when its copies have landed; the MMA issuer
        // fences the async proxy after the barrier before the tensor cores read the stage
        cp_async_arrive_noinc(full_bar(s));
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    cp_async_wait<0>();
  } else if (TR::transform_a && warp >= 6 && warp < 10) {
    // ------------------------------------------------------- A = SwiGLU(H) producers (down-projection)
    // Thread gt takes 16-byte piece j (eight columns) of rows rsub + 16q (q = 0..7) of the 128-row A tile at
    // every k-block: it loads those columns of the cached gate and up halves of H, forms SiLU(g) * u in fp32,
    // rounds to bf16 and writes the piece at its 128-byte-swizzled place in the stage, as a TMA load would.
    const int gt = threadIdx.x - 192;
    const int j = gt & 7;
    const int rsub = gt >> 3;
    const uint32_t swz = static_cast<uint32_t>((j ^ (rsub & 7)) << 4);
    const uint8_t *hbase = static_cast<const uint8_t *>(a.Hin);
    const size_t hld = static_cast<size_t>(2 * a.n) * 2;  // bytes per row of H
    int s = 0;
    uint32_t ph = 0;
    bool aborted = false;
    // the 128-byte gate and up segments of a row's next k-block go to L2 ahead of their loads (one thread per row)
    auto prefetch_kblock = [&](const Tile &tt, int kb) {
      if (j != 0) return;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int r = tt.row0 + rsub + 16 * q;
        if (r < tt.row_end) {
          const uint8_t *hp = hbase + static_cast<size_t>(r) * hld + static_cast<size_t>(kb * kBK) * 2;
          prefetch_l2(hp);
          prefetch_l2(hp + static_cast<size_t>(a.n) * 2);
        }
      }
    };
    for (int pair = first_pair, ti = 0; pair < total && !aborted; pair += pair_step, ++ti) {
      const Tile t = tile_at<MODE, BN, MB>(a, tile_cache, cached, ti, pair, rank, total_m, poff);
      if (t.kblocks == 0) continue;
      for (int kb = 0; kb < t.kblocks; ++kb) {
        uint4 g[8], u[8];
        const size_t col = static_cast<size_t>(kb * kBK + j * 8) * 2;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int r = t.row0 + rsub + 16 * q;
          if (r < t.row_end) {  // rows past the expert are never read (they may lie past the end of H)
            const uint8_t *hp = hbase + static_cast<size_t>(r) * hld + col;
            g[q] = __ldcg(reinterpret_cast<const uint4 *>(hp));
            u[q] = __ldcg(reinterpret_cast<const uint4 *>(hp + static_cast<size_t>(a.n) * 2));
          } else {
            g[q] = make_uint4(0u, 0u, 0u, 0u);
            u[q] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        if (kb + 1 < t.kblocks) prefetch_kblock(t, kb + 1);
        if (!mbar_wait(empty_bar(s), ph ^ 1u) || *abort_flag) {
          set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
          *abort_flag = 1;
          aborted = true;
          break;
        }
        const uint32_t dst = sA + s * SM::kABytesMB + rsub * 128 + swz;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t gw[4] = {g[q].x, g[q].y, g[q].z, g[q].w};
          const uint32_t uw[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
          float o[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            o[2 * i] = silu_tanh(bf16_lo(gw[i])) * bf16_lo(uw[i]);
            o[2 * i + 1] = silu_tanh(bf16_hi(gw[i])) * bf16_hi(uw[i]);
          }
          st_shared_v4(dst + q * 2048, __uint_as_float(pack_bf16x2(o[0], o[1])), __uint_as_float(pack_bf16x2(o[2], o[3])),
                       __uint_as_float(pack_bf16x2(o[4], o[5])), __uint_as_float(pack_bf16x2(o[6], o[7])));
        }
        fence_proxy_async_smem();  // these generic-proxy writes are read by the tensor cores (async proxy)
        mbar_arrive(full_bar(s));
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------------------------- MMA issuer
    // (CTA pairs: the leader issues the pair's M = 256 MMAs and commits to both CTAs' barriers)
    if (lane == 0 && (CG == 1 || rank == 0)) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM * CG, BN, TR::a_mn, TR::b_mn);
      int s = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t bph = 0;
      bool aborted = false;
      for (int pair = first_pair, ti = 0; pair < total && !aborted; pair += pair_step, ++ti) {
        const Tile t = tile_at<MODE, BN, MB>(a, tile_cache, cached, ti, pair, rank, total_m, poff);
        if (t.kblocks == 0) continue;
        // CTA pairs: both barriers also receive the peer's arrivals (cluster-scope acquire)
        if (!(CG == 2 ? mbar_wait_cluster(tempty_bar(buf), bph ^ 1u) : mbar_wait(tempty_bar(buf), bph ^ 1u)) ||
            *abort_flag) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * kBufCols;
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if (!(CG == 2 ? mbar_wait_cluster(full_bar(s), ph) : mbar_wait(full_bar(s), ph)) || *abort_flag) {
            aborted = true;
            break;
          }
          if (TR::producers) fence_proxy_async_smem();  // generic-proxy writes (cp.async, st.shared) -> tensor-core reads
          tc_fence_after();
          const uint32_t a_st = sA + s * SM::kABytesMB;
          const uint32_t b_st = sB + s * SM::kBBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t bd = TR::b_mn ? smem_desc_sw128(b_st + k * 2048, 8192, 1024)
                                         : smem_desc_sw128(b_st + k * 32, 16, 1024);
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
              const uint32_t a_blk = a_st + mb * kABytes;
              const uint64_t ad = TR::a_mn ? smem_desc_sw128(a_blk + k * 2048, 8192, 1024)
                                           : smem_desc_sw128(a_blk + k * 32, 16, 1024);
              if (CG == 2) umma_bf16_pair(d_tmem + mb * BN, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
              else umma_bf16(d_tmem + mb * BN, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          // the stage is free once these MMAs have read it
          if (CG == 2) {
            umma_commit_pair(empty_bar(s));
            umma_commit_pair(mapa_shared(empty_bar(s), 1));
          } else {
            umma_commit(empty_bar(s));
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (aborted) break;
        if (CG == 2) {
          umma_commit_pair(tfull_bar(buf));
          umma_commit_pair(mapa_shared(tfull_bar(buf), 1));
        } else {
          umma_commit(tfull_bar(buf));
        }
        if (++buf == kBufs) {
          buf = 0;
          bph ^= 1u;
        }
      }
      if (aborted) {
        set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else if (TR::producers ? ((warp >= 2 && warp < 6) || (kEpiWarps == 8 && warp >= 10 && warp < 14))
                        : (warp >= 2 && warp < 2 + kEpiWarps)) {
    // ---------------------------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // weight gradients with eight epilogue warps: warps 2..5 drain M block 0, warps 10..13 M block 1
    const int mb_lo = (TR::varlen_k && kEpiWarps == 8 && warp >= 10) ? 1 : 0;
    const int mb_hi = (TR::varlen_k && kEpiWarps == 8) ? mb_lo + 1 : MB;
    const int row = q * 32 + lane;
    int buf = 0;
    uint32_t bph = 0;
    uint32_t hin_par = 0u;                       // dH epilogue: bit b = parity of H buffer b's next fill
    bool h_pre = false;  // dH epilogue: the tile's first chunk of H was requested at the end of the previous tile
    const int p_rows = MODE == kDH ? __ldg(&a.offsets[a.E]) : 0;  // dH: rows routed in total
    const uint64_t pol_acc = policy_evict_last();  // keep the fp32 accumulator slab in L2
    const uint64_t pol_stream = policy_evict_first();  // streamed epilogue traffic (H, A, dH, s*A) is touched once here
    for (int pair = first_pair, ti = 0; pair < total; pair += pair_step, ++ti) {
      const Tile t = tile_at<MODE, BN, MB>(a, tile_cache, cached, ti, pair, rank, total_m, poff);
      // weight gradients: the output of this tile and its row length
      const int dw_m = MODE == kDW ? (t.w2 ? a.n : a.d) : a.Mdim;
      const int dw_n = MODE == kDW ? (t.w2 ? a.d : 2 * a.n) : a.Ndim;
      uint8_t *dw_out = static_cast<uint8_t *>((MODE == kDW && t.w2) ? a.out1 : a.out0);
      if (t.kblocks == 0) {
        if (TR::varlen_k) {  // an expert without rows has an exactly zero weight gradient
          for (int mb = mb_lo; mb < mb_hi; ++mb) {
            uint8_t *dst = dw_out + (((size_t)t.e * dw_m + t.m0 + mb * kBM + row) * dw_n + t.n0) * 2;
            for (int c = 0; c < BN * 2; c += 16) st_v4(dst + c, 0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      // scatter-add GEMMs: the row's token and score are read before the accumulator wait (their latency
      // overlaps it)
      constexpr bool kScatter = (MODE == kDown || MODE == kDX || MODE == kDownH);
      int tok = -1;
      float sc = 1.f;
      if (kScatter && t.row0 + row < t.row_end) {
        tok = __ldg(&a.row_token[t.row0 + row]);
        if (MODE != kDX) sc = __ldg(&a.row_score[t.row0 + row]);
      }
      const float dh_sc = (MODE == kDH && t.row0 + row < t.row_end) ? __ldg(&a.row_score[t.row0 + row]) : 0.f;
      bool released = false;  // TMEM handed back to the MMA issuer before the end of the tile
      int ok = 1;
      if (lane == 0) ok = mbar_wait(tfull_bar(buf), bph) && !*abort_flag;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
          *abort_flag = 1;
          if (MODE == kDH && h_pre) mbar_wait(hin_bar(q, 0), hin_par & 1u);  // the requested H chunk lands first
        }
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf) * kBufCols;

      if (MODE == kUp) {
        const int r = t.row0 + row;
        const bool valid = r < t.row_end;
        const bool full_warp = t.row0 + q * 32 + 31 < t.row_end;  // all 32 rows belong to this expert
        const int wrow = t.row0 + q * 32;
        const int j0 = t.n0 / 2;
        const uint32_t out_st = base + SM::kStgOff + q * kUpWarpBytes;
        const int sw = (lane >> 1) & 3;  // 64-byte swizzle: piece p of row `lane` at piece p ^ ((lane >> 1) & 3)
        uint8_t *hrow = static_cast<uint8_t *>(a.out0) + (size_t)r * (2 * a.n) * 2;
        uint8_t *arow = static_cast<uint8_t *>(a.out1) + (size_t)r * a.n * 2;
        const bool store_a = a.out1 != nullptr;  // A is not kept when the down-projection recomputes it from H
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tacc + c * 32, g);
          tmem_ld32(tacc + BN / 2 + c * 32, u);
          tmem_ld_wait();
          uint32_t hg[16], hu[16], av[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            const float a0 = __fdividef(g0, 1.f + __expf(-g0)) * u0;
            const float a1 = __fdividef(g1, 1.f + __expf(-g1)) * u1;
            hg[i] = pack_bf16x2(g0, g1);
            hu[i] = pack_bf16x2(u0, u1);
            av[i] = pack_bf16x2(a0, a1);
          }
          const int j = j0 + c * 32;
          if (full_warp) {
            if (lane == 0) bulk_wait_read<0>();  // the previous chunk's stores have read the staging tile
            __syncwarp();
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const uint32_t o = lane * 64 + ((p ^ sw) << 4);
              st_shared_v4(out_st + o, __uint_as_float(hg[4 * p]), __uint_as_float(hg[4 * p + 1]),
                           __uint_as_float(hg[4 * p + 2]), __uint_as_float(hg[4 * p + 3]));
              st_shared_v4(out_st + 2048 + o, __uint_as_float(hu[4 * p]), __uint_as_float(hu[4 * p + 1]),
                           __uint_as_float(hu[4 * p + 2]), __uint_as_float(hu[4 * p + 3]));
              st_shared_v4(out_st + 4096 + o, __uint_as_float(av[4 * p]), __uint_as_float(av[4 * p + 1]),
                           __uint_as_float(av[4 * p + 2]), __uint_as_float(av[4 * p + 3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm.dh, out_st, j, wrow, pol_stream);
              tma_store_2d(&tm.dh, out_st + 2048, a.n + j, wrow, pol_stream);
              if (store_a) tma_store_2d(&tm.sa, out_st + 4096, j, wrow, pol_stream);
              bulk_commit();
            }
          } else if (valid) {
            // a warp whose rows run past the expert: per-row stores keep the next expert's rows intact
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              st_v4_hint(hrow + (size_t)j * 2 + v * 16, hg[4 * v], hg[4 * v + 1], hg[4 * v + 2], hg[4 * v + 3],
                         pol_stream);
              st_v4_hint(hrow + (size_t)(a.n + j) * 2 + v * 16, hu[4 * v], hu[4 * v + 1], hu[4 * v + 2], hu[4 * v + 3],
                         pol_stream);
              if (store_a)
                st_v4_hint(arow + (size_t)j * 2 + v * 16, av[4 * v], av[4 * v + 1], av[4 * v + 2], av[4 * v + 3],
                           pol_stream);
            }
          }
          __syncwarp();
        }
      } else if (kScatter) {
        if (t.row0 + row < t.row_end && (tok < 0 || tok >= a.T)) {
          set_status(a.status, MOE_ERR_BAD_METADATA);
          tok = -1;
        }
        // epilogue warp index 0..7: warps 2..9, or 2..5 and 10..13 beside the producer warps
        const int ew = (TR::producers && warp >= 10) ? warp - 6 : warp - 2;
        const int half = ew >> 2;  // which half of the BN columns this warp drains
        const uint32_t stg = base + SM::kStgOff + (ew * 32 + lane) * kStgRowBytes;
        if (DET) {
          // 32 columns per bulk add: 32 64-bit integers fill the 256-byte staging row
          long long *grow = a.out_i64 + (size_t)(tok >= 0 ? tok : 0) * a.d + t.n0 + half * (BN / 2);
          bool range_ok = true;
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {
            uint32_t v[32];
            tmem_ld32(tacc + half * (BN / 2) + c * 32, v);
            tmem_ld_wait();
            bulk_wait_read<0>();  // the previous bulk add has read the staging row
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const long long q0 = to_fixed(sc * __uint_as_float(v[2 * i]), range_ok);
              const long long q1 = to_fixed(sc * __uint_as_float(v[2 * i + 1]), range_ok);
              st_shared_v2_u64(stg + i * 16, static_cast<unsigned long long>(q0), static_cast<unsigned long long>(q1));
            }
            fence_proxy_async_smem();
            if (tok >= 0) bulk_reduce_add_u64(grow + c * 32, stg, 256, pol_acc);
            bulk_commit();
          }
          if (!range_ok && tok >= 0) set_status(a.status, MOE_ERR_RANGE);  // rows that are written
        } else {
          float *grow = a.out_f32 + (size_t)(tok >= 0 ? tok : 0) * a.d + t.n0 + half * (BN / 2);
          static_assert(!kScatter || BN == 256, "the scatter epilogue drains 128 columns per warp");
          if (MODE == kDownH) {
            // 448 threads leave no room for all 128 columns in registers: 64 columns per TMEM wait
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
              uint32_t v0[32], v1[32];
              const uint32_t col = half * (BN / 2) + c * 64;
              tmem_ld32(tacc + col, v0);
              tmem_ld32(tacc + col + 32, v1);
              tmem_ld_wait();
              bulk_wait_read<0>();  // the previous bulk add has read the staging row
#pragma unroll
              for (int i = 0; i < 8; ++i)
                st_shared_v4(stg + i * 16, sc * __uint_as_float(v0[4 * i]), sc * __uint_as_float(v0[4 * i + 1]),
                             sc * __uint_as_float(v0[4 * i + 2]), sc * __uint_as_float(v0[4 * i + 3]));
#pragma unroll
              for (int i = 0; i < 8; ++i)
                st_shared_v4(stg + 128 + i * 16, sc * __uint_as_float(v1[4 * i]), sc * __uint_as_float(v1[4 * i + 1]),
                             sc * __uint_as_float(v1[4 * i + 2]), sc * __uint_as_float(v1[4 * i + 3]));
              fence_proxy_async_smem();
              if (tok >= 0) bulk_reduce_add_f32(grow + c * 64, stg, 256, pol_acc);
              bulk_commit();
            }
          } else {
            // all 128 columns of this warp's half in one wait, then TMEM goes back to the MMA issuer while the two
            // 64-column reduce-adds go out through the staging row
            uint32_t v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tacc + half * (BN / 2) + c * 32, v[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (CG == 2 && rank != 0) mbar_arrive_remote(mapa_shared(tempty_bar(buf), 0));
              else mbar_arrive(tempty_bar(buf));
            }
            released = true;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              bulk_wait_read<0>();  // the previous bulk add has read the staging row
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  st_shared_v4(stg + h * 128 + i * 16, sc * __uint_as_float(v[2 * c + h][4 * i]),
                               sc * __uint_as_float(v[2 * c + h][4 * i + 1]), sc * __uint_as_float(v[2 * c + h][4 * i + 2]),
                               sc * __uint_as_float(v[2 * c + h][4 * i + 3]));
              fence_proxy_async_smem();
              if (tok >= 0) bulk_reduce_add_f32(grow + c * 64, stg, 256, pol_acc);
              bulk_commit();
            }
          }
        }
      } else if (MODE == kDH) {
        const int r = t.row0 + row;
        const bool valid = r < t.row_end;
        const bool full_warp = t.row0 + q * 32 + 31 < t.row_end;  // all 32 rows belong to this expert
        const float sc = dh_sc;
        // rows past the last expert (up to the end of its last tile) get zeros: the weight-gradient GEMMs read
        // them as the zero tail of that expert's last 64-row block
        const bool zero_row = !valid && t.row_end == p_rows && r < a.p_cap;
        const int wrow = t.row0 + q * 32;                          // first row of this warp's 32
        const uint32_t wbase = base + SM::kStgOff + q * kDhWarpBytes;
        const uint32_t out_st = wbase + 4096;                      // dH gate | dH up staging
        // 64-byte swizzle: 16-byte piece p of row `lane` sits at piece p ^ ((lane >> 1) & 3)
        const int sw = (lane >> 1) & 3;
        // chunk c (32 columns of the gate half and the same of the up half) of the H rows [wr, wr + 32) of a tile
        auto issue_h_at = [&](int n0, int wr, int c, int b) {
          const uint32_t hb = hin_bar(q, b);
          mbar_arrive_expect_tx(hb, 4096);
          tma_load_2d(wbase + b * 4096, &tm.h, n0 + c * 32, wr, hb, pol_stream);
          tma_load_2d(wbase + b * 4096 + 2048, &tm.h, a.n + n0 + c * 32, wr, hb, pol_stream);
        };
        auto issue_h = [&](int c, int b) { issue_h_at(t.n0, wrow, c, b); };
        if (lane == 0 && !h_pre) {
          fence_proxy_async_smem();  // the previous tile's reads of the buffer come before this refill
          issue_h(0, 0);
        }
        h_pre = false;
        uint8_t *dhrow = static_cast<uint8_t *>(a.out0) + (size_t)r * (2 * a.n) * 2;
        uint8_t *sarow = static_cast<uint8_t *>(a.out1) + (size_t)r * a.n * 2;
        float ds = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int b = 0;
          uint32_t v[32];
          tmem_ld32(tacc + c * 32, v);
          const bool got = mbar_wait(hin_bar(q, b), (hin_par >> b) & 1u);
          hin_par ^= 1u << b;
          if (!got) {
            set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
          }
          tmem_ld_wait();
          uint32_t hg[16], hu[16];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float4 g4 = ld_shared_v4(wbase + b * 4096 + lane * 64 + ((p ^ sw) << 4));
            const float4 u4 = ld_shared_v4(wbase + b * 4096 + 2048 + lane * 64 + ((p ^ sw) << 4));
            hg[4 * p] = __float_as_uint(g4.x);
            hg[4 * p + 1] = __float_as_uint(g4.y);
            hg[4 * p + 2] = __float_as_uint(g4.z);
            hg[4 * p + 3] = __float_as_uint(g4.w);
            hu[4 * p] = __float_as_uint(u4.x);
            hu[4 * p + 1] = __float_as_uint(u4.y);
            hu[4 * p + 2] = __float_as_uint(u4.z);
            hu[4 * p + 3] = __float_as_uint(u4.w);
          }
          __syncwarp();  // every lane has read this chunk of H: the buffer can be refilled
          if (c + 1 < BN / 32) {
            if (lane == 0) {
              fence_proxy_async_smem();  // the warp's generic-proxy reads are ordered before the TMA refill
              issue_h(c + 1, 0);
            }
          } else if (pair + pair_step < total) {
            // the next tile's first chunk, while this tile's last chunk is computed and stored
            if (lane == 0) {
              const Tile tn = tile_at<MODE, BN, MB>(a, tile_cache, cached, ti + 1, pair + pair_step, rank, total_m, poff);
              fence_proxy_async_smem();
              issue_h_at(tn.n0, tn.row0 + q * 32, 0, 0);
            }
            h_pre = true;
          }
          uint32_t dg[16], du[16], sa[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float o_g[2], o_u[2], o_a[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float gg = h ? bf16_hi(hg[i]) : bf16_lo(hg[i]);
              const float uu = h ? bf16_hi(hu[i]) : bf16_lo(hu[i]);
              const float dap = __uint_as_float(v[2 * i + h]);
              const float sig = __fdividef(1.f, 1.f + __expf(-gg));
              const float silu = gg * sig;
              const float act = silu * uu;
              ds += dap * act;
              const float da = sc * dap;
              o_g[h] = da * uu * sig * (1.f + gg * (1.f - sig));
              o_u[h] = da * silu;
              o_a[h] = sc * act;
            }
            dg[i] = pack_bf16x2(o_g[0], o_g[1]);
            du[i] = pack_bf16x2(o_u[0], o_u[1]);
            sa[i] = pack_bf16x2(o_a[0], o_a[1]);
          }
          const int j = t.n0 + c * 32;
          if (full_warp) {
            if (lane == 0) bulk_wait_read<0>();  // the previous chunk's stores have read the staging tile
            __syncwarp();
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const uint32_t o = lane * 64 + ((p ^ sw) << 4);
              st_shared_v4(out_st + o, __uint_as_float(dg[4 * p]), __uint_as_float(dg[4 * p + 1]),
                           __uint_as_float(dg[4 * p + 2]), __uint_as_float(dg[4 * p + 3]));
              st_shared_v4(out_st + 2048 + o, __uint_as_float(du[4 * p]), __uint_as_float(du[4 * p + 1]),
                           __uint_as_float(du[4 * p + 2]), __uint_as_float(du[4 * p + 3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm.dh, out_st, j, wrow, pol_stream);
              tma_store_2d(&tm.dh, out_st + 2048, a.n + j, wrow, pol_stream);
              bulk_commit();
              bulk_wait_read<0>();  // the dH gate tile has been read: s*A reuses its 2 KB
            }
            __syncwarp();
#pragma unroll
            for (int p = 0; p < 4; ++p)
              st_shared_v4(out_st + lane * 64 + ((p ^ sw) << 4), __uint_as_float(sa[4 * p]),
                           __uint_as_float(sa[4 * p + 1]), __uint_as_float(sa[4 * p + 2]), __uint_as_float(sa[4 * p + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm.sa, out_st, j, wrow, pol_stream);
              bulk_commit();
            }
          } else if (valid) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              st_v4(dhrow + (size_t)j * 2 + w * 16, dg[4 * w], dg[4 * w + 1], dg[4 * w + 2], dg[4 * w + 3]);
              st_v4(dhrow + (size_t)(a.n + j) * 2 + w * 16, du[4 * w], du[4 * w + 1], du[4 * w + 2], du[4 * w + 3]);
              st_v4(sarow + (size_t)j * 2 + w * 16, sa[4 * w], sa[4 * w + 1], sa[4 * w + 2], sa[4 * w + 3]);
            }
          } else if (zero_row) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              st_v4(dhrow + (size_t)j * 2 + w * 16, 0u, 0u, 0u, 0u);
              st_v4(dhrow + (size_t)(a.n + j) * 2 + w * 16, 0u, 0u, 0u, 0u);
              st_v4(sarow + (size_t)j * 2 + w * 16, 0u, 0u, 0u, 0u);
            }
          }
          __syncwarp();
        }
        if (valid) {
          // deterministic: one partial per column tile, summed in tile order afterwards
          if (DET) a.dS_part[(size_t)r * (a.Ndim / BN) + t.n0 / BN] = ds;
          else atomicAdd(&a.dS[r], ds);
        }
      } else {
        // weight gradients: bf16 rows of dW_e (M block mb sits in TMEM columns [mb * BN, (mb + 1) * BN)), stored
        // as 32 x 32 boxes of the [E * M, N] output view through two staging tiles per warp
        // Two 32-column chunks per TMEM wait, stored as two boxes from the warp's two staging tiles.
        const CUtensorMap *omap = (MODE == kDW && t.w2) ? &tm.sa : &tm.dh;
        const int ew = (warp >= 10) ? 4 + q : q;  // this warp's staging slot
        const uint32_t stg = base + SM::kStgOff + ew * kDwWarpBytes;
        const int sw = (lane >> 1) & 3;  // 64-byte swizzle
#pragma unroll 1
        for (int mb = mb_lo; mb < mb_hi; ++mb) {
#pragma unroll 1
          for (int c = 0; c < BN / 32; c += 2) {
            uint32_t v0[32], v1[32];
            tmem_ld32(tacc + mb * BN + c * 32, v0);
            tmem_ld32(tacc + mb * BN + (c + 1) * 32, v1);
            tmem_ld_wait();
            uint32_t p0[16], p1[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              p0[i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
              p1[i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
            }
            if (lane == 0) bulk_wait_read<0>();  // the previous pair of boxes has been read from both tiles
            __syncwarp();
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const uint32_t o = lane * 64 + ((w ^ sw) << 4);
              st_shared_v4(stg + o, __uint_as_float(p0[4 * w]), __uint_as_float(p0[4 * w + 1]),
                           __uint_as_float(p0[4 * w + 2]), __uint_as_float(p0[4 * w + 3]));
              st_shared_v4(stg + 2048 + o, __uint_as_float(p1[4 * w]), __uint_as_float(p1[4 * w + 1]),
                           __uint_as_float(p1[4 * w + 2]), __uint_as_float(p1[4 * w + 3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int orow = t.e * dw_m + t.m0 + mb * kBM + q * 32;
              tma_store_2d(omap, stg, t.n0 + c * 32, orow, policy_evict_first());
              tma_store_2d(omap, stg + 2048, t.n0 + (c + 1) * 32, orow, policy_evict_first());
              bulk_commit();
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !released) {
        if (CG == 2 && rank != 0) mbar_arrive_remote(mapa_shared(tempty_bar(buf), 0));  // the leader's MMAs wait
        else mbar_arrive(tempty_bar(buf));
      }
      if (++buf == kBufs) {
        buf = 0;
        bph ^= 1u;
      }
    }
    bulk_wait<0>();  // every bulk store / reduce-add of this thread has landed before the end
  }

  __syncthreads();
  if (warp == 1 && *abort_flag && lane == 0 && (CG == 1 || rank == 0)) {
    if (CG == 2) umma_commit_pair(drain_bar);
    else umma_commit(drain_bar);  // all MMAs this CTA issued are complete once this arrives
    mbar_wait(drain_bar, 0);
  }
  if (CG == 2) {  // neither CTA frees its TMEM (or exits) while the leader's MMAs may still write the peer's
    tc_fence_before();
    cluster_sync();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (CG == 2) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Host launcher for one instantiation: one CTA per SM, an even number of CTAs (CTA 2i + rank takes tile
// `rank` of each of its pairs).  The shared-memory attribute and the grid size are set up once per device.
template <int MODE, int BN, int STAGES, int MB = 1, bool DET = false, int CG = 1>
int launch_gemm(const GemmArgs &a, const TensorMaps &tm, cudaStream_t stream) {
  using SM = Smem<BN, STAGES, epi_bytes<MODE, MB>(), MB, tile_cache_bytes<MODE>(), CG>;
  auto kernel = moe_gemm_kernel<MODE, BN, STAGES, MB, DET, CG>;
  static DeviceCache grid_cache;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return record_cuda_error(err);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_DEVICE;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // CTA pairs: clusters of two
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.blockDim = dim3(cta_threads<MODE, MB>(), 1, 1);
  cfg.dynamicSmemBytes = SM::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = CG == 2 ? 2 : 1;
  const int grid = grid_cache.get(dev, [&]() -> int {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    if (e != cudaSuccess) return -static_cast<int>(e);
    if (CG == 2) {
      // persistent: exactly the pairs that can be resident at once (an SM left over in a GPC takes no pair)
      int clusters = 0;
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
      e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &q);
      if (e != cudaSuccess) return -static_cast<int>(e);
      if (clusters <= 0) return -static_cast<int>(cudaErrorInvalidConfiguration);
      return 2 * clusters;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, cta_threads<MODE, MB>(), SM::kBytes);
    if (e != cudaSuccess || per_sm <= 0) per_sm = 1;
    return 2 * ((num_sms() * per_sm) / 2);
  });
  if (grid <= 0) return record_cuda_error(static_cast<cudaError_t>(-grid));
  cfg.gridDim = dim3(grid, 1, 1);
  static const char *const kNames[] = {"gemm_up",  "gemm_down", "gemm_dh", "gemm_dx",
                                       "gemm_dw1", "gemm_dw2",  "gemm_dw", "gemm_down_h"};
  prof_begin(kNames[MODE], stream);
  err = cudaLaunchKernelEx(&cfg, kernel, tm, a);
  prof_end(stream);
  count_launch();
  if (err == cudaSuccess) err = cudaGetLastError();
  if (err != cudaSuccess) return record_cuda_error(err);
  return MOE_OK;
}

}  // namespace moe
