/*
 * moe.h - C ABI of the GB300 (sm_103a) fine-grained MoE expert layer (SonicMoE hot path).
 *
 * The layer, per token t with routed rows r (one row per (token, expert) pair):
 *     H_r = X_t W1_e            (gate | up, [2n])
 *     A_r = SiLU(H_r[:n]) * H_r[n:]
 *     O_t = sum_r s_r A_r W2_e
 * as set out in "SonicMoE: Accelerating MoE with IO and Tile-aware Optimizations" (ICLR 2026 reading note),
 * section "Method details / overall framework" (up-projection, down-projection, expert aggregation; dH,
 * dX~, dX, dW1, dW2), with routing from "Key design 1: Token Rounding routing", the fused epilogues of
 * "Key design 2: IO-aware fused kernels" and the X/H-only activation cache of "Key design 3:
 * minimal-activation-cache backward".
 *
 * Entry points
 *   routing      moe_route, moe_route_ex (stochastic rounding's uniforms), moe_route_noalloc; capacity and
 *                workspace queries
 *   layer        moe_forward, moe_backward, and their _ex forms with flags (MOE_FLAG_DETERMINISTIC)
 *   router       moe_router_forward (logits = X W_r), moe_router_backward (dlogits, dX += dz W_r^T, dW_r)
 *   diagnostics  moe_get_status, moe_strerror, moe_last_cuda_error, moe_kernel_launch_count, moe_profile_*,
 *                moe_selftest_bounded_wait
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library allocates no device memory.
 *     Tensors are contiguous and row-major.  "bf16" arguments hold IEEE bfloat16 bit patterns (moe_bf16).
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream) and returns a status code (MOE_OK = 0) for host-side validation and launch errors.  Errors
 *     found on the device (bad routing metadata, a bounded wait that ran out) are written to the routing
 *     status block and read with moe_get_status().
 *   - Shapes: E <= 1024, 1 <= K <= min(E, 32), d % 256 == 0, n % 128 == 0, M_tile = 128.  Other shapes
 *     return MOE_ERR_UNSUPPORTED_SHAPE.
 *   - Only an sm_100-family device with compute capability 10.3 is accepted (MOE_ERR_DEVICE otherwise).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;

enum moe_status_code {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer, T/E/K <= 0, K > E, unknown mode, missing uniforms     */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the limits above                                     */
  MOE_ERR_WORKSPACE = 3,          /* workspace pointer null or smaller than the *_workspace_size query  */
  MOE_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed (moe_last_cuda_error() has it)   */
  MOE_ERR_NONFINITE_LOGITS = 5,   /* device: a router logit is NaN or +-inf                             */
  MOE_ERR_DEVICE_TIMEOUT = 6,     /* device: a bounded pipeline wait ran out; the kernel returned early */
  MOE_ERR_BAD_METADATA = 7,       /* device: a row's token id or an offset is out of range              */
  MOE_ERR_DEVICE = 8,             /* current device is not compute capability 10.3 (GB300)              */
  MOE_ERR_RANGE = 9               /* device: deterministic mode met a contribution of magnitude >= 2^21 */
};

/*
 * Routing modes.  Token rounding ("Key design 1") rounds each expert's token-choice count f_e to a multiple of
 * M_tile and then keeps token-choice tokens ahead of expert-choice candidates; the rounding subroutine is a
 * choice the method is robust to ("Loss function / training strategy"), so every rule below is offered.  A
 * rounding that would need more than T tokens takes the floor under every rule.  Expert choice is the "EC"
 * baseline of the ablation table.
 */
enum moe_route_mode {
  MOE_ROUTE_TC = 0,               /* token choice: each token's top-K experts                                 */
  MOE_ROUTE_TR = 1,               /* token rounding, nearest multiple (ceil only when strictly closer)        */
  MOE_ROUTE_TR_UP = 2,            /* token rounding, always the ceiling                                       */
  MOE_ROUTE_TR_DOWN = 3,          /* token rounding, always the floor                                         */
  MOE_ROUTE_TR_STOCHASTIC = 4,    /* token rounding, ceiling iff u_e * M_tile < f_e - floor (u_e per expert,  */
                                  /* uniform in [0,1), passed to moe_route_ex): expected count f_e            */
  MOE_ROUTE_EC = 5                /* expert choice: each expert's C = min(T, floor(T*K/E)) tokens with the    */
                                  /* largest logits (ties to the lower token id); gate = the token's softmax  */
                                  /* over all E logits                                                        */
};

#define MOE_M_TILE 128
#define MOE_STATUS_WORDS 4

/*
 * Routing metadata (all device pointers, caller-allocated).  P_cap comes from moe_route_capacity().
 *   topk_idx   int32 [T*K]   token t's k-th expert, best first (logit descending, expert ascending on ties)
 *   topk_score fp32  [T*K]   softmax over the token's K selected logits
 *   tc_counts  int32 [E]     token-choice count f_e of each expert
 *   counts     int32 [E]     rows per expert (TC: f_e; TR modes: r_e = f_e rounded to M_tile; EC: C)
 *   offsets    int32 [E+1]   exclusive prefix sum of counts; offsets[E] = P (rows of expert e are
 *                            [offsets[e], offsets[e+1]), ordered by ascending token id)
 *   tile_offsets int32 [E+1] exclusive prefix sum of ceil(counts/M_tile) (the grouped-GEMM schedule)
 *   row_token  int32 [P_cap] token of each row
 *   row_slot   int32 [P_cap] k with topk_idx[token*K+k] == expert, or -1 for a pair added by rounding
 *   row_score  fp32  [P_cap] the row's gate score s_r (a pair added by rounding uses its token's
 *                            token-choice softmax normaliser; EC: softmax over all E logits)
 *   status     int32 [MOE_STATUS_WORDS]  [0] device error code, [1] P, [2] total M-tiles, [3] reserved
 * Rows at and beyond P are left untouched.
 */
typedef struct moe_routing {
  int32_t *topk_idx;
  float *topk_score;
  int32_t *tc_counts;
  int32_t *counts;
  int32_t *offsets;
  int32_t *tile_offsets;
  int32_t *row_token;
  int32_t *row_slot;
  float *row_score;
  int32_t *status;
} moe_routing;

/* Upper bound on P: T*K for TC, TR_DOWN and EC; T*K + E*M_tile/2 for TR (the nearest rule pads an expert by
 * less than M_tile/2 rows); T*K + E*(M_tile-1) for TR_UP and TR_STOCHASTIC. */
int moe_route_capacity(int T, int E, int K, int mode, size_t *p_cap);

/* Bytes of scratch moe_route needs (per-CTA and per-chunk expert histograms, per-token normalisers; every
 * mode but TC adds the membership bitmap and an expert-major copy of the logit order keys, 4*T*E bytes). */
int moe_route_workspace_size(int T, int E, int K, int mode, size_t *bytes);

/*
 * moe_route - routing metadata from router logits ("Key design 1: Token Rounding routing").
 *   logits  fp32 [T, E] device.  Must be finite (else MOE_ERR_NONFINITE_LOGITS in status[0]).
 *   mode    a moe_route_mode other than MOE_ROUTE_TR_STOCHASTIC (which needs moe_route_ex).  Every mode but TC
 *           supports T <= 49152.
 *   r       filled routing struct; every pointer non-null.  status is cleared by this call.
 *   ws      device scratch of at least moe_route_workspace_size() bytes (contents need not be zero).
 *   P_host  optional host pointer: if non-null, the call synchronises `stream` and stores P there.
 * Bit-exact and deterministic: same logits give the same metadata on every run.  Under EC, row_slot names the
 * token-choice slot of a pair that token choice also picked (-1 otherwise) and tc_counts still holds f_e.
 */
int moe_route(const float *logits, int T, int E, int K, int mode, const moe_routing *r, void *ws,
              size_t ws_bytes, int32_t *P_host, void *stream);

/*
 * moe_route_ex - moe_route with the random draws of stochastic rounding.
 *   uniforms  fp32 [E] device, one uniform draw in [0, 1) per expert (the caller's generator): expert e pads
 *             to the ceiling iff uniforms[e] * M_tile < f_e - floor.  Required for MOE_ROUTE_TR_STOCHASTIC
 *             (MOE_ERR_INVALID_ARG when NULL), ignored by the other modes.
 * Every other argument and result as moe_route; same uniforms and logits give the same metadata.
 */
int moe_route_ex(const float *logits, const float *uniforms, int T, int E, int K, int mode, const moe_routing *r,
                 void *ws, size_t ws_bytes, int32_t *P_host, void *stream);

/*
 * moe_route_noalloc - moe_route for callers that may not allocate device memory.  The paper has no
 * counterpart: this is a packaging variant of the routing call.
 *   Who needs it: code embedded in a host program whose allocator owns all device memory (raw cudaMalloc
 *   is forbidden), or a path with a fixed memory budget where no allocation may happen.  Such callers
 *   still pass the logits and the routing outputs (r); only the routing scratch changes hands.
 *   Scratch: a static device array of MOE_ROUTE_NOALLOC_SCRATCH_BYTES (16 MiB) inside the library, which
 *   every GPU that loads the library holds until the process exits.  When moe_route_workspace_size exceeds
 *   it, token rounding leaves out its expert-major copy of the logit keys (4*T*E bytes) and reads the logits
 *   in place (same results, slower selection); shapes that still do not fit return MOE_ERR_WORKSPACE before
 *   any device work.
 *   Set-up: the first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *   that device current; make that first call before any stream capture.
 *   Sharing: all calls in the process share the one array per device and it keeps the last call's
 *   contents (this call clears whatever must start at zero).  Calls that overlap on the GPU (different
 *   streams, or different host threads on one device) race on the array and corrupt each other.
 *   Never calls cudaMalloc, cudaFree or any allocating routine.  Other arguments and results as moe_route
 *   (MOE_ROUTE_TR_STOCHASTIC is not available here: it needs the uniforms of moe_route_ex).
 */
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES (16u << 20)
int moe_route_noalloc(const float *logits, int T, int E, int K, int mode, const moe_routing *r, int32_t *P_host,
                      void *stream);

/* Forward scratch: A [P_cap, n] bf16 and the fp32 accumulation buffer of O [T, d]. */
int moe_forward_workspace_size(int T, int d, int n, int E, int K, size_t p_cap, size_t *bytes);
/* Same for the given flags (MOE_FLAG_DETERMINISTIC: the accumulation buffer of O holds 64-bit integers;
 * MOE_FLAG_A_FROM_H: no A buffer). */
int moe_forward_workspace_size_ex(int T, int d, int n, int E, int K, size_t p_cap, unsigned flags, size_t *bytes);

/*
 * moe_forward - O = sum_k s_k SwiGLU(X W1_e) W2_e  ("Method details / overall framework").
 *   X   bf16 [T, d];  W1 bf16 [E, d, 2n] (columns [0,n) gate, [n,2n) up);  W2 bf16 [E, n, d]
 *   r   routing from moe_route on the same T, E, K
 *   O   bf16 [T, d] output (a token with no rows gets zeros)
 *   H   bf16 [P_cap, 2n] output: the pre-activation up-projection, the one per-row tensor kept for the
 *       backward ("Key design 3"); rows >= P untouched
 *   ws  scratch of moe_forward_workspace_size() bytes
 * Y [P, d] is never written: the down-projection adds s_r * A_r W2_e straight into O's fp32 buffer.
 */
int moe_forward(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2, const moe_routing *r, int T,
                int d, int n, int E, int K, size_t p_cap, moe_bf16 *O, moe_bf16 *H, void *ws,
                size_t ws_bytes, void *stream);
/* moe_forward with flags (0, MOE_FLAG_DETERMINISTIC, MOE_FLAG_A_FROM_H or both); ws sized by
 * moe_forward_workspace_size_ex with the same flags.  moe_backward_ex does not take MOE_FLAG_A_FROM_H. */
int moe_forward_ex(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2, const moe_routing *r, int T, int d,
                   int n, int E, int K, size_t p_cap, moe_bf16 *O, moe_bf16 *H, void *ws, size_t ws_bytes,
                   unsigned flags, void *stream);

/*
 * Deterministic aggregation (flag of moe_forward_ex / moe_backward_ex; the pages have no counterpart: they
 * leave the order of the aggregation's additions open).  O and dX sum a token's rows from different experts,
 * whose contributions land in whatever order the GPU schedules them; fp32 addition depends on that order, so the
 * default path can differ in the last bits from run to run.  With this flag every contribution is added as a
 * 64-bit fixed-point integer with 32 fractional bits (integer addition does not depend on order) and dS sums its
 * per-column-tile partials in a fixed order: O, H, dX, dW1, dW2 and dS are then bitwise identical on every run.
 * Cost: twice the reduce-add bytes and accumulator memory.  Range: one contribution s_r * y_r (or a row of
 * dH W1^T) must stay below 2^21 in magnitude, else MOE_ERR_RANGE in the status block.
 */
#define MOE_FLAG_DETERMINISTIC 1u

/*
 * A kept on chip (flag of moe_forward_ex; "Key design 3: minimal-activation-cache backward" keeps only X, H and
 * the routing metadata, and "Key design 2" fuses elementwise work into the GEMMs).  By default the
 * up-projection's epilogue also writes A = SiLU(H_gate) * H_up [P, n] bf16 to the workspace, and the
 * down-projection reads it back (once per column slab).  With this flag A is never written: producer warps of the
 * down-projection load the cached H rows and compute A in fp32 straight into the tensor cores' shared-memory
 * operand, once per 256-column tile of O.  The forward then moves no A bytes (P*n*2 written, read twice at d =
 * 1536) but reads H (twice A's bytes) in its place and recomputes SwiGLU per column tile; A is formed from the
 * bf16 H rather than from the fp32 accumulators (as the backward also does), so O differs in the last bits.
 */
#define MOE_FLAG_A_FROM_H 2u

/* Backward scratch: dH [P_cap, 2n] bf16, s*A [P_cap, n] bf16 and the fp32 accumulation buffer of dX. */
int moe_backward_workspace_size(int T, int d, int n, int E, int K, size_t p_cap, size_t *bytes);
/* Same for the given flags (MOE_FLAG_DETERMINISTIC adds the dS partials and a 64-bit dX accumulator). */
int moe_backward_workspace_size_ex(int T, int d, int n, int E, int K, size_t p_cap, unsigned flags, size_t *bytes);

/*
 * moe_backward - gradients of the layer for upstream gradient dO, routing held fixed
 * ("Key design 2" for the dH epilogue, "Key design 3" for the cache).
 *   dO  bf16 [T, d];  X, W1, W2 as in moe_forward;  H the forward's H output
 *   dX  bf16 [T, d];  dW1 bf16 [E, d, 2n];  dW2 bf16 [E, n, d]  (an expert with no rows gets zeros)
 *   dS  fp32 [P_cap]: dL/ds_r per row, computed as <dO_t W2_e^T, SwiGLU(H_r)> without Y or dY
 *   ws  scratch of moe_backward_workspace_size() bytes
 */
int moe_backward(const moe_bf16 *dO, const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2,
                 const moe_bf16 *H, const moe_routing *r, int T, int d, int n, int E, int K, size_t p_cap,
                 moe_bf16 *dX, moe_bf16 *dW1, moe_bf16 *dW2, float *dS, void *ws, size_t ws_bytes,
                 void *stream);
/* moe_backward with flags (0 or MOE_FLAG_DETERMINISTIC); ws sized by moe_backward_workspace_size_ex. */
int moe_backward_ex(const moe_bf16 *dO, const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W2, const moe_bf16 *H,
                    const moe_routing *r, int T, int d, int n, int E, int K, size_t p_cap, moe_bf16 *dX, moe_bf16 *dW1,
                    moe_bf16 *dW2, float *dS, void *ws, size_t ws_bytes, unsigned flags, void *stream);

/*
 * The router on either side of the layer ("Method details / overall framework": router scoring of the input
 * tokens feeds the routing step).  Shapes: E % 8 == 0, E <= 1024, d % 256 == 0.
 *
 * moe_router_forward - logits = X W_r on the tensor cores, fp32 accumulation.
 *   X  bf16 [T, d];  W_r bf16 [d, E];  logits fp32 [T, E] output (the input of moe_route / moe_route_ex)
 *   status  optional device int32: a bounded wait that ran out writes MOE_ERR_DEVICE_TIMEOUT there
 */
int moe_router_forward(const moe_bf16 *X, const moe_bf16 *Wr, int T, int d, int E, float *logits, int32_t *status,
                       void *stream);

/* Router backward scratch: dz in bf16 [T, E] and up to 32 token-split partials of dW_r [d, E] (fp32). */
int moe_router_backward_workspace_size(int T, int d, int E, size_t *bytes);

/*
 * moe_router_backward - gradients through the gates, the routing held fixed (selection is piecewise constant).
 * A row r = (t, e) has the gate s_r = exp(z_te) / sum_{j in N(t)} exp(z_tj), N(t) = the token's K token-choice
 * experts (MOE_ROUTE_TC and every token-rounding mode) or all E experts (MOE_ROUTE_EC), so
 *     dz_tj = [a row (t, j) exists] dS_tj s_tj - [j in N(t)] s_tj G_t,   G_t = sum over the token's rows of dS_r s_r.
 *   dS       fp32 [P_cap] from moe_backward (dL/ds_r per row);  r, K, mode, p_cap: the routing call's
 *   logits   fp32 [T, E], the routing call's input (read under MOE_ROUTE_EC only)
 *   X, W_r   as in moe_router_forward
 *   dlogits  fp32 [T, E] output: dz
 *   dX       bf16 [T, d] in/out: the layer's dX from moe_backward; dz W_r^T is added to it
 *   dWr      fp32 [d, E] output: X^T dz
 *   ws       scratch of moe_router_backward_workspace_size() bytes
 * Row metadata out of range is skipped and reported as MOE_ERR_BAD_METADATA in the routing status block.
 * Every output is reproducible bit for bit: G_t is summed in a fixed order, and dWr adds its token splits'
 * partials in split order.
 */
int moe_router_backward(const float *dS, const moe_routing *r, const float *logits, const moe_bf16 *X,
                        const moe_bf16 *Wr, int T, int d, int E, int K, int mode, size_t p_cap, float *dlogits,
                        moe_bf16 *dX, float *dWr, void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream` and read the routing status block: device error code and P (either may be NULL). */
int moe_get_status(const moe_routing *r, int32_t *code, int32_t *P, void *stream);

/* Human-readable text of a status code (static storage). */
const char *moe_strerror(int code);

/*
 * Self-test of the bounded device waits (no counterpart in the paper).  Launches one CTA that waits on an
 * mbarrier nothing will ever arrive on, with the same bounded wait the GEMM pipelines use: after
 * MOE_WAIT_TIMEOUT_NS (2 s) it gives up, writes MOE_ERR_DEVICE_TIMEOUT to status[0] (a device int32 the
 * caller zeroes) and returns, leaving the CUDA context usable.  Asynchronous on `stream`.
 */
int moe_selftest_bounded_wait(int32_t *status, void *stream);

/* The cudaError_t of the last MOE_ERR_CUDA on this thread (0 if none). */
int moe_last_cuda_error(void);

/* Number of kernels the library launched since load (a counter for benchmarks and tests). */
uint64_t moe_kernel_launch_count(void);

/*
 * Per-kernel timing for benchmarks.  moe_profile_enable(1) clears earlier results and, until
 * moe_profile_enable(0), brackets every kernel the library launches with two CUDA events on the launch
 * stream.  moe_profile_enable(0) waits for those events and aggregates them per kernel name; the summary is
 * then read with moe_profile_count() and moe_profile_entry(i, ...) (name copied NUL-terminated into a
 * caller buffer of name_len bytes, number of launches, summed milliseconds).  Off by default; the host
 * cost is two event records per launch while on.
 */
int moe_profile_enable(int on);
int moe_profile_count(void);
int moe_profile_entry(int i, char *name, size_t name_len, int *launches, double *total_ms);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
