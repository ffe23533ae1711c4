"""Plain fp64 CPU oracle of the SonicMoE fine-grained MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute this module: only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.  It shares no code with
the CUDA library and does not import the package.

Sources (the pages this restates; section names as printed on each page):

* [NOTE-FW]  "SonicMoE: Accelerating MoE with IO and Tile-aware Optimizations", ICLR 2026 reading note
  (papernotes.org), section "Method details / overall framework": the layer is split into up-projection,
  down-projection and expert aggregation (forward) and dH, dX~, aggregation dX, dW1, dW2 (backward).
* [NOTE-TR]  same page, "Key design 1: Token Rounding routing": token-choice top-K first, then a per-expert
  expert-choice ordering with the token-choice tokens always ahead of expert-choice candidates, then
  round_and_sparsify to the nearest multiple of M_tile (pad when the distance up is strictly smaller).
* [NOTE-IO]  same page, "Key design 2: IO-aware fused kernels": SwiGLU in the up-projection epilogue; the
  dH epilogue produces dH and dS = <dA, A'>.
* [NOTE-BW]  same page, "Key design 3: minimal-activation-cache backward": FLOPs (6+12)TnKd; only X, H and
  routing metadata are cached, about 2Td + 4TKn bytes; dS and dH are computed without Y or dY.
* [ABSTRACT] arXiv abstract (mlsanity.com index page): token rounding and the memory-efficient backward.

Everything is float64; inputs are the exact float64 values of the bf16 / fp32 tensors.  No blocking,
fusion or reordering beyond the definitions: the forward gathers X_e explicitly, materialises Y, and the
backward follows the chain rule through Y.  ``numpy.matmul`` is the one library primitive used.

Readings taken where the pages are silent (each listed in the design notes of the repository):
  * H is the pre-activation up-projection output [P, 2n] = (gate | up); A = SiLU(gate) * up.
  * Expert choice for top-K uses the raw logits, larger first, ties to the lower expert index.
  * Gate scores: softmax over the K selected logits of the token.
  * Token rounding ranks each expert's candidates by (in token choice, logit, -token) descending; a tie
    f_e - floor = ceil - f_e rounds down; a pad that would exceed T rounds down; an expert-choice pair
    added by rounding gets the token's token-choice softmax normaliser.
  * Rows of one expert are ordered by ascending token id.
  * Rounding subroutines other than the nearest multiple (the note, "Loss function / training strategy",
    says token rounding is robust to which one is used): always up, always down, and stochastic (up with
    probability (f - floor)/M_tile, from one uniform draw per expert passed in, so the expected count is f).
    Padding beyond T tokens is impossible under every rule, which then rounds down.
  * The router (the flowchart's "router scoring") is z = X W_r with W_r [d, E]; its backward holds the routing
    fixed and differentiates only the gates (selection is piecewise constant in z).
  * Expert choice (the "EC" rows of the note's ablation table): each expert takes the C = floor(T K / E)
    tokens with the largest logits in its column (ties to the lower token id); a routed pair's gate is the
    token's softmax over all E logits.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------------------------------
# library primitive: every matrix product of the oracle goes through here (tests count MACs with it)
# --------------------------------------------------------------------------------------------------


def _matmul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.matmul(a, b)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


# --------------------------------------------------------------------------------------------------
# routing  [NOTE-TR]
# --------------------------------------------------------------------------------------------------


def topk_token_choice(z: np.ndarray, K: int) -> np.ndarray:
    """Token choice: each token's K experts with the largest logits, best first; ties go to the lower
    expert index.  K passes of a first-maximum search with the chosen entry removed."""
    z = np.asarray(z, dtype=np.float64)
    T, E = z.shape
    if not np.all(np.isfinite(z)):
        raise ValueError("non-finite router logits")
    work = z.copy()
    idx = np.empty((T, K), dtype=np.int64)
    rows = np.arange(T)
    for k in range(K):
        j = np.argmax(work, axis=1)  # first occurrence of the maximum -> lowest expert index on ties
        idx[:, k] = j
        work[rows, j] = -np.inf
    return idx


def token_normaliser(z: np.ndarray, topk_idx: np.ndarray):
    """Per token: its largest selected logit z0 and sum_k exp(z_k - z0) over its K selected experts."""
    z = np.asarray(z, dtype=np.float64)
    T = z.shape[0]
    zs = z[np.arange(T)[:, None], topk_idx]
    z0 = zs[:, 0]
    den = np.exp(zs - z0[:, None]).sum(axis=1)
    return z0, den


def gate_scores(z: np.ndarray, topk_idx: np.ndarray) -> np.ndarray:
    """s_{t,k} = softmax over the token's K selected logits."""
    z = np.asarray(z, dtype=np.float64)
    T = z.shape[0]
    zs = z[np.arange(T)[:, None], topk_idx]
    z0, den = token_normaliser(z, topk_idx)
    return np.exp(zs - z0[:, None]) / den[:, None]


ROUNDING_RULES = ("nearest", "up", "down", "stochastic")


def round_and_sparsify(f: np.ndarray, m_tile: int, T: int, rule: str = "nearest", u=None) -> np.ndarray:
    """Each expert's count f rounded to a multiple of M_tile: floor or ceil.

    nearest:     ceil when ceil - f < f - floor (strict), else floor (the pages' rule)
    up / down:   ceil / floor
    stochastic:  ceil when u * M_tile < f - floor for the expert's uniform u in [0, 1), so that ceil is taken
                 with probability (f - floor) / M_tile and the expected count is f
    A ceil beyond T tokens is impossible, so every rule takes the floor there."""
    f = np.asarray(f, dtype=np.int64)
    lo = (f // m_tile) * m_tile
    hi = -((-f) // m_tile) * m_tile
    if rule == "nearest":
        up = (hi - f) < (f - lo)
    elif rule == "up":
        up = hi > f
    elif rule == "down":
        up = np.zeros(f.shape, dtype=bool)
    elif rule == "stochastic":
        u = np.asarray(u, dtype=np.float64)
        if u.shape != f.shape:
            raise ValueError("stochastic rounding needs one uniform per expert")
        up = u * m_tile < (f - lo)
    else:
        raise ValueError(rule)
    up = up & (hi <= T)
    return np.where(up, hi, lo)


def _pack(T, E, K, topk_idx, topk_score, counts, tc_counts, expert_rows, m_tile):
    """Lay the per-expert row lists out as grouped rows (expert-major, ascending token within an expert)."""
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    tiles = -((-counts) // m_tile)
    tile_offsets = np.zeros(E + 1, dtype=np.int64)
    tile_offsets[1:] = np.cumsum(tiles)
    P = int(offsets[-1])
    row_token = np.empty(P, dtype=np.int64)
    row_slot = np.empty(P, dtype=np.int64)
    row_score = np.empty(P, dtype=np.float64)
    row_expert = np.empty(P, dtype=np.int64)
    for e in range(E):
        toks, slots, scores = expert_rows[e]
        s = slice(offsets[e], offsets[e + 1])
        row_token[s] = toks
        row_slot[s] = slots
        row_score[s] = scores
        row_expert[s] = e
    return dict(T=T, E=E, K=K, m_tile=m_tile, topk_idx=topk_idx, topk_score=topk_score,
                counts=counts, tc_counts=tc_counts, offsets=offsets, tile_offsets=tile_offsets, P=P,
                row_token=row_token, row_slot=row_slot, row_score=row_score, row_expert=row_expert)


def route_tc(z: np.ndarray, K: int, m_tile: int = 128) -> dict:
    """Token-choice routing [NOTE-TR]: top-K, scores, per-expert counts, exclusive-scan offsets, rows."""
    z = np.asarray(z, dtype=np.float64)
    T, E = z.shape
    idx = topk_token_choice(z, K)
    score = gate_scores(z, idx)
    member = np.zeros((T, E), dtype=bool)
    slot_of = np.full((T, E), -1, dtype=np.int64)
    for k in range(K):
        member[np.arange(T), idx[:, k]] = True
        slot_of[np.arange(T), idx[:, k]] = k
    counts = member.sum(axis=0).astype(np.int64)
    expert_rows = []
    for e in range(E):
        toks = np.nonzero(member[:, e])[0]            # ascending token id
        slots = slot_of[toks, e]
        expert_rows.append((toks, slots, score[toks, slots]))
    return _pack(T, E, K, idx, score, counts, counts.copy(), expert_rows, m_tile)


def route_tr(z: np.ndarray, K: int, m_tile: int = 128, rule: str = "nearest", u=None) -> dict:
    """Token rounding [NOTE-TR]: token choice, then per expert an expert-choice ranking of all tokens with
    token-choice tokens first, then keep the first r_e = round_and_sparsify(f_e) of that ranking (under the
    given rounding rule)."""
    z = np.asarray(z, dtype=np.float64)
    T, E = z.shape
    idx = topk_token_choice(z, K)
    score = gate_scores(z, idx)
    z0, den = token_normaliser(z, idx)
    member = np.zeros((T, E), dtype=bool)
    slot_of = np.full((T, E), -1, dtype=np.int64)
    for k in range(K):
        member[np.arange(T), idx[:, k]] = True
        slot_of[np.arange(T), idx[:, k]] = k
    f = member.sum(axis=0).astype(np.int64)
    r = round_and_sparsify(f, m_tile, T, rule, u)
    tok = np.arange(T)
    expert_rows = []
    for e in range(E):
        # primary key: in token choice (first); then logit descending; then token ascending
        order = np.lexsort((tok, -z[:, e], ~member[:, e]))
        kept = np.sort(order[: r[e]])
        slots = slot_of[kept, e]
        s = np.exp(z[kept, e] - z0[kept]) / den[kept]
        expert_rows.append((kept, slots, s))
    out = _pack(T, E, K, idx, score, r.astype(np.int64), f, expert_rows, m_tile)
    return out


def softmax_all(z: np.ndarray) -> np.ndarray:
    """Per token: softmax over all E logits."""
    z = np.asarray(z, dtype=np.float64)
    ex = np.exp(z - z.max(axis=1, keepdims=True))
    return ex / ex.sum(axis=1, keepdims=True)


def ec_capacity(T: int, E: int, K: int) -> int:
    """Tokens each expert takes under expert choice: the token-choice average T K / E, rounded down."""
    return min(T, (T * K) // E)


def route_ec(z: np.ndarray, K: int, m_tile: int = 128) -> dict:
    """Expert choice: every expert takes the C tokens with the largest logits in its column (ties to the
    lower token id); a pair's gate is the token's softmax over all E logits.  Token choice is still
    computed (topk_idx, topk_score, tc_counts) and names the slot of a pair that token choice also picked."""
    z = np.asarray(z, dtype=np.float64)
    T, E = z.shape
    idx = topk_token_choice(z, K)
    score = gate_scores(z, idx)
    prob = softmax_all(z)
    slot_of = np.full((T, E), -1, dtype=np.int64)
    for k in range(K):
        slot_of[np.arange(T), idx[:, k]] = k
    f = (slot_of >= 0).sum(axis=0).astype(np.int64)
    C = ec_capacity(T, E, K)
    tok = np.arange(T)
    expert_rows = []
    for e in range(E):
        order = np.lexsort((tok, -z[:, e]))            # logit descending, then token ascending
        kept = np.sort(order[:C])
        expert_rows.append((kept, slot_of[kept, e], prob[kept, e]))
    counts = np.full(E, C, dtype=np.int64)
    return _pack(T, E, K, idx, score, counts, f, expert_rows, m_tile)


# routing modes: token choice, token rounding under each rounding rule, expert choice
ROUTE_MODES = ("tc", "tr", "tr_up", "tr_down", "tr_stoch", "ec")


def route(z: np.ndarray, K: int, mode: str = "tc", m_tile: int = 128, u=None) -> dict:
    """Routing metadata in one of ROUTE_MODES; `u` holds the per-expert uniforms of "tr_stoch"."""
    if mode == "tc":
        return route_tc(z, K, m_tile)
    if mode == "tr":
        return route_tr(z, K, m_tile)
    if mode == "tr_up":
        return route_tr(z, K, m_tile, "up")
    if mode == "tr_down":
        return route_tr(z, K, m_tile, "down")
    if mode == "tr_stoch":
        return route_tr(z, K, m_tile, "stochastic", u)
    if mode == "ec":
        return route_ec(z, K, m_tile)
    raise ValueError(mode)


# --------------------------------------------------------------------------------------------------
# forward  [NOTE-FW]
# --------------------------------------------------------------------------------------------------


def forward(X, W1, W2, row_token, row_expert, row_score):
    """O_t = sum over the token's rows r of s_r * (SiLU(X_t W1_e[:, :n]) * (X_t W1_e[:, n:])) W2_e.

    Returns O [T, d] together with the per-row H [P, 2n], A [P, n] and Y [P, d]."""
    X = np.asarray(X, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    T, d = X.shape
    E, _, n2 = W1.shape
    n = n2 // 2
    P = len(row_token)
    H = np.zeros((P, n2))
    A = np.zeros((P, n))
    Y = np.zeros((P, d))
    O = np.zeros((T, d))
    for e in np.unique(row_expert):
        sel = np.nonzero(row_expert == e)[0]
        toks = row_token[sel]
        Xe = X[toks]                                   # explicit gather of the expert's tokens
        He = _matmul(Xe, W1[e])                        # up-projection
        Ae = silu(He[:, :n]) * He[:, n:]               # SwiGLU
        Ye = _matmul(Ae, W2[e])                        # down-projection
        H[sel], A[sel], Y[sel] = He, Ae, Ye
    for e in np.unique(row_expert):                    # expert aggregation (tokens are distinct per expert)
        sel = np.nonzero(row_expert == e)[0]
        O[row_token[sel]] += row_score[sel, None] * Y[sel]
    return dict(O=O, H=H, A=A, Y=Y)


# --------------------------------------------------------------------------------------------------
# backward through Y by the chain rule  [NOTE-FW], [NOTE-BW]
# --------------------------------------------------------------------------------------------------


def backward(dO, X, W1, W2, row_token, row_expert, row_score, fwd):
    """Gradients of L = <dO, O> with the routing held fixed.

    dY_r = s_r dO_t;  dS_r = <dO_t, Y_r>;  dW2_e = sum_r A_r^T dY_r;  dA_r = dY_r W2_e^T;
    dgate = dA * up * sig(gate) * (1 + gate (1 - sig(gate)));  dup = dA * SiLU(gate);
    dW1_e = sum_r X_t^T dH_r;  dX_t = sum_r dH_r W1_e^T."""
    dO = np.asarray(dO, np.float64)
    X = np.asarray(X, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    T, d = X.shape
    E, _, n2 = W1.shape
    n = n2 // 2
    P = len(row_token)
    H, A, Y = fwd["H"], fwd["A"], fwd["Y"]
    dX = np.zeros((T, d))
    dW1 = np.zeros_like(W1)
    dW2 = np.zeros_like(W2)
    dS = np.zeros(P)
    dH = np.zeros((P, n2))
    dXt = np.zeros((P, d))
    for e in np.unique(row_expert):
        sel = np.nonzero(row_expert == e)[0]
        toks = row_token[sel]
        dOe = dO[toks]
        dYe = row_score[sel, None] * dOe
        dS[sel] = (dOe * Y[sel]).sum(axis=1)
        dW2[e] = _matmul(A[sel].T, dYe)
        dAe = _matmul(dYe, W2[e].T)
        g, u = H[sel, :n], H[sel, n:]
        sg = sigmoid(g)
        dg = dAe * u * sg * (1.0 + g * (1.0 - sg))
        du = dAe * g * sg
        dHe = np.concatenate([dg, du], axis=1)
        dH[sel] = dHe
        dW1[e] = _matmul(X[toks].T, dHe)
        dXt[sel] = _matmul(dHe, W1[e].T)
    for e in np.unique(row_expert):                    # aggregation of dX~ (tokens distinct per expert)
        sel = np.nonzero(row_expert == e)[0]
        dX[row_token[sel]] += dXt[sel]
    return dict(dX=dX, dW1=dW1, dW2=dW2, dS=dS, dH=dH)


def ds_via_h(dO, W2, row_token, row_expert, H):
    """The method's dS path [NOTE-IO]: dS_r = <dO_t W2_e^T, SiLU(gate_r) * up_r>, from H, no Y."""
    dO = np.asarray(dO, np.float64)
    W2 = np.asarray(W2, np.float64)
    n = W2.shape[1]
    dS = np.zeros(len(row_token))
    for e in np.unique(row_expert):
        sel = np.nonzero(row_expert == e)[0]
        dA = _matmul(dO[row_token[sel]], W2[e].T)
        a = silu(H[sel, :n]) * H[sel, n:]
        dS[sel] = (dA * a).sum(axis=1)
    return dS


# --------------------------------------------------------------------------------------------------
# router  [NOTE-FW] (flowchart: input tokens and router scoring feed the routing step)
# --------------------------------------------------------------------------------------------------


def router_logits(X, Wr):
    """The router's scores: z = X W_r, [T, d] x [d, E] -> [T, E]."""
    return _matmul(np.asarray(X, np.float64), np.asarray(Wr, np.float64))


def router_dz(z, rt: dict, dS, mode: str, tokens=None):
    """Gradient of L = sum_r dS_r s_r with respect to the logits, the routing held fixed.

    A row r = (t, e) has the gate s_r = exp(z_te) / sum_{j in N(t)} exp(z_tj), where the normaliser set N(t) is
    the token's K token-choice experts (token choice and every token-rounding rule: a pair added by rounding
    shares its token's token-choice normaliser) or all E experts (expert choice).  By the chain rule
    dz_tj = sum over the token's rows r of dS_r * s_r * ([j = e_r] - [j in N(t)] * s(t, j)).
    Returns dz [T, E] (rows outside `tokens`, when given, stay zero)."""
    z = np.asarray(z, np.float64)
    dS = np.asarray(dS, np.float64)
    T, E = z.shape
    dz = np.zeros((T, E))
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, np.int64)
    want = np.zeros(T, dtype=bool)
    want[tokens] = True
    rows_of = {}
    for r in np.nonzero(want[rt["row_token"]])[0]:
        rows_of.setdefault(int(rt["row_token"][r]), []).append(int(r))
    for t in tokens:
        t = int(t)
        N = np.arange(E) if mode == "ec" else np.asarray(rt["topk_idx"][t])
        m = z[t, N].max()
        den = np.exp(z[t, N] - m).sum()
        s_N = np.exp(z[t, N] - m) / den
        for r in rows_of.get(t, []):
            e = int(rt["row_expert"][r])
            s_r = np.exp(z[t, e] - m) / den
            dz[t, e] += dS[r] * s_r
            dz[t, N] -= dS[r] * s_r * s_N
    return dz


def router_backward(z, rt: dict, dS, X, Wr, mode: str):
    """Router gradients: dz (router_dz), its contribution to dX (dz W_r^T) and dW_r = X^T dz."""
    dz = router_dz(z, rt, dS, mode)
    dX = _matmul(dz, np.asarray(Wr, np.float64).T)
    dWr = _matmul(np.asarray(X, np.float64).T, dz)
    return dict(dz=dz, dX=dX, dWr=dWr)


# --------------------------------------------------------------------------------------------------
# accounting  [NOTE-BW]
# --------------------------------------------------------------------------------------------------


def layer_flops(P: int, n: int, d: int):
    """Forward 6Pnd, backward 12Pnd (P = TK under token choice, giving (6+12)TnKd)."""
    return 6 * P * n * d, 12 * P * n * d


def cached_activation_bytes(T: int, d: int, n: int, P: int) -> int:
    """Bytes kept from forward to backward by the method, metadata excluded: X (2Td, bf16) and H
    (P x 2n bf16 = 4Pn); with P = TK this is 2Td + 4TKn."""
    return 2 * T * d + 4 * P * n


# --------------------------------------------------------------------------------------------------
# convenience: the whole layer on one routing
# --------------------------------------------------------------------------------------------------


def layer(X, W1, W2, dO, rt: dict):
    fwd = forward(X, W1, W2, rt["row_token"], rt["row_expert"], rt["row_score"])
    bwd = backward(dO, X, W1, W2, rt["row_token"], rt["row_expert"], rt["row_score"], fwd)
    return fwd, bwd

