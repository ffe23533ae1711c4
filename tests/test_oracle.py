"""Pins of the CPU oracle to facts it does not compute itself: library routines on special cases, brute
force on tiny inputs, hand-worked fixtures, finite differences, an independent autograd derivation,
closed forms and the token-rounding invariants.  Some tests plant a mistake in the oracle (on the CPU)
to show that a pin catches it."""
import itertools

import numpy as np
import pytest
import scipy.special
import torch

from conftest import load_golden
from fine_grained_mixture_gb300 import synth
from oracle import moe_oracle as orc

# ----------------------------------------------------------------------------------------------- routing


@pytest.mark.parametrize("name", ["tiny", "fine7b", "sparse", "skew", "coarse"])
def test_topk_equals_stable_argsort_on_workload_logits(name):
    w = synth.WORKLOADS[name]
    z = synth.make_logits_only(w, seed=0).numpy()
    got = orc.topk_token_choice(z, w.K)
    ref = np.argsort(-z.astype(np.float64), axis=1, kind="stable")[:, : w.K]
    assert np.array_equal(got, ref)


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(1)
    for _ in range(200):
        T, E, K = 3, 5, int(rng.integers(1, 5))
        z = rng.choice([-1.0, -0.0, 0.0, 0.5, 1.0], size=(T, E)).astype(np.float32)   # -0.0 ties +0.0
        got = orc.topk_token_choice(z, K)
        for t in range(T):
            # brute force: the K-subset whose (logit desc, expert asc) key list is smallest, listed in key order
            best = None
            for S in itertools.combinations(range(E), K):
                key = sorted((-float(z[t, e]), e) for e in S)
                if best is None or key < best:
                    best = key
            assert [e for _, e in best] == list(got[t])


def test_scores_are_softmax_of_selected():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((64, 16)).astype(np.float32)
    idx = orc.topk_token_choice(z, 4)
    s = orc.gate_scores(z, idx)
    sel = np.take_along_axis(z.astype(np.float64), idx, axis=1)
    assert np.allclose(s, scipy.special.softmax(sel, axis=1), rtol=1e-14, atol=0)
    assert np.allclose(s.sum(1), 1.0, rtol=0, atol=1e-14)


@pytest.mark.parametrize("f,M,T,r", [
    (0, 128, 10**6, 0), (1, 128, 10**6, 0), (63, 128, 10**6, 0), (64, 128, 10**6, 0),   # tie -> floor
    (65, 128, 10**6, 128), (127, 128, 10**6, 128), (128, 128, 10**6, 128), (129, 128, 10**6, 128),
    (192, 128, 10**6, 128), (193, 128, 10**6, 256), (100, 128, 120, 0),                  # ceil > T -> floor
    (3, 4, 100, 4), (5, 4, 100, 4), (2, 4, 100, 0), (6, 4, 100, 4), (7, 4, 100, 8),
])
def test_round_and_sparsify_table(f, M, T, r):
    assert int(orc.round_and_sparsify(np.array([f]), M, T)[0]) == r


def _check_tr_invariants(z, K, M, rule="nearest", u=None):
    tc = orc.route_tc(z, K, M)
    tr = orc.route_tr(z, K, M, rule, u)
    T, E = z.shape
    z64 = z.astype(np.float64)
    f, r = tc["counts"], tr["counts"]
    assert np.array_equal(tr["tc_counts"], f)
    assert np.all(r % M == 0)
    hi = -((-f) // M) * M
    lo = (f // M) * M
    near = hi <= T                                            # padding possible
    if rule == "nearest":
        assert np.all(np.abs(r - f)[near] <= M // 2)          # never more than half a tile away
    elif rule == "up":
        assert np.all(r[near] == hi[near])
    elif rule == "down":
        assert np.all(r == lo)
    else:
        assert np.all((r == lo) | (r == hi))
    assert np.all(np.abs(r - f) < M)                          # deviation within one tile
    for e in range(E):
        tc_set = tc["row_token"][tc["offsets"][e]:tc["offsets"][e + 1]]
        kept = tr["row_token"][tr["offsets"][e]:tr["offsets"][e + 1]]
        assert np.all(np.diff(kept) > 0)                      # ascending token ids
        tcs, ks = set(tc_set.tolist()), set(kept.tolist())
        if r[e] >= f[e]:
            assert tcs <= ks                                  # every TC token kept before any EC token
            added = np.array(sorted(ks - tcs), dtype=np.int64)
            rest = np.array(sorted(set(range(T)) - ks), dtype=np.int64)
            if len(added) and len(rest):
                assert z64[added, e].min() >= z64[rest, e].max()
        else:
            assert ks <= tcs                                  # drops only among TC tokens ...
            dropped = np.array(sorted(tcs - ks), dtype=np.int64)
            if len(dropped) and len(kept):
                assert z64[kept, e].min() >= z64[dropped, e].max()   # ... the weakest ones
        sl = slice(tr["offsets"][e], tr["offsets"][e + 1])
        for t, k, s in zip(tr["row_token"][sl], tr["row_slot"][sl], tr["row_score"][sl]):
            if k >= 0:
                assert tc["topk_idx"][t, k] == e and s == tc["topk_score"][t, k]
            else:
                assert e not in tc["topk_idx"][t]
    return tc, tr


@pytest.mark.parametrize("name", ["tiny", "sparse", "skew", "fine7b"])
def test_tr_invariants_on_workloads(name):
    w = synth.WORKLOADS[name]
    _check_tr_invariants(synth.make_logits_only(w, 0).numpy(), w.K, synth.M_TILE)


def test_tr_invariants_random_seeds():
    rng = np.random.default_rng(3)
    for seed in range(40):
        T = int(rng.integers(1, 700))
        E = int(rng.integers(2, 20))
        K = int(rng.integers(1, min(E, 6) + 1))
        M = int(rng.choice([4, 16, 128]))
        z = rng.standard_normal((T, E)).astype(np.float32)
        if seed % 4 == 0:
            z = np.round(z * 2) / 2                          # heavy ties
        _check_tr_invariants(z, K, M)


@pytest.mark.parametrize("rule", orc.ROUNDING_RULES)
def test_tr_rule_invariants_random_seeds(rule):
    rng = np.random.default_rng(13)
    for seed in range(25):
        T = int(rng.integers(1, 500))
        E = int(rng.integers(2, 16))
        K = int(rng.integers(1, min(E, 5) + 1))
        M = int(rng.choice([4, 16, 128]))
        z = rng.standard_normal((T, E)).astype(np.float32)
        if seed % 3 == 0:
            z = np.round(z * 2) / 2                          # heavy ties
        u = rng.random(E).astype(np.float32)
        _check_tr_invariants(z, K, M, rule, u)


@pytest.mark.parametrize("rule,f,M,T,u,r", [
    ("up", 0, 128, 10**6, 0, 0), ("up", 1, 128, 10**6, 0, 128), ("up", 127, 128, 10**6, 0, 128),
    ("up", 128, 128, 10**6, 0, 128), ("up", 129, 128, 10**6, 0, 256), ("up", 100, 128, 120, 0, 0),   # ceil > T
    ("down", 0, 128, 10**6, 0, 0), ("down", 127, 128, 10**6, 0, 0), ("down", 128, 128, 10**6, 0, 128),
    ("down", 255, 128, 10**6, 0, 128),
    # stochastic: ceil iff u * M < f - floor; u = 0.5 pads when f - floor > 64, u = 0 whenever f is not a multiple
    ("stochastic", 64, 128, 10**6, 0.5, 0), ("stochastic", 65, 128, 10**6, 0.5, 128), ("stochastic", 1, 128, 10**6, 0.0, 128),
    ("stochastic", 128, 128, 10**6, 0.0, 128), ("stochastic", 127, 128, 10**6, 0.9921875, 0),  # 0.9921875*128 = 127
    ("stochastic", 127, 128, 120, 0.0, 0), ("stochastic", 3, 4, 100, 0.74, 4), ("stochastic", 3, 4, 100, 0.75, 0),
])
def test_rounding_rules_table(rule, f, M, T, u, r):
    got = orc.round_and_sparsify(np.array([f]), M, T, rule, np.array([u], dtype=np.float32))
    assert int(got[0]) == r


@pytest.mark.parametrize("M", [4, 16, 128])
def test_stochastic_rounding_is_unbiased_over_a_uniform_grid(M):
    """Closed form: with the uniforms u_i = (i + 1/2)/M, i = 0..M-1, exactly f - floor of them pad, so the mean
    of the rounded count over the grid is f itself (the expected count equals the token-choice count)."""
    grid = (np.arange(M) + 0.5) / M
    for f in range(0, 3 * M + 1):
        r = [int(orc.round_and_sparsify(np.array([f]), M, 10**6, "stochastic", np.array([u]))[0]) for u in grid]
        assert sum(r) == f * M


def test_ec_per_expert_top_c_is_stable_argsort_and_gate_is_softmax():
    rng = np.random.default_rng(14)
    for seed in range(20):
        T, E, K = int(rng.integers(1, 300)), int(rng.integers(1, 12)), 1
        K = int(rng.integers(1, E + 1))
        z = rng.standard_normal((T, E)).astype(np.float32)
        if seed % 3 == 0:
            z = np.round(z * 2) / 2                          # heavy ties
        rt = orc.route_ec(z, K, 16)
        C = min(T, T * K // E)
        assert np.all(rt["counts"] == C) and rt["P"] == E * C
        prob = scipy.special.softmax(z.astype(np.float64), axis=1)
        for e in range(E):
            ref = np.sort(np.argsort(-z[:, e].astype(np.float64), kind="stable")[:C])
            sl = slice(rt["offsets"][e], rt["offsets"][e + 1])
            assert np.array_equal(rt["row_token"][sl], ref)
            assert np.allclose(rt["row_score"][sl], prob[ref, e], rtol=1e-14, atol=0)
            for t, k in zip(rt["row_token"][sl], rt["row_slot"][sl]):
                assert (k == -1 and e not in rt["topk_idx"][t]) or rt["topk_idx"][t, k] == e


@pytest.mark.parametrize("rule", orc.ROUNDING_RULES)
def test_tr_bruteforce_tiny(rule):
    rng = np.random.default_rng(4)
    for _ in range(40):
        T, E, K, M = int(rng.integers(2, 11)), 3, int(rng.integers(1, 3)), 4
        z = rng.choice([-1.0, -0.5, 0.0, 0.25, 0.5, 1.0], size=(T, E)).astype(np.float32)
        tc = orc.route_tc(z, K, M)
        tr = orc.route_tr(z, K, M, rule, rng.random(E))
        member = np.zeros((T, E), bool)
        for t in range(T):
            member[t, tc["topk_idx"][t]] = True
        for e in range(E):
            r = int(tr["counts"][e])
            # brute force: the r-subset whose descending key list is lexicographically largest
            best = None
            for S in itertools.combinations(range(T), r):
                key = sorted(((int(member[t, e]), float(z[t, e]), -t) for t in S), reverse=True)
                if best is None or key > best:
                    best, bestS = key, S
            kept = tr["row_token"][tr["offsets"][e]:tr["offsets"][e + 1]]
            assert list(kept) == sorted(bestS)


def test_tr_expected_total_unchanged():
    rng = np.random.default_rng(5)
    T, E, K, M = 4096, 64, 4, 128
    diffs = []
    for _ in range(100):
        z = rng.standard_normal((T, E)).astype(np.float32)
        tc = orc.route_tc(z, K, M)
        r = orc.round_and_sparsify(tc["counts"], M, T)
        diffs.append(int(r.sum()) - T * K)
    diffs = np.array(diffs, dtype=np.float64)
    # rounding to the nearest tile moves each expert by at most M/2 either way; the mean change of the
    # total stays within a few standard errors of zero (plus the half-token tie bias per expert)
    se = diffs.std(ddof=1) / np.sqrt(len(diffs))
    assert abs(diffs.mean()) <= 4 * se + E * 0.5
    assert abs(diffs.mean()) / (T * K) < 0.01


@pytest.mark.parametrize("mode", orc.ROUTE_MODES)
def test_offsets_and_tile_offsets_by_walking_the_rows(mode):
    """offsets and tile_offsets counted by walking each expert's rows: the expert's rows are the next counts[e]
    rows, and cutting them into M_tile blocks from the first row gives full blocks and at most one partial one."""
    rng = np.random.default_rng(7)
    for T, E, K, M in ((300, 8, 2, 128), (50, 6, 3, 4), (9, 5, 1, 4)):
        z = rng.standard_normal((T, E)).astype(np.float32)
        rt = orc.route(z, K, mode, M, u=rng.random(E).astype(np.float32))
        row, tile = 0, 0
        for e in range(E):
            assert rt["offsets"][e] == row and rt["tile_offsets"][e] == tile
            start = row
            while row < start + rt["counts"][e]:
                block = min(M, start + rt["counts"][e] - row)   # one block: M rows, or the partial last one
                assert 0 < block <= M
                assert all(rt["row_expert"][row:row + block] == e)
                row += block
                tile += 1
        assert rt["offsets"][E] == row == rt["P"] and rt["tile_offsets"][E] == tile


@pytest.mark.parametrize("fixture", ["tr_pad_and_drop.txt", "tr_tie_rounds_down.txt", "tr_rules_and_ec.txt"])
def test_routing_golden(fixture):
    g = load_golden(fixture)
    z = np.array(g["logits"], dtype=np.float32)
    for mode, exp in g["expect"].items():
        exp = dict(exp)
        u = np.array(exp.pop("u"), dtype=np.float32) if "u" in exp else None
        rt = orc.route(z, g["K"], mode, g["m_tile"], u=u)
        for key, val in exp.items():
            got = rt[key]
            if key in ("row_score", "topk_score"):
                assert np.allclose(np.ravel(got), val, rtol=1e-15, atol=0), key
            else:
                assert list(np.ravel(got).astype(np.int64)) == [int(v) for v in val], (mode, key)


# ------------------------------------------------------------------------------------- layer arithmetic


def _tiny_problem(seed=0, T=8, d=8, n=4, E=4, K=2):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, E)).astype(np.float32)
    rt = orc.route_tc(z, K, 4)
    X = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, d, 2 * n)) / np.sqrt(d)
    W2 = rng.standard_normal((E, n, d)) / np.sqrt(n)
    dO = rng.standard_normal((T, d))
    return rt, X, W1, W2, dO


def _loss(X, W1, W2, dO, rt, s=None):
    s = rt["row_score"] if s is None else s
    f = orc.forward(X, W1, W2, rt["row_token"], rt["row_expert"], s)
    return float((dO * f["O"]).sum())


def test_golden_single_row():
    g = load_golden("swiglu_single_row.txt")
    X = np.array(g["x"]).reshape(1, 2)
    W1 = np.array(g["W1"]).reshape(1, 2, 2)
    W2 = np.array(g["W2"]).reshape(1, 1, 2)
    dO = np.array(g["dO"]).reshape(1, 2)
    tok, ex, sc = np.array([0]), np.array([0]), np.array([1.0])
    f = orc.forward(X, W1, W2, tok, ex, sc)
    b = orc.backward(dO, X, W1, W2, tok, ex, sc, f)
    assert np.allclose(f["O"][0], g["O"], rtol=1e-15)
    assert np.allclose(b["dS"], g["dS"], rtol=1e-15)
    assert np.allclose(b["dH"][0], g["dgate"] + g["dup"], rtol=1e-14)
    assert np.allclose(b["dW2"][0, 0], [g["dS"][0]] * 2, rtol=1e-15)


@pytest.mark.parametrize("seed", [0, 1])
def test_finite_differences(seed):
    rt, X, W1, W2, dO = _tiny_problem(seed)
    f, b = orc.layer(X, W1, W2, dO, rt)
    h = 1e-6

    def fd(arr, setter):
        g = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            old = arr[i]
            arr[i] = old + h
            lp = setter()
            arr[i] = old - h
            lm = setter()
            arr[i] = old
            g[i] = (lp - lm) / (2 * h)
        return g

    L = lambda: _loss(X, W1, W2, dO, rt)
    for name, arr in (("dX", X), ("dW1", W1), ("dW2", W2)):
        g = fd(arr, L)
        err = np.abs(g - b[name]).max() / np.abs(b[name]).max()
        assert err <= 1e-6, (name, err)
    s = rt["row_score"].copy()
    g = fd(s, lambda: _loss(X, W1, W2, dO, rt, s))
    assert np.abs(g - b["dS"]).max() / np.abs(b["dS"]).max() <= 1e-6


def test_independent_autograd_derivation():
    """A per-token dense formulation differentiated by torch autograd in fp64 (not the oracle's chain rule)."""
    rt, X, W1, W2, dO = _tiny_problem(7, T=16, d=16, n=8, E=6, K=3)
    f, b = orc.layer(X, W1, W2, dO, rt)
    Xt = torch.tensor(X, requires_grad=True)
    W1t = torch.tensor(W1, requires_grad=True)
    W2t = torch.tensor(W2, requires_grad=True)
    st = torch.tensor(rt["topk_score"], requires_grad=True)
    n = W1.shape[2] // 2
    outs = []
    for t in range(X.shape[0]):
        acc = torch.zeros(X.shape[1], dtype=torch.float64)
        for k in range(rt["K"]):
            e = int(rt["topk_idx"][t, k])
            h = Xt[t] @ W1t[e]
            acc = acc + st[t, k] * ((torch.nn.functional.silu(h[:n]) * h[n:]) @ W2t[e])
        outs.append(acc)
    O = torch.stack(outs)
    (O * torch.tensor(dO)).sum().backward()
    assert np.allclose(O.detach().numpy(), f["O"], rtol=1e-12, atol=1e-13)
    assert np.allclose(Xt.grad.numpy(), b["dX"], rtol=1e-11, atol=1e-12)
    assert np.allclose(W1t.grad.numpy(), b["dW1"], rtol=1e-11, atol=1e-12)
    assert np.allclose(W2t.grad.numpy(), b["dW2"], rtol=1e-11, atol=1e-12)
    ds_dense = st.grad.numpy()[rt["row_token"], rt["row_slot"]]
    assert np.allclose(ds_dense, b["dS"], rtol=1e-11, atol=1e-12)


def test_dense_swiglu_mlp_special_case():
    """K = E = 1 with score 1: the layer is a dense SwiGLU MLP."""
    rng = np.random.default_rng(9)
    T, d, n = 12, 16, 8
    X = rng.standard_normal((T, d))
    W1 = rng.standard_normal((1, d, 2 * n))
    W2 = rng.standard_normal((1, n, d))
    rt = orc.route_tc(np.zeros((T, 1), np.float32), 1, 4)
    assert np.all(rt["row_score"] == 1.0)
    f = orc.forward(X, W1, W2, rt["row_token"], rt["row_expert"], rt["row_score"])
    lin = torch.nn.functional.linear
    xt = torch.tensor(X)
    h_gate = lin(xt, torch.tensor(W1[0][:, :n].T))
    h_up = lin(xt, torch.tensor(W1[0][:, n:].T))
    ref = lin(torch.nn.functional.silu(h_gate) * h_up, torch.tensor(W2[0].T)).numpy()
    assert np.allclose(f["O"], ref, rtol=1e-12, atol=1e-12)


def test_ds_via_h_equals_ds_via_y():
    rt, X, W1, W2, dO = _tiny_problem(11, T=32, d=24, n=8, E=5, K=2)
    f, b = orc.layer(X, W1, W2, dO, rt)
    ds2 = orc.ds_via_h(dO, W2, rt["row_token"], rt["row_expert"], f["H"])
    assert np.abs(ds2 - b["dS"]).max() <= 1e-12 * np.abs(b["dS"]).max()


def test_flop_count_by_counting_macs(monkeypatch):
    rt, X, W1, W2, dO = _tiny_problem(12, T=20, d=16, n=8, E=4, K=2)
    macs = []
    real = orc._matmul

    def counting(a, b):
        macs.append(a.shape[0] * a.shape[1] * b.shape[1])
        return real(a, b)

    monkeypatch.setattr(orc, "_matmul", counting)
    f = orc.forward(X, W1, W2, rt["row_token"], rt["row_expert"], rt["row_score"])
    fwd_macs = sum(macs)
    macs.clear()
    orc.backward(dO, X, W1, W2, rt["row_token"], rt["row_expert"], rt["row_score"], f)
    bwd_macs = sum(macs)
    P, n, d = rt["P"], 8, 16
    ff, bf = orc.layer_flops(P, n, d)
    assert 2 * fwd_macs == ff and 2 * bwd_macs == bf
    assert P == 20 * 2 and ff + bf == 18 * 20 * n * 2 * d       # (6+12) T n K d under token choice


def test_cached_bytes_are_x_and_h():
    T, d, n, K = 64, 32, 16, 4
    X = torch.empty((T, d), dtype=torch.bfloat16)
    H = torch.empty((T * K, 2 * n), dtype=torch.bfloat16)
    assert orc.cached_activation_bytes(T, d, n, T * K) == X.nbytes + H.nbytes


# ------------------------------------------------------------------------- planted mistakes are caught


def test_planted_sign_error_in_dgate_is_caught(monkeypatch):
    rt, X, W1, W2, dO = _tiny_problem(0)
    real_sigmoid = orc.sigmoid
    monkeypatch.setattr(orc, "sigmoid", lambda x: 1.0 - real_sigmoid(x))   # a wrong sigmoid in the backward
    f, b = orc.layer(X, W1, W2, dO, rt)
    h = 1e-6
    i = (0, 1, 0)
    old = W1[i]
    W1[i] = old + h
    lp = _loss(X, W1, W2, dO, rt)
    W1[i] = old - h
    lm = _loss(X, W1, W2, dO, rt)
    W1[i] = old
    assert abs((lp - lm) / (2 * h) - b["dW1"][i]) > 1e-4


def test_planted_transposed_tie_break_is_caught(monkeypatch):
    g = load_golden("tr_tie_rounds_down.txt")
    z = np.array(g["logits"], dtype=np.float32)
    real = orc.topk_token_choice

    def last_max(z, K):                              # ties to the higher expert index
        return real(np.asarray(z)[:, ::-1], K)[:, :] * -1 + (np.asarray(z).shape[1] - 1)

    monkeypatch.setattr(orc, "topk_token_choice", last_max)
    rt = orc.route_tc(z, g["K"], g["m_tile"])
    assert list(rt["topk_idx"].ravel()) != [int(v) for v in g["expect"]["tc"]["topk_idx"]]


# ------------------------------------------------------------------------------------------------ router


def _gate_loss(z, rt, dS, mode):
    """L = sum_r dS_r s_r, each gate exp(z_te - logsumexp of the token's normaliser set) via scipy."""
    L = 0.0
    for r in range(rt["P"]):
        t, e = int(rt["row_token"][r]), int(rt["row_expert"][r])
        N = np.arange(z.shape[1]) if mode == "ec" else rt["topk_idx"][t]
        L += dS[r] * np.exp(z[t, e] - scipy.special.logsumexp(z[t, N]))
    return L


def _router_problem(seed, mode, T=10, d=6, E=5, K=2, M=4):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, d))
    Wr = rng.standard_normal((d, E)) / np.sqrt(d)
    z = orc.router_logits(X, Wr)
    rt = orc.route(z.astype(np.float32), K, mode, M, u=rng.random(E))
    dS = rng.standard_normal(rt["P"])
    return X, Wr, z, rt, dS


@pytest.mark.parametrize("mode", ["tc", "tr", "tr_up", "ec"])
def test_router_dz_matches_finite_differences(mode):
    X, Wr, z, rt, dS = _router_problem(21, mode)
    dz = orc.router_dz(z, rt, dS, mode)
    h = 1e-6
    g = np.zeros_like(z)
    for i in np.ndindex(z.shape):
        zp, zm = z.copy(), z.copy()
        zp[i] += h
        zm[i] -= h
        g[i] = (_gate_loss(zp, rt, dS, mode) - _gate_loss(zm, rt, dS, mode)) / (2 * h)
    assert np.abs(g - dz).max() <= 1e-7 * max(np.abs(dz).max(), 1.0)


@pytest.mark.parametrize("mode", ["tc", "ec"])
def test_router_dz_equals_torch_softmax_autograd(mode):
    X, Wr, z, rt, dS = _router_problem(22, mode, T=24, E=7, K=3)
    zt = torch.tensor(z, requires_grad=True)
    if mode == "ec":
        s = torch.softmax(zt, dim=1)
        gates = s[torch.tensor(rt["row_token"]), torch.tensor(rt["row_expert"])]
    else:
        idx = torch.tensor(rt["topk_idx"])
        s = torch.softmax(torch.gather(zt, 1, idx), dim=1)
        gates = s[torch.tensor(rt["row_token"]), torch.tensor(rt["row_slot"])]
    (gates * torch.tensor(dS)).sum().backward()
    assert np.allclose(zt.grad.numpy(), orc.router_dz(z, rt, dS, mode), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("mode", orc.ROUTE_MODES)
def test_router_dz_rows_sum_to_zero(mode):
    """Adding a constant to all of a token's logits leaves every gate unchanged, so each row of dz sums to 0."""
    X, Wr, z, rt, dS = _router_problem(23, mode, T=64, E=8, K=3, M=8)
    dz = orc.router_dz(z, rt, dS, mode)
    assert np.abs(dz.sum(axis=1)).max() <= 1e-14 * max(np.abs(dz).max(), 1.0)
    assert np.abs(dz).max() > 0


def test_router_dz_is_zero_for_top1_token_choice():
    """K = 1: every gate is exp(z_te)/exp(z_te) = 1, whatever the logits."""
    X, Wr, z, rt, dS = _router_problem(24, "tc", K=1)
    assert np.all(orc.router_dz(z, rt, dS, "tc") == 0.0)


@pytest.mark.parametrize("mode", ["tc", "tr_down", "ec"])
def test_router_backward_through_x_and_wr(mode):
    X, Wr, z, rt, dS = _router_problem(25, mode, T=8, d=5, E=4, K=2)
    out = orc.router_backward(z, rt, dS, X, Wr, mode)
    assert np.allclose(orc.router_logits(X, Wr), torch.nn.functional.linear(torch.tensor(X), torch.tensor(Wr.T)).numpy(),
                       rtol=1e-14, atol=1e-15)
    h = 1e-6
    for name, arr in (("dX", X), ("dWr", Wr)):
        g = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            old = arr[i]
            arr[i] = old + h
            lp = _gate_loss(orc.router_logits(X, Wr), rt, dS, mode)
            arr[i] = old - h
            lm = _gate_loss(orc.router_logits(X, Wr), rt, dS, mode)
            arr[i] = old
            g[i] = (lp - lm) / (2 * h)
        assert np.abs(g - out[name]).max() <= 1e-7 * max(np.abs(out[name]).max(), 1.0), name


# -------------------------------------------------------------------- restriction used by sampled checks


def test_oracle_on_rows_equals_the_full_layer_where_the_rows_decide():
    """The full-size GPU checks run the oracle on a subset of rows: those of some tokens (their O and dX rows,
    and the rows' H and dS) or of one expert (its dW1 and dW2).  On a small layer that subset computation must
    equal the full oracle there, up to the last bits of fp64 (the library matmul may block a different number of
    rows differently)."""
    close = lambda a, b: np.allclose(a, b, rtol=1e-12, atol=1e-14)   # noqa: E731
    from gpu_util import oracle_on_rows

    w = synth.custom(300, 64, 32, 8, 2, skew=True)
    inp = synth.make_inputs(w, 3)
    ref = orc.route(inp["logits"].numpy(), w.K, "tr", 16)
    f64 = lambda t: t.double().numpy()                      # noqa: E731
    full_f, full_b = orc.layer(f64(inp["X"]), f64(inp["W1"]), f64(inp["W2"]), f64(inp["dO"]), ref)
    toks = np.array([0, 7, 150, 299])
    rows = np.nonzero(np.isin(ref["row_token"], toks))[0]
    _, fwd, bwd = oracle_on_rows(inp, ref, rows)
    assert close(fwd["O"][toks], full_f["O"][toks]) and close(bwd["dX"][toks], full_b["dX"][toks])
    assert close(fwd["H"], full_f["H"][rows]) and close(bwd["dS"], full_b["dS"][rows])
    assert not close(fwd["O"][toks] * 1.001, full_f["O"][toks])
    for e in np.nonzero(ref["counts"])[0][:3]:
        erows = np.arange(ref["offsets"][e], ref["offsets"][e + 1])
        experts, _, be = oracle_on_rows(inp, ref, erows)
        assert list(experts) == [e]
        assert close(be["dW1"][0], full_b["dW1"][e]) and close(be["dW2"][0], full_b["dW2"][e])
