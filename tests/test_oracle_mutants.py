"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle's source (a dropped term, a wrong sign, a wrong index or axis, swapped
operands, a flipped comparison or tie-break), re-runs the named pins of tests/test_oracle.py against that wrong
oracle in a child pytest process, and requires that at least one of them fails.  The pins compare the oracle with
facts it does not compute itself (finite differences, autograd, library routines, brute force, hand-worked
fixtures, closed forms), so a mistake that none of them notices would be a hole in the parity evidence.
"""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle", "moe_oracle.py")

FD = "finite_differences or autograd"
# (what the mistake is, the oracle's line, the line with the mistake, the pins expected to notice it)
MUTANTS = [
    # forward
    ("silu with the wrong sign", "return x / (1.0 + np.exp(-x))", "return x / (1.0 + np.exp(x))",
     "dense_swiglu or golden_single_row"),
    ("gate and up swapped in SwiGLU", "Ae = silu(He[:, :n]) * He[:, n:]", "Ae = He[:, :n] * silu(He[:, n:])",
     "dense_swiglu or ds_via_h or " + FD),
    ("tokens gathered by row index", "Xe = X[toks]", "Xe = X[sel]", FD),
    ("score dropped from the aggregation", "O[row_token[sel]] += row_score[sel, None] * Y[sel]",
     "O[row_token[sel]] += Y[sel]", FD),
    # backward
    ("score dropped from dY", "dYe = row_score[sel, None] * dOe", "dYe = dOe", FD),
    ("dS weighted by the score", "dS[sel] = (dOe * Y[sel]).sum(axis=1)", "dS[sel] = (dYe * Y[sel]).sum(axis=1)",
     "ds_via_h or " + FD),
    ("dW2 from the unweighted dO", "dW2[e] = _matmul(A[sel].T, dYe)", "dW2[e] = _matmul(A[sel].T, dOe)", FD),
    ("dgate without its second term", "dg = dAe * u * sg * (1.0 + g * (1.0 - sg))", "dg = dAe * u * sg", FD),
    ("dup with the wrong sign", "du = dAe * g * sg", "du = -dAe * g * sg", FD),
    ("dW1 gathers X by row index", "dW1[e] = _matmul(X[toks].T, dHe)", "dW1[e] = _matmul(X[sel].T, dHe)", FD),
    ("dX rows overwritten, not summed", "dX[row_token[sel]] += dXt[sel]", "dX[row_token[sel]] = dXt[sel]", FD),
    ("dS via H without SiLU", "a = silu(H[sel, :n]) * H[sel, n:]", "a = H[sel, :n] * H[sel, n:]", "ds_via_h"),
    # token-choice routing
    ("top-K ties to the higher expert", "j = np.argmax(work, axis=1)",
     "j = work.shape[1] - 1 - np.argmax(work[:, ::-1], axis=1)", "topk_bruteforce or routing_golden"),
    ("top-K keeps the chosen expert in play", "work[rows, j] = -np.inf", "work[rows, j] = work[rows, j]",
     "topk_equals_stable_argsort"),
    ("gate normaliser over all experts", "den = np.exp(zs - z0[:, None]).sum(axis=1)",
     "den = np.exp(z - z0[:, None]).sum(axis=1)", "scores_are_softmax or routing_golden"),
    ("an expert's rows in descending token order", "toks = np.nonzero(member[:, e])[0]",
     "toks = np.nonzero(member[:, e])[0][::-1]", "routing_golden"),
    ("row score taken from slot 0", "expert_rows.append((toks, slots, score[toks, slots]))",
     "expert_rows.append((toks, slots, score[toks, 0]))", "routing_golden"),
    ("M-tile count rounded down", "tiles = -((-counts) // m_tile)", "tiles = counts // m_tile",
     "walking_the_rows"),
    ("offsets as an inclusive scan", "offsets[1:] = np.cumsum(counts)", "offsets[:-1] = np.cumsum(counts)",
     "walking_the_rows or routing_golden"),
    # token rounding
    ("a rounding tie pads up", "up = (hi - f) < (f - lo)", "up = (hi - f) <= (f - lo)",
     "round_and_sparsify_table or routing_golden"),
    ("padding beyond T allowed", "up = up & (hi <= T)", "up = up", "round_and_sparsify_table or rules_table"),
    ("stochastic comparison flipped", "up = u * m_tile < (f - lo)", "up = u * m_tile > (f - lo)",
     "rules_table or unbiased"),
    ("always-down pads up", "up = np.zeros(f.shape, dtype=bool)", "up = np.ones(f.shape, dtype=bool)",
     "rules_table"),
    ("expert-choice candidates ranked before token choice", "order = np.lexsort((tok, -z[:, e], ~member[:, e]))",
     "order = np.lexsort((tok, -z[:, e], member[:, e]))", "tr_invariants or tr_bruteforce or routing_golden"),
    ("token-rounding ties to the higher token", "order = np.lexsort((tok, -z[:, e], ~member[:, e]))",
     "order = np.lexsort((-tok, -z[:, e], ~member[:, e]))", "tr_bruteforce or routing_golden"),
    ("token-rounding candidates by ascending logit", "order = np.lexsort((tok, -z[:, e], ~member[:, e]))",
     "order = np.lexsort((tok, z[:, e], ~member[:, e]))", "tr_invariants or tr_bruteforce or routing_golden"),
    ("kept rows left in rank order", "kept = np.sort(order[: r[e]])", "kept = order[: r[e]]",
     "tr_bruteforce or routing_golden"),
    ("added pair scored with its own logit as the maximum", "s = np.exp(z[kept, e] - z0[kept]) / den[kept]",
     "s = 1.0 / den[kept]", "tr_bruteforce or routing_golden"),
    # expert choice
    ("expert-choice capacity rounded up", "return min(T, (T * K) // E)", "return min(T, -((-T * K) // E))",
     "ec_per_expert or routing_golden"),
    ("expert-choice gate normalised over tokens", "return ex / ex.sum(axis=1, keepdims=True)",
     "return ex / ex.sum(axis=0, keepdims=True)", "ec_per_expert or routing_golden"),
    ("expert choice ties to the higher token", "order = np.lexsort((tok, -z[:, e]))",
     "order = np.lexsort((-tok, -z[:, e]))", "ec_per_expert or routing_golden"),
    # router
    ("router: the own-logit term with the wrong sign", "dz[t, e] += dS[r] * s_r", "dz[t, e] -= dS[r] * s_r",
     "router_dz"),
    ("router: the normaliser term dropped", "dz[t, N] -= dS[r] * s_r * s_N", "dz[t, N] -= 0.0 * s_N", "router_dz"),
    ("router: expert choice normalised over the top-K",
     'N = np.arange(E) if mode == "ec" else np.asarray(rt["topk_idx"][t])', 'N = np.asarray(rt["topk_idx"][t])',
     "router_dz"),
    ("router: dX with the wrong sign", "dX = _matmul(dz, np.asarray(Wr, np.float64).T)",
     "dX = -_matmul(dz, np.asarray(Wr, np.float64).T)", "router_backward_through"),
    ("router: dW_r from the logits", "dWr = _matmul(np.asarray(X, np.float64).T, dz)",
     "dWr = _matmul(np.asarray(X, np.float64).T, z - z.mean())", "router_backward_through"),
    # more lines of the same functions
    ("gate exponent with the wrong sign", "return np.exp(zs - z0[:, None]) / den[:, None]",
     "return np.exp(z0[:, None] - zs) / den[:, None]", "scores_are_softmax or routing_golden"),
    ("token-rounding slot looked up in expert 0", "slots = slot_of[kept, e]", "slots = slot_of[kept, 0]",
     "routing_golden or tr_bruteforce"),
    ("expert-choice slot looked up in expert 0", "expert_rows.append((kept, slot_of[kept, e], prob[kept, e]))",
     "expert_rows.append((kept, slot_of[kept, 0], prob[kept, e]))", "routing_golden or ec_per_expert"),
    ("router: token rounding normalised over all experts",
     'N = np.arange(E) if mode == "ec" else np.asarray(rt["topk_idx"][t])', "N = np.arange(E)", "router_dz"),
    ("down-projection fed the gate instead of A", "Ye = _matmul(Ae, W2[e])", "Ye = _matmul(He[:, :n], W2[e])",
     "dense_swiglu or ds_via_h or " + FD),
    ("dX from the gate half of dH only", "dXt[sel] = _matmul(dHe, W1[e].T)",
     "dXt[sel] = _matmul(np.concatenate([dg, 0 * du], axis=1), W1[e].T)", FD),
    # accounting
    ("backward FLOPs counted as the forward's", "return 6 * P * n * d, 12 * P * n * d",
     "return 6 * P * n * d, 6 * P * n * d", "flop_count"),
    ("H cached at half its size", "return 2 * T * d + 4 * P * n", "return 2 * T * d + 2 * P * n", "cached_bytes"),
]


def test_every_planted_line_is_in_the_oracle():
    with open(ORACLE) as f:
        src = f.read()
    for name, old, new, _ in MUTANTS:
        assert src.count(old) == 1, name
        assert old != new, name


def _run_pins_against(old, new, pins):
    env = dict(os.environ, MOE_ORACLE_MUTANT=json.dumps([old, new]))
    tag = f"{abs(hash((old, new))):x}"   # each child gets a temporary directory of its own
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"), "-x", "-q",
           "-p", "no:cacheprovider", "-m", "not gpu", "-k", pins,
           "--basetemp", os.path.join(ROOT, ".pytest_tmp_children", tag)]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def outcomes():
    """Every mutant's child run, several at a time (they are independent processes)."""
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as pool:
        futures = {name: pool.submit(_run_pins_against, old, new, pins) for name, old, new, pins in MUTANTS}
        return {name: f.result() for name, f in futures.items()}


@pytest.mark.parametrize("name,pins", [(m[0], m[3]) for m in MUTANTS], ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(outcomes, name, pins):
    r = outcomes[name]
    # exit code 1: tests ran and at least one failed (5 would mean the pin expression selected nothing)
    assert r.returncode == 1, f"{name}: pins {pins!r} did not fail (exit {r.returncode})\n{r.stdout[-3000:]}"
