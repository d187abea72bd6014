"""Pins of the oracle's router logits and selection (no GPU).

Selection rule: page spark_model/layers/moe_v41.rs, fn softplus and fn
route_from_logits -- scores sqrt(softplus(l / temp)), keys score + bias, ids
stably sorted by descending key, the first k picked, weights = unbiased
scores renormalised (+1e-20) when norm_topk_prob and k > 1, times
route_scale.
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from moe_decode_quantized_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _nearest_f32(fr: Fraction) -> set:
    """The f32 value(s) nearest to an exact rational."""
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    dist = [abs(Fraction(float(c)) - fr) for c in cands]
    best = min(dist)
    return {float(c) for c, d in zip(cands, dist) if d == best}


def test_router_logits_are_correctly_rounded_exact_sums():
    seed = 11
    m, n, dim = 3, 8, 512
    x = synth.x_bf16(seed, 0, m, dim)
    w = synth.router_bf16(seed, 0, n, dim)
    got = oracle.router_logits(x, w)
    xv, wv = _bf16_vals(x), _bf16_vals(w)
    for t in range(m):
        for e in range(n):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xv[t], wv[e]))
            assert float(got[t, e]) in _nearest_f32(exact), (t, e)


def test_golden_tiny_selection():
    vals = {}
    with open(os.path.join(GOLD, "route_tiny.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                vals[k] = [float(a) for a in v]
    c = oracle.cfg(256, 256, 4, 3, True, 1.0, 2.5, 7.0)
    picks, weights, scores, flags = oracle.route(c, np.array([vals["logits"]], np.float32),
                                                 np.array(vals["bias"], np.float32))
    assert list(picks[0]) == [int(v) for v in vals["picks"]]
    assert list(scores[0]) == [5.0, 6.0, 7.0, 8.0]
    den = np.float32(np.float32(vals["weights_den"][0]) + np.float32(1e-20))
    want = [np.float32(np.float32(np.float32(v) / den) * np.float32(2.5)) for v in vals["weights_num"]]
    assert [w.view(np.uint32) for w in weights[0]] == [w.view(np.uint32) for w in want]
    assert flags[0] == 0


def _keys(scores, bias):
    return (scores.astype(np.float32) + bias.astype(np.float32)).astype(np.float32)


def test_brute_force_over_all_subsets_tiny_layer():
    """n = 16, k = 2 (the tiny layer): the pick set is the one 2-subset whose members all
    rank before every other expert (larger key, or equal key and lower id)."""
    c = oracle.cfg(256, 256, 16, 2)
    rng = np.random.default_rng(12)
    for trial in range(40):
        logits = (rng.standard_normal((1, 16)) * 1.5).astype(np.float32)
        bias = synth.uniform_f32(synth.tensor_key(trial, 0, synth.T_BIAS), 16, -0.1, 0.1)
        if trial % 4 == 0:     # force ties
            logits = synth.round_to_grid(logits, 0.5)
            bias = synth.round_to_grid(bias, 0.25)
        picks, weights, scores, _ = oracle.route(c, logits, bias)
        key = _keys(scores[0], bias)

        def before(a, b):
            return key[a] > key[b] or (key[a] == key[b] and a < b)
        ok = [S for S in itertools.combinations(range(16), 2)
              if all(before(i, j) for i in S for j in range(16) if j not in S)]
        assert len(ok) == 1
        assert set(picks[0]) == set(ok[0])
        assert before(picks[0][0], picks[0][1])


@pytest.mark.parametrize("norm", [True, False])
def test_invariants_full_size(norm):
    """384 experts, top 6: distinct picks, non-increasing keys, ties by ascending id, the
    ranking equal to Python's stable sort, weights summing to route_scale."""
    c = oracle.cfg(4096, 2048, 384, 6, norm, 1.0, 2.5, 7.0)
    seed = 13
    for batch in range(4):
        logits = (synth.normal_f32(synth.tensor_key(seed, batch, synth.T_LOGITS), 8 * 384, 1.3)
                  .reshape(8, 384))
        bias = synth.bias_f32(seed, batch, 384)
        picks, weights, scores, flags = oracle.route(c, logits, bias)
        for t in range(8):
            key = _keys(scores[t], bias)
            order = sorted(range(384), key=lambda e: -float(key[e]))   # stable: ties keep id order
            assert list(picks[t]) == order[:6]
            assert len(set(picks[t])) == 6
            s = scores[t][picks[t]]
            if norm:
                tot = np.float64(weights[t].astype(np.float64).sum())
                assert abs(tot - 2.5) <= 6 * 2 * np.spacing(np.float32(2.5))
                assert np.all(weights[t] > 0)
            else:
                np.testing.assert_array_equal(weights[t], (s * np.float32(2.5)).astype(np.float32))


def test_tie_stress_ranking():
    """Logits and bias on a 2^-4 grid: many exact key ties; equal keys rank by ascending id."""
    c = oracle.cfg(4096, 2048, 384, 6, True, 1.0, 2.5, 7.0)
    logits = synth.tie_logits(21, 0, 8, 384)
    bias = synth.round_to_grid(synth.bias_f32(21, 0, 384))
    picks, weights, scores, flags = oracle.route(c, logits, bias)
    n_ties = 0
    for t in range(8):
        key = _keys(scores[t], bias)
        order = sorted(range(384), key=lambda e: -float(key[e]))
        assert list(picks[t]) == order[:6]
        n_ties += sum(1 for a, b in zip(order[:7], order[1:8]) if key[a] == key[b])
    assert n_ties > 0, "the tie-stress input must produce ties near the top"


def test_topk_one_is_not_renormalised():
    c = oracle.cfg(256, 256, 16, 1, True, 1.0, 2.5, 7.0)
    logits = np.linspace(-2, 2, 16, dtype=np.float32)[None]
    bias = np.zeros(16, np.float32)
    picks, weights, scores, _ = oracle.route(c, logits, bias)
    assert picks[0, 0] == 15
    assert weights[0, 0] == np.float32(scores[0, 15] * np.float32(2.5))


def test_nonfinite_logits_are_flagged_and_nan_ranks_last():
    c = oracle.cfg(256, 256, 16, 3, True, 1.0, 2.5, 7.0)
    logits = np.zeros((2, 16), np.float32)
    logits[0, 3] = np.nan
    logits[0, 5] = np.inf
    logits[1, :] = np.nan
    logits[1, 7] = 1.0
    bias = np.zeros(16, np.float32)
    picks, weights, scores, flags = oracle.route(c, logits, bias)
    assert flags[0] & 2 and flags[1] & 2
    assert picks[0, 0] == 5                 # +inf key first
    assert 3 not in picks[0]                # NaN never beats a number
    assert list(picks[1]) == [7, 0, 1]      # one number, then NaNs by ascending id


def test_temperature_divides_in_f32():
    s1, _ = oracle.score(3.0, 2.0)
    s2, _ = oracle.score(1.5, 1.0)
    assert s1 == s2


@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_weight_tolerance_covers_logit_perturbations(temp):
    """The bound the GPU tests use for weights against the oracle (helpers'
    assert_weights_close): perturbing the oracle's logits by at most dl moves
    each renormalised weight by at most dl / temp relatively (plus roundings),
    whenever the picks stay the same."""
    from helpers import assert_weights_close
    import moe_decode_quantized_gb300 as moe
    cfg = moe.Config(dim=4096, inter=2048, n_routed=384, topk=6, gate_temp=temp)
    c = oracle.cfg(4096, 2048, 384, 6, True, temp, 2.5, 7.0)
    rng = np.random.default_rng(5)
    checked = 0
    for trial in range(40):
        logits = rng.normal(0, 1.5, (1, 384)).astype(np.float32)
        bias = rng.uniform(-0.1, 0.1, 384).astype(np.float32)
        dl = float(10.0 ** rng.uniform(-7, -4))
        moved = (logits + rng.uniform(-dl, dl, logits.shape)).astype(np.float32)
        dl_real = float(np.abs(moved.astype(np.float64) - logits).max())
        p0, w0, _, _ = oracle.route(c, logits, bias)
        p1, w1, _, _ = oracle.route(c, moved, bias)
        if list(p0[0]) != list(p1[0]):
            continue
        assert_weights_close(cfg, w1[0], w0[0], dl_real)
        checked += 1
    assert checked >= 30


def _golden_plan():
    rows = {}
    with open(os.path.join(GOLD, "plan_m2.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *vals = line.split()
                rows[key] = vals
    return rows


def test_plan_layout_golden_m2():
    """The two-token header / plan / pointer table worked by hand
    (tests/golden/plan_m2.txt) against the oracle's plan."""
    g = _golden_plan()
    m, k, n = int(g["m"][0]), int(g["k"][0]), int(g["n"][0])
    picks = np.array([[int(v) for v in g[f"picks{t}"]] for t in range(m)], np.int32)
    weights = np.array([[float(v) for v in g[f"weights{t}"]] for t in range(m)], np.float32)
    slots = np.array([int(v) for v in g["slots"]], np.int32)
    arena = [int(v, 16) for v in g["arena"]]
    hdr, pw, pr, ptrs, ne = oracle.plan(picks, weights, None, slots, arena, n)
    hw = 1 + 3 * k
    for t in range(m):
        assert [int(v) for v in hdr[t * hw:(t + 1) * hw]] == [int(v, 0) for v in g[f"row{t}"]], t
    po, cap = m * hw, m * k
    assert ne == int(g["ne"][0]) == hdr[po]
    assert list(hdr[po + 1:po + 2 + ne]) == [int(v) for v in g["pair_start"]]
    assert list(hdr[po + 2 + cap:po + 2 + cap + ne]) == [int(v) for v in g["plan_expert"]]
    # words the layout leaves unused are not written
    assert list(hdr[po + 2 + ne:po + 2 + cap]) == [-7] * (cap - ne)
    assert list(hdr[po + 2 + cap + ne:]) == [-7] * (cap - ne)
    assert list(pr) == [int(v) for v in g["plan_rows"]]
    assert list(pw) == [float(v) for v in g["plan_w"]]
    for which, off in (("gate", 0), ("up", cap), ("down", 2 * cap)):
        assert [int(v) for v in ptrs[off:off + ne]] == [int(v, 16) for v in g[which]], which


def test_plan_flags_and_single_token():
    """At m = 1 the layout is the pages' own (1 + 3k header words, then the
    plan's ne and its one-pair-per-expert starts); the non-finite flag
    carries into the status word."""
    picks = np.array([[4, 0, 2]], np.int32)
    weights = np.array([[0.5, 0.25, 0.25]], np.float32)
    slots = np.array([3, -1, 1, -1, 0], np.int32)
    hdr, pw, pr, ptrs, ne = oracle.plan(picks, weights, np.array([2]), slots, (0, 0x100, 0, 0x10, 0x20), 5)
    assert hdr[0] == 2                          # non-finite; every pick resident
    assert list(hdr[7:10]) == [3, 1, 0]         # slots of 0, 2, 4 in ascending id
    hdr2 = oracle.plan(np.array([[1, 4, 2]], np.int32), weights, None, slots, (0, 0x100, 0, 0x10, 0x20), 5)[0]
    assert hdr2[0] == 1 and list(hdr2[7:10]) == [0, 1, 0]  # expert 1 missing: slot 0 and the miss bit
    assert ne == 3 and list(hdr[11:15]) == [0, 1, 2, 3]
    assert len(hdr) == 18 and list(hdr[15:18]) == [0, 2, 4]
    assert list(pw) == [0.25, 0.25, 0.5] and list(pr) == [0, 0, 0]


def test_pick_comparison_allows_an_order_swap_only_between_near_equal_keys():
    """The GPU tests compare picks in order, except where two of the k best
    keys are closer than the logit tolerance can resolve: then as a set, with
    the weights matched by pick."""
    from helpers import match_picks, near_tie, order_near_tie, tiny_cfg
    cfg = tiny_cfg(1)  # 16 experts, top 2
    bias = np.zeros(16, np.float32)
    logits = np.zeros((1, 16), np.float32)
    logits[0, 3], logits[0, 7] = 2.0, np.float32(2.0) + np.float32(2.0 ** -22)
    assert order_near_tie(cfg, logits, bias, 0) and not near_tie(cfg, logits, bias, 0)
    w, rw = match_picks(cfg, [3, 7], [0.4, 0.6], [7, 3], [0.6, 0.4], logits, bias, 0)
    assert w.tolist() == rw.tolist()
    with pytest.raises(AssertionError):
        match_picks(cfg, [3, 8], [0.4, 0.6], [7, 3], [0.6, 0.4], logits, bias, 0)
    logits[0, 7] = 3.0  # well separated: the order itself must match
    assert not order_near_tie(cfg, logits, bias, 0)
    with pytest.raises(AssertionError):
        match_picks(cfg, [3, 7], [0.4, 0.6], [7, 3], [0.6, 0.4], logits, bias, 0)
