"""Pins of the float64 oracle to facts fixed outside the oracle itself.

Each test ties an oracle function to a value the pages print (fixtures under
tests/golden/, each citing its section), a closed form, brute-force
enumeration, or an invariant of the method.  No GPU is used.
"""

import itertools
import math

import numpy as np
import pytest

from oracle import moe_oracle as O

ABS3 = 5e-4  # the pages print 3 decimals


# ---------------------------------------------------------------------------
# Gating worked example ("路由器怎样选专家：top-k 与两种门控")
# ---------------------------------------------------------------------------

def test_worked_example_softmax(golden):
    g = golden("moe10_gating_worked_example.json")
    z = np.array([g["logits"]])
    p = O.softmax(z)[0]
    np.testing.assert_allclose(p, g["softmax"]["scores"], atol=ABS3)
    idx = O.topk_experts(z, g["k"])
    assert idx[0].tolist() == g["chosen"]
    w = O.topk_weights(O.softmax(z), idx, renormalize=True)[0]
    np.testing.assert_allclose(w, g["softmax"]["renormalized"], atol=ABS3)


def test_worked_example_sigmoid_scaled(golden):
    g = golden("moe10_gating_worked_example.json")
    z = np.array([g["logits"]])
    s = O.sigmoid(z)[0]
    np.testing.assert_allclose(s, g["sigmoid"]["scores"], atol=ABS3)
    idx = O.topk_experts(z, g["k"])
    assert idx[0].tolist() == g["chosen"]
    w1 = O.topk_weights(O.sigmoid(z), idx, renormalize=True)[0]
    np.testing.assert_allclose(w1, g["sigmoid"]["renormalized"], atol=ABS3)
    rsf = g["sigmoid"]["routed_scaling_factor"]
    w = O.topk_weights(O.sigmoid(z), idx, renormalize=True, routed_scaling_factor=rsf)[0]
    np.testing.assert_allclose(w, g["sigmoid"]["scaled"], atol=ABS3)
    # the page: the selected weights sum to 1 (softmax) or 2.5 (DeepSeek-V3)
    assert abs(w.sum() - 2.5) < 1e-12


@pytest.mark.parametrize("gate,rsf,key", [("softmax", 1.0, "renormalized"),
                                          ("sigmoid", 2.5, "scaled")])
def test_worked_example_through_route(golden, gate, rsf, key):
    # the full routing entry (gate dispatch, top-k, weights) on the page's example
    g = golden("moe10_gating_worked_example.json")
    z = np.array([g["logits"]])
    r = O.route(z, g["k"], gate, True, rsf, None)
    np.testing.assert_allclose(r["scores"][0], g[gate]["scores"], atol=ABS3)
    assert r["topk_idx"][0].tolist() == g["chosen"]
    np.testing.assert_allclose(r["topk_w"][0], g[gate][key], atol=ABS3)
    with pytest.raises(ValueError):
        O.gate_scores(z, "relu")


def test_top2_softmax_renorm_closed_form():
    # renormalised top-2 softmax weight of the best expert is sigma(z1 - z2):
    # exp(z1) / (exp(z1) + exp(z2)) = 1 / (1 + exp(z2 - z1)); independent of
    # the other logits.
    rng = np.random.default_rng(1)
    z = rng.normal(size=(50, 6))
    idx = O.topk_experts(z, 2)
    w = O.topk_weights(O.softmax(z), idx, renormalize=True)
    for t in range(z.shape[0]):
        z1, z2 = z[t, idx[t, 0]], z[t, idx[t, 1]]
        assert z1 >= z2
        assert abs(w[t, 0] - 1.0 / (1.0 + math.exp(z2 - z1))) < 1e-14
        assert abs(w[t].sum() - 1.0) < 1e-14


def test_softmax_sigmoid_closed_values():
    # sigma(ln 3) = 3/4 and sigma(-ln 3) = 1/4 exactly; softmax of [ln a_i]
    # is a_i / sum a.
    s = O.sigmoid(np.array([math.log(3.0), -math.log(3.0), 0.0]))
    np.testing.assert_allclose(s, [0.75, 0.25, 0.5], rtol=1e-15)
    a = np.array([1.0, 2.0, 3.0, 4.0])
    np.testing.assert_allclose(O.softmax(np.log(a)[None])[0], a / 10.0, rtol=1e-14)
    # shift invariance of softmax only holds if the max shift is exact
    np.testing.assert_allclose(O.softmax(np.log(a)[None] + 700.0)[0], a / 10.0, rtol=1e-13)


def test_mean_prob_sums_to_one_softmax():
    rng = np.random.default_rng(2)
    z = rng.normal(size=(37, 9))
    P = O.mean_router_prob(O.softmax(z))
    assert abs(P.sum() - 1.0) < 1e-13
    # sigmoid means are each in (0, 1) and equal the plain column mean
    P2 = O.mean_router_prob(O.sigmoid(z))
    assert np.all((P2 > 0) & (P2 < 1))


# ---------------------------------------------------------------------------
# Top-k selection against brute force over all expert subsets
# ---------------------------------------------------------------------------

def _brute_topk(zrow, k):
    """Best k-subset by sum of logits; among equal sums, the lexicographically
    smallest sorted index tuple (the lowest-index tie rule)."""
    best, best_key = None, None
    for sub in itertools.combinations(range(len(zrow)), k):
        key = (-sum(zrow[list(sub)]), sub)
        if best_key is None or key < best_key:
            best, best_key = sub, key
    return sorted(best, key=lambda e: (-zrow[e], e))


@pytest.mark.parametrize("E,k", [(4, 2), (8, 2), (6, 3), (5, 1), (7, 7)])
def test_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 100 + k)
    z = rng.normal(size=(40, E))
    # forced ties: quantised logits and all-equal rows
    zq = np.round(rng.normal(size=(40, E)) * 2) / 2
    zeq = np.zeros((3, E))
    for arr in (z, zq, zeq):
        idx = O.topk_experts(arr, k)
        for t in range(arr.shape[0]):
            assert idx[t].tolist() == _brute_topk(arr[t], k)


def test_topk_ties_go_to_lower_index():
    z = np.array([[1.0, 3.0, 3.0, 1.0, 3.0]])
    assert O.topk_experts(z, 2)[0].tolist() == [1, 2]
    assert O.topk_experts(z, 4)[0].tolist() == [1, 2, 4, 0]


# ---------------------------------------------------------------------------
# Capacity and dispatch ("负载不均：路由坍缩与丢 token")
# ---------------------------------------------------------------------------

def test_capacity_worked_example(golden):
    g = golden("moe10_capacity_example.json")
    idx = np.array(g["choice"]).reshape(g["T"], g["k"])
    for case in g["cases"]:
        C = O.expert_capacity(g["T"], g["E"], case["capacity_factor"])
        assert C == case["capacity"]
        r = O.dispatch(idx, g["E"], C)
        dropped = [t for t in range(g["T"]) if r["drop_mask"][t]]
        assert dropped == case["dropped_tokens"]
        assert int(r["drops"].sum()) == case["n_dropped"]


def test_capacity_formula_values():
    assert O.expert_capacity(8, 4, 1.25) == 3          # 2 x 1.25 = 2.5 -> 3
    assert O.expert_capacity(16384, 64, 1.25) == 320   # Switch-shaped layer
    assert O.expert_capacity(8, 4, None) is None


def _check_dispatch_invariants(idx, E, C, r):
    T, k = idx.shape
    A = T * k
    counts, drops, offsets, perm = r["counts"], r["drops"], r["offsets"], r["perm"]
    assert counts.sum() + drops.sum() == A
    if C is not None:
        assert np.all(counts <= C)
        # an expert drops only when full
        assert np.all((drops == 0) | (counts == C))
    assert offsets[0] == 0 and np.all(np.diff(offsets) == counts)
    n = offsets[E]
    kept = sorted(int(a) for a in perm[:n])
    assert kept == [a for a in range(A) if r["drop_mask"][a] == 0]
    flat = idx.reshape(A)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)       # ascending assignment id
    for a in range(A):
        if r["drop_mask"][a]:
            assert r["row_of"][a] == -1
        else:
            assert perm[r["row_of"][a]] == a
    # fill order: every dropped assignment comes after all kept ones of its expert
    for e in range(E):
        ids = [a for a in range(A) if flat[a] == e]
        dm = [r["drop_mask"][a] for a in ids]
        assert dm == sorted(dm)


@pytest.mark.parametrize("cf", [None, 0.5, 1.0, 1.25, 3.0])
def test_dispatch_invariants_random(cf):
    rng = np.random.default_rng(7)
    T, E, k = 53, 6, 2
    z = rng.normal(size=(T, E)) + np.linspace(1.5, 0, E)   # skewed load
    idx = O.topk_experts(z, k)
    C = O.expert_capacity(T, E, cf)
    r = O.dispatch(idx, E, C)
    _check_dispatch_invariants(idx, E, C, r)


def test_dispatch_capacity_zero_and_large():
    idx = np.array([[0, 1], [1, 0], [0, 2]])
    r0 = O.dispatch(idx, 3, 0)
    assert r0["counts"].tolist() == [0, 0, 0] and r0["drops"].tolist() == [3, 2, 1]
    r9 = O.dispatch(idx, 3, 99)
    assert r9["drops"].sum() == 0
    assert r9["perm"][:6].tolist() == [0, 3, 4, 1, 2, 5]


# ---------------------------------------------------------------------------
# Balance term ("辅助损失") and parameter accounting ("总参数和激活参数怎样算")
# ---------------------------------------------------------------------------

def test_aux_loss_worked_values(golden):
    for c in golden("moe10_aux_loss_example.json")["cases"]:
        assert abs(O.switch_balance_term(c["f"], c["P"]) - c["value"]) < 1e-12


def test_load_fractions_from_counts():
    f = O.load_fractions(np.array([3, 1, 1, 1]), np.array([2, 0, 0, 0]))
    np.testing.assert_allclose(f, [5 / 8, 1 / 8, 1 / 8, 1 / 8], rtol=1e-15)


def test_mixtral_param_closed_form(golden):
    m = golden("moe10_param_counts.json")["mixtral_8x7b"]
    d, E, k, F = m["d"], m["E"], m["k"], m["F"]
    assert O.moe_layer_params(d, 1, F) - d == m["per_expert"]
    assert O.moe_layer_params(d, E, 0) == m["router_per_layer"]
    rest = m["attention_per_layer"] + m["norms_per_layer"]
    total = m["layers"] * (rest + O.moe_layer_params(d, E, F)) + m["embed_and_head"] + m["final_norm"]
    active = m["layers"] * (rest + O.moe_layer_params(d, E, F, k=k)) + m["embed_and_head"] + m["final_norm"]
    assert total == m["total"]
    assert active == m["active"]


def test_deepseek_v3_param_closed_form(golden):
    m = golden("moe10_param_counts.json")["deepseek_v3"]
    d, E, k, F, Fs, L = m["d"], m["E"], m["k"], m["F"], m["F_s"], m["moe_layers"]
    assert O.moe_layer_params(d, 1, F) - d == m["per_expert"]
    fixed = m["mla_all_layers"] + m["dense_ffn_first_3"] + m["embed_and_head"] + m["norms"]
    assert fixed + L * O.moe_layer_params(d, E, F, Fs) == m["total"]
    assert fixed + L * O.moe_layer_params(d, E, F, Fs, k=k) == m["active"]


def test_decode_expert_usage(golden):
    u = golden("moe10_param_counts.json")["decode_usage"]
    for B, pct in u["batch_to_percent"].items():
        frac = O.expected_touched_experts(u["E"], u["k"], int(B)) / u["E"]
        assert round(100 * frac) == pct


# ---------------------------------------------------------------------------
# Expert FFN closed forms
# ---------------------------------------------------------------------------

def test_silu_closed_values():
    # SiLU(u) = u sigma(u); sigma(ln 3) = 3/4 exactly
    u = np.array([math.log(3.0), -math.log(3.0), 0.0])
    np.testing.assert_allclose(O.silu(u), [0.75 * math.log(3.0), -0.25 * math.log(3.0), 0.0],
                               rtol=1e-15, atol=1e-300)


def test_swiglu_permutation_experts():
    # One-hot weights make every projection a coordinate pick, so the FFN is a
    # closed form that changes if any operand is transposed:
    #   gate_f = x[pg[f]], up_f = x[pu[f]], y_i = h[pd[i]]
    d, F = 3, 4
    pg, pu, pd = [2, 0, 1, 2], [1, 1, 0, 2], [3, 0, 2]
    Wg = np.zeros((F, d)); Wu = np.zeros((F, d)); Wd = np.zeros((d, F))
    for f in range(F):
        Wg[f, pg[f]] = 1.0
        Wu[f, pu[f]] = 1.0
    for i in range(d):
        Wd[i, pd[i]] = 1.0
    x = np.array([[math.log(3.0), 2.0, -math.log(3.0)]])
    sil = {0: 0.75 * math.log(3.0), 2: -0.25 * math.log(3.0)}   # SiLU(x[c]) for c=0,2
    sil[1] = 2.0 / (1.0 + math.exp(-2.0))
    h = [sil[pg[f]] * x[0, pu[f]] for f in range(F)]
    want = [h[pd[i]] for i in range(d)]
    np.testing.assert_allclose(O.swiglu_ffn(x, Wg, Wu, Wd)[0], want, rtol=1e-14)


def test_router_logits_hand_example():
    x = np.array([[1.0, 2.0]])
    W = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])   # [E=3, d=2]
    assert O.router_logits(x, W)[0].tolist() == [1.0, 2.0, 3.0]
    assert O.router_logits(x, W, np.array([0.5, 0.0, -1.0]))[0].tolist() == [1.5, 2.0, 2.0]


# ---------------------------------------------------------------------------
# Layer special cases
# ---------------------------------------------------------------------------

def _rand_layer(rng, T, d, E, F, Fs=0):
    x = rng.normal(size=(T, d))
    wr = rng.normal(size=(E, d)) / math.sqrt(d)
    ex = [(rng.normal(size=(F, d)) / math.sqrt(d), rng.normal(size=(F, d)) / math.sqrt(d),
           rng.normal(size=(d, F)) / math.sqrt(F)) for _ in range(E)]
    sh = None
    if Fs:
        sh = (rng.normal(size=(Fs, d)) / math.sqrt(d), rng.normal(size=(Fs, d)) / math.sqrt(d),
              rng.normal(size=(d, Fs)) / math.sqrt(Fs))
    return x, wr, ex, sh


def test_single_expert_is_dense_swiglu():
    rng = np.random.default_rng(3)
    x, wr, ex, _ = _rand_layer(rng, 9, 5, 1, 7)
    r = O.moe_layer_forward(x, wr, ex, k=1, gate="softmax", renormalize=True)
    np.testing.assert_allclose(r["y"], O.swiglu_ffn(x, *ex[0]), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("gate,rsf", [("softmax", 1.0), ("sigmoid", 2.5)])
def test_identical_experts_sum_of_weights(gate, rsf):
    rng = np.random.default_rng(4)
    x, wr, ex, sh = _rand_layer(rng, 11, 6, 5, 8, Fs=4)
    same = [ex[0]] * 5
    r = O.moe_layer_forward(x, wr, same, k=3, gate=gate, renormalize=True,
                            routed_scaling_factor=rsf, shared=sh)
    want = rsf * O.swiglu_ffn(x, *ex[0]) + O.swiglu_ffn(x, *sh)
    np.testing.assert_allclose(r["y"], want, rtol=1e-12, atol=1e-13)


def test_k_equals_E_is_full_softmax_mixture():
    rng = np.random.default_rng(5)
    x, wr, ex, _ = _rand_layer(rng, 7, 4, 3, 6)
    r = O.moe_layer_forward(x, wr, ex, k=3, gate="softmax", renormalize=True)
    z = x @ wr.T
    p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
    want = sum(p[:, [e]] * O.swiglu_ffn(x, *ex[e]) for e in range(3))
    np.testing.assert_allclose(r["y"], want, rtol=1e-12, atol=1e-13)


def test_capacity_zero_leaves_shared_only():
    rng = np.random.default_rng(6)
    x, wr, ex, sh = _rand_layer(rng, 6, 4, 3, 5, Fs=3)
    r = O.moe_layer_forward(x, wr, ex, k=2, gate="softmax", renormalize=True,
                            capacity=0, shared=sh)
    np.testing.assert_allclose(r["y"], O.swiglu_ffn(x, *sh), rtol=1e-14)
    r2 = O.moe_layer_forward(x, wr, ex, k=2, gate="softmax", renormalize=True, capacity=0)
    assert np.all(r2["y"] == 0.0)


@pytest.mark.parametrize("cap,gate,renorm,rsf", [(None, "softmax", True, 1.0),
                                                 (3, "softmax", False, 1.0),
                                                 (4, "sigmoid", True, 2.5)])
def test_two_formulations_agree(cap, gate, renorm, rsf):
    rng = np.random.default_rng(8)
    x, wr, ex, sh = _rand_layer(rng, 17, 6, 5, 7, Fs=5)
    bias = -1.2 * np.log(np.arange(5) + 1.0)
    r = O.moe_layer_forward(x, wr, ex, k=2, gate=gate, renormalize=renorm,
                            routed_scaling_factor=rsf, capacity=cap,
                            router_bias=bias, shared=sh)
    y2 = O.moe_layer_forward_token_loop(x, wr, ex, k=2, gate=gate, renormalize=renorm,
                                        routed_scaling_factor=rsf, capacity=cap,
                                        router_bias=bias, shared=sh)
    np.testing.assert_allclose(r["y"], y2, rtol=1e-12, atol=1e-13)


def test_token_subset_matches_full():
    rng = np.random.default_rng(9)
    x, wr, ex, sh = _rand_layer(rng, 20, 4, 4, 6, Fs=2)
    full = O.moe_layer_forward(x, wr, ex, k=2, gate="softmax", renormalize=True,
                               capacity=6, shared=sh)
    sub = O.moe_layer_forward(x, wr, ex, k=2, gate="softmax", renormalize=True,
                              capacity=6, shared=sh, tokens=[19, 3, 11])
    np.testing.assert_allclose(sub["y"], full["y"][[19, 3, 11]], rtol=1e-14)


def test_dropped_assignment_contributes_zero_no_rerenorm():
    # token 2's first choice is dropped at capacity 2; its second choice keeps
    # its original weight (no second renormalisation).
    d, F, E = 2, 3, 3
    x = np.array([[1.0, 0.0], [1.0, 0.1], [1.0, -0.2]])
    wr = np.array([[2.0, 0.0], [0.0, 1.0], [0.0, -1.0]])
    rng = np.random.default_rng(10)
    ex = [(rng.normal(size=(F, d)), rng.normal(size=(F, d)), rng.normal(size=(d, F)))
          for _ in range(E)]
    r = O.moe_layer_forward(x, wr, ex, k=2, gate="softmax", renormalize=True, capacity=2)
    assert r["topk_idx"][:, 0].tolist() == [0, 0, 0]
    assert r["drop_mask"].reshape(3, 2)[2].tolist() == [1, 0]
    g = r["topk_w"]
    assert r["topk_idx"][2].tolist() == [0, 2]
    want = g[2, 1] * O.swiglu_ffn(x[2:3], *ex[2])[0]
    np.testing.assert_allclose(r["y"][2], want, rtol=1e-14)


# ---------------------------------------------------------------------------
# DeepSeek-V3 auxiliary-loss-free bias and group-limited selection
# ([moe10] "DeepSeek-V3 的无辅助损失偏置")
# ---------------------------------------------------------------------------

def test_bias_update_printed_trace(golden):
    fx = golden("moe10_bias_update_trace.json")
    steps = fx["steps"]
    for before, after in zip(steps[:-1], steps[1:]):
        b = O.update_score_bias(np.array(before["bias"]), np.array(before["load"]), fx["gamma"])
        np.testing.assert_allclose(b, after["bias"], rtol=0, atol=1e-12)


def test_bias_trace_replayed_with_constructed_scores(golden):
    # the page's three load vectors come out of ranking by s + b, with the
    # bias stepped between batches (the scores are a constructed witness)
    fx = golden("moe10_bias_update_trace.json")
    s = np.array(fx["constructed_scores"])
    b = np.zeros(fx["E"])
    for step in fx["steps"]:
        np.testing.assert_allclose(b, step["bias"], atol=1e-12)
        idx = O.topk_experts_biased(s, b, fx["k"])
        load = np.bincount(idx[:, 0], minlength=fx["E"])
        np.testing.assert_array_equal(load, step["load"])
        b = O.update_score_bias(b, load, fx["gamma"])


def test_bias_at_mean_load_unchanged():
    b = O.update_score_bias(np.array([0.1, -0.2, 0.3]), np.array([2, 2, 2]), 0.5)
    np.testing.assert_array_equal(b, [0.1, -0.2, 0.3])


def test_weights_use_raw_scores_not_biased_keys():
    # a large bias pulls expert 3 into every token's choice; its weight is
    # still its own raw score over the raw scores of the chosen pair
    rng = np.random.default_rng(5)
    s = O.sigmoid(rng.normal(size=(20, 6)))
    bias = np.array([0, 0, 0, 10.0, 0, 0])
    r = O.route(np.log(s / (1 - s)), 2, "sigmoid", True, 2.5, None, score_bias=bias)
    assert np.all(r["topk_idx"][:, 0] == 3)
    for t in range(20):
        e0, e1 = r["topk_idx"][t]
        np.testing.assert_allclose(r["topk_w"][t], 2.5 * np.array([s[t, e0], s[t, e1]]) /
                                   (s[t, e0] + s[t, e1]), rtol=1e-12)


def test_zero_bias_no_groups_equals_logit_topk():
    rng = np.random.default_rng(6)
    z = rng.normal(size=(50, 16))
    a = O.topk_experts(z, 4)
    b = O.topk_experts_biased(O.sigmoid(z), np.zeros(16), 4)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("E,n_group,topk_group,k", [(8, 4, 2, 3), (12, 3, 2, 4), (16, 8, 4, 8),
                                                    (6, 2, 1, 2)])
def test_group_limited_selection_brute_force(E, n_group, topk_group, k):
    # independent formulation: a group's score is the best pair sum inside it;
    # the kept groups are the topk_group-subset with the largest total; the
    # chosen experts are the k-subset of their experts with the largest total
    rng = np.random.default_rng(E * 100 + k)
    s = rng.uniform(size=(30, E))
    bias = rng.normal(scale=0.1, size=E)
    keys = s + bias[None, :]
    gs = E // n_group
    idx = O.topk_experts_biased(s, bias, k, n_group, topk_group)
    gsc = O.group_scores(keys, n_group)
    for t in range(30):
        for g in range(n_group):
            members = range(g * gs, (g + 1) * gs)
            best = max(keys[t, i] + keys[t, j] for i, j in itertools.combinations(members, 2))
            assert gsc[t, g] == pytest.approx(best, abs=1e-15)
        kept = max(itertools.combinations(range(n_group), topk_group),
                   key=lambda c: sum(gsc[t, g] for g in c))
        pool = [e for e in range(E) if e // gs in kept]
        chosen = max(itertools.combinations(pool, k), key=lambda c: sum(keys[t, e] for e in c))
        assert sorted(idx[t]) == sorted(chosen)
        assert all(keys[t, idx[t, j]] >= keys[t, idx[t, j + 1]] for j in range(k - 1))


def test_deepseek_v3_groups_limit_each_token_to_four_groups():
    # 256 experts in 8 groups of 32, 4 groups kept, top-8: every token's
    # experts lie in at most 4 groups ([routing]: at most 4 nodes per token)
    rng = np.random.default_rng(7)
    s = O.sigmoid(rng.normal(size=(40, 256)))
    idx = O.topk_experts_biased(s, rng.normal(scale=0.01, size=256), 8, 8, 4)
    assert all(len(set(int(e) // 32 for e in row)) <= 4 for row in idx)


# ---------------------------------------------------------------------------
# Shared-expert gate ([moe10] "细粒度专家与共享专家") and the balance loss scalar
# ([moe10] "辅助损失")
# ---------------------------------------------------------------------------

def _tiny_layer(seed, T=24, d=16, E=4, F=8, Fs=8):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, d))
    wr = rng.normal(size=(E, d)) / 4
    ex = [(rng.normal(size=(F, d)) / 4, rng.normal(size=(F, d)) / 4, rng.normal(size=(d, F)) / 3)
          for _ in range(E)]
    sh = (rng.normal(size=(Fs, d)) / 4, rng.normal(size=(Fs, d)) / 4, rng.normal(size=(d, Fs)) / 3)
    return x, wr, ex, sh


def test_shared_gate_zero_weights_halves_shared_expert():
    # sigmoid(0) = 1/2 exactly: the gated layer equals routed + S(x) / 2
    x, wr, ex, sh = _tiny_layer(8)
    full = O.moe_layer_forward(x, wr, ex, k=2, gate="sigmoid", renormalize=True,
                               routed_scaling_factor=2.5, shared=sh)["y"]
    gated = O.moe_layer_forward(x, wr, ex, k=2, gate="sigmoid", renormalize=True,
                                routed_scaling_factor=2.5, shared=sh,
                                shared_gate=np.zeros(x.shape[1]))["y"]
    np.testing.assert_allclose(gated, full - 0.5 * O.swiglu_ffn(x, *sh), rtol=1e-12, atol=1e-12)


def test_shared_gate_closed_value():
    # x . w = ln 3 gives the weight 3/4
    d = 5
    x = np.zeros((1, d))
    x[0, 2] = math.log(3.0)
    w = np.zeros(d)
    w[2] = 1.0
    assert O.shared_gate_weights(x, w)[0] == pytest.approx(0.75, abs=1e-15)


def test_shared_gate_two_formulations_agree():
    x, wr, ex, sh = _tiny_layer(9)
    wsg = np.random.default_rng(10).normal(size=x.shape[1]) / 4
    a = O.moe_layer_forward(x, wr, ex, k=2, gate="softmax", renormalize=True, shared=sh,
                            shared_gate=wsg)["y"]
    b = O.moe_layer_forward_token_loop(x, wr, ex, k=2, gate="softmax", renormalize=True,
                                       shared=sh, shared_gate=wsg)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_balance_loss_worked_values(golden):
    # the page's three cases through counts/drops and mean probabilities:
    # 8 assignments on 4 experts, alpha = 0.01
    for counts, P, want in [([2, 2, 2, 2], [0.25] * 4, 1.0), ([5, 1, 1, 1], [0.55, 0.15, 0.15, 0.15], 1.6),
                            ([8, 0, 0, 0], [1, 0, 0, 0], 4.0)]:
        assert O.balance_loss(np.array(counts), np.zeros(4), np.array(P), 0.01) == \
            pytest.approx(0.01 * want, rel=1e-12)
    # dropped assignments still count as assigned
    assert O.balance_loss(np.array([3, 1, 1, 1]), np.array([2, 0, 0, 0]),
                          np.array([0.55, 0.15, 0.15, 0.15]), 1.0) == pytest.approx(1.6, rel=1e-12)


# ---------------------------------------------------------------------------
# FP8 E4M3 expert weights ([moe10] "推理时": DeepSeek-V3 ships FP8 weights)
# ---------------------------------------------------------------------------

def test_e4m3_landmark_values():
    v = O.e4m3_to_f64(np.array([0x38, 0x7E, 0x01, 0x08, 0x07, 0x00, 0x80, 0xB8, 0x40, 0x30]))
    np.testing.assert_array_equal(v, [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, 7 * 2.0 ** -9, 0.0, -0.0,
                                      -1.0, 2.0, 0.5])
    assert np.all(np.isnan(O.e4m3_to_f64(np.array([0x7F, 0xFF]))))


def test_e4m3_matches_torch_for_every_code():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(ours)
    assert finite.sum() == 254
    np.testing.assert_array_equal(ours[finite], theirs[finite])
    assert np.all(np.isnan(theirs[~finite]))


def test_e4m3_positive_codes_strictly_increase():
    v = O.e4m3_to_f64(np.arange(0, 127))
    assert np.all(np.diff(v) > 0)


def test_dequantize_rows_scales_each_output_channel():
    codes = np.array([[0x38, 0x40], [0x30, 0xB8]], dtype=np.uint8)
    np.testing.assert_array_equal(O.dequantize_rows(codes, [3.0, 0.25]),
                                  [[3.0, 6.0], [0.125, -0.25]])


# ---------------------------------------------------------------------------
# Expert-choice routing ([routing]: each expert takes the fixed number of
# tokens it wants most)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,C", [(6, 3, 2), (7, 2, 3), (5, 4, 5), (8, 3, 0)])
def test_expert_choice_brute_force(T, E, C):
    rng = np.random.default_rng(T * 10 + E)
    s = rng.uniform(size=(T, E))
    ec = O.expert_choice(s, C)
    for e in range(E):
        best = max(itertools.combinations(range(T), C), key=lambda c: sum(s[t, e] for t in c))
        assert list(ec["tokens"][e]) == sorted(best)
        np.testing.assert_array_equal(ec["weights"][e], s[ec["tokens"][e], e])
    assert ec["picked"].sum() == E * C            # balanced: every expert exactly C


def test_expert_choice_ties_go_to_lower_token():
    s = np.array([[0.5, 0.1], [0.5, 0.9], [0.5, 0.9], [0.2, 0.9]])
    ec = O.expert_choice(s, 2)
    assert list(ec["tokens"][0]) == [0, 1]
    assert list(ec["tokens"][1]) == [1, 2]
    assert list(ec["picked"]) == [1, 2, 1, 0]      # token 3 taken by no expert


def test_expert_choice_capacity_default():
    assert O.expert_choice_capacity(16384, 64, 1) == 256
    assert O.expert_choice_capacity(10, 4, 2) == 5     # ceil(20 / 4)
    assert O.expert_choice_capacity(10, 3, 2) == 7     # ceil(20 / 3)
    assert O.expert_choice_capacity(4, 2, 2, 9) == 4   # at most T


def test_expert_choice_full_capacity_is_full_softmax_mixture():
    # C = T: every expert takes every token, so y = sum_e p_e E_e(x), which is
    # token-choice top-E with renormalisation (the weights already sum to 1)
    x, wr, ex, _ = _tiny_layer(20, T=9, E=4)
    T = x.shape[0]
    a = O.moe_layer_expert_choice(x, wr, ex, C=T, gate="softmax")["y"]
    b = O.moe_layer_forward(x, wr, ex, k=4, gate="softmax", renormalize=True)["y"]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_expert_choice_layer_matches_token_loop():
    x, wr, ex, sh = _tiny_layer(21, T=12, E=4)
    r = O.moe_layer_expert_choice(x, wr, ex, C=5, gate="sigmoid", shared=sh)
    s = O.sigmoid(O.router_logits(x, wr))
    want = np.zeros_like(r["y"])
    for t in range(x.shape[0]):
        for e in range(4):
            if t in set(r["tokens"][e].tolist()):
                want[t] += s[t, e] * O.swiglu_ffn(x[t:t + 1], *ex[e])[0]
        want[t] += O.swiglu_ffn(x[t:t + 1], *sh)[0]
    np.testing.assert_allclose(r["y"], want, rtol=1e-12, atol=1e-12)
