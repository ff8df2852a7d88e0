"""Float64 CPU oracle for the forward pass of a sparsely-gated MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path imports,
calls or links this module; only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg do.  It shares no code with the CUDA path.

Everything here is plain NumPy in float64, written as the pages state the
method, step by step, with no blocking, fusion or reordering:

  [moe10]  "10. 混合专家 MoE：总参数与激活参数" (niuwancheng.cn)
  [routing] the amazingdata.cn article on why routing is the hardest part of MoE
  [lesson] "MoE为什么只激活一部分专家" (hi-bin.com lesson notes)
  [explain] "为什么大模型参数这么多却不太慢？MoE 混合专家架构原理拆解" (wuaizhan.com)

Layout conventions (nn.Linear orientation, out x in): x [T,d], w_router [E,d],
expert e: w_gate [F,d], w_up [F,d], w_down [d,F]; shared expert likewise.

Readings taken where the pages are silent:
  * top-k ties go to the lower expert index; the chosen list is ordered by
    logit descending, then index ascending;
  * the selection key is the raw logit z (softmax and sigmoid are strictly
    increasing in z, so the chosen set is the one the pages describe); with a
    DeepSeek-V3 score bias or expert groups it is s + b, as the pages state;
  * the bias step leaves an expert exactly at the mean load unchanged;
  * routed_scaling_factor multiplies the routed weights only; the shared
    expert is added with weight 1;
  * capacity = ceil((T / E) * capacity_factor) in IEEE double; slots are
    filled in ascending assignment id a = t*k + j (token order);
  * a dropped assignment contributes zero and the surviving weights of that
    token are not renormalised again; y excludes the residual.

Parity pins: every function below is pinned by tests in tests/test_oracle_*.py
against values the pages print, closed forms, brute force or invariants.
"""

from __future__ import annotations

import math
from typing import Dict, Iterable, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# Router: logits = x . W^T  ([moe10] "把一个大 FFN 换成一组小 FFN", the block
# sketch's first line; [routing] the router's first step writes x . W_g with
# W_g stored d x E, which is the transpose of the layout used here).
# ---------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray,
                  bias: Optional[np.ndarray] = None) -> np.ndarray:
    """z[t,e] = sum_c x[t,c] * w_router[e,c] (+ bias[e])."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float64)
    z = x @ w.T
    if bias is not None:
        z = z + np.asarray(bias, dtype=np.float64)[None, :]
    return z


# ---------------------------------------------------------------------------
# Gating scores ([moe10] "路由器怎样选专家：top-k 与两种门控"):
#   softmax  p_i = exp(z_i) / sum_j exp(z_j)
#   sigmoid  s_i = 1 / (1 + exp(-z_i)), each expert scored on its own
# ---------------------------------------------------------------------------

def softmax(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)       # shift for range only; cancels
    ez = np.exp(z - m)
    return ez / np.sum(ez, axis=-1, keepdims=True)


def sigmoid(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def gate_scores(z: np.ndarray, gate: str) -> np.ndarray:
    if gate == "softmax":
        return softmax(z)
    if gate == "sigmoid":
        return sigmoid(z)
    raise ValueError(f"unknown gate {gate!r}")


# ---------------------------------------------------------------------------
# Top-k selection ([moe10] block sketch `probs.topk(k)`; [lesson] y_t sums over
# TopK(s_t); k is num_experts_per_tok).
# ---------------------------------------------------------------------------

def topk_experts(z: np.ndarray, k: int) -> np.ndarray:
    """idx[t, :] = the k experts with the largest logit, in descending order.

    Equal logits are ordered by ascending expert index, so a tie always goes
    to the lower index.  Implemented as the plain definition: sort the pairs
    (-z[t,e], e) lexicographically and keep the first k.
    """
    z = np.asarray(z, dtype=np.float64)
    T, E = z.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    idx = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-z[t, e], e))
        idx[t] = order[:k]
    return idx


def topk_weights(scores: np.ndarray, idx: np.ndarray, renormalize: bool,
                 routed_scaling_factor: float = 1.0) -> np.ndarray:
    """Combine weights g[t,j] of the chosen experts.

    With renormalisation ([moe10] top-k section, whose worked example divides
    the two chosen scores by their sum; the block sketch's `w / w.sum(-1)`): g_j = score_j / sum_sel score, then
    multiplied by routed_scaling_factor (DeepSeek-V3: 2.5).  Without it
    ([explain] "门控是怎么挑专家的": out = sum score_i * expert_i): g_j = score_j
    (times the factor, which is 1 for the configurations that skip renorm).
    """
    scores = np.asarray(scores, dtype=np.float64)
    T, k = idx.shape
    g = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        sel = np.array([scores[t, idx[t, j]] for j in range(k)])
        if renormalize:
            g[t] = sel / np.sum(sel)
        else:
            g[t] = sel
    return g * routed_scaling_factor


# ---------------------------------------------------------------------------
# DeepSeek-V3 auxiliary-loss-free selection ([moe10] "DeepSeek-V3 的无辅助损失
# 偏置"; [routing] the paragraph on auxiliary-loss-free load balancing).  Each
# expert carries a bias b_e that enters only the ranking, s_e + b_e; the
# combine weights keep the raw score s_e.  With groups, the experts are split
# into n_group equal consecutive groups, a group is scored by the sum of its
# two best ranking values, the topk_group best groups are kept, and the k
# experts are chosen among the kept groups only (node-limited routing: a token
# reaches at most topk_group groups).
# ---------------------------------------------------------------------------

def group_scores(keys: np.ndarray, n_group: int) -> np.ndarray:
    """score[t, g] = the two largest keys[t, e] of group g, added."""
    keys = np.asarray(keys, dtype=np.float64)
    T, E = keys.shape
    if n_group < 1 or E % n_group != 0 or E // n_group < 2:
        raise ValueError("groups must split E evenly into groups of at least 2")
    gs = E // n_group
    out = np.empty((T, n_group), dtype=np.float64)
    for t in range(T):
        for g in range(n_group):
            vals = sorted(keys[t, g * gs:(g + 1) * gs], reverse=True)
            out[t, g] = vals[0] + vals[1]
    return out


def topk_experts_biased(scores: np.ndarray, score_bias: Optional[np.ndarray], k: int,
                        n_group: int = 1, topk_group: int = 1) -> np.ndarray:
    """idx[t, :] = the k experts with the largest s + b among the kept groups.

    Ties (of experts and of groups) go to the lower index, as in
    ``topk_experts``; the chosen list is ordered by s + b descending.
    """
    scores = np.asarray(scores, dtype=np.float64)
    T, E = scores.shape
    keys = scores + (0.0 if score_bias is None else np.asarray(score_bias, np.float64)[None, :])
    allowed = [list(range(E)) for _ in range(T)]
    if n_group > 1:
        if not (1 <= topk_group <= n_group):
            raise ValueError("need 1 <= topk_group <= n_group")
        gsc = group_scores(keys, n_group)
        gs = E // n_group
        for t in range(T):
            kept = sorted(range(n_group), key=lambda g: (-gsc[t, g], g))[:topk_group]
            allowed[t] = [e for e in range(E) if e // gs in kept]
    idx = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        if k > len(allowed[t]):
            raise ValueError("k exceeds the experts of the kept groups")
        order = sorted(allowed[t], key=lambda e: (-keys[t, e], e))
        idx[t] = order[:k]
    return idx


def update_score_bias(score_bias: np.ndarray, load: np.ndarray, gamma: float) -> np.ndarray:
    """One bias step after a batch: an expert above the mean load loses gamma,
    one below it gains gamma ([moe10] "DeepSeek-V3 的无辅助损失偏置");
    an expert exactly at the mean is left unchanged."""
    load = np.asarray(load, dtype=np.float64)
    return np.asarray(score_bias, dtype=np.float64) - gamma * np.sign(load - np.mean(load))


# ---------------------------------------------------------------------------
# Expert-choice routing ([routing], the paragraph on expert choice: each
# expert takes a fixed number of the tokens it scores highest, which balances
# the load by construction; a token may be taken by no expert).
# ---------------------------------------------------------------------------

def expert_choice_capacity(T: int, E: int, k: int, capacity: Optional[int] = None) -> int:
    """Tokens each expert takes: the given capacity, else ceil(T * k / E)
    (as many slots as token-choice top-k would fill on average); at most T."""
    c = int(math.ceil(T * k / E)) if capacity is None else int(capacity)
    return max(0, min(c, T))


def expert_choice(scores: np.ndarray, C: int) -> Dict[str, np.ndarray]:
    """Expert e takes the C tokens with the largest scores[t, e], ties to the
    lower token index; its tokens are listed in ascending token order.

      tokens[e, i]  the i-th token of expert e
      weights[e, i] scores[tokens[e, i], e], the combine weight
      picked[t]     how many experts took token t
    """
    scores = np.asarray(scores, dtype=np.float64)
    T, E = scores.shape
    tokens = np.empty((E, C), dtype=np.int64)
    for e in range(E):
        best = sorted(range(T), key=lambda t: (-scores[t, e], t))[:C]
        tokens[e] = sorted(best)
    weights = np.take_along_axis(scores.T, tokens, axis=1)
    picked = np.bincount(tokens.ravel(), minlength=T) if C > 0 else np.zeros(T, np.int64)
    return {"tokens": tokens, "weights": weights, "picked": picked}


def moe_layer_expert_choice(x: np.ndarray, w_router: np.ndarray, experts, C: int, gate: str,
                            shared=None, tokens: Optional[Sequence[int]] = None,
                            logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """y_t = sum over the experts e that took t of scores[t, e] * E_e(x_t)
    (+ the shared expert), computed per expert over its chosen tokens."""
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    z = router_logits(x, w_router) if logits is None else np.asarray(logits, np.float64)
    scores = gate_scores(z, gate)
    ec = expert_choice(scores, C)
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    pos = {int(t): i for i, t in enumerate(toks)}
    y = np.zeros((len(toks), x.shape[1]), dtype=np.float64)
    for e in range(z.shape[1]):
        rows = [int(t) for t in ec["tokens"][e] if int(t) in pos]
        if not rows:
            continue
        out = swiglu_ffn(x[rows], *experts[e])
        for i, t in enumerate(rows):
            y[pos[t]] += scores[t, e] * out[i]
    if shared is not None:
        y += swiglu_ffn(x[toks], *shared)
    ec.update(y=y, scores=scores, logits=z, mean_prob=mean_router_prob(scores))
    return ec


def mean_router_prob(scores: np.ndarray) -> np.ndarray:
    """P_e = (1/T) sum_t score[t,e], the batch-mean router probability that
    the load statistics use ([moe10] "辅助损失", definition of P_i)."""
    scores = np.asarray(scores, dtype=np.float64)
    return np.mean(scores, axis=0)


# ---------------------------------------------------------------------------
# Capacity and dispatch ([moe10] "负载不均：路由坍缩与丢 token": capacity =
# tokens per batch / experts x capacity factor, 2 x 1.25 = 2.5 rounded up to 3;
# over-capacity tokens skip the expert and ride the residual.  [routing] gives
# the same formula and the same dropping rule.)
# ---------------------------------------------------------------------------

def expert_capacity(T: int, E: int, capacity_factor: Optional[float]) -> Optional[int]:
    """ceil((T / E) * capacity_factor) in IEEE double; None = unlimited."""
    if capacity_factor is None:
        return None
    return int(math.ceil((float(T) / float(E)) * float(capacity_factor)))


def dispatch(idx: np.ndarray, E: int, capacity: Optional[int]) -> Dict[str, np.ndarray]:
    """Group assignments by expert, filling slots in ascending assignment id.

    Assignment a = t*k + j is token t's j-th choice.  Walking a upward, the
    assignment takes the next free slot of its expert; once an expert holds
    ``capacity`` assignments, later ones are dropped.  Returns

      counts[e]   kept assignments of expert e (<= capacity)
      drops[e]    dropped assignments of expert e
      offsets     exclusive prefix sum of counts, length E + 1
      perm[r]     assignment id held by grouped row r (r < offsets[E])
      drop_mask[a] 1 where a was dropped
      row_of[a]   grouped row of a, or -1 when dropped
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    A = T * k
    flat = idx.reshape(A)
    counts = np.zeros(E, dtype=np.int64)
    drops = np.zeros(E, dtype=np.int64)
    slot = np.full(A, -1, dtype=np.int64)
    drop_mask = np.zeros(A, dtype=np.uint8)
    for a in range(A):
        e = int(flat[a])
        if capacity is None or counts[e] < capacity:
            slot[a] = counts[e]
            counts[e] += 1
        else:
            drop_mask[a] = 1
            drops[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    perm = np.full(A, -1, dtype=np.int64)
    row_of = np.full(A, -1, dtype=np.int64)
    for a in range(A):
        if drop_mask[a] == 0:
            r = offsets[flat[a]] + slot[a]
            perm[r] = a
            row_of[a] = r
    return {"counts": counts, "drops": drops, "offsets": offsets, "perm": perm,
            "drop_mask": drop_mask, "row_of": row_of, "slot": slot}


# ---------------------------------------------------------------------------
# Expert FFN: SwiGLU, gate and up d -> F, SiLU(gate) * up, down F -> d
# ([moe10] "把一个大 FFN 换成一组小 FFN": each expert has the dense model's
# FFN structure, 3 x d x F parameters).  SiLU(u) = u * sigmoid(u).
# ---------------------------------------------------------------------------

def silu(u: np.ndarray) -> np.ndarray:
    u = np.asarray(u, dtype=np.float64)
    return u * sigmoid(u)


def swiglu_ffn(x_rows: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray,
               w_down: np.ndarray) -> np.ndarray:
    """E(x) = (SiLU(x W_gate^T) * (x W_up^T)) W_down^T for each row of x."""
    x_rows = np.asarray(x_rows, dtype=np.float64)
    g = x_rows @ np.asarray(w_gate, dtype=np.float64).T
    u = x_rows @ np.asarray(w_up, dtype=np.float64).T
    h = silu(g) * u
    return h @ np.asarray(w_down, dtype=np.float64).T


# ---------------------------------------------------------------------------
# Routing for a whole batch.
# ---------------------------------------------------------------------------

def route(z: np.ndarray, k: int, gate: str, renormalize: bool,
          routed_scaling_factor: float, capacity: Optional[int],
          score_bias: Optional[np.ndarray] = None, n_group: int = 1,
          topk_group: int = 1) -> Dict[str, np.ndarray]:
    """Scores, top-k, weights, mean probability and dispatch from logits z.

    Without a score bias or groups the k largest logits are chosen; with
    either, the k largest s + b among the kept groups (``topk_experts_biased``).
    The weights always come from the raw scores.
    """
    z = np.asarray(z, dtype=np.float64)
    E = z.shape[1]
    scores = gate_scores(z, gate)
    if score_bias is None and n_group <= 1:
        idx = topk_experts(z, k)
    else:
        idx = topk_experts_biased(scores, score_bias, k, n_group, topk_group)
    g = topk_weights(scores, idx, renormalize, routed_scaling_factor)
    out = {"logits": z, "scores": scores, "topk_idx": idx, "topk_w": g,
           "mean_prob": mean_router_prob(scores)}
    out.update(dispatch(idx, E, capacity))
    return out


# ---------------------------------------------------------------------------
# The layer: y_t = sum_{i in TopK} g_{t,i} E_i(x_t)  (+ shared expert)
# ([lesson] "Router 怎样给 Token 选专家"; [routing] output = sum g_i Expert_i(x);
# [moe10] "细粒度专家与共享专家": the shared expert's output is added directly).
# ---------------------------------------------------------------------------

def moe_layer_forward(x: np.ndarray, w_router: np.ndarray, experts,
                      k: int, gate: str, renormalize: bool,
                      routed_scaling_factor: float = 1.0,
                      capacity: Optional[int] = None,
                      router_bias: Optional[np.ndarray] = None,
                      shared=None,
                      tokens: Optional[Sequence[int]] = None,
                      logits: Optional[np.ndarray] = None,
                      score_bias: Optional[np.ndarray] = None,
                      n_group: int = 1, topk_group: int = 1,
                      shared_gate: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Per-expert grouped formulation (the block sketch's loop over experts).

    ``experts[e]`` returns (w_gate_e, w_up_e, w_down_e) as float64 arrays and
    is called at most once per expert.  ``shared`` is None or the shared
    expert's (w_gate, w_up, w_down).  Routing is always computed for the
    whole batch (capacity depends on earlier tokens); the output y is
    computed for ``tokens`` only (default: all), in that order.  ``logits``,
    when given, replaces x . W^T (+ bias).  ``shared_gate`` (a [d] vector)
    scales the shared expert's output per token by sigmoid(x_t . w) ([moe10]
    "细粒度专家与共享专家": a token-dependent sigmoid gate in front of the
    shared expert); without it the shared output is added with weight 1.
    """
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    z = router_logits(x, w_router, router_bias) if logits is None else np.asarray(logits, np.float64)
    r = route(z, k, gate, renormalize, routed_scaling_factor, capacity, score_bias, n_group,
              topk_group)
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    pos = {int(t): i for i, t in enumerate(toks)}
    y = np.zeros((len(toks), x.shape[1]), dtype=np.float64)
    idx, g, drop = r["topk_idx"], r["topk_w"], r["drop_mask"].reshape(T, k)
    E = z.shape[1]
    for e in range(E):
        rows, slots = [], []
        for t in toks:
            for j in range(k):
                if idx[t, j] == e and drop[t, j] == 0:
                    rows.append(int(t))
                    slots.append(j)
        if not rows:
            continue
        wg, wu, wd = experts[e]
        out = swiglu_ffn(x[rows], wg, wu, wd)
        for i, (t, j) in enumerate(zip(rows, slots)):
            y[pos[t]] += g[t, j] * out[i]
    if shared is not None:
        sy = swiglu_ffn(x[toks], *shared)
        if shared_gate is not None:
            sy = shared_gate_weights(x[toks], shared_gate)[:, None] * sy
        y += sy
    r["y"] = y
    r["tokens"] = toks
    return r


def shared_gate_weights(x_rows: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Per-token weight of the shared expert: sigmoid(x_t . w)."""
    return sigmoid(np.asarray(x_rows, np.float64) @ np.asarray(w, np.float64))


def moe_layer_forward_token_loop(x: np.ndarray, w_router: np.ndarray, experts,
                                 k: int, gate: str, renormalize: bool,
                                 routed_scaling_factor: float = 1.0,
                                 capacity: Optional[int] = None,
                                 router_bias: Optional[np.ndarray] = None,
                                 shared=None,
                                 shared_gate: Optional[np.ndarray] = None) -> np.ndarray:
    """Second formulation: per token, per choice, no grouping or permutation.

    Used only to cross-check ``moe_layer_forward`` on small inputs; both must
    agree to float64 rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape
    z = router_logits(x, w_router, router_bias)
    scores = gate_scores(z, gate)
    idx = topk_experts(z, k)
    g = topk_weights(scores, idx, renormalize, routed_scaling_factor)
    E = z.shape[1]
    taken = [0] * E
    y = np.zeros((T, d), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if capacity is not None and taken[e] >= capacity:
                continue
            taken[e] += 1
            wg, wu, wd = experts[e]
            y[t] += g[t, j] * swiglu_ffn(x[t:t + 1], wg, wu, wd)[0]
        if shared is not None:
            gate = 1.0
            if shared_gate is not None:
                gate = 1.0 / (1.0 + math.exp(-float(np.dot(x[t], shared_gate))))
            y[t] += gate * swiglu_ffn(x[t:t + 1], *shared)[0]
    return y


# ---------------------------------------------------------------------------
# Load statistics derived from the emitted counts and mean probabilities.
# ---------------------------------------------------------------------------

def load_fractions(counts: np.ndarray, drops: np.ndarray) -> np.ndarray:
    """f_e = share of all assignments that chose expert e (kept + dropped)."""
    load = np.asarray(counts, dtype=np.float64) + np.asarray(drops, dtype=np.float64)
    return load / np.sum(load)


def balance_loss(counts: np.ndarray, drops: np.ndarray, mean_prob: np.ndarray,
                 alpha: float) -> float:
    """L_aux = alpha * N * sum_i f_i * P_i ([moe10] "辅助损失"), from the emitted
    per-expert counts, drops and mean router probabilities."""
    return alpha * switch_balance_term(load_fractions(counts, drops), mean_prob)


def switch_balance_term(f: np.ndarray, P: np.ndarray) -> float:
    """N * sum_i f_i * P_i, the part of the Switch auxiliary loss that the
    worked example of [moe10] "辅助损失" evaluates (1.0 uniform, 4.0 collapsed)."""
    f = np.asarray(f, dtype=np.float64)
    P = np.asarray(P, dtype=np.float64)
    return float(len(f) * np.sum(f * P))


# ---------------------------------------------------------------------------
# FP8 (E4M3) expert weights ([moe10] "推理时：显存按总参数，计算按激活参数":
# DeepSeek-V3 ships its weights in FP8, about one byte per parameter).  A
# stored weight is an 8-bit E4M3 code times a per-output-channel scale.
# E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0
# holds the subnormals m * 2^-9; S.1111.111 is NaN (no infinities); the
# largest finite value is 448.
# ---------------------------------------------------------------------------

def _e4m3_value(c: np.ndarray) -> np.ndarray:
    """Value of each E4M3 code, straight from the format: sign bit, 4-bit
    exponent of bias 7, 3-bit mantissa; exponent 0 is subnormal (m * 2^-9);
    S.1111.111 is NaN."""
    c = np.asarray(c, dtype=np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.power(2.0, e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    v = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 7) == 7), np.nan, v)


# the definition above evaluated once for every one of the 256 codes
_E4M3_VALUES = _e4m3_value(np.arange(256))


def e4m3_to_f64(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8 array): the format's definition
    (``_e4m3_value``), looked up per code."""
    return _E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def dequantize_rows(codes, scale) -> np.ndarray:
    """w[r, c] = e4m3(codes[r, c]) * scale[r] (one scale per output channel)."""
    return e4m3_to_f64(codes) * np.asarray(scale, dtype=np.float64)[:, None]


# ---------------------------------------------------------------------------
# Parameter accounting ([moe10] "总参数和激活参数怎样算").
# ---------------------------------------------------------------------------

def moe_layer_params(d: int, E: int, F: int, F_s: int = 0, k: Optional[int] = None) -> int:
    """Parameters of one MoE FFN layer: router E*d plus 3*d*F per expert
    (all E experts, or only k of them for the active count) plus the shared
    expert's 3*d*F_s."""
    n_exp = E if k is None else k
    return E * d + n_exp * 3 * d * F + 3 * d * F_s


def expected_touched_experts(E: int, k: int, B: int) -> float:
    """Expected number of distinct experts touched by B independent tokens
    each choosing k of E uniformly ([moe10] "推理时：显存按总参数，计算按激活参数")."""
    return E * (1.0 - (1.0 - k / E) ** B)
