"""Helpers shared by the GPU parity tests (comparison rules and oracle calls)."""

from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
import torch

import top_routing_expert_gate_b300 as moe
from oracle import moe_oracle as O
from workloads.generate import ExpertWeights, shared_weights, to_f64

# Layer output tolerance: max |err| <= 2e-2 * RMS(y_ref), mean |err| <= 2e-3 * RMS(y_ref)
MAX_REL_RMS = 2e-2
MEAN_REL_RMS = 2e-3
# Routing end to end: tokens whose k-th / (k+1)-th score margin exceeds this
# must route identically; router weights within 1e-3 absolute.
MARGIN = 1e-3
WEIGHT_ABS = 1e-3


def assert_layer_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = "y"):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    rms = math.sqrt(float(np.mean(y_ref ** 2)))
    err = np.abs(y_gpu - y_ref)
    mx, mean = float(err.max()), float(err.mean())
    assert rms > 0
    assert mx <= MAX_REL_RMS * rms, f"{what}: max|err| {mx:.3e} > {MAX_REL_RMS} * rms {rms:.3e}"
    assert mean <= MEAN_REL_RMS * rms, \
        f"{what}: mean|err| {mean:.3e} > {MEAN_REL_RMS} * rms {rms:.3e}"
    return mx / rms, mean / rms


def assert_capacity_layer_close(y_gpu: np.ndarray, y_ref: np.ndarray, drop_mask: np.ndarray,
                                what: str = "y"):
    """With a capacity: tokens whose every choice was dropped must be exactly
    zero without a shared expert; with one they carry only the shared
    expert's output, held to the layer tolerance relative to their own RMS.
    The other tokens are held to the layer tolerance relative to their own
    RMS (the dropped tokens' exact zeros would otherwise deflate the RMS of
    the comparison)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    all_dropped = np.all(np.asarray(drop_mask).reshape(y_ref.shape[0], -1) != 0, axis=1)
    if all_dropped.any():
        if np.all(y_ref[all_dropped] == 0.0):
            assert np.all(y_gpu[all_dropped] == 0.0), f"{what}: dropped tokens must be 0"
        else:
            assert_layer_close(y_gpu[all_dropped], y_ref[all_dropped], what + " (all dropped)")
    if (~all_dropped).any():
        assert_layer_close(y_gpu[~all_dropped], y_ref[~all_dropped], what)


def score_margins(scores: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Per token: score of the k-th chosen expert minus the best unchosen score
    (inf when every expert is chosen)."""
    T, k = idx.shape
    E = scores.shape[1]
    if k == E:
        return np.full(T, np.inf)
    m = np.empty(T)
    for t in range(T):
        chosen = set(int(e) for e in idx[t])
        kth = scores[t, idx[t, k - 1]]
        rest = max(scores[t, e] for e in range(E) if e not in chosen)
        m[t] = kth - rest
    return m


def same_sets(gi: np.ndarray, ri: np.ndarray) -> np.ndarray:
    """Per token: the chosen expert sets agree (order ignored)."""
    return np.all(np.sort(gi, axis=1) == np.sort(ri, axis=1), axis=1)


def order_separated(scores: np.ndarray, idx: np.ndarray, margin: float) -> np.ndarray:
    """Per token: consecutive chosen scores differ by more than ``margin``, so
    the order inside the chosen list is fixed too."""
    T, k = idx.shape
    if k == 1:
        return np.ones(T, dtype=bool)
    sel = np.take_along_axis(scores, idx, axis=1)
    return np.all(sel[:, :-1] - sel[:, 1:] > margin, axis=1)


def oracle_capacity(shape, T: Optional[int] = None) -> Optional[int]:
    T = shape.T if T is None else T
    return O.expert_capacity(T, shape.E, shape.capacity_factor)


def _codes(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


class DequantExperts:
    """Per-expert float64 weights of an E4M3 layer: the oracle's decoding of
    the stored codes times the per-row scales, one expert at a time."""

    def __init__(self, inputs):
        self.q = (inputs["w_gate"], inputs["w_up"], inputs["w_down"])
        self.s = (inputs["w_gate_scale"], inputs["w_up_scale"], inputs["w_down_scale"])

    def __len__(self) -> int:
        return self.q[0].shape[0]

    def __getitem__(self, e: int):
        return tuple(O.dequantize_rows(_codes(q[e]), to_f64(s[e])) for q, s in zip(self.q, self.s))


def layer_experts(inputs):
    """The routed experts as float64 weights (exact widening, or E4M3 decoding)."""
    if inputs.get("w_gate_scale") is not None:
        return DequantExperts(inputs)
    return ExpertWeights(inputs["w_gate"], inputs["w_up"], inputs["w_down"])


def layer_shared(inputs):
    if inputs.get("ws_gate") is None:
        return None
    if inputs.get("ws_gate_scale") is not None:
        return tuple(O.dequantize_rows(_codes(inputs[k]), to_f64(inputs[k + "_scale"]))
                     for k in ("ws_gate", "ws_up", "ws_down"))
    return shared_weights(inputs)


def oracle_layer(shape, inputs, tokens: Optional[Sequence[int]] = None,
                 logits: Optional[np.ndarray] = None):
    """Run the float64 oracle on the (bf16/fp32/E4M3) inputs, widened exactly.

    ``logits`` (the library's fp32 router logits, router bias included)
    replace the oracle's own x . W^T: routing is then decided on the same
    numbers on both sides, so its outputs must agree bit for bit."""
    T = inputs["x"].shape[0]
    return O.moe_layer_forward(
        to_f64(inputs["x"]), to_f64(inputs["w_router"]),
        layer_experts(inputs),
        k=shape.k, gate=shape.gate, renormalize=shape.renormalize,
        routed_scaling_factor=shape.rsf, capacity=oracle_capacity(shape, T),
        router_bias=to_f64(inputs["router_bias"]), shared=layer_shared(inputs),
        tokens=tokens, logits=logits, score_bias=to_f64(inputs.get("score_bias")),
        n_group=max(shape.n_group, 1), topk_group=shape.topk_group,
        shared_gate=to_f64(inputs.get("shared_gate")))


def oracle_route(shape, logits: np.ndarray):
    """The oracle's routing and dispatch of the whole batch from given logits."""
    T = logits.shape[0]
    return O.route(logits, shape.k, shape.gate, shape.renormalize, shape.rsf,
                   oracle_capacity(shape, T))


def library_routing(cfg, inputs, ws):
    """The library's routing of the whole batch through the split entry
    points: fp32 logits (x . W^T plus the router bias, the numbers the layer
    ranks), top-k indices and weights, mean probability, and the dispatch
    arrays.  Enqueued on the current stream; synchronise before reading."""
    w = moe.LayerWeights.from_inputs(inputs)
    r = moe.route(cfg, inputs["x"], w.w_router, w.router_bias, ws=ws, score_bias=w.score_bias)
    r.update(moe.dispatch(cfg, r["topk_idx"], ws=ws))
    return r


# Router weights from the same fp32 logits: fp32 exp and division against
# float64, a few ulp apart.
WEIGHT_REL_SHARED = 2e-6


def assert_routing_bit_exact(lib, ref, T: int, k: int):
    """Check (a): fed the same fp32 logits, top-k indices, counts, drops,
    offsets, permutation and drop mask agree bit for bit; the weights within
    a few ulp."""
    A = T * k
    np.testing.assert_array_equal(np_i(lib["topk_idx"]), ref["topk_idx"])
    np.testing.assert_array_equal(np_i(lib["counts"]), ref["counts"])
    np.testing.assert_array_equal(np_i(lib["drops"]), ref["drops"])
    np.testing.assert_array_equal(np_i(lib["offsets"]), ref["offsets"])
    n = int(ref["offsets"][-1])
    np.testing.assert_array_equal(np_i(lib["perm"])[:n], ref["perm"][:n])
    np.testing.assert_array_equal(np_i(lib["drop_mask"])[:A], ref["drop_mask"])
    np.testing.assert_allclose(np_f(lib["topk_w"]), ref["topk_w"], rtol=WEIGHT_REL_SHARED,
                               atol=2e-7)


def ragged_tail_tokens(ref, k: int) -> np.ndarray:
    """For every expert that kept a row, the token of its last grouped row:
    that row lies in the expert's last (ragged) row tile, next to the first
    row of the following expert, in every tile layout."""
    offs, perm = ref["offsets"], ref["perm"]
    toks = [int(perm[offs[e + 1] - 1]) // k for e in range(len(offs) - 1) if offs[e + 1] > offs[e]]
    return np.unique(np.asarray(toks, dtype=np.int64))


def check_tokens(ref, T: int, k: int, n: int, seed: int = 0) -> np.ndarray:
    """Tokens whose outputs a sampled comparison checks: each expert's
    ragged-tail token, the first and last token (the shared expert's first
    and last row tile), up to 8 tokens with a dropped choice and up to 8
    whose every choice was dropped, then random tokens up to ``n`` in all."""
    rng = np.random.default_rng(seed)
    pick = set(ragged_tail_tokens(ref, k).tolist()) | {0, T - 1}
    drop = np.asarray(ref["drop_mask"]).reshape(T, k) != 0
    for mask in (drop.any(axis=1) & ~drop.all(axis=1), drop.all(axis=1)):
        cand = np.flatnonzero(mask)
        if len(cand):
            pick |= set(rng.choice(cand, min(8, len(cand)), replace=False).tolist())
    rest = np.setdiff1d(np.arange(T), np.fromiter(pick, dtype=np.int64))
    if len(pick) < n and len(rest):
        pick |= set(rng.choice(rest, min(n - len(pick), len(rest)), replace=False).tolist())
    return np.sort(np.fromiter(pick, dtype=np.int64))


def biased_margins(scores: np.ndarray, bias: Optional[np.ndarray], idx: np.ndarray,
                   n_group: int, topk_group: int) -> np.ndarray:
    """Per token, for selection by s + b among kept groups: the smaller of
    (k-th chosen key - best unchosen key of the kept groups) and, with groups,
    (last kept group score - best dropped group score).  Decisions within
    this margin depend on the rounding of s + b."""
    T, k = idx.shape
    E = scores.shape[1]
    keys = scores + (0.0 if bias is None else bias[None, :])
    m = np.full(T, np.inf)
    if n_group > 1:
        gsc = O.group_scores(keys, n_group)
        gs = E // n_group
    for t in range(T):
        allowed = np.ones(E, dtype=bool)
        if n_group > 1:
            order = sorted(range(n_group), key=lambda g: (-gsc[t, g], g))
            kept = order[:topk_group]
            if topk_group < n_group:
                m[t] = gsc[t, kept[-1]] - gsc[t, order[topk_group]]
            allowed = np.array([e // gs in kept for e in range(E)])
        rest = [keys[t, e] for e in range(E) if allowed[e] and e not in set(idx[t].tolist())]
        if rest:
            m[t] = min(m[t], keys[t, idx[t, k - 1]] - max(rest))
    return m


def np_i(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def np_f(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()
