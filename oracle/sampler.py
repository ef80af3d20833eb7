"""ORACLE -- test infrastructure only.

The sampler chain applied to one logits row, in plain numpy. Only ``tests/`` use it; the
product library never loads it and shares no code with it.

The article ("llama.cpp AI LLM Engine -- how it works", section "Sampler chain", after step 14
on ``llama_get_logits_ith``) describes sampling as a sequence of steps over one row of logits:
  1. a repeat penalty lowers the logits of tokens that already appeared;
  2. cut-offs drop candidates: top-k keeps the k largest logits, top-p (nucleus) keeps the
     tokens whose accumulated probability reaches p, min-p drops everything far below the
     leader;
  3. temperature divides the remaining logits (> 1 flattens, < 1 sharpens);
  4. one token is chosen: the largest logit (greedy) or a random draw with the softmax
     probabilities of the remaining logits.
Where the article leaves a step open, the reading taken (each one listed with the others in
the design notes):
  * penalty: a token of the history has its logit divided by the penalty when positive and
    multiplied by it otherwise (both lower it for a penalty > 1), once per distinct token; the
    result is a float32 like the stored logit (one IEEE operation, emulated exactly);
  * candidate order: larger logit first, the lower token id first among equal logits
    (-0.0 and +0.0 are equal);
  * top-p keeps the shortest prefix of that order whose probability mass (softmax over the
    candidates left by top-k) reaches p -- at least one token;
  * min-p keeps the candidates with logit >= max + ln(min_p), i.e. probability >= min_p times
    the leader's -- at least the leader;
  * the weights of the draw are exp((l - max) / temperature); the random number u in [0, 1)
    is an input; the draw walks the remaining candidates in increasing token id and returns
    the first whose running weight sum exceeds u times the total (the last one if rounding
    leaves none);
  * temperature <= 0 is the greedy choice: the leader, which every cut-off keeps.
The probabilities are computed in float64.

``nudge`` moves the three floating-point decisions by a relative amount (the top-p target,
the min-p threshold and the draw target); ``acceptable_tokens`` lists every token a correct
float32 implementation may return where a decision falls within rounding of its boundary.
"""
from __future__ import annotations

import math

import numpy as np


def penalize(logits: np.ndarray, history, penalty: float) -> np.ndarray:
    """Step 1: float32 logits with the repeat penalty applied to each distinct history token."""
    out = np.array(logits, dtype=np.float32, copy=True)
    if penalty == 1.0 or history is None:
        return out
    r = np.float32(penalty)
    V = out.shape[0]
    for t in sorted(set(int(x) for x in np.asarray(history).ravel())):
        if 0 <= t < V:
            out[t] = out[t] / r if out[t] > 0 else out[t] * r
    return out


def candidate_order(vals: np.ndarray) -> np.ndarray:
    """Token ids by decreasing logit, lower id first among equal logits."""
    ids = np.arange(vals.shape[0])
    return np.lexsort((ids, -vals.astype(np.float64)))


def prepare(logits, history=None, penalty_repeat: float = 1.0):
    """Step 1 and the candidate order: (penalised float32 logits, ids in candidate order)."""
    vals = penalize(logits, history, penalty_repeat)
    return vals, candidate_order(vals)


def chain_after_penalty(vals, order, top_k: int = 0, top_p: float = 1.0, min_p: float = 0.0, temp: float = 1.0,
                        u: float = 0.0, nudge=(0.0, 0.0, 0.0)) -> int:
    """Steps 2-4 on prepared logits (see prepare)."""
    V = vals.shape[0]
    keep = V
    if 0 < top_k < V:                                              # top-k
        keep = top_k
    v = vals[order].astype(np.float64)
    m = v[0]
    if temp <= 0 or not math.isfinite(m):                           # greedy
        return int(order[0])
    if top_p < 1.0:                                                 # top-p over the top-k survivors
        w = np.exp(v[:keep] - m)
        cum = np.cumsum(w)
        target = top_p * cum[-1] * (1.0 + nudge[0])
        n = int(np.searchsorted(cum, target, side="left"))         # first index with cum >= target
        keep = min(keep, max(1, n + 1))
    if min_p > 0.0:                                                 # min-p
        thr = m + math.log(min_p)
        thr += nudge[1] * max(1.0, abs(thr))
        keep = min(keep, max(1, int(np.count_nonzero(v[:keep] >= thr))))
    cand = np.sort(order[:keep])                                    # the draw walks ids upwards
    w = np.exp((vals[cand].astype(np.float64) - m) / temp)
    cum = np.cumsum(w)
    target = float(u) * cum[-1] * (1.0 + nudge[2])
    j = int(np.searchsorted(cum, target, side="right"))            # first index with cum > target
    return int(cand[min(j, keep - 1)])


def sample_chain(logits, history=None, penalty_repeat: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                 min_p: float = 0.0, temp: float = 1.0, u: float = 0.0, nudge=(0.0, 0.0, 0.0)) -> int:
    """The token the chain picks from one float32 logits row (see the module notes)."""
    vals, order = prepare(logits, history, penalty_repeat)
    return chain_after_penalty(vals, order, top_k, top_p, min_p, temp, u, nudge)


def acceptable_tokens(logits, history=None, penalty_repeat: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                      min_p: float = 0.0, temp: float = 1.0, u: float = 0.0, rel: float = 1e-4) -> set[int]:
    """Every token the chain may return when each floating-point decision -- the top-p target,
    the min-p threshold, the draw target -- moves by up to `rel` of its size: the tokens a
    float32 implementation may answer. Every survivor count between the extremes of the two
    cut-offs and every draw position between the extremes of the target are included; away
    from the boundaries this is the single token sample_chain returns."""
    vals, order = prepare(logits, history, penalty_repeat)
    V = vals.shape[0]
    v = vals[order].astype(np.float64)
    m = v[0]
    if temp <= 0 or not math.isfinite(m):
        return {int(order[0])}
    keep0 = top_k if 0 < top_k < V else V
    keeps_p = [keep0]
    if top_p < 1.0:
        cum = np.cumsum(np.exp(v[:keep0] - m))
        lo = int(np.searchsorted(cum, top_p * cum[-1] * (1.0 - rel), side="left"))
        hi = int(np.searchsorted(cum, top_p * cum[-1] * (1.0 + rel), side="left"))
        keeps_p = [min(keep0, max(1, n + 1)) for n in range(lo, hi + 1)]
    finals = set()
    for k1 in sorted(set(keeps_p)):
        if min_p > 0.0:
            thr = m + math.log(min_p)
            d = rel * max(1.0, abs(thr))
            lo = max(1, int(np.count_nonzero(v[:k1] >= thr + d)))
            hi = max(1, int(np.count_nonzero(v[:k1] >= thr - d)))
            finals.update(min(k1, k2) for k2 in range(lo, hi + 1))
        else:
            finals.add(k1)
    out = set()
    for keep in sorted(finals):
        cand = np.sort(order[:keep])
        cum = np.cumsum(np.exp((vals[cand].astype(np.float64) - m) / temp))
        t = float(u) * cum[-1]
        j0 = int(np.searchsorted(cum, t * (1.0 - rel), side="right"))
        j1 = int(np.searchsorted(cum, t * (1.0 + rel), side="right"))
        out.update(int(cand[min(j, keep - 1)]) for j in range(j0, j1 + 1))
    return out
