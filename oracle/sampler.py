"""Reference sampler: temperature, top-k, nucleus cut, Gumbel-max (test oracle).

Steps, in the order the pages give them:

1. Temperature.  Grok-1 "第 8 章 runners.py 推理引擎", section 8.3
   (``sample_token``): the logits are divided by the temperature before any
   filtering; section 8.3.1.1 fixes the order, temperature first, then the
   nucleus filter on the scaled distribution.  T -> 0 is greedy (section
   8.1.1 and 8.3), so T == 0 is taken as exactly ``argmax`` (lowest index on
   ties).
2. Top-k.  nanochat "04 · Engine", section 3 (``sample_next_token``): only the
   k largest logits stay candidates.  The pages do not say how ties at the
   k-th value are broken; this oracle keeps exactly k, ordering by value
   (descending) and then by index (ascending).  k <= 0 or k >= V is "off".
3. Nucleus.  Grok-1 section 8.3.1 (``top_p_filter``): sort ascending, take
   softmax probabilities, find the first index whose running sum reaches
   ``1 - p``, keep every logit ``>=`` the logit there.  Restated in
   descending order (the form used here): the kept set is the smallest
   descending prefix whose probability mass exceeds p, widened to every
   element equal to its last value.  After a top-k cut the probabilities are
   those of the renormalised top-k set.  p >= 1 is "off".
4. Gumbel-max draw.  nano-vllm "Model Runner" notes, section "run model":
   the sampler divides by the temperature, takes the softmax and draws with
   the Gumbel-max trick.  Here: token = argmax over kept j of
   ``x_j / T + g_j``, with g_j = -log(-log u_j) and u_j from the Philox
   stream in ``oracle.philox`` (lowest index wins an exact tie).

Extras of Grok-1 section 8.3 (``sample_token``), all optional:

5. Mask.  After the temperature, ``where(mask, logits, -1e10)``: a masked id
   keeps a logit of -1e10, so it is cut by every filter and never drawn while
   any allowed id remains (all masked: every id is equal, the draw uniform).
   Greedy rows (T == 0) take the argmax over the allowed ids (id 0 when none
   is allowed).
6. ``token_prob``: the drawn id's probability under ``softmax`` of the
   filtered logits (kept ids as they are, every other id at -1e10, so
   probability 0); greedy rows give 1.
7. Top-8 (``TOP_K = 8``, section 8.3.2): ``jax.lax.top_k`` of those
   probabilities: the 8 largest, an equal pair in index order (the ids of
   probability 0 therefore follow in index order).  Greedy rows: the drawn id
   with probability 1, then the lowest other ids with 0.

All arithmetic is float64 on the exactly upcast logits.
"""
from __future__ import annotations

import numpy as np

from . import philox


def greedy(x: np.ndarray) -> int:
    """argmax with the lowest index on ties."""
    return int(np.argmax(np.asarray(x, dtype=np.float64)))


def order_desc(x: np.ndarray) -> np.ndarray:
    """Indices by value descending, then index ascending."""
    x = np.asarray(x, dtype=np.float64)
    return np.lexsort((np.arange(x.shape[0]), -x))


def topk_set(x: np.ndarray, k: int) -> np.ndarray:
    """Indices kept by top-k (exactly k, lowest index first among ties)."""
    order = order_desc(x)
    if k <= 0 or k >= x.shape[0]:
        return order
    return order[:k]


def nucleus_cut(xs: np.ndarray, kept: np.ndarray, p: float):
    """Apply the nucleus cut to the candidate set ``kept`` (in descending order).

    xs are the temperature-scaled logits.  Returns (new kept indices, info)
    where info holds the masses on both sides of the cut, so callers can tell
    whether float rounding could have moved it.
    """
    vals = xs[kept]
    z = vals - vals.max()
    probs = np.exp(z)
    probs = probs / probs.sum()
    cum = np.cumsum(probs)
    over = np.nonzero(cum > p)[0]
    if over.size == 0:
        return kept, {"mass_before": float(cum[-1]), "mass_after": float(cum[-1]),
                      "cut_all": True}
    t = int(over[0])
    threshold = vals[t]
    keep_mask = vals >= threshold
    # mass strictly above the threshold value, and mass up to and including it
    above = float(probs[vals > threshold].sum())
    upto = float(probs[keep_mask].sum())
    return kept[keep_mask], {"mass_before": above, "mass_after": upto,
                             "cut_all": False}


NEG = -1e10          # the masked / filtered logit of sample_token


def masked_scaled(x: np.ndarray, temperature: float, mask=None) -> np.ndarray:
    """x / T with masked ids at -1e10 (mask: bool per id, True = allowed)."""
    xs = np.asarray(x, dtype=np.float64) / float(temperature)
    if mask is not None:
        xs = np.where(np.asarray(mask, dtype=bool), xs, NEG)
    return xs


def kept_set(x: np.ndarray, temperature: float, top_k: int, top_p: float, mask=None):
    """Ids that survive the mask, top-k and nucleus filters (T > 0), plus the
    nucleus diagnostics (None when the nucleus is off)."""
    xs = masked_scaled(x, temperature, mask)
    kept = topk_set(xs, int(top_k))
    ninfo = None
    if float(top_p) < 1.0:
        kept, ninfo = nucleus_cut(xs, kept, float(top_p))
    return xs, kept, ninfo


def sample_row(x: np.ndarray, temperature: float, top_k: int, top_p: float,
               seed: int, offset: int, return_info: bool = False, mask=None):
    """One row's token id (and diagnostics used by the parity tests)."""
    x = np.asarray(x, dtype=np.float64)
    T = float(temperature)
    info = {"greedy": False, "nucleus": None, "top2_gap": np.inf,
            "top1_score": 0.0, "kept": None}
    if T < 0:
        raise ValueError("negative temperature")
    if T == 0.0:
        if mask is not None and np.any(mask):
            tok = greedy(np.where(np.asarray(mask, dtype=bool), x, -np.inf))
        else:
            tok = greedy(x) if mask is None else 0
        info["greedy"] = True
        return (tok, info) if return_info else tok
    xs, kept, info["nucleus"] = kept_set(x, T, top_k, top_p, mask)
    kept_sorted = np.sort(kept)
    g = philox.gumbel(seed, offset, kept_sorted)
    score = xs[kept_sorted] + g
    best = int(np.argmax(score))          # first maximum = lowest index
    tok = int(kept_sorted[best])
    if score.shape[0] > 1:
        two = np.partition(score, -2)[-2:]
        info["top2_gap"] = float(two[1] - two[0])
    info["top1_score"] = float(score[best])
    info["kept"] = kept_sorted
    return (tok, info) if return_info else tok


def filtered_probs(x: np.ndarray, temperature: float, top_k: int, top_p: float, mask=None) -> np.ndarray:
    """softmax of the filtered logits: kept ids as scaled, every other id at
    -1e10 (T > 0)."""
    xs, kept, _ = kept_set(x, temperature, top_k, top_p, mask)
    f = np.full_like(xs, NEG)
    f[kept] = xs[kept]
    z = np.exp(f - f.max())
    return z / z.sum()


def sample_outputs(x: np.ndarray, temperature: float, top_k: int, top_p: float,
                   seed: int, offset: int, mask=None, return_info: bool = False):
    """(token, token_prob, top-8 probabilities, top-8 ids) of one row.

    The top-8 order is the mathematical one: ids of positive probability
    (kept and allowed) by scaled logit descending, then index; then the ids
    of probability 0 (filtered or masked) by index.  (Float underflow of a
    kept id's probability does not move it into the second group.)"""
    res = sample_row(x, temperature, top_k, top_p, seed, offset, return_info=True, mask=mask)
    tok, info = res
    V = np.asarray(x).shape[0]
    if float(temperature) == 0.0:
        probs = np.zeros(V)
        probs[tok] = 1.0
        positive = np.array([tok])
        xs = np.zeros(V)
    else:
        probs = filtered_probs(x, temperature, top_k, top_p, mask)
        xs, kept, _ = kept_set(x, temperature, top_k, top_p, mask)
        allowed = np.ones(V, dtype=bool) if mask is None else np.asarray(mask, dtype=bool)
        if not allowed.any():
            allowed = np.ones(V, dtype=bool)       # all masked: every id equal (uniform)
        positive = np.array(sorted(set(kept.tolist()) & set(np.nonzero(allowed)[0].tolist())), dtype=np.int64)
    pos_order = positive[np.lexsort((positive, -xs[positive]))] if positive.size else positive
    rest = np.setdiff1d(np.arange(V), positive)
    order = np.concatenate([pos_order, rest])[:8].astype(np.int64)
    out = (tok, float(probs[tok]), probs[order], order)
    return (out, info) if return_info else out


def truncated_probs(x: np.ndarray, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    """Probability of each id under the truncated, renormalised softmax
    (the distribution the Gumbel-max draw samples from)."""
    x = np.asarray(x, dtype=np.float64)
    xs = x / float(temperature)
    kept = topk_set(x, int(top_k))
    if float(top_p) < 1.0:
        kept, _ = nucleus_cut(xs, kept, float(top_p))
    out = np.zeros_like(xs)
    z = xs[kept] - xs[kept].max()
    w = np.exp(z)
    out[kept] = w / w.sum()
    return out


def sample_batch(logits: np.ndarray, temperature, top_k, top_p, seeds, offsets,
                 return_info: bool = False):
    res = [sample_row(logits[i], temperature[i], top_k[i], top_p[i],
                      int(seeds[i]), int(offsets[i]), return_info)
           for i in range(logits.shape[0])]
    if return_info:
        return np.array([r[0] for r in res], dtype=np.int64), [r[1] for r in res]
    return np.array(res, dtype=np.int64)
