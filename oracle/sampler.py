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


def sample_row(x: np.ndarray, temperature: float, top_k: int, top_p: float,
               seed: int, offset: int, return_info: bool = False):
    """One row's token id (and diagnostics used by the parity tests)."""
    x = np.asarray(x, dtype=np.float64)
    T = float(temperature)
    info = {"greedy": False, "nucleus": None, "top2_gap": np.inf,
            "top1_score": 0.0, "kept": None}
    if T < 0:
        raise ValueError("negative temperature")
    if T == 0.0:
        tok = greedy(x)
        info["greedy"] = True
        return (tok, info) if return_info else tok
    xs = x / T
    kept = topk_set(x, int(top_k))
    if float(top_p) < 1.0:
        kept, ninfo = nucleus_cut(xs, kept, float(top_p))
        info["nucleus"] = ninfo
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
