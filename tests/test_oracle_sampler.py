"""Pins for the oracle's Philox stream and sampler.

Philox is pinned to published known-answer vectors; the sampler to closed
forms (T -> 0, k = 1, p -> 0 give greedy; p = 1, k = 0 keep everything), a
hand-computed nucleus example, the page's own ascending-sort formulation of
the nucleus filter (an independent algorithm), and a chi-square test of
Gumbel-max against the truncated softmax it must sample from.
"""
import numpy as np
import pytest
import torch
from scipy import stats

from conftest import golden_lines
from oracle import philox, sampler


def test_philox_known_answer_vectors():
    for ln in golden_lines("philox_kat.txt"):
        w = [int(x, 16) for x in ln.split()]
        ctr, key, expect = w[:4], w[4:6], w[6:]
        got = [int(x) for x in philox.philox4x32_10(ctr, key)]
        assert got == expect, (ln, [hex(g) for g in got])


def test_stream_word_layout():
    # w_j is word j % 4 of Philox(counter=(j//4, lo(off), hi(off), 0), key=(lo(seed), hi(seed)))
    seed, off = 0x0123456789ABCDEF, 0x0000000500000007
    ids = np.arange(12)
    w = philox.stream_words(seed, off, ids)
    for j in ids:
        ref = philox.philox4x32_10((j // 4, off & 0xFFFFFFFF, off >> 32, 0),
                                   (seed & 0xFFFFFFFF, seed >> 32))
        assert int(w[j]) == int(ref[j % 4])


def test_uniforms_open_interval_exact_and_uniform():
    u = philox.uniforms(12345, 0, np.arange(200_000))
    assert np.all(u > 0) and np.all(u < 1)
    k = u * 2 ** 23 - 0.5
    assert np.array_equal(k, np.round(k))          # exact 23-bit grid
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    counts, _ = np.histogram(u, bins=50, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-3


def test_greedy_ties_lowest_index():
    x = np.array([1.0, 3.0, -2.0, 3.0, 0.5])
    assert sampler.sample_row(x, 0.0, 0, 1.0, 1, 0) == 1


def test_temperature_to_zero_is_greedy():
    rng = np.random.default_rng(0)
    for s in range(20):
        x = rng.standard_normal(500) * 2
        tok = sampler.sample_row(x, 1e-6, 0, 1.0, s, s)
        assert tok == int(np.argmax(x))


def test_top_k_one_and_tiny_p_are_greedy():
    rng = np.random.default_rng(1)
    for s in range(20):
        x = rng.standard_normal(300)
        assert sampler.sample_row(x, 1.5, 1, 1.0, s, 0) == int(np.argmax(x))
        assert sampler.sample_row(x, 1.5, 0, 1e-9, s, 0) == int(np.argmax(x))


def test_p_one_and_k_zero_keep_full_vocab():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(257)
    _, info = sampler.sample_row(x, 1.0, 0, 1.0, 3, 4, return_info=True)
    assert len(info["kept"]) == 257
    _, info = sampler.sample_row(x, 1.0, 10_000, 1.0, 3, 4, return_info=True)
    assert len(info["kept"]) == 257


def test_nucleus_hand_example():
    # probabilities 0.5, 0.3, 0.15, 0.05 (T = 1): the smallest descending prefix
    # with mass > p is {0} for p < 0.5, {0,1} for 0.5 <= p < 0.8, {0,1,2} below 0.95.
    x = np.log(np.array([0.15, 0.5, 0.05, 0.3]))   # shuffled positions: ids 1,3,0,2
    cases = {0.4: {1}, 0.6: {1, 3}, 0.79: {1, 3}, 0.81: {0, 1, 3}, 0.94: {0, 1, 3}, 0.96: {0, 1, 2, 3}}
    for p, expect in cases.items():
        kept, _ = sampler.nucleus_cut(x, sampler.order_desc(x), p)
        assert set(kept.tolist()) == expect, p


def _page_top_p_filter(x, p):
    """Grok-1 section 8.3.1 formulation, written from the page's description:
    sort ascending, softmax, first index whose running sum is >= 1 - p, keep
    every logit >= the logit at that index."""
    srt = np.sort(x)
    probs = np.exp(srt - srt.max())
    probs /= probs.sum()
    idx = int(np.argmax(np.cumsum(probs) >= 1 - p))
    return set(np.nonzero(x >= srt[idx])[0].tolist())


def test_nucleus_matches_page_ascending_formulation():
    rng = np.random.default_rng(3)
    n_checked = 0
    for trial in range(300):
        V = int(rng.integers(2, 400))
        x = rng.standard_normal(V).astype(np.float32) * rng.uniform(0.5, 4)
        x = torch.from_numpy(x).to(torch.bfloat16).double().numpy()   # many ties
        p = float(rng.uniform(0.05, 0.99))
        kept, info = sampler.nucleus_cut(x, sampler.order_desc(x), p)
        # skip rows whose cut sits within rounding of p (the two formulations
        # accumulate in different orders)
        if min(abs(info["mass_before"] - p), abs(info["mass_after"] - p)) < 1e-9:
            continue
        assert set(kept.tolist()) == _page_top_p_filter(x, p)
        n_checked += 1
    assert n_checked > 250


def test_top_k_ties_keep_lowest_indices():
    x = np.array([1.0, 2.0, 2.0, 0.0, 2.0, 2.0, 3.0])
    assert sampler.topk_set(x, 3).tolist() == [6, 1, 2]
    assert sampler.topk_set(x, 1).tolist() == [6]


def test_top_k_then_top_p_on_renormalised_set():
    x = np.log(np.array([0.4, 0.3, 0.2, 0.1]))
    # top-2 renormalises to 4/7, 3/7: p = 0.5 keeps only id 0; p = 0.6 keeps both
    _, info = sampler.sample_row(x, 1.0, 2, 0.5, 0, 0, return_info=True)
    assert info["kept"].tolist() == [0]
    _, info = sampler.sample_row(x, 1.0, 2, 0.6, 0, 0, return_info=True)
    assert info["kept"].tolist() == [0, 1]


@pytest.mark.parametrize("T,k,p", [(1.0, 0, 1.0), (0.7, 0, 0.8), (1.3, 5, 1.0), (1.0, 6, 0.9)])
def test_gumbel_max_chi_square_against_truncated_softmax(T, k, p):
    rng = np.random.default_rng(4)
    x = rng.standard_normal(12) * 1.5
    probs = sampler.truncated_probs(x, T, k, p)
    n = 20_000
    draws = np.array([sampler.sample_row(x, T, k, p, 99, off) for off in range(n)])
    assert np.all(probs[draws] > 0)                 # never outside the kept set
    support = np.nonzero(probs > 0)[0]
    counts = np.array([(draws == j).sum() for j in support])
    expected = probs[support] * n
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    assert stats.chisquare(obs, exp).pvalue > 1e-3


# ---- sample_token extras: mask, token_prob, top-8 (Grok-1 section 8.3)

def _page_probs(x, T, p, mask):
    """The page's sample_token order written out with the page-form filter:
    x / T, masked ids to -1e10, ascending-sort nucleus, softmax."""
    xs = np.asarray(x, dtype=np.float64) / T
    xs = np.where(mask, xs, -1e10)
    if p < 1.0:
        keep = _page_top_p_filter(xs, p)
        xs = np.where(np.isin(np.arange(xs.shape[0]), list(keep)), xs, -1e10)
    z = np.exp(xs - xs.max())
    return z / z.sum()


def test_token_prob_and_top8_match_the_page_formula():
    rng = np.random.default_rng(21)
    checked = 0
    for trial in range(200):
        V = int(rng.integers(9, 300))
        x = torch.from_numpy((rng.standard_normal(V) * rng.uniform(0.5, 3)).astype(np.float32))
        x = x.to(torch.bfloat16).double().numpy()
        T = float(rng.uniform(0.3, 2.0))
        p = float(rng.choice([1.0, 0.9, 0.5]))
        mask = rng.random(V) > 0.3
        mask[int(rng.integers(V))] = True
        (tok, tp, p8, i8), info = sampler.sample_outputs(x, T, 0, p, 5, trial, mask=mask, return_info=True)
        n = info["nucleus"]
        if n is not None and min(abs(n["mass_before"] - p), abs(n["mass_after"] - p)) < 1e-9:
            continue
        ref = _page_probs(x, T, p, mask)
        assert mask[tok] and ref[tok] > 0
        np.testing.assert_allclose(tp, ref[tok], rtol=1e-12)
        # lax.top_k: largest first, equal values in index order
        order = np.lexsort((np.arange(V), -ref))[:8]
        np.testing.assert_allclose(p8, ref[order], rtol=1e-12, atol=0)
        assert i8.tolist() == order.tolist()
        checked += 1
    assert checked > 150


def test_all_allowed_mask_changes_nothing():
    rng = np.random.default_rng(22)
    x = rng.standard_normal(50)
    for T, k, p in [(1.0, 0, 1.0), (0.8, 7, 0.9), (0.0, 0, 1.0)]:
        a = sampler.sample_outputs(x, T, k, p, 3, 4)
        b = sampler.sample_outputs(x, T, k, p, 3, 4, mask=np.ones(50, bool))
        assert a[0] == b[0] and a[1] == b[1]
        assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])


def test_masked_ids_are_never_drawn_and_the_rest_keep_their_ratios():
    rng = np.random.default_rng(23)
    x = rng.standard_normal(10) * 1.2
    mask = np.array([1, 0, 1, 1, 0, 1, 1, 1, 0, 1], bool)
    n = 20_000
    draws = np.array([sampler.sample_row(x, 1.0, 0, 1.0, 17, off, mask=mask) for off in range(n)])
    assert mask[draws].all()
    w = np.exp(x - x.max()) * mask
    expected = w / w.sum() * n
    obs = np.array([(draws == j).sum() for j in range(10)])
    assert stats.chisquare(obs[mask], expected[mask]).pvalue > 1e-3


def test_all_masked_row_draws_uniformly_and_greedy_takes_id_zero():
    n = 12_000
    draws = np.array([sampler.sample_row(np.arange(6.0), 0.9, 0, 1.0, 8, off, mask=np.zeros(6, bool))
                      for off in range(n)])
    assert stats.chisquare(np.bincount(draws, minlength=6), np.full(6, n / 6)).pvalue > 1e-3
    assert sampler.sample_row(np.arange(6.0), 0.0, 0, 1.0, 8, 0, mask=np.zeros(6, bool)) == 0
    assert sampler.sample_row(np.arange(6.0), 0.0, 0, 1.0, 8, 0,
                              mask=np.array([1, 1, 0, 0, 0, 0], bool)) == 1


def test_top8_closed_forms():
    x = np.array([0.0, 5.0, 1.0, 5.0, 3.0, -2.0, 4.0, 2.0, 6.0, -1.0])
    # greedy: the drawn id with probability 1, then the lowest other ids
    tok, tp, p8, i8 = sampler.sample_outputs(x, 0.0, 0, 1.0, 1, 0)
    assert tok == 8 and tp == 1.0 and i8.tolist() == [8, 0, 1, 2, 3, 4, 5, 6]
    assert p8.tolist() == [1.0] + [0.0] * 7
    # top-k 3: the three kept ids by value (5.0 tie in index order), then ids 0, 2, ... at 0
    tok, tp, p8, i8 = sampler.sample_outputs(x, 1.0, 3, 1.0, 1, 0)
    assert i8.tolist() == [8, 1, 3, 0, 2, 4, 5, 6]
    w = np.exp(np.array([6.0, 5.0, 5.0]) - 6.0)
    np.testing.assert_allclose(p8[:3], w / w.sum(), rtol=1e-15)
    assert np.all(p8[3:] == 0) and abs(p8.sum() - 1) < 1e-15
