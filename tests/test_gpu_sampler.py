"""Fused sampler on the GPU against the oracle.

Greedy ids are bit-exact.  Stochastic ids must equal the oracle's for the
same Philox stream except where the oracle's two best perturbed scores are
closer than 1e-5 * max(1, |s1|), or the nucleus cut mass lies within 1e-6 of
p (float rounding can move either decision); such rows are counted, and must
be rare.  A chi-square test over 1e5 draws checks the distribution.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import workloads
from workloads import configs
from gpu_helpers import require_gpu, sampling_exempt

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev_params(si, B=None):
    B = si.logits.shape[0] if B is None else B
    return (torch.from_numpy(si.temperature).to(DEV), torch.from_numpy(si.top_k).to(DEV),
            torch.from_numpy(si.top_p).to(DEV), torch.from_numpy(si.seeds.view(np.int64)).to(DEV),
            torch.from_numpy(si.offsets.view(np.int64)).to(DEV))


_exempt = sampling_exempt


@pytest.mark.parametrize("name", list(configs.CONFIGS))
def test_greedy_bit_exact(name):
    pk = require_gpu()
    si = workloads.make_sampler_inputs(configs.CONFIGS[name])
    B = si.logits.shape[0]
    T, k, p, s, o = _dev_params(si)
    tok = pk.sample(si.logits.to(DEV), torch.zeros_like(T), k, p, s, o).cpu().numpy()
    x = si.logits.double().numpy()
    ref = [oracle.sampler.greedy(x[i]) for i in range(B)]
    assert tok.tolist() == ref


@pytest.mark.parametrize("name", list(configs.CONFIGS))
def test_stochastic_matches_oracle(name):
    pk = require_gpu()
    si = workloads.make_sampler_inputs(configs.CONFIGS[name])
    T, k, p, s, o = _dev_params(si)
    tok = pk.sample(si.logits.to(DEV), T, k, p, s, o).cpu().numpy()
    x = si.logits.double().numpy()
    mism, exempt = 0, 0
    for i in range(x.shape[0]):
        ref, info = oracle.sampler.sample_row(x[i], float(si.temperature[i]), int(si.top_k[i]),
                                              float(si.top_p[i]), int(si.seeds[i]), int(si.offsets[i]),
                                              return_info=True)
        if int(tok[i]) != ref:
            if _exempt(info, float(si.top_p[i])):
                exempt += 1
            else:
                mism += 1
    assert mism == 0
    assert exempt <= max(1, x.shape[0] // 20)


def test_many_seeds_and_offsets_match_oracle():
    """Same row under 512 (seed, offset) pairs: exercises the Philox stream."""
    pk = require_gpu()
    rng = np.random.default_rng(11)
    V, R = 3001, 512
    row = torch.from_numpy((rng.standard_normal(V) * 1.5).astype(np.float32)).to(torch.bfloat16)
    logits = row.unsqueeze(0).repeat(R, 1)
    seeds = rng.integers(0, 2**63, size=R, dtype=np.int64)
    offs = rng.integers(0, 2**40, size=R, dtype=np.int64)
    T32, p32 = float(np.float32(0.9)), float(np.float32(0.97))
    T = torch.full((R,), T32, device=DEV)
    tok = pk.sample(logits.to(DEV), T, torch.full((R,), 100, dtype=torch.int32, device=DEV),
                    torch.full((R,), 0.97, device=DEV), torch.from_numpy(seeds).to(DEV),
                    torch.from_numpy(offs).to(DEV)).cpu().numpy()
    x = row.double().numpy()
    bad = 0
    for i in range(R):
        ref, info = oracle.sampler.sample_row(x, T32, 100, p32, int(seeds[i]), int(offs[i]),
                                              return_info=True)
        if int(tok[i]) != ref and not _exempt(info, p32):
            bad += 1
    assert bad == 0


@pytest.mark.parametrize("dtype,T,k,p", [(torch.float32, 1.0, 0, 1.0), (torch.bfloat16, 0.7, 0, 0.8),
                                         (torch.float16, 1.3, 5, 1.0), (torch.bfloat16, 1.0, 6, 0.9)])
def test_chi_square_1e5_draws(dtype, T, k, p):
    pk = require_gpu()
    rng = np.random.default_rng(5)
    V, R = 40, 100_000
    row = torch.from_numpy((rng.standard_normal(V) * 1.5).astype(np.float32)).to(dtype)
    logits = row.unsqueeze(0).repeat(R, 1).to(DEV)
    tok = pk.sample(logits, torch.full((R,), T, device=DEV), torch.full((R,), k, dtype=torch.int32, device=DEV),
                    torch.full((R,), p, device=DEV), torch.full((R,), 1234, dtype=torch.int64, device=DEV),
                    torch.arange(R, dtype=torch.int64, device=DEV)).cpu().numpy()
    probs = oracle.sampler.truncated_probs(row.double().numpy(), float(np.float32(T)), k, float(np.float32(p)))
    assert np.all(probs[tok] > 0)
    support = np.nonzero(probs > 0)[0]
    counts = np.bincount(tok, minlength=V)[support]
    expected = probs[support] * R
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    assert stats.chisquare(obs, exp).pvalue > 1e-3


def test_top_k_tie_group_straddling_the_cut():
    """Ten equal logits at the k-th value: exactly the lowest-index ones stay."""
    pk = require_gpu()
    V, R = 300, 4000
    x = torch.full((V,), -3.0)
    x[[250, 5, 77]] = 2.0                       # three clear leaders
    ties = [290, 12, 150, 33, 199, 8, 64, 111, 275, 40]
    x[ties] = 1.0
    logits = x.to(torch.bfloat16).unsqueeze(0).repeat(R, 1).to(DEV)
    tok = pk.sample(logits, torch.full((R,), 3.0, device=DEV), torch.full((R,), 7, dtype=torch.int32, device=DEV),
                    torch.ones(R, device=DEV), torch.full((R,), 99, dtype=torch.int64, device=DEV),
                    torch.arange(R, dtype=torch.int64, device=DEV)).cpu().numpy()
    allowed = {250, 5, 77} | set(sorted(ties)[:4])
    assert set(tok.tolist()) == allowed
    ref = oracle.sampler.topk_set(x.double().numpy(), 7)
    assert set(ref.tolist()) == allowed


def test_degenerate_rows():
    pk = require_gpu()
    # vocab 1; all-equal logits (greedy -> 0, sampling uniform over ids); p = 0 keeps the top group
    one = torch.zeros(3, 1, dtype=torch.float32, device=DEV)
    T = torch.tensor([0.0, 1.0, 5.0], device=DEV)
    z = torch.zeros(3, dtype=torch.int64, device=DEV)
    tok = pk.sample(one, T, torch.zeros(3, dtype=torch.int32, device=DEV), torch.ones(3, device=DEV), z, z)
    assert tok.cpu().tolist() == [0, 0, 0]
    flat = torch.zeros(2, 50, dtype=torch.float16, device=DEV)
    tok = pk.sample(flat, torch.tensor([0.0, 1.0], device=DEV), torch.zeros(2, dtype=torch.int32, device=DEV),
                    torch.ones(2, device=DEV), z[:2], z[:2])
    assert tok.cpu().tolist()[0] == 0
    x = torch.randn(64, 500, device=DEV)
    x[:, 17] = 100.0
    tok = pk.sample(x, torch.ones(64, device=DEV), torch.zeros(64, dtype=torch.int32, device=DEV),
                    torch.zeros(64, device=DEV), torch.arange(64, device=DEV), torch.zeros(64, dtype=torch.int64, device=DEV))
    assert (tok == 17).all()
    # negative zero and positive zero are the same value
    y = torch.tensor([[-0.0, 0.0, -1.0]], dtype=torch.bfloat16, device=DEV)
    tok = pk.sample(y, torch.zeros(1, device=DEV), torch.zeros(1, dtype=torch.int32, device=DEV),
                    torch.ones(1, device=DEV), z[:1], z[:1])
    assert tok.item() == 0


def test_unaligned_rows_use_the_scalar_path():
    pk = require_gpu()
    rng = np.random.default_rng(3)
    base = torch.from_numpy(rng.standard_normal((8, 1001)).astype(np.float32)).to(torch.bfloat16)
    logits = base.to(DEV)[:, 1:]                 # rows start 2 bytes past a 16-byte boundary
    z = torch.zeros(8, dtype=torch.int64, device=DEV)
    tok = pk.sample(logits, torch.zeros(8, device=DEV), torch.zeros(8, dtype=torch.int32, device=DEV),
                    torch.ones(8, device=DEV), z, z).cpu().tolist()
    ref = [oracle.sampler.greedy(base[i, 1:].double().numpy()) for i in range(8)]
    assert tok == ref


def test_window_fallback_when_top_k_lies_below_the_window():
    """Keys more than 32768 steps below the max force the radix fallback."""
    pk = require_gpu()
    V, R = 4096, 3000
    x = torch.full((V,), -65000.0)
    x[1234] = 65000.0
    logits = x.to(torch.float16).unsqueeze(0).repeat(R, 1).to(DEV)
    tok = pk.sample(logits, torch.full((R,), 1e6, device=DEV), torch.full((R,), 5, dtype=torch.int32, device=DEV),
                    torch.ones(R, device=DEV), torch.full((R,), 5, dtype=torch.int64, device=DEV),
                    torch.arange(R, dtype=torch.int64, device=DEV)).cpu().numpy()
    ref = set(oracle.sampler.topk_set(x.to(torch.float16).double().numpy(), 5).tolist())
    assert ref == {1234, 0, 1, 2, 3}
    assert set(tok.tolist()) == ref


def test_radix_top_k_ties_straddle_ranks():
    """A k-th value too far below the max for the window (radix selection),
    held by a tie group that starts inside one rank's slice and runs on into
    the next: the lowest-index ties are kept across the rank boundary."""
    pk = require_gpu()
    V, R = 151936, 64
    x = torch.full((V,), -60000.0)
    x[70000:] = -30000.0
    top = [7, 100000, 151000]
    x[top] = 65000.0
    t = 8000
    k = len(top) + t
    logits = x.to(torch.float16).unsqueeze(0).repeat(R, 1).to(DEV)
    seeds = torch.arange(R, dtype=torch.int64) * 31 + 5
    offs = torch.arange(R, dtype=torch.int64)
    T = 1e6
    tok = pk.sample(logits, torch.full((R,), T, device=DEV), torch.full((R,), k, dtype=torch.int32, device=DEV),
                    torch.ones(R, device=DEV), seeds.to(DEV), offs.to(DEV)).cpu().numpy()
    xd = x.to(torch.float16).double().numpy()
    allowed = set(oracle.sampler.topk_set(xd, k).tolist())
    assert sorted(a for a in allowed if a not in top) == list(range(70000, 70000 + t))
    assert set(tok.tolist()) <= allowed
    assert max(int(a) for a in tok if a not in top) > 76000     # past a two-way split of the row
    for i in range(8):
        ref, info = oracle.sampler.sample_row(xd, float(np.float32(T)), k, 1.0, int(seeds[i]), int(offs[i]),
                                              return_info=True)
        assert int(tok[i]) == ref or _exempt(info, 1.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_unaligned_rows_stochastic_match_oracle(dtype):
    """Rows that cannot be bulk-copied take the generic radix path."""
    pk = require_gpu()
    rng = np.random.default_rng(9)
    R, V = 24, 5001
    base = torch.from_numpy((rng.standard_normal((R, V + 1)) * 2).astype(np.float32)).to(dtype)
    logits = base.to(DEV)[:, 1:]
    T = torch.from_numpy(rng.uniform(0.5, 1.5, R).astype(np.float32))
    K = torch.from_numpy(rng.choice([0, 7, 40], R).astype(np.int32))
    P = torch.from_numpy(rng.choice([1.0, 0.9, 0.6], R).astype(np.float32))
    S = torch.from_numpy(rng.integers(0, 2**62, R, dtype=np.int64))
    O = torch.from_numpy(rng.integers(0, 2**30, R, dtype=np.int64))
    tok = pk.sample(logits, T.to(DEV), K.to(DEV), P.to(DEV), S.to(DEV), O.to(DEV)).cpu().numpy()
    bad = 0
    for i in range(R):
        ref, info = oracle.sampler.sample_row(base[i, 1:].double().numpy(), float(T[i]), int(K[i]), float(P[i]),
                                              int(S[i]), int(O[i]), return_info=True)
        if int(tok[i]) != ref and not _exempt(info, float(P[i])):
            bad += 1
    assert bad == 0


def _branch_case(name):
    """Full-width rows that steer the 16-bit windowed path into each of its
    branches: the first-window list overflowing, a nucleus cut past the
    first window (second counting stage), top-k with nucleus and a tie
    group resolved from the tie list, and a tie group too large for it."""
    rng = np.random.default_rng(17)
    R, V = 6, 151936
    if name == "list_overflow":            # every id within two binades of the max
        x = 8.0 + 0.5 * rng.standard_normal((R, V))
        return torch.from_numpy(x.astype(np.float32)).to(torch.float16), 1.0, 0, 0.9
    if name == "second_stage":             # nearly flat weights: the cut lies ~5 binades below the max
        x = np.exp2(rng.uniform(-7.0, 3.0, (R, V)))
        return torch.from_numpy(x.astype(np.float32)).to(torch.float16), 50.0, 0, 0.6
    if name == "topk_nucleus_ties":        # bf16 with many equal values near the k-th
        x = np.round(2.0 * rng.standard_normal((R, V)), 1)
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16), 1.0, 300, 0.9
    if name == "huge_tie_group":           # 50k ids at the k-th value
        x = np.full((R, V), -3.0)
        x[:, rng.choice(V, 50_000, replace=False)] = 1.0
        for r in range(R):
            x[r, rng.choice(V, 20, replace=False)] = 2.0
        return torch.from_numpy(x.astype(np.float32)).to(torch.float16), 1.0, 1000, 1.0
    raise KeyError(name)


@pytest.mark.parametrize("name", ["list_overflow", "second_stage", "topk_nucleus_ties", "huge_tie_group"])
def test_windowed_path_branches_match_oracle(name):
    pk = require_gpu()
    logits, T, k, p = _branch_case(name)
    R = logits.shape[0]
    seeds = torch.arange(1, R + 1, dtype=torch.int64) * 7919
    offs = torch.arange(R, dtype=torch.int64) * 3
    tok = pk.sample(logits.to(DEV), torch.full((R,), T, device=DEV), torch.full((R,), k, dtype=torch.int32, device=DEV),
                    torch.full((R,), p, device=DEV), seeds.to(DEV), offs.to(DEV)).cpu().numpy()
    bad = 0
    for i in range(R):
        ref, info = oracle.sampler.sample_row(logits[i].double().numpy(), float(np.float32(T)), k,
                                              float(np.float32(p)), int(seeds[i]), int(offs[i]), return_info=True)
        if int(tok[i]) != ref and not _exempt(info, float(np.float32(p))):
            bad += 1
    assert bad == 0


# ---- sample_token extras (NEXT f2): mask, token_prob, top-8

def _extras_rows(name, R, V, dtype, rng):
    if name == "normal":
        x = rng.standard_normal((R, V)) * 2.0
    elif name == "bf16_ties":
        x = np.round(rng.standard_normal((R, V)) * 2.0, 1)
    else:
        raise KeyError(name)
    return torch.from_numpy(x.astype(np.float32)).to(dtype)


@pytest.mark.parametrize("dtype,V,case", [(torch.float16, 151936, "normal"), (torch.bfloat16, 65536, "bf16_ties"),
                                          (torch.float32, 5000, "normal"), (torch.bfloat16, 2048, "normal")])
def test_sample_ex_matches_oracle(dtype, V, case):
    pk = require_gpu()
    rng = np.random.default_rng(31)
    R = 12
    logits = _extras_rows(case, R, V, dtype, rng)
    T = rng.choice([0.0, 0.6, 1.0, 1.4], R).astype(np.float32)
    K = rng.choice([0, 5, 50, 300], R).astype(np.int32)
    P = rng.choice([1.0, 0.9, 0.5], R).astype(np.float32)
    allowed = rng.random((R, V)) > rng.choice([0.0, 0.3, 0.9], R)[:, None]
    allowed[3] = False                                     # a row with nothing allowed
    T[3] = 0.8
    T[4] = 0.0
    allowed[4] = rng.random(V) > 0.5                        # a greedy row with a mask
    S = rng.integers(0, 2**62, R, dtype=np.int64)
    O = rng.integers(0, 2**30, R, dtype=np.int64)
    mask_words = pk.pack_mask(torch.from_numpy(allowed)).to(DEV)
    tok, tp, p8, i8 = pk.sample_ex(logits.to(DEV), torch.from_numpy(T).to(DEV), torch.from_numpy(K).to(DEV),
                                   torch.from_numpy(P).to(DEV), torch.from_numpy(S).to(DEV),
                                   torch.from_numpy(O).to(DEV), mask_words=mask_words)
    tok, tp, p8, i8 = tok.cpu().numpy(), tp.cpu().numpy(), p8.cpu().numpy(), i8.cpu().numpy()
    # the ids equal plain sampling on the same inputs with masked logits at -inf
    x = logits.double().numpy()
    checked = 0
    for r in range(R):
        (rt, rp, r8p, r8i), info = oracle.sampler.sample_outputs(x[r], float(T[r]), int(K[r]), float(P[r]), int(S[r]),
                                                                  int(O[r]), mask=allowed[r], return_info=True)
        if r == 3:                                          # nothing allowed: uniform draw
            assert 0 <= tok[r] < V and abs(tp[r] - 1.0 / V) < 1e-9 and i8[r].tolist() == list(range(8))
            continue
        if int(tok[r]) != rt:
            assert _exempt(info, float(P[r]))
            continue
        assert allowed[r, tok[r]]
        np.testing.assert_allclose(tp[r], rp, rtol=1e-5, atol=1e-30)
        assert i8[r].tolist() == r8i.tolist()
        np.testing.assert_allclose(p8[r], r8p, rtol=1e-5, atol=1e-30)
        checked += 1
    assert checked >= R - 3


def test_all_allowed_mask_gives_the_same_ids_as_plain_sampling():
    pk = require_gpu()
    si = workloads.make_sampler_inputs(configs.QWEN3)
    T, k, p, s, o = _dev_params(si)
    L = si.logits.to(DEV)
    plain = pk.sample(L, T, k, p, s, o)
    words = pk.pack_mask(torch.ones(L.shape, dtype=torch.bool)).to(DEV)
    masked, _, _, _ = pk.sample_ex(L, T, k, p, s, o, mask_words=words, with_probs=False)
    assert torch.equal(plain, masked)


def test_masked_ids_are_never_drawn_chi_square():
    pk = require_gpu()
    rng = np.random.default_rng(32)
    V, R = 40, 100_000
    row = torch.from_numpy((rng.standard_normal(V) * 1.5).astype(np.float32)).to(torch.bfloat16)
    allowed = torch.from_numpy(rng.random(V) > 0.4)
    logits = row.unsqueeze(0).repeat(R, 1).to(DEV)
    words = pk.pack_mask(allowed.unsqueeze(0).repeat(R, 1)).to(DEV)
    tok, _, _, _ = pk.sample_ex(logits, torch.full((R,), 0.9, device=DEV), torch.zeros(R, dtype=torch.int32, device=DEV),
                                torch.full((R,), 0.95, device=DEV), torch.full((R,), 5, dtype=torch.int64, device=DEV),
                                torch.arange(R, dtype=torch.int64, device=DEV), mask_words=words, with_probs=False)
    tok = tok.cpu().numpy()
    probs = oracle.sampler.filtered_probs(row.double().numpy(), float(np.float32(0.9)), 0, float(np.float32(0.95)),
                                          allowed.numpy())
    assert np.all(allowed.numpy()[tok]) and np.all(probs[tok] > 0)
    support = np.nonzero(probs > 0)[0]
    counts = np.bincount(tok, minlength=V)[support]
    expected = probs[support] * R
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    assert stats.chisquare(obs, exp).pvalue > 1e-3


def test_nothing_allowed_draws_uniformly():
    pk = require_gpu()
    V, R = 24, 60_000
    logits = torch.randn(R, V, device=DEV).to(torch.float16)
    words = pk.pack_mask(torch.zeros(R, V, dtype=torch.bool)).to(DEV)
    tok, tp, _, i8 = pk.sample_ex(logits, torch.ones(R, device=DEV), torch.zeros(R, dtype=torch.int32, device=DEV),
                                  torch.ones(R, device=DEV), torch.full((R,), 9, dtype=torch.int64, device=DEV),
                                  torch.arange(R, dtype=torch.int64, device=DEV), mask_words=words)
    counts = np.bincount(tok.cpu().numpy(), minlength=V)
    assert stats.chisquare(counts, np.full(V, R / V)).pvalue > 1e-3
    assert torch.allclose(tp, torch.full_like(tp, 1.0 / V))
    assert torch.equal(i8[0].cpu(), torch.arange(8, dtype=torch.int32))


def test_single_and_multi_wave_launches_match_oracle():
    """The same rows sampled in a batch that one wave of clusters covers and
    inside a batch of several waves (which the library runs with two CTAs of
    512 threads per SM instead of one of 1024): greedy ids bit-exact, drawn ids
    equal to the oracle's except for the exempt near-ties, in both."""
    pk = require_gpu()
    cfg = configs.QWEN3
    si = workloads.make_sampler_inputs(cfg, num_rows=48)
    x = si.logits.double().numpy()
    ref = [oracle.sampler.sample_row(x[i], float(si.temperature[i]), int(si.top_k[i]), float(si.top_p[i]),
                                     int(si.seeds[i]), int(si.offsets[i]), return_info=True) for i in range(48)]
    greedy_ref = [oracle.sampler.greedy(x[i]) for i in range(48)]
    for copies in (1, 10):                                     # 48 rows; 480 rows (several waves)
        logits = si.logits.repeat(copies, 1).to(DEV)
        rep = lambda a: torch.from_numpy(np.tile(a, copies)).to(DEV)
        T, k, p = rep(si.temperature), rep(si.top_k), rep(si.top_p)
        s, o = rep(si.seeds.view(np.int64)), rep(si.offsets.view(np.int64))
        tok = pk.sample(logits, T, k, p, s, o).cpu().numpy()
        g = pk.sample(logits, torch.zeros_like(T), k, p, s, o).cpu().numpy()
        for c in range(copies):
            assert g[c * 48:(c + 1) * 48].tolist() == greedy_ref
            bad = 0
            for i in range(48):
                t = int(tok[c * 48 + i])
                if t != ref[i][0] and not sampling_exempt(ref[i][1], float(si.top_p[i])):
                    bad += 1
            assert bad == 0, (copies, c)


@pytest.mark.parametrize("dtype,T", [(torch.bfloat16, 1.0), (torch.float16, 2.0), (torch.bfloat16, 0.5)])
def test_untruncated_draws_match_oracle(dtype, T):
    """No top-k and no nucleus (the plain temperature softmax): most ids are
    candidates, so the kernel draws word by word with one Philox call per
    four ids; the ids still follow the Philox stream id by id."""
    pk = require_gpu()
    rng = np.random.default_rng(21)
    R, V = 96, 6000
    logits = torch.from_numpy((rng.standard_normal((R, V)) * 2).astype(np.float32)).to(dtype)
    seeds = rng.integers(0, 2**62, size=R, dtype=np.int64)
    offs = rng.integers(0, 2**40, size=R, dtype=np.int64)
    T32 = float(np.float32(T))
    tok = pk.sample(logits.to(DEV), torch.full((R,), T, device=DEV), torch.zeros(R, dtype=torch.int32, device=DEV),
                    torch.ones(R, device=DEV), torch.from_numpy(seeds).to(DEV),
                    torch.from_numpy(offs).to(DEV)).cpu().numpy()
    x = logits.double().numpy()
    bad = exempt = 0
    for i in range(R):
        ref, info = oracle.sampler.sample_row(x[i], T32, 0, 1.0, int(seeds[i]), int(offs[i]), return_info=True)
        if int(tok[i]) != ref:
            if sampling_exempt(info, 1.0):
                exempt += 1
            else:
                bad += 1
    assert bad == 0 and exempt <= 2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_chi_square_untruncated_16bit(dtype):
    pk = require_gpu()
    rng = np.random.default_rng(8)
    V, R = 48, 100_000
    row = torch.from_numpy((rng.standard_normal(V) * 1.2).astype(np.float32)).to(dtype)
    logits = row.unsqueeze(0).repeat(R, 1).to(DEV)
    tok = pk.sample(logits, torch.ones(R, device=DEV), torch.zeros(R, dtype=torch.int32, device=DEV),
                    torch.ones(R, device=DEV), torch.full((R,), 77, dtype=torch.int64, device=DEV),
                    torch.arange(R, dtype=torch.int64, device=DEV)).cpu().numpy()
    probs = oracle.sampler.truncated_probs(row.double().numpy(), 1.0, 0, 1.0)
    counts = np.bincount(tok, minlength=V)
    expected = probs * R
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    assert stats.chisquare(obs, exp).pvalue > 1e-3
