"""Pins for the oracle's paged decode attention and LSE merge.

The oracle is checked against things other than itself: PyTorch's
scaled_dot_product_attention (a library routine) on the de-paged contiguous
K/V, closed forms (one token, equal keys, empty context), invariances
(physical block permutation) and the softmax identity for split contexts.
"""
import numpy as np
import pytest
import torch

from oracle import attention


def _random_paged(rng, B, Hq, Hkv, D, bs, ctx, pool_extra=3):
    nblk = [-(-c // bs) for c in ctx]
    nb = sum(nblk) + pool_extra
    perm = rng.permutation(nb)
    width = max(max(nblk), 1) + 1
    tables = np.full((B, width), -1, np.int64)
    pos = 0
    for i in range(B):
        tables[i, :nblk[i]] = perm[pos:pos + nblk[i]]
        pos += nblk[i]
    kc = rng.standard_normal((nb, bs, Hkv, D))
    vc = rng.standard_normal((nb, bs, Hkv, D))
    q = rng.standard_normal((B, Hq, D))
    return q, kc, vc, tables, np.array(ctx)


def _contiguous(kc, vc, table, c):
    bs = kc.shape[1]
    rows = [(table[j // bs], j % bs) for j in range(c)]
    K = np.stack([kc[b, r] for b, r in rows])   # [c, Hkv, D]
    V = np.stack([vc[b, r] for b, r in rows])
    return K, V


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (6, 1), (8, 2)])
def test_matches_torch_sdpa_gqa(Hq, Hkv):
    rng = np.random.default_rng(Hq * 10 + Hkv)
    B, D, bs = 4, 16, 4
    ctx = [1, 5, 12, 9]
    q, kc, vc, tables, ctx = _random_paged(rng, B, Hq, Hkv, D, bs, ctx)
    scale = 0.37
    out = attention.decode_attention(q, kc, vc, tables, ctx, scale)
    for i in range(B):
        K, V = _contiguous(kc, vc, tables[i], ctx[i])
        qt = torch.from_numpy(q[i]).unsqueeze(0).unsqueeze(2)          # [1, Hq, 1, D]
        Kt = torch.from_numpy(K).permute(1, 0, 2).unsqueeze(0)         # [1, Hkv, c, D]
        Vt = torch.from_numpy(V).permute(1, 0, 2).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, Kt, Vt, scale=scale, enable_gqa=True)[0, :, 0].numpy()
        np.testing.assert_allclose(out[i], ref, rtol=1e-12, atol=1e-12)


def test_single_token_returns_v_exactly():
    rng = np.random.default_rng(3)
    q, kc, vc, tables, ctx = _random_paged(rng, 2, 4, 2, 8, 4, [1, 1])
    out = attention.decode_attention(q, kc, vc, tables, ctx, 1.0)
    for i in range(2):
        for h in range(4):
            assert np.array_equal(out[i, h], vc[tables[i, 0], 0, h // 2])


def test_empty_context_gives_zeros():
    rng = np.random.default_rng(4)
    q, kc, vc, tables, ctx = _random_paged(rng, 2, 2, 2, 8, 4, [0, 3])
    kc[...] = np.nan     # nothing may be read for the empty row
    vc[...] = np.nan
    kc[tables[1, 0]] = 1.0
    vc[tables[1, 0]] = 2.0
    out = attention.decode_attention(q, kc, vc, tables, ctx, 1.0)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.allclose(out[1], 2.0)


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(5)
    q, kc, vc, tables, ctx = _random_paged(rng, 1, 2, 1, 8, 4, [11])
    kc[...] = 0.25
    out = attention.decode_attention(q, kc, vc, tables, ctx, 1.0)
    K, V = _contiguous(kc, vc, tables[0], 11)
    np.testing.assert_allclose(out[0, 0], V[:, 0].mean(axis=0), rtol=1e-13)


def test_invariant_under_physical_block_permutation():
    rng = np.random.default_rng(6)
    q, kc, vc, tables, ctx = _random_paged(rng, 3, 4, 2, 8, 4, [7, 13, 4])
    out = attention.decode_attention(q, kc, vc, tables, ctx, 0.5)
    nb = kc.shape[0]
    perm = rng.permutation(nb)             # new position of each old block
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tables2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1)
    out2 = attention.decode_attention(q, kc2, vc2, tables2, ctx, 0.5)
    np.testing.assert_array_equal(out, out2)


def test_tail_rows_and_unused_table_entries_are_not_read():
    rng = np.random.default_rng(7)
    q, kc, vc, tables, ctx = _random_paged(rng, 1, 2, 2, 8, 4, [6])
    ref = attention.decode_attention(q, kc, vc, tables, ctx, 1.0)
    last = tables[0, 1]
    kc[last, 2:] = np.nan
    vc[last, 2:] = np.nan
    out = attention.decode_attention(q, kc, vc, tables, ctx, 1.0)
    np.testing.assert_array_equal(out, ref)


def test_large_scores_are_stable():
    rng = np.random.default_rng(8)
    q, kc, vc, tables, ctx = _random_paged(rng, 1, 1, 1, 4, 4, [9])
    kc *= 1e3
    out = attention.decode_attention(q, kc, vc, tables, ctx, 1.0)
    assert np.all(np.isfinite(out))
    K, V = _contiguous(kc, vc, tables[0], 9)
    s = K[:, 0] @ q[0, 0]
    np.testing.assert_allclose(out[0, 0], V[int(np.argmax(s)), 0], rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("cuts", [[5], [1, 2, 3], [17, 18], [3, 9, 20, 31]])
def test_lse_merge_of_split_context_equals_full(cuts):
    rng = np.random.default_rng(len(cuts))
    ctx = 32
    K = rng.standard_normal((ctx, 16)) * 3
    V = rng.standard_normal((ctx, 16))
    q = rng.standard_normal(16)
    full = attention.attend(q, K, V, 0.7)
    edges = [0] + cuts + [ctx]
    parts = [attention.partial_state(q, K[a:b], V[a:b], 0.7) for a, b in zip(edges[:-1], edges[1:])]
    np.testing.assert_allclose(attention.lse_merge(parts), full, rtol=1e-12, atol=1e-13)


# ---- sliding window (newest W positions of the context)

@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_window_matches_sdpa_with_a_window_mask(Hq, Hkv):
    """SDPA over the whole contiguous context with a boolean mask that allows
    only positions >= ctx - W: the window as a library routine computes it."""
    rng = np.random.default_rng(40 + Hq)
    B, D, bs = 5, 16, 4
    ctx = [1, 7, 12, 9, 20]
    q, kc, vc, tables, ctx = _random_paged(rng, B, Hq, Hkv, D, bs, ctx)
    scale = 0.41
    for W in (1, 3, 8, 50):
        out = attention.decode_attention(q, kc, vc, tables, ctx, scale, window=W)
        for i in range(B):
            K, V = _contiguous(kc, vc, tables[i], ctx[i])
            c = ctx[i]
            qt = torch.from_numpy(q[i]).unsqueeze(0).unsqueeze(2)
            Kt = torch.from_numpy(K).permute(1, 0, 2).unsqueeze(0)
            Vt = torch.from_numpy(V).permute(1, 0, 2).unsqueeze(0)
            allow = torch.from_numpy(np.arange(c) >= c - W).view(1, 1, 1, c)
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, Kt, Vt, attn_mask=allow, scale=scale, enable_gqa=True)[0, :, 0].numpy()
            np.testing.assert_allclose(out[i], ref, rtol=1e-12, atol=1e-12)


def test_window_equals_full_attention_on_the_last_w_tokens_relaid():
    """The windowed row equals the unwindowed oracle on a fresh cache that
    holds only the newest W tokens, laid out from position 0 in new blocks."""
    rng = np.random.default_rng(44)
    B, Hq, Hkv, D, bs = 3, 4, 2, 8, 4
    ctx = [30, 9, 17]
    q, kc, vc, tables, ctx = _random_paged(rng, B, Hq, Hkv, D, bs, ctx)
    W = 10
    out = attention.decode_attention(q, kc, vc, tables, ctx, 0.3, window=W)
    for i in range(B):
        K, V = _contiguous(kc, vc, tables[i], ctx[i])
        K, V = K[-W:], V[-W:]
        n = K.shape[0]
        nb = -(-n // bs)
        kc2 = np.zeros((nb, bs, Hkv, D))
        vc2 = np.zeros((nb, bs, Hkv, D))
        for j in range(n):
            kc2[j // bs, j % bs] = K[j]
            vc2[j // bs, j % bs] = V[j]
        ref = attention.decode_attention(q[i:i + 1], kc2, vc2, np.arange(nb)[None, :], np.array([n]), 0.3)
        np.testing.assert_allclose(out[i], ref[0], rtol=1e-13, atol=1e-13)


def test_window_closed_forms():
    rng = np.random.default_rng(45)
    q, kc, vc, tables, ctx = _random_paged(rng, 3, 4, 2, 8, 4, [6, 13, 1])
    full = attention.decode_attention(q, kc, vc, tables, ctx, 0.5)
    # a window at least the context is no window; W <= 0 is no window
    for W in (13, 100, 0, -1):
        np.testing.assert_array_equal(attention.decode_attention(q, kc, vc, tables, ctx, 0.5, window=W), full)
    # a window of one returns the newest token's V row exactly
    one = attention.decode_attention(q, kc, vc, tables, ctx, 0.5, window=1)
    for i in range(3):
        c = ctx[i]
        blk, row = tables[i][(c - 1) // 4], (c - 1) % 4
        for h in range(4):
            np.testing.assert_array_equal(one[i, h], vc[blk, row, h // 2])
