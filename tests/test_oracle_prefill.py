"""Pins for the oracle's varlen paged prefill (slot mapping and attention).

The oracle is checked against things other than itself: PyTorch's
scaled_dot_product_attention with ``is_causal=True`` (a library routine) on
contiguous K/V; the already pinned decode oracle (one new token per sequence
is a decode step); closed forms (window 1, a single token); invariances
(chunked prefill equals one-shot prefill, a prefix-cache hit reproduces the
full prefill's rows, physical blocks may be permuted); and the pages'
statement that ``cu_seqlens_k[-1] > cu_seqlens_q[-1]`` exactly when some
sequence has cached tokens.
"""
import numpy as np
import pytest
import torch

from oracle import attention, paging, prefill, store


def _layout(rng, k_lens, bs, extra=3):
    """Shuffled block tables covering k_lens tokens per sequence."""
    nblk = [-(-k // bs) for k in k_lens]
    nb = sum(nblk) + extra
    perm = rng.permutation(nb)
    width = max(max(nblk), 1) + 1
    tables = np.full((len(k_lens), width), -1, np.int64)
    at = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[at:at + n]
        at += n
    return tables, nb


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


def _case(seed, q_lens, cached, Hq, Hkv, D, bs):
    """Contiguous per-sequence K/V, a paged cache holding the cached prefix
    and the new rows written through the oracle's own slot mapping + store."""
    rng = np.random.default_rng(seed)
    k_lens = [q + c for q, c in zip(q_lens, cached)]
    tables, nb = _layout(rng, k_lens, bs)
    kc = np.full((nb, bs, Hkv, D), np.nan)
    vc = np.full((nb, bs, Hkv, D), np.nan)
    Kfull = [rng.standard_normal((k, Hkv, D)) for k in k_lens]
    Vfull = [rng.standard_normal((k, Hkv, D)) for k in k_lens]
    for i, c in enumerate(cached):                       # the cached prefix
        for p in range(c):
            s = paging.slot_of_position(tables[i], p, bs)
            kc[s // bs, s % bs] = Kfull[i][p]
            vc[s // bs, s % bs] = Vfull[i][p]
    cu_q, cu_k = _cu(q_lens), _cu(k_lens)
    slots = prefill.prefill_slot_mapping(tables, cu_q, cu_k, bs)
    k_new = np.concatenate([Kfull[i][cached[i]:] for i in range(len(q_lens))]) \
        if sum(q_lens) else np.zeros((0, Hkv, D))
    v_new = np.concatenate([Vfull[i][cached[i]:] for i in range(len(q_lens))]) \
        if sum(q_lens) else np.zeros((0, Hkv, D))
    store.kv_store(k_new, v_new, slots, kc, vc)
    Qfull = [rng.standard_normal((k, Hq, D)) for k in k_lens]
    q = np.concatenate([Qfull[i][cached[i]:] for i in range(len(q_lens))]) \
        if sum(q_lens) else np.zeros((0, Hq, D))
    return dict(q=q, kc=kc, vc=vc, tables=tables, cu_q=cu_q, cu_k=cu_k,
                Kfull=Kfull, Vfull=Vfull, Qfull=Qfull, slots=slots)


def _sdpa_causal(Q, K, V, scale):
    """torch causal SDPA in float64 on one contiguous sequence: [n, Hq, D]."""
    qt = torch.from_numpy(Q).permute(1, 0, 2).unsqueeze(0)
    kt = torch.from_numpy(K).permute(1, 0, 2).unsqueeze(0)
    vt = torch.from_numpy(V).permute(1, 0, 2).unsqueeze(0)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, is_causal=True, scale=scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (6, 1), (8, 2)])
def test_no_cache_matches_torch_causal_sdpa(Hq, Hkv):
    q_lens = [1, 7, 13, 4]
    c = _case(11 + Hq + Hkv, q_lens, [0] * 4, Hq, Hkv, 16, 4)
    out = prefill.prefill_attention(c["q"], c["kc"], c["vc"], c["tables"],
                                    c["cu_q"], c["cu_k"], 0.41)
    for i in range(4):
        ref = _sdpa_causal(c["Qfull"][i], c["Kfull"][i], c["Vfull"][i], 0.41)
        got = out[c["cu_q"][i]:c["cu_q"][i + 1]]
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (6, 2)])
def test_prefix_hit_reproduces_full_prefill_rows(Hq, Hkv):
    """New tokens after a cached prefix get exactly the rows a full causal
    prefill of the whole sequence gives them."""
    q_lens, cached = [5, 3, 9, 1], [8, 0, 4, 12]
    c = _case(5, q_lens, cached, Hq, Hkv, 8, 4)
    assert prefill.has_prefix_hits(c["cu_q"], c["cu_k"])
    out = prefill.prefill_attention(c["q"], c["kc"], c["vc"], c["tables"],
                                    c["cu_q"], c["cu_k"], 0.3)
    for i in range(4):
        ref = _sdpa_causal(c["Qfull"][i], c["Kfull"][i], c["Vfull"][i], 0.3)
        got = out[c["cu_q"][i]:c["cu_q"][i + 1]]
        np.testing.assert_allclose(got, ref[cached[i]:], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("window", [0, 1, 3, 6, 100])
def test_every_token_equals_a_decode_step(window):
    """Token at position p attends like a decode step with context p + 1
    (the decode oracle is pinned on its own, window included)."""
    q_lens, cached = [6, 2, 9], [3, 7, 0]
    c = _case(7, q_lens, cached, 4, 2, 8, 4)
    out = prefill.prefill_attention(c["q"], c["kc"], c["vc"], c["tables"],
                                    c["cu_q"], c["cu_k"], 0.5, window=window)
    seq, pos = prefill.token_positions(c["cu_q"], c["cu_k"])
    for t in range(len(seq)):
        ref = attention.decode_attention(c["q"][t:t + 1], c["kc"], c["vc"],
                                         c["tables"][seq[t]:seq[t] + 1],
                                         np.array([pos[t] + 1]), 0.5, window=window)
        np.testing.assert_allclose(out[t], ref[0], rtol=1e-12, atol=1e-12)


def test_window_one_returns_own_value_row():
    q_lens, cached = [5, 3], [2, 0]
    c = _case(9, q_lens, cached, 4, 2, 8, 4)
    out = prefill.prefill_attention(c["q"], c["kc"], c["vc"], c["tables"],
                                    c["cu_q"], c["cu_k"], 1.0, window=1)
    seq, pos = prefill.token_positions(c["cu_q"], c["cu_k"])
    for t in range(len(seq)):
        for h in range(4):
            assert np.array_equal(out[t, h], c["Vfull"][seq[t]][pos[t], h // 2])


def test_chunked_prefill_equals_one_shot():
    """Prefill in chunks (each earlier chunk is a cached prefix of the next)
    gives the one-shot outputs."""
    rng = np.random.default_rng(21)
    Hq, Hkv, D, bs, n = 4, 2, 8, 4, 23
    tables, nb = _layout(rng, [n], bs)
    K = rng.standard_normal((n, Hkv, D))
    V = rng.standard_normal((n, Hkv, D))
    Q = rng.standard_normal((n, Hq, D))

    def run(chunks):
        kc = np.full((nb, bs, Hkv, D), np.nan)
        vc = np.full((nb, bs, Hkv, D), np.nan)
        outs, done = [], 0
        for m in chunks:
            cu_q, cu_k = np.array([0, m]), np.array([0, done + m])
            slots = prefill.prefill_slot_mapping(tables, cu_q, cu_k, bs)
            store.kv_store(K[done:done + m], V[done:done + m], slots, kc, vc)
            outs.append(prefill.prefill_attention(Q[done:done + m], kc, vc, tables,
                                                  cu_q, cu_k, 0.7))
            done += m
        return np.concatenate(outs)

    one = run([n])
    np.testing.assert_array_equal(run([5, 4, 14]), one)
    np.testing.assert_array_equal(run([1] * n), one)


def test_block_permutation_invariance():
    q_lens, cached = [7, 5], [3, 6]
    a = _case(31, q_lens, cached, 4, 4, 8, 4)
    out = prefill.prefill_attention(a["q"], a["kc"], a["vc"], a["tables"],
                                    a["cu_q"], a["cu_k"], 0.6)
    perm = np.random.default_rng(0).permutation(a["kc"].shape[0])
    inv = np.argsort(perm)
    kc2, vc2 = a["kc"][perm], a["vc"][perm]
    t2 = np.where(a["tables"] >= 0, inv[np.maximum(a["tables"], 0)], -1)
    out2 = prefill.prefill_attention(a["q"], kc2, vc2, t2, a["cu_q"], a["cu_k"], 0.6)
    np.testing.assert_array_equal(out, out2)


def test_single_first_token_is_its_value_row():
    c = _case(3, [1], [0], 2, 1, 8, 4)
    out = prefill.prefill_attention(c["q"], c["kc"], c["vc"], c["tables"],
                                    c["cu_q"], c["cu_k"], 1.0)
    for h in range(2):
        assert np.array_equal(out[0, h], c["Vfull"][0][0, 0])


def test_slot_mapping_one_token_each_equals_decode_slots():
    rng = np.random.default_rng(4)
    k_lens = [5, 1, 17, 8]
    tables, _ = _layout(rng, k_lens, 4)
    cu_q, cu_k = _cu([1] * 4), _cu(k_lens)
    np.testing.assert_array_equal(
        prefill.prefill_slot_mapping(tables, cu_q, cu_k, 4),
        paging.decode_slot_mapping(tables, np.array(k_lens), 4))


def test_slot_mapping_contiguous_tables_closed_form():
    """Row i owning blocks [8 i, 8 i + 8): slot = 8 i bs + position."""
    bs, q_lens, cached = 16, [30, 1, 64, 0, 17], [5, 0, 40, 3, 100]
    tables = np.array([[8 * i + j for j in range(8)] for i in range(5)])
    cu_q, cu_k = _cu(q_lens), _cu([q + c for q, c in zip(q_lens, cached)])
    got = prefill.prefill_slot_mapping(tables, cu_q, cu_k, bs)
    want = [8 * i * bs + cached[i] + j for i in range(5) for j in range(q_lens[i])]
    np.testing.assert_array_equal(got, want)


def test_chunk_slots_partition_the_one_shot_slots():
    rng = np.random.default_rng(8)
    tables, _ = _layout(rng, [37], 8)
    one = prefill.prefill_slot_mapping(tables, [0, 37], [0, 37], 8)
    parts = [prefill.prefill_slot_mapping(tables, [0, m], [0, d + m], 8)
             for d, m in [(0, 10), (10, 20), (30, 7)]]
    np.testing.assert_array_equal(np.concatenate(parts), one)
    assert len(set(one.tolist())) == 37


def test_prefix_hit_test_matches_the_cached_count():
    """The pages give two equivalent tests for a batch with cached prefixes."""
    rng = np.random.default_rng(12)
    for _ in range(200):
        B = int(rng.integers(1, 6))
        q = rng.integers(0, 5, B)
        c = rng.integers(0, 3, B) * rng.integers(0, 2, B)
        cu_q, cu_k = _cu(q), _cu(q + c)
        assert prefill.has_prefix_hits(cu_q, cu_k) == (int(c.sum()) > 0)


def test_empty_sequences_and_bad_lengths():
    c = _case(2, [0, 3, 0], [4, 0, 0], 2, 2, 8, 4)
    out = prefill.prefill_attention(c["q"], c["kc"], c["vc"], c["tables"],
                                    c["cu_q"], c["cu_k"], 1.0)
    assert out.shape == (3, 2, 8)
    with pytest.raises(ValueError):
        prefill.sequence_lengths([0, 3], [0, 2])
    with pytest.raises(ValueError):
        prefill.sequence_lengths([1, 3], [1, 4])
