"""Pins for the oracle's slot arithmetic, cache sizing and scalar store."""
import numpy as np
import pytest
import torch

from conftest import golden_lines
from oracle import paging, store


def test_slot_worked_example():
    # nano-vllm "Model Runner" notes, "allocated kv cache": pos 299, table [5, 10], block 256 -> 2603
    (line,) = golden_lines("slot_example.txt")
    pos, table, bs, logical, physical, offset, slot = line.split()
    table = [int(t) for t in table.split(",")]
    pos, bs = int(pos), int(bs)
    assert pos // bs == int(logical)
    assert table[pos // bs] == int(physical)
    assert pos % bs == int(offset)
    assert paging.slot_of_position(table, pos, bs) == int(slot)


def test_decode_slot_mapping_positions():
    # new token sits at position ctx-1 ("prefill and decode": n-1 cached + 1 now)
    tables = np.array([[5, 10, -1], [7, -1, -1], [3, 4, 9], [2, -1, -1]], dtype=np.int32)
    ctx = np.array([300, 1, 513, 0], dtype=np.int32)
    got = paging.decode_slot_mapping(tables, ctx, 256)
    assert got.tolist() == [10 * 256 + 43, 7 * 256 + 0, 9 * 256 + 0, -1]


def test_slot_mapping_brute_force_flat_positions():
    # Brute force: lay every sequence's blocks out explicitly and count positions.
    rng = np.random.default_rng(0)
    bs, nb = 16, 64
    perm = rng.permutation(nb)
    ctx = [1, 15, 16, 17, 33, 100]
    tables, pos = [], 0
    for c in ctx:
        n = -(-c // bs)
        tables.append(list(perm[pos:pos + n]) + [-1] * (8 - n))
        pos += n
    tables = np.array(tables, dtype=np.int32)
    got = paging.decode_slot_mapping(tables, np.array(ctx), bs)
    for i, c in enumerate(ctx):
        flat = [b * bs + r for b in tables[i] if b >= 0 for r in range(bs)]
        assert got[i] == flat[c - 1]


def _sizing():
    out = {}
    for ln in golden_lines("cache_sizing.txt"):
        name, factors, value = [s.strip() for s in ln.split("|")]
        kv = dict(f.split("=") for f in factors.split())
        out[name] = ({k: int(v) for k, v in kv.items()}, value)
    return out


def test_block_bytes_qwen3():
    f, v = _sizing()["qwen3_block_bytes"]
    got = paging.paged_block_bytes(f["layers"], f["block"], f["kv_heads"], f["head_dim"], f["itemsize"])
    assert got == int(v) == 29_360_128


def test_grok_cache_bytes_and_gqa_ratio():
    s = _sizing()
    f, v = s["grok1_cache_bytes"]
    got = paging.contiguous_cache_bytes(f["layers"], f["max_len"], f["kv_heads"], f["head_dim"],
                                        f["itemsize"], f["batch"])
    assert got == int(v) == 2 * 1024 ** 3
    f2, v2 = s["grok1_mha_cache_bytes"]
    got2 = paging.contiguous_cache_bytes(f2["layers"], f2["max_len"], f2["kv_heads"], f2["head_dim"],
                                         f2["itemsize"], f2["batch"])
    assert got2 == int(v2) == 6 * got


def test_grok_waste_and_logits_row():
    s = _sizing()
    f, v = s["grok1_waste_fraction"]
    assert abs((f["max_len"] - f["used"]) / f["max_len"] - float(v)) < 1e-4
    f, v = s["grok1_logits_row_bytes"]
    assert f["vocab"] * f["itemsize"] == int(v) == 512 * 1024


def test_blocks_needed():
    assert [paging.blocks_needed(c, 16) for c in (0, 1, 16, 17, 32, 33)] == [0, 1, 1, 2, 2, 3]


# ---------------------------------------------------------------- store

def _raw16(t):
    return t.view(torch.int16).numpy().copy()


def test_store_readback_is_bit_exact_bf16_and_nan_payloads():
    rng = np.random.default_rng(1)
    nb, bs, H, D = 6, 4, 2, 8
    kc = torch.from_numpy(rng.standard_normal((nb, bs, H, D), dtype=np.float32)).to(torch.bfloat16)
    vc = kc.clone()
    k = torch.from_numpy(rng.standard_normal((3, H, D), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((3, H, D), dtype=np.float32)).to(torch.bfloat16)
    kraw, vraw = _raw16(k), _raw16(v)
    kraw[0, 0, 0] = 0x7FC1            # a NaN with a payload: a bit copy keeps it
    kc_raw, vc_raw = _raw16(kc), _raw16(vc)
    before = kc_raw.copy()
    slots = np.array([5, -1, 22], dtype=np.int64)
    store.kv_store(kraw, vraw, slots, kc_raw, vc_raw)
    assert np.array_equal(kc_raw[1, 1], kraw[0]) and np.array_equal(vc_raw[1, 1], vraw[0])
    assert np.array_equal(kc_raw[5, 2], kraw[2]) and np.array_equal(vc_raw[5, 2], vraw[2])
    # everything else untouched
    mask = np.ones((nb, bs), bool)
    mask[1, 1] = mask[5, 2] = False
    assert np.array_equal(kc_raw[mask], before[mask])


def test_store_rejects_bad_slots():
    kc = np.zeros((2, 4, 1, 2), np.float32)
    vc = kc.copy()
    k = np.ones((2, 1, 2), np.float32)
    with pytest.raises(IndexError):
        store.kv_store(k, k, np.array([0, 8]), kc, vc)
    with pytest.raises(ValueError):
        store.kv_store(k, k, np.array([3, 3]), kc, vc)
