"""Pins for the oracle's host block manager (prefix sharing, clone-N, CoW).

Checked against things other than the oracle's own bookkeeping: an
independent content model (what each physical block's rows hold, updated
only by the writes a runner would do -- new tokens into their slots, the
copy-on-write copies the manager asks for), a recount of references from the
live block tables, and the free list equal to the blocks nobody references.
"""
import numpy as np

from oracle.block_manager import BlockManager


class ContentModel:
    """Rows of token ids per physical block, written the way the device does:
    a prompt writes its uncached tokens, a decode step its one token, a
    copy-on-write copies the first `rows` rows."""

    def __init__(self, nb, bs):
        self.rows = [[None] * bs for _ in range(nb)]
        self.bs = bs

    def write(self, table, pos, tok):
        self.rows[table[pos // self.bs]][pos % self.bs] = tok

    def copy(self, src, dst, rows):
        for r in range(rows):
            self.rows[dst][r] = self.rows[src][r]

    def read(self, table, n):
        return [self.rows[table[p // self.bs]][p % self.bs] for p in range(n)]


def _check(bm, live, content):
    refs = [0] * bm.nb
    for toks, table in live.values():
        for b in table:
            refs[b] += 1
        assert content.read(table, len(toks)) == toks          # every sequence reads its own tokens
        assert len(table) == -(-len(toks) // bm.bs)
    if hasattr(bm, "ref"):                                    # the oracle: its lists directly
        assert refs == bm.ref
        assert sorted(bm.free) == [b for b in range(bm.nb) if refs[b] == 0]
        assert len(set(bm.free)) == len(bm.free)
    else:                                                      # the native manager: its queries
        assert refs == [bm.ref_count(b) for b in range(bm.nb)]
        assert bm.num_free() == sum(1 for r in refs if r == 0)


def run_random_workload(make_bm, seed, steps=400, nb=48, bs=4, check=True):
    """Random prompts with shared prefixes, decode appends, forks and frees.
    Returns the trace of every manager answer (for comparing two managers)."""
    rng = np.random.default_rng(seed)
    bm = make_bm(nb, bs)
    content = ContentModel(nb, bs) if check else None
    live, trace, next_id = {}, [], 0
    prefixes = [list(rng.integers(0, 50, int(rng.integers(1, 14)))) for _ in range(4)]
    for step in range(steps):
        op = rng.choice(["alloc", "append", "fork", "free"], p=[0.3, 0.4, 0.1, 0.2])
        if op == "alloc" or not live:
            base = list(prefixes[int(rng.integers(4))]) if rng.random() < 0.7 else []
            toks = base + list(rng.integers(0, 50, int(rng.integers(1, 10))))
            res = bm.allocate(toks)
            trace.append(("alloc", None if res is None else (list(res[0]), res[1])))
            if res is not None:
                table, cached = res
                if check:
                    for p in range(cached, len(toks)):
                        content.write(table, p, toks[p])
                live[next_id] = (toks, list(table))
                next_id += 1
        else:
            sid = list(live)[int(rng.integers(len(live)))]
            toks, table = live[sid]
            if op == "append":
                nt = toks + [int(rng.integers(0, 50))]
                t2, cp = bm.append(nt, table)
                trace.append(("append", None if t2 is None else (list(t2), cp)))
                if t2 is not None:
                    if check:
                        if cp is not None:
                            content.copy(*cp)
                        content.write(t2, len(nt) - 1, nt[-1])
                    live[sid] = (nt, list(t2))
            elif op == "fork":
                t2 = bm.fork(table)
                trace.append(("fork", list(t2)))
                live[next_id] = (list(toks), list(t2))
                next_id += 1
            else:
                bm.release(table)
                trace.append(("free", None))
                del live[sid]
        trace.append(("free_count", bm.num_free()))
        if check:
            _check(bm, live, content)
    return trace


def test_random_workloads_keep_contents_refs_and_free_list_consistent():
    for seed in range(6):
        run_random_workload(BlockManager, seed)


def test_identical_prompts_share_full_blocks_but_recompute_the_last_token():
    bm = BlockManager(16, 4)
    t1, c1 = bm.allocate(list(range(12)))            # three full blocks
    t2, c2 = bm.allocate(list(range(12)))
    assert c1 == 0 and c2 == 8                      # the block holding the last token is not reused
    assert t2[:2] == t1[:2] and t2[2] != t1[2]
    t3, c3 = bm.allocate(list(range(13)))
    assert c3 == 12 and t3[:3] == t1[:3]            # one token after three full blocks


def test_freed_blocks_stay_reusable_until_handed_out_again():
    bm = BlockManager(4, 2)
    t, _ = bm.allocate([5, 6, 7, 8, 9])             # blocks 0, 1, 2
    bm.release(t)
    assert bm.free == [3, 2, 1, 0]
    t2, c2 = bm.allocate([5, 6, 7, 8, 1])
    assert c2 == 4 and t2[:2] == [0, 1] and bm.free == [2]
    assert t2 == [0, 1, 3]                          # the fresh tail block is the FIFO front
    t3, c3 = bm.allocate([7, 7])
    assert t3 == [2] and c3 == 0


def test_fork_then_append_copies_a_shared_partial_block_once():
    bm = BlockManager(8, 4)
    t, _ = bm.allocate([1, 2, 3, 4, 5, 6])          # blocks 0 (full), 1 (two rows)
    f = bm.fork(t)
    assert bm.ref[:2] == [2, 2]
    t2, cp = bm.append([1, 2, 3, 4, 5, 6, 7], f)
    assert cp == (1, 2, 2) and t2 == [0, 2] and bm.ref[:3] == [2, 1, 1]
    t3, cp3 = bm.append([1, 2, 3, 4, 5, 6, 7, 8], t2)   # now private: no copy
    assert cp3 is None and t3 == [0, 2]
    t4, cp4 = bm.append([1, 2, 3, 4, 5, 6, 9], t)   # the original row: block 1 is private again
    assert cp4 is None and t4 == [0, 1]


def test_no_space_changes_nothing():
    bm = BlockManager(3, 4)
    t, _ = bm.allocate(list(range(9)))              # 3 blocks
    before = (list(bm.free), list(bm.ref), dict(bm.cache))
    assert bm.allocate([1]) is None
    assert (list(bm.free), list(bm.ref), dict(bm.cache)) == before
    toks = list(range(10))
    t2, cp = bm.append(toks, t)                     # lands in the last block's free row: no block needed
    assert t2 == t and cp is None
    toks += [10, 11, 12]
    assert bm.append(toks[:11], t2)[0] == t2 and bm.append(toks[:12], t2)[0] == t2
    assert bm.append(toks[:13], t2) == (None, None)   # a 4th block: none free


# ---- the native manager against the oracle (host code: no GPU needed)

def test_native_block_manager_matches_the_oracle_step_by_step():
    import paged_kv_decode_store_gb300 as pk
    for seed in range(8):
        for nb, bs in [(48, 4), (20, 2), (96, 16)]:
            want = run_random_workload(BlockManager, seed, nb=nb, bs=bs, check=False)
            got = run_random_workload(pk.BlockManager, seed, nb=nb, bs=bs, check=True)
            assert got == want


def test_native_block_manager_rejects_bad_tables():
    import paged_kv_decode_store_gb300 as pk
    from paged_kv_decode_store_gb300 import _capi
    bm = pk.BlockManager(4, 2)
    t, _ = bm.allocate([1, 2, 3])
    import pytest
    with pytest.raises(_capi.PkvdError):
        bm.release([t[0], 9])                      # a block outside the pool: nothing released
    assert bm.ref_count(t[0]) == 1
    with pytest.raises(_capi.PkvdError):
        bm.fork([3])                               # an unreferenced block cannot be cloned
    assert bm.allocate([1] * 20) is None and bm.num_free() == 2


def _shared_prefix_brute(tables, ctx, bs):
    """Longest run of leading blocks equal in every row and full before each
    row's newest token, by brute force, in tokens."""
    B = len(tables)
    if B < 2:
        return 0
    best = 0
    for nb in range(0, min(len(t) for t in tables) + 1):
        ok = all(int(c) - 1 >= nb * bs for c in ctx) and \
            all(all(tables[i][j] == tables[0][j] and tables[0][j] >= 0 for i in range(B)) for j in range(nb))
        if ok:
            best = nb * bs
    return best


def test_shared_prefix_of_a_batch():
    """pkvd_bm_shared_prefix against brute force: forked rows share their
    prompt's blocks, private blocks differ, short rows cap the prefix."""
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_decode_store_gb300 import shared_prefix_len
    rng = np.random.default_rng(3)
    for trial in range(200):
        bs = int(rng.choice([16, 32]))
        B = int(rng.integers(1, 6))
        width = int(rng.integers(1, 12))
        shared = int(rng.integers(0, width + 1))
        base = rng.permutation(1000)[:width]
        tables = []
        for i in range(B):
            t = base.copy()
            t[shared:] = rng.permutation(1000)[:width - shared] + 1000 * (i + 1)   # private blocks
            if rng.random() < 0.2 and width:
                t[int(rng.integers(0, width))] = -1
            tables.append(t)
        ctx = rng.integers(0, width * bs + 1, size=B)
        got = shared_prefix_len(np.array(tables, dtype=np.int32), ctx.astype(np.int32), bs)
        want = _shared_prefix_brute([list(t) for t in tables], ctx, bs)
        assert got == want, (trial, got, want)
