"""Pins of the oracle's prefix cache ("PagedAttention" S06, "What's next":
block contents are hashed so that two requests with a common prefix share
the same physical blocks; a chat server that sends one system prompt over
and over stops paying its prefill).

Each pin is fixed by the pages or by hand, not by the oracle: the sharing
the pages describe, hand-worked eviction orders, a closed form for a
system-prompt trace, and a brute-force property on random traces (every
slot a sequence reads holds K/V computed from that sequence's own prefix).
"""
import numpy as np
import pytest

import oracle


def _bm(N, B):
    return oracle.BlockManager(N, B, np.arange(N, dtype=np.int32))


def _prefill(bm, seq, tokens):
    """Admit through the cache, append the rest, register the full blocks."""
    n_cached = bm.add_seq_cached(seq, tokens)
    if len(tokens) > n_cached:
        bm.append(seq, len(tokens) - n_cached)
    bm.commit(seq, tokens)
    return n_cached


def _named_plus_idle_is_pool(bm, live):
    named = {int(b) for s in live for b in bm.table(s)}
    st = bm.cache_stats()
    assert len(named) + len(bm.free_list()) + st["unreferenced"] == bm.num_blocks
    return named


def test_common_prefix_shares_physical_blocks():
    bm = _bm(32, 4)
    a = list(range(100, 110))                      # 2 full blocks + 2 tokens
    assert _prefill(bm, 0, a) == 0
    b = a[:8] + [7, 7, 7]
    assert _prefill(bm, 1, b) == 8
    ta, tb = bm.table(0), bm.table(1)
    assert np.array_equal(ta[:2], tb[:2]) and ta[2] != tb[2]
    assert [bm.refcount(int(x)) for x in ta[:2]] == [2, 2]
    assert bm.cache_stats()["hits"] == 2


def test_same_block_after_a_different_prefix_is_a_miss():
    bm = _bm(32, 4)
    x, y, z = [1, 2, 3, 4], [5, 6, 7, 8], [9, 9, 9, 9]
    _prefill(bm, 0, x + y)
    assert _prefill(bm, 1, z + y) == 0               # same second block, other first block
    assert not set(bm.table(0)) & set(bm.table(1))
    assert _prefill(bm, 2, x + [5, 6, 7, 0]) == 4    # first block only
    assert bm.table(2)[0] == bm.table(0)[0]


def test_a_hit_needs_the_whole_prefix_not_just_the_block():
    """x is cached at depth 0 (from x + q) and a block holding y is cached at
    depth 1 (from w + y); x + y shares only x."""
    bm = _bm(32, 4)
    x, y, q, w = [1, 2, 3, 4], [5, 6, 7, 8], [0, 0, 0, 0], [9, 9, 9, 9]
    _prefill(bm, 0, x + q)
    _prefill(bm, 1, w + y)
    assert _prefill(bm, 2, x + y) == 4
    assert bm.table(2)[0] == bm.table(0)[0]
    assert bm.table(2)[1] not in (bm.table(0)[1], bm.table(1)[1])


def test_only_full_blocks_are_cached():
    bm = _bm(16, 4)
    p = [3, 1, 4, 1, 5, 9, 2]                        # one full block + 3 tokens
    _prefill(bm, 0, p)
    assert bm.cache_stats()["cached"] == 1
    assert _prefill(bm, 1, p) == 4
    assert bm.table(1)[1] != bm.table(0)[1]


def test_a_prompt_is_served_after_its_first_request_ended():
    N, B = 20, 4
    bm = _bm(N, B)
    system = list(range(50, 62))                     # 3 blocks
    _prefill(bm, 0, system + [1, 2])
    first = bm.table(0)[:3].copy()
    bm.free_seq(0)
    assert bm.num_free() == N                        # unreferenced cached blocks still count as free
    assert bm.cache_stats()["unreferenced"] == 3
    assert _prefill(bm, 1, system + [8]) == 12
    assert np.array_equal(bm.table(1)[:3], first)
    assert bm.cache_stats()["unreferenced"] == 0


def test_eviction_takes_the_free_list_first_then_least_recently_released_deepest_first():
    bm = _bm(6, 2)
    _prefill(bm, 0, [1, 2, 3, 4, 5, 6])              # blocks 0, 1, 2
    bm.free_seq(0)
    _prefill(bm, 1, [7, 8, 9, 10])                   # blocks 3, 4
    bm.free_seq(1)
    assert list(bm.free_list()) == [5]
    bm.add_seq(2)
    bm.append(2, 8)
    assert list(bm.table(2)) == [5, 2, 1, 0]
    assert bm.cache_stats()["evictions"] == 3
    assert _prefill(bm, 3, [1, 2, 3, 4]) == 0        # the first request's prompt is gone
    bm.free_seq(3)
    bm2 = _bm(6, 2)                                  # the second request's prompt survives
    _prefill(bm2, 0, [1, 2, 3, 4, 5, 6])
    bm2.free_seq(0)
    _prefill(bm2, 1, [7, 8, 9, 10])
    bm2.free_seq(1)
    bm2.add_seq(2)
    bm2.append(2, 8)
    assert _prefill(bm2, 3, [7, 8, 9, 10]) == 4
    assert list(bm2.table(3)) == [3, 4]


def test_out_of_blocks_counts_evictable_blocks_and_is_all_or_nothing():
    bm = _bm(4, 2)
    _prefill(bm, 0, [1, 2, 3, 4])
    bm.free_seq(0)
    bm.add_seq(1)
    with pytest.raises(oracle.OracleError):
        bm.append(1, 9)                              # 5 blocks of 4
    assert bm.cache_stats() == {"cached": 2, "unreferenced": 2, "hits": 0, "evictions": 0}
    bm.append(1, 8)
    assert bm.cache_stats()["evictions"] == 2


@pytest.mark.parametrize("R,k,B", [(10, 4, 16), (64, 8, 16), (25, 3, 4)])
def test_system_prompt_trace_closed_form(R, k, B):
    """R requests = one system prompt of k full blocks + a private suffix of
    u_i tokens: the first request allocates everything, the others hit k
    blocks each, and prefill writes S + sum(u) tokens instead of R*S + sum(u)."""
    rng = np.random.default_rng(R * 7 + k)
    S = k * B
    system = list(rng.integers(0, 32000, S))
    u = rng.integers(1, 3 * B, R)
    bm = _bm(k + int(sum(-(-u // B))) + 5, B)
    written = 0
    for i in range(R):
        toks = system + list(rng.integers(0, 32000, int(u[i])))
        written += len(toks) - _prefill(bm, i, toks)
    assert bm.cache_stats()["hits"] == (R - 1) * k
    assert written == S + int(u.sum())
    used = _named_plus_idle_is_pool(bm, range(R))
    assert len(used) == k + int(sum(-(-u // B)))


def test_without_commits_the_cache_changes_nothing():
    rng = np.random.default_rng(11)
    N, B = 40, 4
    a, b = _bm(N, B), _bm(N, B)
    for i in range(12):
        toks = list(rng.integers(0, 9, int(rng.integers(1, 15))))
        assert a.add_seq_cached(i, toks) == 0
        b.add_seq(i)
        try:
            ra = a.append(i, len(toks))
        except oracle.OracleError:
            with pytest.raises(oracle.OracleError):
                b.append(i, len(toks))
            continue
        rb = b.append(i, len(toks))
        assert np.array_equal(ra[0], rb[0])
        if rng.random() < 0.4:
            a.free_seq(i)
            b.free_seq(i)
        assert np.array_equal(a.free_list(), b.free_list())


@pytest.mark.parametrize("seed", range(6))
def test_every_slot_holds_kv_of_the_sequences_own_prefix(seed):
    """Random admissions (prompts that share prefixes of a few base strings),
    decode appends, forks (with CoW copies), commits and retirements in a
    small pool, so blocks are shared, released, evicted and reused. K/V at
    position t of a sequence is modelled as the tuple of its tokens 0..t;
    after every operation each slot every live sequence names must hold
    exactly that tuple for that sequence."""
    rng = np.random.default_rng(seed)
    B = int(rng.choice([2, 4, 8]))
    N = int(rng.integers(12, 40))
    bm = oracle.BlockManager(N, B, rng.permutation(N).astype(np.int32))
    bases = [list(rng.integers(0, 5, 6 * B)) for _ in range(3)]
    content = {}
    toks = {}
    nid = 0

    def write(seq, slots, first):
        for i, sl in enumerate(slots):
            content[int(sl)] = tuple(toks[seq][: first + i + 1])

    def cow(pair):
        if pair is not None:
            src, dst = pair
            for o in range(B):
                if src * B + o in content:
                    content[dst * B + o] = content[src * B + o]
                else:
                    content.pop(dst * B + o, None)

    for _ in range(300):
        r = rng.random()
        live = list(toks)
        try:
            if r < 0.3 or not live:
                base = bases[int(rng.integers(len(bases)))]
                cut = int(rng.integers(0, len(base)))
                prompt = base[:cut] + list(rng.integers(0, 5, int(rng.integers(0, 2 * B))))
                if not prompt:
                    continue
                seq, nid = nid, nid + 1
                toks[seq] = prompt
                n_cached = bm.add_seq_cached(seq, prompt)
                try:
                    if len(prompt) > n_cached:
                        slots, pair = bm.append(seq, len(prompt) - n_cached)
                        cow(pair)
                        write(seq, slots, n_cached)
                except oracle.OracleError:
                    bm.free_seq(seq)
                    del toks[seq]
                    continue
                if rng.random() < 0.8:
                    bm.commit(seq, prompt)
            else:
                seq = int(rng.choice(live))
                if r < 0.6:
                    n = int(rng.integers(1, B + 2))
                    old = len(toks[seq])
                    new = list(rng.integers(0, 5, n))
                    slots, pair = bm.append(seq, n)
                    toks[seq] = toks[seq] + new
                    cow(pair)
                    write(seq, slots, old)
                    if rng.random() < 0.5:
                        bm.commit(seq, toks[seq])
                elif r < 0.7:
                    child, nid = nid, nid + 1
                    bm.fork(seq, child)
                    toks[child] = list(toks[seq])
                else:
                    bm.free_seq(seq)
                    del toks[seq]
        except oracle.OracleError:
            pass
        named = _named_plus_idle_is_pool(bm, toks)
        refs = {}
        for s in toks:
            assert bm.seq_len(s) == len(toks[s])
            t = bm.table(s)
            for b in t:
                refs[int(b)] = refs.get(int(b), 0) + 1
            for pos in range(len(toks[s])):
                slot = int(t[pos // B]) * B + pos % B
                assert content.get(slot) == tuple(toks[s][: pos + 1]), (s, pos)
        for b in named:
            assert bm.refcount(b) == refs[b]
