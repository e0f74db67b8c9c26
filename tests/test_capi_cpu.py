"""libpagedkv on the CPU: it builds, loads, exports every declared symbol, and
its host block manager agrees bit for bit with the oracle's.

No GPU entry point runs here except the host-side argument checks that
return before any CUDA call.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from workloads import WORKLOAD_NAMES, make_workload, prefill_plan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    pk.build()
    return pk.lib()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pk_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert _declared_symbols() == sorted(pk.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in _declared_symbols():
        assert hasattr(L, name), name
    assert pk.pk_status_string(0) == "ok"
    assert pk.pk_status_string(3) == "out of blocks"


def _replay_both(wl):
    """Runs the workload's prefill plan and one step on both block managers."""
    ours = pk.BlockManager(wl.num_blocks, wl.block_size, wl.alloc_order())
    ref = oracle.BlockManager(wl.num_blocks, wl.block_size, wl.alloc_order())
    for op in prefill_plan(wl):
        if op[0] == "add":
            ours.add_seq(op[1])
            ref.add_seq(op[1])
        elif op[0] == "fork":
            ours.fork(op[1], op[2])
            ref.fork(op[1], op[2])
        elif op[0] == "free":
            ours.free_seq(op[1])
            ref.free_seq(op[1])
        elif op[0] == "admit":
            toks = wl.chat_tokens(op[1])
            n = ours.add_seq_cached(op[1], toks)
            assert n == ref.add_seq_cached(op[1], toks)
            if len(toks) > n:
                s1, _ = ours.append(op[1], len(toks) - n)
                s2, _ = ref.append(op[1], len(toks) - n)
                assert np.array_equal(s1, s2)
            ours.commit(op[1], toks)
            ref.commit(op[1], toks)
        else:
            s1, c1 = ours.append(op[1], op[2])
            s2, c2 = ref.append(op[1], op[2])
            assert np.array_equal(s1, s2) and c1 == c2
    slots, pairs = ours.append_batch(range(wl.num_seqs))
    ref_slots, ref_pairs = [], []
    for s in range(wl.num_seqs):
        sl, cow = ref.append(s, 1)
        ref_slots.append(sl[0])
        if cow is not None:
            ref_pairs.append(cow)
    assert slots.tolist() == ref_slots
    assert [tuple(p) for p in pairs.tolist()] == ref_pairs
    return ours, ref


@pytest.mark.parametrize("name,B", [(n, None) for n in WORKLOAD_NAMES if n != "prefix"] +
                         [("prefix", 8), ("prefix", 16), ("prefix", 32)])
def test_block_manager_matches_oracle_on_workloads(L, name, B):
    wl = make_workload(name, block_size=B)
    ours, ref = _replay_both(wl)
    ctx = wl.ctx_lens
    maxb = -(-int(ctx.max()) // wl.block_size)
    tables, lens = ours.export_tables(range(wl.num_seqs), maxb)
    assert np.array_equal(tables, ref.export_tables(range(wl.num_seqs), maxb))
    assert np.array_equal(lens, ctx.astype(np.int32))
    assert ours.num_free() == ref.num_free()
    for b in range(0, wl.num_blocks, max(1, wl.num_blocks // 500)):
        assert ours.refcount(b) == ref.refcount(b)
    ours.check_invariants()
    assert ours.cache_stats() == ref.cache_stats()
    st = ours.stats()
    assert st["live_tokens"] == int(ctx.sum())
    assert st["cow_copies"] == ref.cow_copies()
    assert st["tail_waste"] == int(sum(-(-int(c) // wl.block_size) * wl.block_size - int(c) for c in ctx))


def test_block_manager_random_ops_match_oracle(L):
    rng = np.random.default_rng(99)
    for trial in range(20):
        B = int(rng.choice([1, 4, 8, 16]))
        N = int(rng.integers(8, 80))
        order = rng.permutation(N).astype(np.int32)
        ours, ref = pk.BlockManager(N, B, order), oracle.BlockManager(N, B, order)
        live, nid = [], 0
        for _ in range(150):
            r = rng.random()
            if r < 0.2 or not live:
                ours.add_seq(nid)
                ref.add_seq(nid)
                live.append(nid)
                nid += 1
            elif r < 0.55:
                s, n = int(rng.choice(live)), int(rng.integers(0, 2 * B + 3))
                try:
                    a = ours.append(s, n)
                except pk.PagedKVError as e:
                    assert e.status == 3
                    with pytest.raises(oracle.OracleError):
                        ref.append(s, n)
                else:
                    b = ref.append(s, n)
                    assert np.array_equal(a[0], b[0]) and a[1] == b[1]
            elif r < 0.7:
                seqs = [int(x) for x in rng.choice(live, size=int(rng.integers(1, len(live) + 1)))]
                free0 = ours.num_free()
                try:
                    slots, pairs = ours.append_batch(seqs)
                except pk.PagedKVError as e:
                    assert e.status == 3 and ours.num_free() == free0  # batch undone
                    continue
                for i, s in enumerate(seqs):
                    sl, cow = ref.append(s, 1)
                    assert slots[i] == sl[0]
                assert len(pairs) == sum(1 for _ in pairs)
            elif r < 0.85:
                p = int(rng.choice(live))
                ours.fork(p, nid)
                ref.fork(p, nid)
                live.append(nid)
                nid += 1
            else:
                s = int(rng.choice(live))
                ours.free_seq(s)
                ref.free_seq(s)
                live.remove(s)
            ours.check_invariants()
            assert ours.num_free() == ref.num_free()
            for s in live:
                assert np.array_equal(ours.table(s), ref.table(s))
                assert ours.seq_len(s) == ref.seq_len(s)


def test_batch_append_is_all_or_nothing(L):
    bm = pk.BlockManager(3, 2, None)
    for s in range(3):
        bm.add_seq(s)
        bm.append(s, 2)            # every sequence holds one full block
    free0, t0 = bm.num_free(), [bm.table(s).tolist() for s in range(3)]
    with pytest.raises(pk.PagedKVError) as ei:
        bm.append_batch([0, 1, 2])  # would need 3 fresh blocks, 0 free
    assert ei.value.status == 3
    assert bm.num_free() == free0 and [bm.table(s).tolist() for s in range(3)] == t0
    assert [bm.seq_len(s) for s in range(3)] == [2, 2, 2]
    bm.check_invariants()


def test_batch_undo_restores_cow_state(L):
    bm = pk.BlockManager(4, 4, None)
    bm.add_seq(0)
    bm.append(0, 6)                # blocks 0, 1 (tail half full)
    bm.fork(0, 1)
    bm.add_seq(2)
    # seq 0 copies its shared tail (takes block 2), seq 2 takes block 3, seq 1
    # then writes its tail in place... and a second token for seq 2 needs none.
    # Ask for one more fresh block than exists: seq 0 CoW, seq 2 new, seq 1
    # in place, then seq 3 unknown -> error, all undone.
    before = (bm.num_free(), bm.table(0).tolist(), bm.table(1).tolist(), bm.refcount(1))
    with pytest.raises(pk.PagedKVError) as ei:
        bm.append_batch([0, 2, 1, 77])
    assert ei.value.status == 4
    assert (bm.num_free(), bm.table(0).tolist(), bm.table(1).tolist(), bm.refcount(1)) == before
    slots, pairs = bm.append_batch([0, 2, 1])
    assert pairs.tolist() == [[1, 2]] and bm.refcount(1) == 1
    bm.check_invariants()


def test_error_statuses(L):
    with pytest.raises(pk.PagedKVError) as ei:
        pk.BlockManager(4, 4, np.array([0, 1, 1, 2], np.int32))
    assert ei.value.status == 1
    bm = pk.BlockManager(4, 4, None)
    with pytest.raises(pk.PagedKVError) as ei:
        bm.append(5, 1)
    assert ei.value.status == 4
    bm.add_seq(5)
    with pytest.raises(pk.PagedKVError) as ei:
        bm.add_seq(5)
    assert ei.value.status == 5
    with pytest.raises(pk.PagedKVError):
        bm.fork(9, 10)
    with pytest.raises(pk.PagedKVError) as ei:
        bm.export_tables([5], 0) if bm.append(5, 1) else None
    assert ei.value.status == 1


def _desc(N=64, B=16, Hk=8, d=128, dt=pk.PK_BF16):
    return pk.CacheDesc(N, B, Hk, d, dt)


def test_partition_resolution_and_workspace_size(L):
    d = _desc()
    assert pk.pk_paged_attention_resolve_partition(8, 64, 32768, 512, d) == 512
    assert pk.pk_paged_attention_resolve_partition(8, 64, 32768, 0, d) == 0
    assert pk.pk_paged_attention_resolve_partition(8, 64, 32768, 40, d) == -1      # not a multiple of B
    # Automatic (no GPU visible: 152 SMs x 3 resident CTAs = 456 slots): 64
    # units of 32K tokens fill the slots once with 7 partitions of 4736 tokens.
    assert pk.pk_paged_attention_resolve_partition(8, 64, 32768, -1, d) == 4736
    assert pk.pk_paged_attention_resolve_partition(2, 16, 32768, -1, d) == 1216    # 16 units: 28 partitions
    assert pk.pk_paged_attention_resolve_partition(1, 8, 4096, -1, d) == 512       # at least 512 tokens
    assert pk.pk_paged_attention_resolve_partition(40, 64, 8192, -1, d) == 0       # 320 units: one per slot
    assert pk.pk_paged_attention_resolve_partition(64, 64, 2048, -1, d) == 0       # 512 units fill the slots
    assert pk.pk_paged_attention_resolve_partition(256, 64, 2048, -1, d) == 0      # 2048 units: whole
    assert pk.pk_paged_attention_resolve_partition(8, 64, 300, -1, d) == 0         # short: no split
    assert pk.pk_paged_attention_resolve_partition(8, 60, 300, -1, d) == -1        # Hq % Hk != 0
    assert pk.pk_paged_attention_resolve_partition(8, 128, 300, -1, d) == -1       # group of 16
    ws = pk.pk_paged_attention_workspace_size(8, 64, 32768, 512, d)
    assert ws == 8 * 64 * 64 * (128 + 2) * 4                   # [S, Hq, P, d+2] fp32 partials
    assert pk.pk_paged_attention_workspace_size(8, 64, 512, 512, d) == 0           # one partition
    assert pk.pk_paged_attention_workspace_size(8, 64, 32768, 0, d) == 0


def test_host_checks_reject_before_launch(L):
    null = ctypes.c_void_p(0)
    bad = _desc(dt=7)
    assert L.pk_reshape_and_cache(null, null, null, 1, null, null, ctypes.byref(bad), null) == 2
    assert L.pk_reshape_and_cache(null, null, null, 0, null, null, ctypes.byref(_desc()), null) == 0
    assert L.pk_reshape_and_cache(null, null, null, 1, null, null, ctypes.byref(_desc()), null) == 1
    assert L.pk_copy_blocks(null, null, null, 0, ctypes.byref(_desc()), null) == 0
    assert L.pk_copy_blocks(null, null, null, -1, ctypes.byref(_desc()), null) == 1
    d = _desc()
    args = [null] * 6 + [ctypes.c_float(0.1), d.block_size, 4, 8, 4, 64, -1, null, 0, ctypes.byref(d), null]
    assert L.pk_paged_attention_decode(*args) == 1          # null pointers
    a2 = list(args)
    a2[9] = 12                                              # 12 query heads over 8 KV heads
    assert L.pk_paged_attention_decode(*a2) == 1
    a3 = list(args)
    a3[8] = 0                                               # empty batch is a no-op
    assert L.pk_paged_attention_decode(*a3) == 0
    a5 = list(a3)
    a5[7] = d.block_size * 2                                # block_size disagrees with the pool's
    assert L.pk_paged_attention_decode(*a5) == 1
    odd = _desc(d=96)
    a4 = list(args)
    a4[15] = ctypes.byref(odd)
    assert L.pk_paged_attention_decode(*a4) == 2            # head_dim 96 not compiled


def test_longest_first_order(L):
    rng = np.random.default_rng(5)
    for n in (0, 1, 7, 300):
        lens = rng.integers(1, 50, size=n).astype(np.int32)   # many ties
        got = pk.pk_longest_first_order(lens)
        assert got.tolist() == np.lexsort((np.arange(n), -lens)).tolist()


def _brute_groups(ref_bm, n, B, max_group, min_blocks):
    """Shared-prefix groups recomputed from the oracle's tables."""
    tables = [ref_bm.table(s).tolist() for s in range(n)]
    lens = [ref_bm.seq_len(s) for s in range(n)]
    buckets, order = {}, []
    for s in range(n):
        if not tables[s]:
            continue
        b0 = tables[s][0]
        if b0 not in buckets:
            buckets[b0] = []
            order.append(b0)
        buckets[b0].append(s)
    groups, seq_prefix = [], [0] * n
    for b0 in order:
        mem = buckets[b0]
        for c in range(0, len(mem), max_group):
            chunk = mem[c:c + max_group]
            if len(chunk) < 2:
                continue
            common = min(len(tables[s]) for s in chunk)
            for j in range(common):
                if any(tables[s][j] != tables[chunk[0]][j] for s in chunk):
                    common = j
                    break
            blocks = min(common, min(lens[s] for s in chunk) // B)
            if blocks < min_blocks:
                continue
            groups.append((chunk, blocks * B))
            for s in chunk:
                seq_prefix[s] = blocks * B
    return groups, seq_prefix


@pytest.mark.parametrize("B,max_group,min_blocks", [(16, 4, 1), (32, 4, 1), (8, 3, 1), (16, 2, 1), (16, 4, 200)])
def test_prefix_groups_match_brute_force(L, B, max_group, min_blocks):
    wl = make_workload("prefix", block_size=B, num_seqs=24)
    ours, ref = _replay_both(wl)
    g = ours.prefix_groups(range(wl.num_seqs), max_group, min_blocks)
    want, want_seq = _brute_groups(ref, wl.num_seqs, B, max_group, min_blocks)
    got = [(g["members"][g["offsets"][i]:g["offsets"][i + 1]].tolist(), int(g["prefix_len"][i]))
           for i in range(g["num_groups"])]
    assert got == want
    assert g["seq_prefix_len"].tolist() == want_seq
    if min_blocks == 1:
        assert g["num_groups"] > 0 and all(p >= (2000 // B - 1) * B for _, p in got)


def test_swap_matches_oracle_on_random_operations(L):
    rng = np.random.default_rng(314)
    for trial in range(12):
        B = int(rng.choice([1, 4, 16]))
        N, H = int(rng.integers(10, 60)), int(rng.integers(4, 50))
        order, horder = rng.permutation(N).astype(np.int32), rng.permutation(H).astype(np.int32)
        ours, ref = pk.BlockManager(N, B, order), oracle.BlockManager(N, B, order)
        ours.set_swap_space(H, horder)
        ref.set_swap_space(H, horder)
        live, nid = [], 0
        for _ in range(150):
            r = rng.random()
            s = int(rng.choice(live)) if live else None
            if r < 0.15 or not live:
                ours.add_seq(nid)
                ref.add_seq(nid)
                live.append(nid)
                nid += 1
                continue
            if r < 0.45:
                n = int(rng.integers(0, 2 * B + 2))
                args = ("append", s, n)
            elif r < 0.55:
                args = ("fork", s, nid)
            elif r < 0.7:
                args = ("swap_out", s)
            elif r < 0.85:
                args = ("swap_in", s)
            else:
                args = ("free_seq", s)
            res = []
            for bm, err in ((ours, pk.PagedKVError), (ref, oracle.OracleError)):
                try:
                    res.append(("ok", getattr(bm, args[0])(*args[1:])))
                except err:
                    res.append(("err", None))
            assert res[0][0] == res[1][0], (args, res)
            if res[0][0] == "ok":
                a, b = res[0][1], res[1][1]
                if args[0] == "append":
                    assert np.array_equal(a[0], b[0]) and a[1] == b[1]
                elif args[0] in ("swap_out", "swap_in"):
                    assert np.array_equal(a, b)
                elif args[0] == "fork":
                    live.append(nid)
                    nid += 1
                elif args[0] == "free_seq":
                    live.remove(s)
            ours.check_invariants()
            assert ours.num_free() == ref.num_free() and ours.host_free() == ref.host_free()
            for q in live:
                assert ours.is_swapped(q) == ref.is_swapped(q)
                assert np.array_equal(ours.table(q), ref.table(q))


@pytest.mark.parametrize("seed", range(8))
def test_prefix_cache_matches_oracle_on_random_traces(L, seed):
    assert _prefix_cache_trace(seed) > 0     # some batches ran out of blocks


def _prefix_cache_trace(seed):
    """Admissions through the cache, commits, decode appends (single and
    batched), forks, swaps and retirements in a small pool (so cached blocks
    are released, revived and evicted): tables, cached counts, free counts
    and cache statistics equal the oracle's after every operation."""
    rng = np.random.default_rng(900 + seed)
    B = int(rng.choice([2, 4, 16]))
    N = int(rng.integers(16, 64))
    order = rng.permutation(N).astype(np.int32)
    ours, ref = pk.BlockManager(N, B, order), oracle.BlockManager(N, B, order)
    H = 32
    ours.set_swap_space(H)
    ref.set_swap_space(H)
    bases = [list(rng.integers(0, 4, 5 * B)) for _ in range(3)]
    toks, nid = {}, 0

    log, failures = [], [0]

    def both(name, *args):
        out = []
        for bm, err in ((ours, pk.PagedKVError), (ref, oracle.OracleError)):
            try:
                out.append(("ok", getattr(bm, name)(*args)))
            except err:
                out.append(("err", None))
        assert out[0][0] == out[1][0], (name, args)
        if out[1][0] == "ok":
            log.append((name, args))
        return out

    for _ in range(250):
        r = rng.random()
        live = [s for s in toks if not ref.is_swapped(s)]
        if r < 0.3 or not live:
            base = bases[int(rng.integers(3))]
            prompt = base[: int(rng.integers(0, len(base)))] + list(rng.integers(0, 4, int(rng.integers(1, 2 * B))))
            assert ours.cache_match(prompt) == ref.add_seq_cached(nid, prompt)
            log.append(("add_seq_cached", (nid, prompt)))
            ours.add_seq_cached(nid, prompt)
            toks[nid] = prompt
            got = both("append", nid, len(prompt) - ref.seq_len(nid))
            if got[0][0] == "ok":
                assert np.array_equal(got[0][1][0], got[1][1][0]) and got[0][1][1] == got[1][1][1]
                if rng.random() < 0.8:
                    both("commit", nid, prompt)
            else:
                toks[nid] = toks[nid][: ref.seq_len(nid)]
            nid += 1
        elif r < 0.5:
            batch = list(rng.choice(live, size=int(rng.integers(1, len(live) + 1))))
            before_free = ref.num_free()
            try:
                slots, pairs = ours.append_batch(batch)
            except pk.PagedKVError:
                # Nothing changed, and one token at a time the oracle runs out too
                # (on a replica rebuilt from the operation log).
                assert ours.num_free() == before_free
                replica = oracle.BlockManager(N, B, order)
                replica.set_swap_space(H)
                for name, args in log:
                    getattr(replica, name)(*args)
                with pytest.raises(oracle.OracleError):
                    for s in batch:
                        replica.append(s, 1)
                failures[0] += 1
                continue
            want, wpairs = [], []
            for s in batch:
                sl, cow = ref.append(s, 1)
                log.append(("append", (s, 1)))
                want.append(sl[0])
                if cow is not None:
                    wpairs.append(cow)
                toks[s] = toks[s] + [int(rng.integers(0, 4))]
            assert np.array_equal(slots, want)
            assert np.array_equal(pairs.reshape(-1, 2), np.array(wpairs, np.int64).reshape(-1, 2))
        elif r < 0.6:
            s = int(rng.choice(live))
            got = both("fork", s, nid)
            if got[0][0] == "ok":
                toks[nid] = list(toks[s])
                nid += 1
        elif r < 0.7:
            s = int(rng.choice(live))
            both("commit", s, toks[s])
        elif r < 0.8:
            s = int(rng.choice(list(toks)))
            name = "swap_in" if ref.is_swapped(s) else "swap_out"
            got = both(name, s)
            if got[0][0] == "ok":
                assert np.array_equal(got[0][1], got[1][1])
        else:
            s = int(rng.choice(list(toks)))
            both("free_seq", s)
            del toks[s]
        ours.check_invariants()
        assert ours.num_free() == ref.num_free()
        assert ours.cache_stats() == ref.cache_stats()
        for s in toks:
            assert ours.is_swapped(s) == ref.is_swapped(s)
            assert np.array_equal(ours.table(s), ref.table(s))
        for b in range(N):
            assert ours.is_cached(b) == ref.is_cached(b)
    assert ref.cache_stats()["evictions"] > 0 and ref.cache_stats()["hits"] > 0
    return failures[0]


def _sim_pair(trace, capacity, policy, B, rule):
    from oracle import allocator_sim
    ours = pk.pk_sim_run(trace, capacity, policy, B, rule)
    ref = allocator_sim.simulate(trace, capacity, policy, B, rule)
    s = dict(ours["summary"])
    assert s.pop("capacity") == (capacity if policy != "paged" else (capacity // B) * B)
    assert s.pop("num_steps") == len(ref["samples"])
    assert s == ref["summary"], (policy, B, rule)
    got = [dict(x, free=x.pop("free_slots")) for x in ours["samples"]]
    assert got == ref["samples"], (policy, B, rule)
    return ours


POLICY_GRID = [("max_reservation", 0), ("exact_contiguous", 0), ("paged", 1), ("paged", 4), ("paged", 8),
               ("paged", 16)]


@pytest.mark.parametrize("rule", ["drop", "stall"])
@pytest.mark.parametrize("seed", range(6))
def test_allocator_sim_matches_oracle_on_random_traces(L, seed, rule):
    rng = np.random.default_rng(4000 + seed)
    C = int(rng.choice([48, 80, 100, 160]))
    trace = []
    for _ in range(int(rng.integers(4, 30))):
        a = int(rng.integers(0, 40))
        m = int(rng.integers(0, C // 3))
        g = int(rng.integers(0, m + 1))
        trace.append(dict(arrival=a, prompt=int(rng.integers(1, C // 4)), max_new=m, gen=g,
                          completion=a + g + int(rng.integers(1, 4))))
    for policy, B in POLICY_GRID:
        _sim_pair(trace, C, policy, B, rule)


@pytest.mark.parametrize("name,n", [("tight", None), ("serving", 120)])
@pytest.mark.parametrize("rule", ["drop", "stall"])
def test_allocator_sim_matches_oracle_on_workload_traces(L, name, n, rule):
    from workloads import allocator_trace
    C, trace = allocator_trace(name, n)
    for policy, B in POLICY_GRID:
        _sim_pair(trace, C, policy, B, rule)


def test_allocator_sim_rejects_malformed_input(L):
    good = [dict(arrival=0, prompt=4, max_new=4, gen=2, completion=3)]
    for bad in ({"prompt": 0}, {"gen": 5}, {"completion": 0}, {"arrival": -1}):
        with pytest.raises(pk.PagedKVError):
            pk.pk_sim_run([dict(good[0], **bad)], 16, "exact_contiguous")
    with pytest.raises(pk.PagedKVError):
        pk.pk_sim_run(good, 3, "paged", 4)
    assert pk.pk_sim_run([], 16, "paged", 4)["summary"]["num_steps"] == 1


@pytest.mark.parametrize("seed", range(5))
def test_work_items_cover_every_partition_once_longest_first(L, seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 5000, int(rng.integers(1, 60))).astype(np.int32)
    for part in (0, 512, 1024, 1728):
        got = pk.pk_attention_work_items(lens, part)
        want = []
        for s, c in enumerate(lens):
            n = -(-int(c) // part) if part else 1
            for j in range(n):
                length = min(part, int(c) - j * part) if part else int(c)
                want.append((-length, -int(c), s, -j))
        want.sort()
        assert [tuple(x) for x in got.tolist()] == [(s, -nj) for _, _, s, nj in want]


def test_attention_plan_choices(L):
    """The host plan on the workloads: long uniform contexts get one wave
    (7 x 4736 tokens), the one 32K request among short ones is cut into
    2048-token items, everything else stays whole (152 SMs x 3 CTAs when no
    GPU is visible); explicit sizes pass through; the items are the work-list
    helper's."""
    want = {"mha7b": 0, "gqa8b": 0, "long": 4736, "chat": 0, "mixed": 2048, "prefix": 0}
    for name, part in want.items():
        wl = make_workload(name)
        d = pk.CacheDesc(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, 1)
        got, items = pk.pk_attention_plan(wl.ctx_lens, wl.num_q_heads, d, -1)
        assert got == part, name
        assert np.array_equal(items, pk.pk_attention_work_items(wl.ctx_lens, got))
    wl = make_workload("mixed")
    d = pk.CacheDesc(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, 1)
    assert pk.pk_attention_plan(wl.ctx_lens, 32, d, 1024)[0] == 1024
    assert pk.pk_attention_plan(wl.ctx_lens, 32, d, 0)[0] == 0
    assert pk.pk_attention_plan(wl.ctx_lens, 32, d, 40000)[0] == 0          # longer than every context
    with pytest.raises(pk.PagedKVError):
        pk.pk_attention_plan(wl.ctx_lens, 32, d, 1000)                    # not a multiple of B


def test_decode_step_prepare_and_launch_pair_up(L):
    """The two halves of pk_decode_step pair up: a launch with nothing
    prepared and a second prepare before the launch are refused before any
    device work; a full prepare appends one token to every sequence and packs
    its slots and lengths into the first staging half."""
    S, maxb, B, nblk = 3, 8, 16, 64
    bm = pk.BlockManager(nblk, B)
    for s in range(S):
        bm.add_seq(s)
        bm.append(s, 15 + s)                      # lengths 15, 16, 17
    before = [bm.table(s).copy() for s in range(S)]
    desc = pk.CacheDesc(nblk, B, 2, 64, pk.PK_BF16)
    mb = int(L.pk_decode_step_meta_bytes(S, maxb))
    meta = np.zeros(mb, dtype=np.uint8)
    buf = pk.StepBuffers()
    buf.meta_host = meta.ctypes.data
    buf.meta_bytes = mb
    ids = np.arange(S, dtype=np.int64)
    args = (bm._h, ids.ctypes.data, S, 4, maxb, 0, ctypes.byref(desc), ctypes.byref(buf))
    assert L.pk_decode_step_launch(S, 4, 0.125, maxb, None, None, ctypes.byref(desc), ctypes.byref(buf),
                                   None) == pk.PK_ERR_INVALID_ARG
    assert L.pk_decode_step_prepare(*args) == pk.PK_OK
    assert [bm.seq_len(s) for s in range(S)] == [16, 17, 18]
    assert buf.tables_resident == 0 and buf.state
    half = mb // 2
    slots = meta[:8 * S].view(np.int64)
    tables = [bm.table(s) for s in range(S)]
    expect = [int(tables[s][t // B]) * B + t % B for s, t in zip(range(S), (15, 16, 17))]
    assert list(slots) == expect
    assert tables[0].tolist() == before[0].tolist()          # 15 -> 16 stays in block 0
    assert len(tables[1]) == len(before[1]) + 1               # 16 -> 17 takes a new block
    assert not meta[half:].any()                              # the second half is untouched
    assert L.pk_decode_step_prepare(*args) == pk.PK_ERR_INVALID_ARG
    assert [bm.seq_len(s) for s in range(S)] == [16, 17, 18]
    bm.check_invariants()
    L.pk_decode_step_release(ctypes.byref(buf))
    assert not buf.state


def test_read_stream_rejects_bad_arguments_before_any_launch(L):
    buf = np.zeros(64, dtype=np.uint8)
    sink = np.zeros(1, dtype=np.uint32)
    assert L.pk_read_stream(None, 64, sink.ctypes.data, None) == pk.PK_ERR_INVALID_ARG
    assert L.pk_read_stream(buf.ctypes.data, 8, sink.ctypes.data, None) == pk.PK_ERR_INVALID_ARG
    assert L.pk_read_stream(buf.ctypes.data, 64, None, None) == pk.PK_ERR_INVALID_ARG
    assert L.pk_read_stream(buf.ctypes.data + 4, 48, sink.ctypes.data, None) == pk.PK_ERR_INVALID_ARG


def test_advance_rejects_bad_arguments_before_any_launch(L):
    # Host buffers stand in for device pointers: every case below returns from
    # the argument checks, before anything is read or launched.
    S, Hq, maxb = 4, 32, 8
    buf = np.zeros(1 << 16, dtype=np.uint8)
    base = (buf.ctypes.data + 255) // 256 * 256
    ptr = [base + 4096 * i for i in range(12)]
    out, q, kn, vn, slots, kc, vc, tables, lens, lens_out, items, ws = ptr
    d = _desc()

    def call(**kw):
        a = dict(out=out, q=q, kn=kn, vn=vn, slots=slots, kc=kc, vc=vc, tables=tables, lens=lens,
                 lens_out=lens_out, scale=0.088, S=S, Hq=Hq, maxb=maxb, max_ctx=100, part=0,
                 items=items, n_items=S, ws=ws, ws_bytes=4096)
        a.update(kw)
        return L.pk_paged_attention_decode_advance(
            a["out"], a["q"], a["kn"], a["vn"], a["slots"], a["kc"], a["vc"], a["tables"], a["lens"],
            a["lens_out"], a["scale"], a["S"], a["Hq"], a["maxb"], a["max_ctx"], a["part"], a["items"],
            a["n_items"], a["ws"], a["ws_bytes"], ctypes.byref(d), None)

    assert call(S=0) == pk.PK_OK                                  # empty batch: nothing to do
    assert call(items=None) == pk.PK_ERR_INVALID_ARG              # the work list is required
    assert call(kn=None) == pk.PK_ERR_INVALID_ARG                 # so are the new K/V and slots
    assert call(vn=None) == pk.PK_ERR_INVALID_ARG
    assert call(slots=None) == pk.PK_ERR_INVALID_ARG
    assert call(lens_out=None) == pk.PK_ERR_INVALID_ARG           # and a separate output length buffer
    assert call(lens_out=lens) == pk.PK_ERR_INVALID_ARG
    assert call(tables=None) == pk.PK_ERR_INVALID_ARG
    assert call(q=q + 4) == pk.PK_ERR_INVALID_ARG                 # 16-byte alignment
    assert call(kn=kn + 8) == pk.PK_ERR_INVALID_ARG
    assert call(scale=float("nan")) == pk.PK_ERR_INVALID_ARG
    assert call(Hq=12) == pk.PK_ERR_INVALID_ARG                   # Hq not a multiple of Hk
    assert call(part=40) == pk.PK_ERR_INVALID_ARG                 # partition not a multiple of B
    assert call(n_items=0) == pk.PK_ERR_UNSUPPORTED               # work-list size out of range
    assert call(n_items=70000) == pk.PK_ERR_UNSUPPORTED


def test_other_entry_points_reject_bad_arguments_before_any_launch(L):
    # As above: host buffers stand in for device memory and no case gets past
    # the argument checks (none reaches a CUDA call).
    buf = np.zeros(1 << 16, dtype=np.uint8)
    base = (buf.ctypes.data + 255) // 256 * 256
    ptr = [base + 2048 * i for i in range(20)]
    out, q, kc, vc, tables, lens, items, ws, kn, vn, slots, goff, gmem, gpre, spre, kh, vh, pairs = ptr[:18]
    d = _desc()                       # 64 blocks of 16 tokens, 8 KV heads, d = 128, bf16
    f = ctypes.c_float(0.088)
    byref = ctypes.byref

    def items_call(**kw):
        a = dict(out=out, q=q, S=4, Hq=32, items=items, n=4, ws=ws)
        a.update(kw)
        return L.pk_paged_attention_decode_items(a["out"], a["q"], kc, vc, tables, lens, f, a["S"], a["Hq"],
                                                  8, 100, 0, a["items"], a["n"], a["ws"], 4096, byref(d),
                                                  pk.IMPLS["auto"], None)

    assert items_call(S=0) == pk.PK_OK
    assert items_call(items=None) == pk.PK_ERR_INVALID_ARG
    assert items_call(out=out + 2) == pk.PK_ERR_INVALID_ARG
    assert items_call(n=0) == pk.PK_ERR_UNSUPPORTED
    assert items_call(Hq=12) == pk.PK_ERR_INVALID_ARG

    def append_call(**kw):
        a = dict(kn=kn, vn=vn, slots=slots, items=items)
        a.update(kw)
        return L.pk_paged_attention_decode_append(out, q, a["kn"], a["vn"], a["slots"], kc, vc, tables, lens, f,
                                                   4, 32, 8, 100, 0, a["items"], 4, ws, 4096, byref(d), None)

    for k in ("kn", "vn", "slots", "items"):
        assert append_call(**{k: None}) == pk.PK_ERR_INVALID_ARG
    assert append_call(vn=vn + 8) == pk.PK_ERR_INVALID_ARG

    def static_call(S=4, Hq=32, max_ctx=100, part=0, B=16):
        return L.pk_paged_attention_decode_static(out, q, kc, vc, tables, lens, f, B, S, Hq, 2048, max_ctx, part,
                                                  byref(d), None)

    assert static_call(Hq=12) == pk.PK_ERR_INVALID_ARG
    assert static_call(B=32) == pk.PK_ERR_INVALID_ARG         # block_size disagrees with the pool's
    assert static_call(part=40) == pk.PK_ERR_INVALID_ARG
    # 64 x 64 heads x 2048 partitions of fp32 partials: far above the fixed scratch.
    assert static_call(S=64, Hq=64, max_ctx=32768, part=16) == pk.PK_ERR_WORKSPACE

    def cascade_call(**kw):
        a = dict(q=q, S=4, part=0, goff=goff, ngroups=1, gmax=2, maxpre=64, ws=ws, ws_bytes=0)
        a.update(kw)
        return L.pk_cascade_attention_decode(out, a["q"], kc, vc, tables, lens, f, a["S"], 32, 8, 100, a["part"],
                                             a["goff"], gmem, gpre, spre, a["ngroups"], a["gmax"], a["maxpre"],
                                             None, a["ws"], a["ws_bytes"], byref(d), None)

    assert cascade_call(S=0, ngroups=0) == pk.PK_OK            # no groups: plain attention, empty batch
    assert cascade_call(ngroups=-1) == pk.PK_ERR_INVALID_ARG
    assert cascade_call(gmax=5) == pk.PK_ERR_UNSUPPORTED       # 5 members x G = 4 > 16 query columns
    assert cascade_call(goff=None) == pk.PK_ERR_INVALID_ARG
    assert cascade_call(q=q + 4) == pk.PK_ERR_INVALID_ARG
    assert cascade_call(part=40) == pk.PK_ERR_INVALID_ARG
    assert cascade_call(ws=None) == pk.PK_ERR_WORKSPACE
    assert cascade_call(ws_bytes=16) == pk.PK_ERR_WORKSPACE

    def swap_call(**kw):
        a = dict(kc=kc, kh=kh, nhost=16, n=2, direction=pk.PK_SWAP_OUT, desc=d)
        a.update(kw)
        return L.pk_swap_blocks(a["kc"], vc, a["kh"], vh, a["nhost"], pairs, a["n"], a["direction"],
                                byref(a["desc"]), None)

    assert swap_call(n=0) == pk.PK_OK
    assert swap_call(n=-1) == pk.PK_ERR_INVALID_ARG
    assert swap_call(nhost=-1) == pk.PK_ERR_INVALID_ARG
    assert swap_call(direction=5) == pk.PK_ERR_INVALID_ARG
    assert swap_call(kh=None) == pk.PK_ERR_INVALID_ARG
    assert swap_call(kc=kc + 4) == pk.PK_ERR_INVALID_ARG
    assert swap_call(desc=_desc(dt=7)) == pk.PK_ERR_UNSUPPORTED
