"""Pins for the oracle's block manager against what the pages fix.

* the simulator snapshot's block tables ("PagedAttention", S06, "Try it");
* the 200-token reply: 13 blocks, 8 wasted of 208 ("paged attention deep");
* the reserved-slots equation B*ceil(L/B) and its tail-waste bound ("The KV
  Cache Is an Allocator Problem");
* reference counts equal the number of tables naming a block after every
  operation ("PagedAttention", "Reference counts must be exact"), and the
  free list never holds a named block ("Paged KV Cache Allocation and the
  Block Table", "Sharing blocks between sequences");
* forks share prefix blocks with refcount > 1 until a writer copies its tail
  block ("paged attention deep", "Copy-on-write for shared prefixes");
* the corrected 80-slot example: contiguous first fit fails, paging succeeds.

The invariants are checked by a brute-force recount from the exported
tables, not by the oracle's own counters.
"""
import json
import os
from collections import Counter

import numpy as np
import pytest

import oracle
from oracle.contiguous import ContiguousPool
from workloads import f32_to_bf16_bits, make_workload, prefill_plan


def _recount(bm, live):
    """Brute-force refcounts from the tables of the live sequences."""
    c = Counter()
    for s in live:
        c.update(int(b) for b in bm.table(s))
    return c


def _check_invariants(bm, live, lens):
    counts = _recount(bm, live)
    free = bm.free_list()
    assert len(set(free.tolist())) == len(free), "a block is on the free list twice"
    for b in range(bm.num_blocks):
        assert bm.refcount(b) == counts.get(b, 0), f"block {b}: refcount {bm.refcount(b)} != {counts.get(b, 0)} tables"
    named = set(counts)
    assert not (named & set(free.tolist())), "a named block is on the free list"
    assert len(named) + len(free) == bm.num_blocks, "a block leaked"
    B = bm.block_size
    for s in live:
        L = lens[s]
        assert bm.seq_len(s) == L
        nblk = len(bm.table(s))
        assert nblk == -(-L // B)
        reserved = B * nblk
        assert 0 <= reserved - L <= B - 1


def test_widget_block_tables(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "widget_block_tables.json")))
    bm = oracle.BlockManager(g["pool_blocks"], g["block_size"], None)
    for i, r in enumerate(g["requests"]):
        bm.add_seq(i)
        bm.append(i, r["tokens"])
    for i, r in enumerate(g["requests"]):
        assert bm.table(i).tolist() == r["table"], r["name"]


def test_two_hundred_token_reply(golden_dir):
    w = json.load(open(os.path.join(golden_dir, "worked_numbers.json")))["reply_200_tokens"]
    bm = oracle.BlockManager(300, w["block_size"], np.random.default_rng(0).permutation(300).astype(np.int32))
    bm.add_seq(0)
    for _ in range(w["tokens"]):
        bm.append(0, 1)
    nblk = len(bm.table(0))
    assert nblk == w["blocks"]
    assert nblk * w["block_size"] == w["reserved_slots"]
    assert nblk * w["block_size"] - w["tokens"] == w["wasted_slots"]
    assert w["wasted_slots"] / w["reserved_slots"] < w["paged_waste_fraction_below"]
    assert w["contiguous_reservation"] - w["tokens"] == w["contiguous_wasted"]
    assert w["contiguous_wasted"] / w["contiguous_reservation"] > w["contiguous_waste_fraction_above"]
    assert w["contiguous_reservation"] // w["block_size"] == w["contiguous_blocks_pinned"]


def test_reservation_waste_and_p1_arithmetic(golden_dir):
    w = json.load(open(os.path.join(golden_dir, "worked_numbers.json")))
    r = w["reservation_40_of_2048"]
    assert round(100 * (r["reserved"] - r["used"]) / r["reserved"]) == r["waste_percent_rounded"]
    a = w["p1_arithmetic"]
    assert a["bytes_per_token"] * a["reservation_tokens"] == a["reservation_bytes"]
    assert a["cache_bytes"] // a["reservation_bytes"] == a["requests_contiguous"]
    bm = oracle.BlockManager(64, a["block_size"], None)
    bm.add_seq(0)
    bm.append(0, a["tokens_per_sequence"])
    per_seq = len(bm.table(0)) * a["block_size"] * a["bytes_per_token"]
    n = a["cache_bytes"] / per_seq
    assert abs(n - a["requests_paged_roughly"]) / a["requests_paged_roughly"] < 0.05


@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16, 32])
def test_tail_waste_bound_every_length(B):
    bm = oracle.BlockManager(200, B, None)
    bm.add_seq(0)
    for L in range(1, 150):
        bm.append(0, 1)
        nblk = len(bm.table(0))
        assert nblk * B == B * -(-L // B)
        assert 0 <= nblk * B - L <= B - 1


def test_slots_are_contiguous_for_identity_order():
    # With ascending hand-out and one sequence, logical and physical agree.
    bm = oracle.BlockManager(10, 4, None)
    bm.add_seq(5)
    slots, _ = bm.append(5, 37)
    assert slots.tolist() == list(range(37))


def test_random_operation_sequences_keep_invariants():
    rng = np.random.default_rng(1234)
    for trial in range(25):
        B = int(rng.choice([1, 2, 4, 8, 16]))
        N = int(rng.integers(8, 64))
        bm = oracle.BlockManager(N, B, rng.permutation(N).astype(np.int32))
        live, lens, next_id = [], {}, 0
        for _ in range(120):
            op = rng.random()
            if op < 0.2 or not live:
                bm.add_seq(next_id)
                live.append(next_id)
                lens[next_id] = 0
                next_id += 1
            elif op < 0.65:
                s = int(rng.choice(live))
                n = int(rng.integers(0, 3 * B + 2))
                before = (bm.num_free(), bm.table(s).tolist())
                try:
                    _, cow = bm.append(s, n)
                    lens[s] += n
                    if cow is not None:
                        src, dst = cow
                        assert bm.refcount(dst) == 1 and src != dst
                except oracle.OracleError as e:
                    assert e.code == oracle.ERR_OUT_OF_BLOCKS
                    assert (bm.num_free(), bm.table(s).tolist()) == before  # all-or-nothing
            elif op < 0.8:
                p = int(rng.choice(live))
                bm.fork(p, next_id)
                live.append(next_id)
                lens[next_id] = lens[p]
                next_id += 1
            else:
                s = int(rng.choice(live))
                bm.free_seq(s)
                live.remove(s)
                del lens[s]
            _check_invariants(bm, live, lens)


def test_fork_shares_prefix_then_copy_on_write():
    B = 16
    bm = oracle.BlockManager(64, B, np.random.default_rng(2).permutation(64).astype(np.int32))
    bm.add_seq(0)
    bm.append(0, 40)             # 2.5 blocks: the tail block is half full
    for c in (1, 2, 3):
        bm.fork(0, c)
    prefix = bm.table(0).tolist()
    assert all(bm.refcount(b) == 4 for b in prefix)
    assert all(bm.table(c).tolist() == prefix for c in (1, 2, 3))
    copies = []
    for s in (0, 1, 2, 3):
        slots, cow = bm.append(s, 1)
        copies.append(cow)
        # The written slot lies in the sequence's (now private) tail block.
        assert slots[0] // B == bm.table(s)[-1] and slots[0] % B == 40 % B
    tail = prefix[-1]
    assert [c is not None for c in copies] == [True, True, True, False]
    assert all(c[0] == tail for c in copies[:3])
    assert len({c[1] for c in copies[:3]}) == 3
    assert bm.table(3)[-1] == tail and bm.refcount(tail) == 1
    assert all(bm.refcount(b) == 4 for b in prefix[:-1])   # full blocks stay shared
    assert bm.cow_copies() == 3
    # Retire a sibling: the shared blocks lose one reference and stay allocated.
    free_before = bm.num_free()
    bm.free_seq(1)
    assert all(bm.refcount(b) == 3 for b in prefix[:-1])
    assert bm.num_free() == free_before + 1       # only its private tail returns


def test_fork_at_block_boundary_needs_no_copy():
    bm = oracle.BlockManager(32, 8, None)
    bm.add_seq(0)
    bm.append(0, 16)
    bm.fork(0, 1)
    _, cow0 = bm.append(0, 1)
    _, cow1 = bm.append(1, 1)
    assert cow0 is None and cow1 is None
    assert bm.table(0)[-1] != bm.table(1)[-1]


def test_exercise_one_four_samples_share_the_prompt(golden_dir):
    e = json.load(open(os.path.join(golden_dir, "worked_numbers.json")))["exercise_1"]
    bm = oracle.BlockManager(400, e["block_size"], None)
    bm.add_seq(0)
    bm.append(0, e["prompt_tokens"])
    for c in range(1, e["samples"]):
        bm.fork(0, c)
    held = set()
    for c in range(e["samples"]):
        held.update(bm.table(c).tolist())
    assert len(held) == e["blocks_shared"]
    assert e["samples"] * len(bm.table(0)) == e["blocks_unshared"]
    s = json.load(open(os.path.join(golden_dir, "worked_numbers.json")))["shared_prompt_four_samples"]
    assert s["prompt_tokens"] * s["samples"] == s["tokens_without_sharing"]
    bm2 = oracle.BlockManager(600, 16, None)
    bm2.add_seq(0)
    bm2.append(0, s["prompt_tokens"])
    for c in range(1, s["samples"]):
        bm2.fork(0, c)
    assert (600 - bm2.num_free()) * 16 == s["tokens_with_sharing_roughly"]


def test_out_of_blocks_is_all_or_nothing():
    bm = oracle.BlockManager(3, 4, None)
    bm.add_seq(0)
    bm.append(0, 9)                    # 3 blocks
    with pytest.raises(oracle.OracleError) as ei:
        bm.append(0, 4)                # needs a 4th block
    assert ei.value.code == oracle.ERR_OUT_OF_BLOCKS
    assert bm.seq_len(0) == 9 and bm.num_free() == 0
    bm.append(0, 3)                    # fills the tail: no new block needed
    assert bm.seq_len(0) == 12


def test_error_codes():
    bm = oracle.BlockManager(4, 4, None)
    with pytest.raises(oracle.OracleError) as ei:
        bm.append(9, 1)
    assert ei.value.code == oracle.ERR_UNKNOWN_SEQ
    bm.add_seq(1)
    with pytest.raises(oracle.OracleError) as ei:
        bm.add_seq(1)
    assert ei.value.code == oracle.ERR_SEQ_EXISTS
    with pytest.raises(oracle.OracleError):
        bm.fork(2, 3)
    with pytest.raises(oracle.OracleError):
        bm.fork(1, 1)


def test_eighty_slot_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "eighty_slot_example.json")))
    pool = ContiguousPool(g["num_slots"])
    for i, n in enumerate(g["reservations"]):
        assert pool.reserve(i, n) is not None
    pool.release(g["release_index"])
    ex = g["expect"]
    assert pool.free_slots() == ex["free_slots"]
    assert pool.largest_hole() == ex["largest_hole"]
    assert (pool.reserve(99, g["request"]) is not None) == ex["contiguous_fits"]

    B = ex["paged_block_size"]
    bm = oracle.BlockManager(g["num_slots"] // B, B, None)
    for i, n in enumerate(g["reservations"]):
        bm.add_seq(i)
        bm.append(i, n)
    bm.free_seq(g["release_index"])
    assert bm.num_free() == ex["paged_free_blocks"]
    bm.add_seq(99)
    bm.append(99, g["request"])
    assert len(bm.table(99)) == ex["paged_blocks_needed"]
    assert ex["paged_fits"]


@pytest.mark.parametrize("B,expect_pairs", [(8, 0), (16, 0), (32, 96)])
def test_prefix_workload_sharing_and_cow(B, expect_pairs):
    wl = make_workload("prefix", block_size=B)
    res = oracle.run_workload(wl, pool=False, attention=False)
    bm = res["bm"]
    nprefix = wl.prefix_len // B
    pairs = list(res["prefill_pairs"]) + [tuple(p) for p in res["cow_pairs"]]
    assert len(pairs) == expect_pairs
    # Full prefix blocks stay shared by all four members of each group.
    for g in range(wl.prefix_groups):
        t0 = bm.table(g * wl.prefix_n)[:nprefix]
        for c in range(1, wl.prefix_n):
            assert np.array_equal(bm.table(g * wl.prefix_n + c)[:nprefix], t0)
        assert all(bm.refcount(int(b)) == wl.prefix_n for b in t0)
    live = list(range(wl.num_seqs))
    _check_invariants(bm, live, {s: int(wl.ctx_lens[s]) for s in live})


def test_prefix_workload_sharing_before_divergence():
    # "Sharing a 2,000-token prompt across four samples turns 8,000 tokens of
    # cache into roughly 2,000": at B=16, 32 groups hold 32 x 125 blocks.
    wl = make_workload("prefix", block_size=16)
    bm = oracle.BlockManager(wl.num_blocks, 16, wl.alloc_order())
    for op in prefill_plan(wl):
        if op[0] == "add":
            bm.add_seq(op[1])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        elif op[3][0] == "prefix":
            bm.append(op[1], op[2])
    assert wl.num_blocks - bm.num_free() == 32 * 125


# ---------------------------------------------------------------------------
# Preemption by swapping ("Paged KV Cache Allocation and the Block Table",
# "What the design costs": the server may swap a sequence's blocks to host
# memory; "PagedAttention", "Exercises" item 3).
# ---------------------------------------------------------------------------
def _check_swap_invariants(bm, live, H):
    device_live = [s for s in live if not bm.is_swapped(s)]
    counts = _recount(bm, device_live)
    for b in range(bm.num_blocks):
        assert bm.refcount(b) == counts.get(b, 0)
    assert len(counts) + bm.num_free() == bm.num_blocks
    host_held = [b for s in live if bm.is_swapped(s) for b in bm.table(s).tolist()]
    assert len(host_held) == len(set(host_held)), "a host block is held twice"
    assert all(0 <= b < H for b in host_held)
    assert len(host_held) + bm.host_free() == H


def _pools(N, B, Hk, d):
    return np.zeros((N, B, Hk, d), np.uint16), np.zeros((N, B, Hk, d), np.uint16)


def test_swap_round_trip_keeps_attention_exact():
    rng = np.random.default_rng(21)
    N, H, B, Hk, d = 40, 24, 4, 2, 8
    bm = oracle.BlockManager(N, B, rng.permutation(N).astype(np.int32))
    bm.set_swap_space(H, rng.permutation(H).astype(np.int32))
    kc, vc = _pools(N, B, Hk, d)
    hk, hv = _pools(H, B, Hk, d)
    lens = [7, 13, 30]
    for s, n in enumerate(lens):
        bm.add_seq(s)
        slots, _ = bm.append(s, n)
        k = f32_to_bf16_bits(rng.standard_normal((n, Hk, d)).astype(np.float32))
        v = f32_to_bf16_bits(rng.standard_normal((n, Hk, d)).astype(np.float32))
        oracle.reshape_and_cache(kc, vc, k, v, slots, N, B)
    q = f32_to_bf16_bits(rng.standard_normal((3, 4, d)).astype(np.float32))
    ctx = np.array(lens, np.int64)
    before = oracle.paged_attention(q, kc, vc, bm.export_tables(range(3), 8), ctx, 0.3, "bf16")
    pairs = bm.swap_out(1)
    assert len(pairs) == 4 and bm.is_swapped(1)
    oracle.swap_copy(hk, hv, kc, vc, pairs)          # device -> host
    _check_swap_invariants(bm, [0, 1, 2], H)
    kc[pairs[:, 0]] = 0                              # the freed blocks get reused / clobbered
    vc[pairs[:, 0]] = 0
    back = bm.swap_in(1)
    assert not bm.is_swapped(1) and np.array_equal(back[:, 0], pairs[:, 1])
    oracle.swap_copy(kc, vc, hk, hv, back)           # host -> device
    _check_swap_invariants(bm, [0, 1, 2], H)
    after = oracle.paged_attention(q, kc, vc, bm.export_tables(range(3), 8), ctx, 0.3, "bf16")
    assert np.array_equal(before, after)


def test_swap_out_of_a_fork_keeps_the_shared_blocks():
    bm = oracle.BlockManager(32, 4, None)
    bm.set_swap_space(16, None)
    bm.add_seq(0)
    bm.append(0, 10)
    bm.fork(0, 1)
    shared = bm.table(0).tolist()
    pairs = bm.swap_out(1)
    assert pairs[:, 0].tolist() == shared
    assert all(bm.refcount(b) == 1 for b in shared)          # the parent still names them
    assert bm.num_free() == 32 - len(shared)                 # nothing was freed
    back = bm.swap_in(1)
    assert not set(back[:, 1].tolist()) & set(shared)        # the child comes back private
    assert all(bm.refcount(int(b)) == 1 for b in back[:, 1])
    _check_swap_invariants(bm, [0, 1], 16)


def test_swap_is_all_or_nothing_and_blocks_the_swapped_sequence():
    bm = oracle.BlockManager(6, 4, None)
    bm.set_swap_space(2, None)
    bm.add_seq(0)
    bm.append(0, 12)                                         # 3 blocks
    with pytest.raises(oracle.OracleError) as ei:
        bm.swap_out(0)                                       # swap space holds 2
    assert ei.value.code == oracle.ERR_OUT_OF_BLOCKS
    assert not bm.is_swapped(0) and bm.host_free() == 2 and bm.num_free() == 3
    bm.add_seq(1)
    bm.append(1, 5)                                          # 2 blocks
    bm.swap_out(1)
    with pytest.raises(oracle.OracleError):
        bm.append(1, 1)                                      # a swapped sequence cannot grow
    with pytest.raises(oracle.OracleError):
        bm.fork(1, 9)
    bm.add_seq(2)
    bm.append(2, 12)                                         # takes the 3 free blocks
    with pytest.raises(oracle.OracleError) as ei:
        bm.swap_in(1)                                        # 2 device blocks needed, 1 free
    assert ei.value.code == oracle.ERR_OUT_OF_BLOCKS and bm.is_swapped(1)
    bm.free_seq(1)                                           # host blocks return
    assert bm.host_free() == 2
    _check_swap_invariants(bm, [0, 2], 2)


def test_exhaustion_recovered_by_swapping():
    # A sequence that keeps generating runs the pool dry; swapping another
    # sequence out lets it continue, and the other comes back once space frees.
    bm = oracle.BlockManager(8, 4, None)
    bm.set_swap_space(8, None)
    for s in (0, 1):
        bm.add_seq(s)
        bm.append(s, 16)                                     # 4 blocks each: pool full
    with pytest.raises(oracle.OracleError):
        bm.append(0, 1)
    bm.swap_out(1)
    bm.append(0, 1)                                          # now fits
    assert bm.seq_len(0) == 17
    bm.free_seq(0)
    bm.swap_in(1)
    assert bm.seq_len(1) == 16 and len(bm.table(1)) == 4
    _check_swap_invariants(bm, [1], 8)


def test_random_operations_with_swaps_keep_invariants():
    rng = np.random.default_rng(77)
    for trial in range(15):
        B = int(rng.choice([1, 4, 8]))
        N, H = int(rng.integers(10, 50)), int(rng.integers(4, 40))
        bm = oracle.BlockManager(N, B, rng.permutation(N).astype(np.int32))
        bm.set_swap_space(H, rng.permutation(H).astype(np.int32))
        live, nid = [], 0
        for _ in range(120):
            r = rng.random()
            try:
                if r < 0.15 or not live:
                    bm.add_seq(nid)
                    live.append(nid)
                    nid += 1
                elif r < 0.45:
                    bm.append(int(rng.choice(live)), int(rng.integers(0, 2 * B + 2)))
                elif r < 0.55:
                    p = int(rng.choice(live))
                    bm.fork(p, nid)
                    live.append(nid)
                    nid += 1
                elif r < 0.7:
                    bm.swap_out(int(rng.choice(live)))
                elif r < 0.85:
                    bm.swap_in(int(rng.choice(live)))
                else:
                    s = int(rng.choice(live))
                    bm.free_seq(s)
                    live.remove(s)
            except oracle.OracleError as e:
                assert e.code in (oracle.ERR_OUT_OF_BLOCKS, oracle.ERR_ARG, oracle.ERR_SEQ_EXISTS)
            _check_swap_invariants(bm, live, H)
