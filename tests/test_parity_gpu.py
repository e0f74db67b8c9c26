"""GPU parity: libpagedkv against the CPU oracle, element by element.

Each case builds the same seeded workload twice -- once through libpagedkv on
the GPU (C++ block manager, CUDA scatter / copy / attention), once through the
oracle on the CPU -- and compares:
* slot mappings, copy-on-write pairs and block tables: bit-exact;
* the whole K and V pools after the step: bit-exact;
* attention outputs: within the tolerances of ``parity_util`` (bf16:
  max-abs 1e-2, rel-L2 2e-3; fp32: 1e-5 / 2e-6).

Reduced cases (a few sequences of each workload, every row compared) run every
kernel variant and partitioning; full-size cases run the benchmark's timed
step exactly and compare every row too (the oracle's rows dealt to the host
cores).
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from paged_kv_cache_113_gb300.harness import DecodeState, from_device
from parity_util import assert_close, as_f64, errors, oracle_every_row
from workloads import Workload, make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.build()
    yield
    torch.cuda.empty_cache()


def _no_device_error():
    kind, idx = pk.pk_get_device_error()
    assert kind == 0, f"device error {pk.DEVERR_NAMES.get(kind, kind)} at {idx}"


def _build_pair(wl, select=None, compare_pool=True, **state_kw):
    """GPU state + oracle replay of one workload step; checks the exact parts."""
    wl.enable_memo()
    ref = oracle.run_workload(wl, attention=select is not None, select=select)
    st = DecodeState(wl, "cuda", **state_kw)
    si = st.prepare_step(0)
    assert np.array_equal(si.slots, ref["slots"]), "step slot mapping differs"
    assert np.array_equal(np.asarray(si.pairs).reshape(-1, 2), ref["cow_pairs"]), "CoW pairs differ"
    assert [tuple(p) for p in st.prefill_pairs] == [tuple(p) for p in ref["prefill_pairs"]]
    for a, b in zip(st.prefill_slots, ref["prefill_slots"]):
        assert np.array_equal(a, b)
    assert np.array_equal(si.tables, ref["tables"]), "block tables differ"
    assert np.array_equal(si.ctx_lens, ref["ctx_lens"].astype(np.int32))
    d = st.upload(si)
    out = st.new_out()
    st.run_step(d, out, st.alloc_workspace(si.max_context_len, -1), -1, "auto")
    torch.cuda.synchronize()
    _no_device_error()
    if compare_pool:
        assert np.array_equal(from_device(st.k_cache), ref["k_cache"]), "K pool differs"
        assert np.array_equal(from_device(st.v_cache), ref["v_cache"]), "V pool differs"
    return st, d, out, ref


def _variants(wl):
    impls = ["simt"] + (["mma"] if wl.dtype == "bf16" else [])
    B = wl.block_size
    parts = [0, -1, 512, 3 * B, B]
    return [(i, p) for i in impls for p in parts]


def _check_all_variants(st, d, ref_out, wl, what):
    results = {}
    for impl, part in _variants(wl):
        out = st.new_out()
        ws = st.alloc_workspace(d["max_context_len"], part)
        st.attention(d, out, ws, part, impl)
        torch.cuda.synchronize()
        _no_device_error()
        results[(impl, part)] = assert_close(from_device(out), ref_out, wl.dtype, f"{what} {impl} part={part}")
    return results


REDUCED = [
    ("tiny", None, None),
    ("mha7b", 6, None),
    ("gqa8b", 24, None),
    ("long", 1, None),
    ("prefix", 8, 8),
    ("prefix", 8, 16),
    ("prefix", 8, 32),
    ("chat", 12, None),
    ("mixed", 40, None),
]


@pytest.mark.parametrize("name,nseq,B", REDUCED)
def test_reduced_workload_all_variants(name, nseq, B):
    wl = make_workload(name, block_size=B, num_seqs=nseq)
    wl.enable_memo()
    st, d, out, ref = _build_pair(wl)
    ref_out = oracle.paged_attention(ref["q"], ref["k_cache"], ref["v_cache"], ref["tables"], ref["ctx_lens"],
                                     wl.scale, wl.dtype)
    assert_close(from_device(out), ref_out, wl.dtype, f"{name} auto")
    _check_all_variants(st, d, ref_out, wl, name)


# Full-size workloads: the benchmark's configurations, every row compared.
FULL = [("mha7b", None, -1), ("gqa8b", None, -1), ("long", None, -1), ("long", None, 512), ("prefix", 8, -1),
        ("prefix", 16, -1), ("prefix", 32, -1), ("chat", None, -1), ("mixed", None, -1)]


@pytest.mark.slow
@pytest.mark.parametrize("name,B,part", FULL)
def test_full_size_every_row(name, B, part):
    """A full-size workload through the benchmark's timed step exactly: the
    step's copy-on-write copies, then the planned work list (pk_attention_plan)
    with the step's scatter fused into the attention launch
    (pk_paged_attention_decode_append). Slots, pairs, tables and both whole
    pools bit for bit against the oracle; every (sequence, query head) row of
    the output within tolerance. Then, on the same state, the (sequence,
    partition) grid at the plan's partition gives the same bits, and the
    grid's own automatic partitioning is again compared row by row.
    ``part`` -1 is the planner's choice; 512 is the 512-token split the
    long-context configuration names."""
    wl = make_workload(name, block_size=B)
    wl.enable_memo()
    ref = oracle.run_workload(wl, attention=False)
    want = oracle_every_row(ref, wl)
    st = DecodeState(wl, "cuda", extra_tokens=64)
    si = st.prepare_step(0)
    assert np.array_equal(si.slots, ref["slots"]), "step slot mapping differs"
    assert np.array_equal(np.asarray(si.pairs).reshape(-1, 2), ref["cow_pairs"]), "CoW pairs differ"
    nb = ref["tables"].shape[1]
    assert np.array_equal(si.tables[:, :nb], ref["tables"]) and (si.tables[:, nb:] == -1).all()
    assert np.array_equal(si.ctx_lens, ref["ctx_lens"].astype(np.int32))
    assert [tuple(p) for p in st.prefill_pairs] == [tuple(p) for p in ref["prefill_pairs"]]
    if name == "prefix" and B == 32:
        assert len(ref["prefill_pairs"]) == 96  # the first divergent tokens copied the shared tail blocks
    d = st.upload(si)
    d["partition"], d["items"] = st.plan(si, part)
    ws = st.alloc_workspace(d["max_context_len"], d["partition"])
    out = st.new_out()
    st.run_step_fused(d, out, ws)
    torch.cuda.synchronize()
    _no_device_error()
    assert np.array_equal(from_device(st.k_cache), ref["k_cache"]), "K pool differs"
    assert np.array_equal(from_device(st.v_cache), ref["v_cache"]), "V pool differs"
    got = from_device(out)
    assert_close(got, want, wl.dtype, f"{name} B={wl.block_size} planned+fused (partition {d['partition']})")
    grid = {k: v for k, v in d.items() if k not in ("items", "partition")}
    same = st.new_out()
    st.attention(grid, same, ws, d["partition"])
    auto = st.new_out()
    st.attention(grid, auto, st.alloc_workspace(d["max_context_len"], -1), -1)
    torch.cuda.synchronize()
    _no_device_error()
    assert np.array_equal(from_device(same), got), "grid launch at the plan's partition differs"
    assert_close(from_device(auto), want, wl.dtype, f"{name} B={wl.block_size} grid (auto)")


def _custom(name, S, Hq, Hk, d, B, lens, N=None, seed=5, dtype="bf16"):
    lens = np.asarray(lens, dtype=np.int64)
    N = N or int(sum(-(-int(c) // B) for c in lens) + 8)
    return Workload(name, S, Hq, Hk, d, B, dtype, N, lens, seed=seed)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_group_headdim_blocksize_grid(G, d, B):
    # Lengths hit the edges: 1, one block, one block + 1, a stage boundary
    # (64), one past it, a ragged tail and a partition boundary (512 + 1).
    lens = [1, B, B + 1, 63, 64, 65, 200, 513]
    wl = _custom(f"grid{G}_{d}_{B}", len(lens), 2 * G, 2, d, B, lens, seed=G * 100 + d + B)
    st, d_, out, ref = _build_pair(wl)
    ref_out = oracle.paged_attention(ref["q"], ref["k_cache"], ref["v_cache"], ref["tables"], ref["ctx_lens"],
                                     wl.scale, wl.dtype)
    _check_all_variants(st, d_, ref_out, wl, wl.name)


def test_fp32_head_dim_128():
    wl = _custom("f32_128", 3, 8, 4, 128, 16, [5, 80, 300], dtype="f32")
    st, d, out, ref = _build_pair(wl)
    ref_out = oracle.paged_attention(ref["q"], ref["k_cache"], ref["v_cache"], ref["tables"], ref["ctx_lens"],
                                     wl.scale, wl.dtype)
    _check_all_variants(st, d, ref_out, wl, wl.name)


@pytest.mark.parametrize("impl", ["simt", "mma"])
def test_block_placement_does_not_change_bits(impl):
    """Same logical data under three physical placements: identical output bits."""
    wl = _custom("perm", 6, 32, 8, 128, 16, [1, 17, 100, 333, 640, 1025], N=600).enable_memo()
    outs = []
    for seed in (1, 2, 3):
        order = np.random.default_rng(seed).permutation(wl.num_blocks).astype(np.int32)
        st = DecodeState(wl, "cuda", alloc_order=order)
        d = st.upload(st.prepare_step(0))
        for part in (0, 128):
            out = st.new_out()
            st.run_step(d, out, st.alloc_workspace(d["max_context_len"], part), part, impl)
            outs.append((part, from_device(out)))
    _no_device_error()
    for part in (0, 128):
        o = [x for p, x in outs if p == part]
        assert np.array_equal(o[0], o[1]) and np.array_equal(o[0], o[2])


@pytest.mark.parametrize("impl", ["simt", "mma"])
def test_nan_in_unwritten_slots_is_never_read(impl):
    """Pools start as NaN: slots past each context end hold NaN and must not leak."""
    wl = _custom("nan", 5, 16, 4, 128, 16, [1, 15, 17, 70, 129]).enable_memo()
    ref = oracle.run_workload(wl)
    st = DecodeState(wl, "cuda", init_value=float("nan"))
    d = st.upload(st.prepare_step(0))
    for part in (0, 32):
        out = st.new_out()
        st.run_step(d, out, st.alloc_workspace(d["max_context_len"], part), part, impl)
        torch.cuda.synchronize()
        assert_close(from_device(out), ref["out"], "bf16", f"nan-pool {impl} {part}")
    _no_device_error()


def test_split_matches_unsplit():
    wl = make_workload("long", num_seqs=1)
    wl.enable_memo()
    st = DecodeState(wl, "cuda")
    d = st.upload(st.prepare_step(0))
    outs = {}
    for part in (0, 512, 2048):
        out = st.new_out()
        st.run_step(d, out, st.alloc_workspace(d["max_context_len"], part), part, "mma")
        outs[part] = as_f64(from_device(out), "bf16")
    _no_device_error()
    for part in (512, 2048):
        mx, rl = errors(outs[part], outs[0])
        assert mx <= 8e-3 and rl <= 2e-3, (part, mx, rl)


@pytest.mark.parametrize("impl", ["simt", "mma"])
def test_launch_order_does_not_change_bits(impl):
    """Longest-first, index order and a random order give identical outputs."""
    wl = make_workload("gqa8b", num_seqs=40)
    wl.enable_memo()
    st = DecodeState(wl, "cuda")
    d = st.upload(st.prepare_step(0))
    rnd = torch.from_numpy(np.random.default_rng(3).permutation(wl.num_seqs).astype(np.int32)).cuda()
    for part in (0, 256):
        outs = []
        for order in (d["order"], None, rnd):
            out = st.new_out()
            pk.pk_paged_attention_decode(out, d["q"], st.k_cache, st.v_cache, d["tables"], d["ctx_lens"],
                                         wl.scale, d["max_context_len"], part,
                                         st.alloc_workspace(d["max_context_len"], part), impl, seq_order=order)
            outs.append(from_device(out))
        _no_device_error()
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_bad_launch_order_is_recorded():
    wl, st, d = _small_state()
    order = torch.tensor([0, 7, 2], dtype=torch.int32, device="cuda")
    out = st.new_out()
    pk.pk_paged_attention_decode(out, d["q"], st.k_cache, st.v_cache, d["tables"], d["ctx_lens"], wl.scale,
                                 d["max_context_len"], 0, None, "mma", seq_order=order)
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "order" and idx == 1


def test_standalone_copy_blocks_each_block_size():
    """96 copies (each group's last prefix block to three fresh blocks), bit-exact."""
    for B in (8, 16, 32):
        wl = make_workload("prefix", block_size=B, num_seqs=32 * 4)
        wl.enable_memo()
        ref = oracle.run_workload(wl, attention=False)
        st = DecodeState(wl, "cuda")
        si = st.prepare_step(0)
        d = st.upload(si)
        st.run_step(d, st.new_out(), st.alloc_workspace(d["max_context_len"], -1))
        free = ref["bm"].free_list()
        pairs = []
        for g in range(wl.prefix_groups):
            src = int(ref["tables"][g * wl.prefix_n][wl.prefix_len // B - 1])
            for c in range(3):
                pairs.append((src, int(free[3 * g + c])))
        pairs = np.array(pairs, np.int64)
        assert len(pairs) == 96
        oracle.copy_blocks(ref["k_cache"], ref["v_cache"], pairs)
        pk.pk_copy_blocks(st.k_cache, st.v_cache, torch.from_numpy(pairs).cuda())
        torch.cuda.synchronize()
        _no_device_error()
        assert np.array_equal(from_device(st.k_cache), ref["k_cache"])
        assert np.array_equal(from_device(st.v_cache), ref["v_cache"])
        del st
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Bad inputs: host checks return a status; device checks skip and record.
# ---------------------------------------------------------------------------
def _small_state():
    wl = _custom("edge", 3, 8, 2, 128, 16, [5, 40, 77]).enable_memo()
    st = DecodeState(wl, "cuda")
    d = st.upload(st.prepare_step(0))
    return wl, st, d


def test_bad_slot_is_skipped_and_recorded():
    wl, st, d = _small_state()
    before = from_device(st.k_cache).copy()
    slots = torch.tensor([-1, wl.num_blocks * wl.block_size, 3], dtype=torch.int64, device="cuda")
    k = torch.ones((3, 2, 128), dtype=torch.bfloat16, device="cuda")
    pk.pk_reshape_and_cache(k, k, slots, st.k_cache, st.v_cache)
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "slot" and idx == 1
    after = from_device(st.k_cache)
    changed = np.argwhere((after != before).any(axis=(2, 3)))
    assert [tuple(x) for x in changed] == [(0, 3)]     # only slot 3 (block 0, offset 3) was written


def test_bad_block_id_is_recorded_without_fault():
    wl, st, d = _small_state()
    for impl in ("simt", "mma"):
        tables = d["tables"].clone()
        tables[1, 1] = wl.num_blocks + 5
        dd = dict(d, tables=tables)
        out = st.new_out()
        st.attention(dd, out, None, 0, impl)
        kind, idx = pk.pk_get_device_error()
        assert pk.DEVERR_NAMES[kind] == "block_id" and idx == 1, impl


def test_bad_context_length_is_recorded_and_zeroed():
    wl, st, d = _small_state()
    for impl in ("simt", "mma"):
        ctx = d["ctx_lens"].clone()
        ctx[2] = 0
        out = st.new_out()
        st.attention(dict(d, ctx_lens=ctx), out, None, 0, impl)
        kind, idx = pk.pk_get_device_error()
        assert pk.DEVERR_NAMES[kind] == "context" and idx == 2
        assert not from_device(out)[2].any()


def test_bad_pair_is_recorded():
    wl, st, d = _small_state()
    pk.pk_copy_blocks(st.k_cache, st.v_cache, torch.tensor([[0, wl.num_blocks]], dtype=torch.int64, device="cuda"))
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "pair" and idx == 0


def test_host_side_rejections():
    wl, st, d = _small_state()
    out = st.new_out()
    with pytest.raises(pk.PagedKVError) as ei:
        pk.pk_paged_attention_decode(out, d["q"], st.k_cache, st.v_cache, d["tables"], d["ctx_lens"], wl.scale,
                                     d["max_context_len"], 16, None)      # splits, no workspace
    assert ei.value.status == 7
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pk.PagedKVError) as ei:
        pk.pk_paged_attention_decode(out, d["q"], st.k_cache, st.v_cache, d["tables"], d["ctx_lens"], wl.scale,
                                     d["max_context_len"], 16, small)
    assert ei.value.status == 7
    with pytest.raises(pk.PagedKVError) as ei:
        pk.pk_paged_attention_decode(out, d["q"], st.k_cache, st.v_cache, d["tables"], d["ctx_lens"], wl.scale,
                                     d["max_context_len"], 24, None)      # not a multiple of B
    assert ei.value.status == 1
    with pytest.raises(ValueError):
        pk.pk_paged_attention_decode(out.cpu(), d["q"], st.k_cache, st.v_cache, d["tables"], d["ctx_lens"],
                                     wl.scale, d["max_context_len"])
    _no_device_error()


def test_chat_prefix_cache_bookkeeping():
    """Requests admitted through the prefix cache: the cache served the same
    blocks on both sides, the GPU pool holds the oracle's bits everywhere, and
    sequences that share a system prompt name the same physical blocks."""
    wl = make_workload("chat", num_seqs=24)
    st, d, out, ref = _build_pair(wl)
    assert st.bm.cache_stats() == ref["bm"].cache_stats()
    assert st.cached_tokens == ref["bm"].cache_stats()["hits"] * wl.block_size
    assert st.cached_tokens > 0
    tables = ref["tables"]
    for p in range(len(wl.chat_prompt_lens)):
        members = [s for s in range(wl.num_seqs) if wl.chat_choice[s] == p]
        full = int(wl.chat_prompt_lens[p]) // wl.block_size
        if len(members) > 1 and full:
            assert (tables[members, :full] == tables[members[0], :full]).all()
    st.bm.check_invariants()


# Every bf16 case on both kernels; the fp32 `tiny` case on the CUDA-core
# kernel only (the tensor-core kernel is bf16 only).
_WORK_LIST_CASES = [(c, impl) for c in [("gqa8b", 40, 256), ("gqa8b", 40, 512), ("long", 2, 4736),
                                        ("prefix", 8, 512), ("mha7b", 8, 0)] for impl in ("mma", "simt")]
_WORK_LIST_CASES.append((("tiny", None, 16), "simt"))


@pytest.mark.parametrize("case,impl", _WORK_LIST_CASES, ids=[f"{c[0]}-{c[2]}-{i}" for c, i in _WORK_LIST_CASES])
def test_work_list_matches_grid_bit_for_bit(case, impl):
    """The (sequence, partition) work list gives the grid launch's result bit
    for bit (the same partials, merged in the same order) and the oracle's
    within tolerance."""
    name, nseq, part = case
    wl = make_workload(name, num_seqs=nseq, block_size=8 if name == "prefix" else None)
    assert impl == "simt" or wl.dtype == "bf16"
    st, d, _, ref = _build_pair(wl, compare_pool=False)
    lens = from_device(d["ctx_lens"])
    items = torch.from_numpy(pk.pk_attention_work_items(lens, st.resolve_partition(d["max_context_len"], part))).cuda()
    ws = st.alloc_workspace(d["max_context_len"], part)
    a, b = st.new_out(), st.new_out()
    st.attention(d, a, ws, part, impl)
    st.attention(dict(d, items=items), b, ws, part, impl)
    torch.cuda.synchronize()
    _no_device_error()
    assert np.array_equal(from_device(a), from_device(b))
    ref_out = oracle.paged_attention(ref["q"], ref["k_cache"], ref["v_cache"], ref["tables"], ref["ctx_lens"],
                                     wl.scale, wl.dtype)
    assert_close(from_device(b), ref_out, wl.dtype, f"{name} work list part={part}")


def test_bad_work_item_is_recorded():
    wl = make_workload("gqa8b", num_seqs=4)
    st, d, _, _ = _build_pair(wl, compare_pool=False)
    items = torch.tensor([[0, 0], [1, 0], [2, 0], [9, 0]], dtype=torch.int32, device="cuda")
    pk.pk_get_device_error()
    st.attention(dict(d, items=items), st.new_out(), None, 0, "mma")
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "order" and idx == 3


FUSED_CASES = [("gqa8b", 40, None, -1), ("gqa8b", 40, None, 256), ("long", 2, None, -1), ("mixed", 40, None, -1),
               ("prefix", 8, 8, -1), ("prefix", 8, 32, 512), ("mha7b", 8, None, -1), ("tiny", None, None, -1),
               ("chat", 12, None, -1)]


@pytest.mark.parametrize("name,nseq,B,part", FUSED_CASES)
def test_scatter_fused_into_attention(name, nseq, B, part):
    """pk_paged_attention_decode_append (the step's scatter inside the
    attention launch) against the separate scatter + attention: pools and
    outputs bit for bit, and the oracle's step within tolerance."""
    wl = make_workload(name, num_seqs=nseq, block_size=B)
    wl.enable_memo()
    ref = oracle.run_workload(wl)
    outs, pools = [], []
    for fused in (False, True):
        st = DecodeState(wl, "cuda")
        si = st.prepare_step(0)
        d = st.upload(si)
        d["partition"], d["items"] = st.plan(si, part)
        ws = st.alloc_workspace(d["max_context_len"], d["partition"])
        out = st.new_out()
        if fused:
            st.run_step_fused(d, out, ws)
        else:
            st.run_step(d, out, ws, d["partition"])
        torch.cuda.synchronize()
        _no_device_error()
        outs.append(from_device(out))
        pools.append((from_device(st.k_cache), from_device(st.v_cache)))
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(pools[0][0], pools[1][0]) and np.array_equal(pools[0][1], pools[1][1])
    assert np.array_equal(pools[1][0], ref["k_cache"]) and np.array_equal(pools[1][1], ref["v_cache"])
    assert_close(outs[1], ref["out"], wl.dtype, f"{name} fused part={part}")


def test_fused_scatter_bad_slot_is_recorded():
    wl = make_workload("gqa8b", num_seqs=4)
    st = DecodeState(wl, "cuda")
    si = st.prepare_step(0)
    d = st.upload(si)
    d["partition"], d["items"] = st.plan(si, -1)
    bad = d["slots"].clone()
    bad[2] = wl.num_blocks * wl.block_size + 5
    pk.pk_get_device_error()
    st.run_step_fused(dict(d, slots=bad), st.new_out(), None)
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "slot" and idx == 2
