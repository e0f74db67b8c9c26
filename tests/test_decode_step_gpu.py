"""pk_decode_step (one native call per decode step from host buffers) against
the step-by-step path (block-manager append, uploads, pk_copy_blocks,
pk_reshape_and_cache, pk_paged_attention_decode): identical outputs and pools
over several steps, including steps with copy-on-write pairs, and the first
step against the oracle."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from paged_kv_cache_113_gb300.harness import DecodeState, from_device, to_device
from parity_util import assert_close, oracle_every_row
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.build()


def _host(a, dtype):
    return to_device(a, dtype, "cpu")


class _Stepwise:
    """The step-by-step path with pk_decode_step's schedule: the first step
    plans (pk_attention_plan), later steps keep its partition and rebuild the
    work list for the current lengths."""

    def __init__(self, state):
        self.st, self.part = state, None

    def step(self, i):
        st = self.st
        si = st.prepare_step(i)
        d = st.upload(si)
        if self.part is None:
            self.part, items = pk.pk_attention_plan(si.ctx_lens, st.wl.num_q_heads, st.desc, -1)
        else:
            items = pk.pk_attention_work_items(si.ctx_lens, self.part)
        d["partition"], d["items"] = self.part, torch.from_numpy(items).cuda()
        out = st.new_out()
        st.run_step(d, out, st.alloc_workspace(d["max_context_len"], self.part))
        return out


@pytest.mark.parametrize("name,nseq,B", [("gqa8b", 24, None), ("prefix", 8, 32), ("long", 1, None),
                                         ("mha7b", 4, None), ("tiny", None, None)])
def test_decode_step_matches_stepwise_path(name, nseq, B):
    wl = make_workload(name, block_size=B, num_seqs=nseq)
    wl.enable_memo()
    steps = 3
    a = DecodeState(wl, "cuda", extra_tokens=steps)
    b = DecodeState(wl, "cuda", extra_tokens=steps)
    stepper = pk.DecodeStepper(b.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, b.max_blocks,
                               b.k_cache, b.v_cache)
    ref_path = _Stepwise(a)
    for i in range(steps):
        out_a = ref_path.step(i)
        q, k, v = wl.step_inputs(i)
        stepper.q_host.copy_(_host(q, wl.dtype))
        stepper.k_host.copy_(_host(k, wl.dtype))
        stepper.v_host.copy_(_host(v, wl.dtype))
        out_b = stepper.step()
        torch.cuda.synchronize()
        assert pk.pk_get_device_error()[0] == 0
        assert np.array_equal(from_device(out_a), from_device(out_b)), f"step {i}"
        if i == 0:
            ref = oracle.run_workload(wl)
            assert_close(from_device(out_b), ref["out"], wl.dtype, f"{name} step 0")
    assert np.array_equal(from_device(a.k_cache), from_device(b.k_cache))
    assert np.array_equal(from_device(a.v_cache), from_device(b.v_cache))
    b.bm.check_invariants()


@pytest.mark.parametrize("name,nseq,B,steps", [("gqa8b", 24, None, 40), ("prefix", 8, 8, 20), ("mixed", 40, None, 20)])
def test_resident_tables_over_many_steps(name, nseq, B, steps):
    """After the first step the tables stay on the device and are advanced by
    the scatter kernel: many steps (crossing block boundaries) still give the
    step-by-step path's outputs bit for bit, and the device tables equal the
    block manager's."""
    wl = make_workload(name, block_size=B, num_seqs=nseq)
    wl.enable_memo()
    a = DecodeState(wl, "cuda", extra_tokens=steps)
    b = DecodeState(wl, "cuda", extra_tokens=steps)
    stepper = pk.DecodeStepper(b.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, b.max_blocks,
                               b.k_cache, b.v_cache)
    ref_path = _Stepwise(a)
    for i in range(steps):
        out_a = ref_path.step(i)
        q, k, v = wl.step_inputs(i)
        stepper.q_host.copy_(_host(q, wl.dtype))
        stepper.k_host.copy_(_host(k, wl.dtype))
        stepper.v_host.copy_(_host(v, wl.dtype))
        out_b = stepper.step()
        assert stepper.buffers.tables_resident == 1
        assert stepper.buffers.plan_partition == ref_path.part
        assert np.array_equal(from_device(out_a), from_device(out_b)), f"step {i}"
    assert pk.pk_get_device_error()[0] == 0
    S, maxb = wl.num_seqs, b.max_blocks
    meta = from_device(stepper.meta_dev)
    lay = _meta_layout(S, maxb)
    tables, lens = b.bm.export_tables(range(S), maxb)
    assert np.array_equal(meta[lay["tables"]: lay["tables"] + 4 * S * maxb].view(np.int32).reshape(S, maxb), tables)
    # The resident steps alternate two length buffers, starting from the full
    # step's upload into the first.
    cur = lay["lens_b"] if (steps - 1) % 2 else lay["lens"]
    assert np.array_equal(meta[cur: cur + 4 * S].view(np.int32), lens)


def _meta_layout(S, maxb):
    """Offsets of the decode-step metadata sections (256-byte aligned, in the
    order slots, pairs, work items, lens, tables, second lens)."""
    up = lambda x: (x + 255) // 256 * 256
    slots = 0
    pairs = up(slots + 8 * S)
    items = up(pairs + 16 * S)
    lens = up(items + 8 * min(S * (1 + maxb // 16), 65535))
    tables = up(lens + 4 * S)
    lens_b = up(tables + 4 * S * maxb)
    assert 2 * up(lens_b + 4 * S) == pk.lib().pk_decode_step_meta_bytes(S, maxb)  # two halves
    return {"slots": slots, "pairs": pairs, "items": items, "lens": lens, "tables": tables, "lens_b": lens_b}


def test_invalidate_after_fork_reuploads_tables():
    wl = make_workload("gqa8b", num_seqs=6)
    wl.enable_memo()
    b = DecodeState(wl, "cuda", extra_tokens=8)
    ids = list(range(wl.num_seqs))
    stepper = pk.DecodeStepper(b.bm, ids, wl.num_q_heads, wl.scale, b.max_blocks, b.k_cache, b.v_cache)
    stepper.step()
    # Free one sequence and fork another into its id: the rows' tables change.
    b.bm.free_seq(2)
    b.bm.fork(4, 2)
    stepper.invalidate()
    stepper.step()
    assert pk.pk_get_device_error()[0] == 0
    S, maxb = wl.num_seqs, b.max_blocks
    lay = _meta_layout(S, maxb)
    meta = from_device(stepper.meta_dev)
    tables, lens = b.bm.export_tables(ids, maxb)
    assert np.array_equal(meta[lay["tables"]: lay["tables"] + 4 * S * maxb].view(np.int32).reshape(S, maxb), tables)
    b.bm.check_invariants()


@pytest.mark.parametrize("B", [8, 16, 32])
def test_scatter_append_updates_tables_like_the_block_manager(B):
    """pk_reshape_and_cache_append against the host block manager on a batch
    with forks (copy-on-write pairs) and sequences opening new blocks."""
    rng = np.random.default_rng(B)
    N, Hk, d = 256, 2, 64
    bm = pk.BlockManager(N, B, rng.permutation(N).astype(np.int32))
    for s, n in enumerate([5, B + 3, 3 * B, 2 * B + 1, 1, 4 * B - 1]):
        bm.add_seq(s)
        bm.append(s, n)
    bm.fork(1, 6)                     # partial tails: the next tokens copy on write
    bm.fork(3, 7)
    bm.add_seq(8)
    bm.append(8, B)                   # the next token opens a block
    ids = list(range(9))
    maxb = 8
    tables0, lens0 = bm.export_tables(ids, maxb)
    slots, pairs = bm.append_batch(ids)
    assert len(pairs) == 2
    tables1, lens1 = bm.export_tables(ids, maxb)
    desc_pool = torch.zeros((N, B, Hk, d), dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(desc_pool)
    kk = torch.randn((len(ids), Hk, d), device="cuda").to(torch.bfloat16)
    vv = torch.randn((len(ids), Hk, d), device="cuda").to(torch.bfloat16)
    dt = torch.from_numpy(tables0).cuda()
    dl = torch.from_numpy(lens0).cuda()
    pk.pk_get_device_error()
    pk.pk_reshape_and_cache_append(kk, vv, torch.from_numpy(slots).cuda(), desc_pool, v_pool, dt, dl)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error()[0] == 0
    assert np.array_equal(dt.cpu().numpy(), tables1)
    assert np.array_equal(dl.cpu().numpy(), lens1)
    flat = desc_pool.view(N * B, Hk, d)
    assert torch.equal(flat[torch.from_numpy(slots).cuda()], kk)


def test_scatter_append_records_a_row_out_of_step():
    B, N = 16, 64
    pool = torch.zeros((N, B, 2, 64), dtype=torch.bfloat16, device="cuda")
    vpool = torch.zeros_like(pool)
    kk = torch.ones((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    tables = torch.tensor([[3, -1], [5, -1]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([4, 7], dtype=torch.int32, device="cuda")
    slots = torch.tensor([3 * B + 4, 5 * B + 9], dtype=torch.int64, device="cuda")   # row 1: offset 9 != 7
    pk.pk_get_device_error()
    pk.pk_reshape_and_cache_append(kk, kk, slots, pool, vpool, tables, lens)
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "context" and idx == 1
    assert lens.tolist() == [5, 7] and tables.tolist() == [[3, -1], [5, -1]]


@pytest.mark.slow
@pytest.mark.parametrize("name,B", [("mha7b", None), ("gqa8b", None), ("long", None), ("mixed", None),
                                    ("chat", None), ("prefix", 32)])
def test_decode_step_full_size_against_the_oracle(name, B):
    """pk_decode_step as the benchmark's e2e leg runs it (full size, planned
    work list, zero-copy from pinned host buffers, the next step prepared
    while the current one runs): its first two steps -- the first uploads
    the tables, the second runs on the device-resident tables in advance
    mode -- against the oracle's two steps on every row, and the pools after
    them bit for bit."""
    wl = make_workload(name, block_size=B)
    wl.enable_memo()
    ref = oracle.run_workload(wl, attention=False)
    b = DecodeState(wl, "cuda", extra_tokens=4)
    stepper = pk.DecodeStepper(b.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, b.max_blocks,
                               b.k_cache, b.v_cache, max_context_len=int(wl.ctx_lens.max()) + 4, zero_copy=True)
    stepper.prepare()
    for step in range(2):
        if step:
            oracle.continue_workload(ref, wl, step, attention=False)
        q, k, v = wl.step_inputs(step)
        stepper.stream.synchronize()
        stepper.q_host.copy_(_host(q, wl.dtype))
        stepper.k_host.copy_(_host(k, wl.dtype))
        stepper.v_host.copy_(_host(v, wl.dtype))
        stepper.launch_prepared()
        # Step 1 is prepared after step 0's launch: on resident tables.
        assert stepper.buffers.tables_resident == 1
        stepper.prepare()
        stepper.stream.synchronize()
        assert pk.pk_get_device_error()[0] == 0
        got = from_device(stepper.out_host)
        assert_close(got, oracle_every_row(ref, wl), wl.dtype, f"{name} pk_decode_step step {step}")
    torch.cuda.synchronize()
    assert np.array_equal(from_device(b.k_cache), ref["k_cache"]), "K pool differs"
    assert np.array_equal(from_device(b.v_cache), ref["v_cache"]), "V pool differs"
    stepper.release()


@pytest.mark.parametrize("name,zero_copy", [("gqa8b", False), ("gqa8b", True), ("long", True), ("tiny", True)])
def test_graph_replay_follows_new_host_buffers(name, zero_copy):
    """Steady steps replay the captured graph; each step passes fresh pinned
    q/k/v tensors, so the graph is re-pointed every step: its input copies
    (copying mode) or its attention kernels' arguments (zero-copy mode; on
    `long` the step splits, so the merge kernel is re-pointed too; `tiny` is
    fp32, the CUDA-core kernel). Outputs equal the step-by-step path bit for
    bit, and the graphs are kept."""
    wl = make_workload(name, num_seqs={"gqa8b": 24, "long": 2}.get(name))
    wl.enable_memo()
    steps = 12
    a = DecodeState(wl, "cuda", extra_tokens=steps)
    b = DecodeState(wl, "cuda", extra_tokens=steps)
    stepper = pk.DecodeStepper(b.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, b.max_blocks,
                               b.k_cache, b.v_cache, zero_copy=zero_copy)
    ref_path = _Stepwise(a)
    counts = []
    for i in range(steps):
        out_a = ref_path.step(i)
        q, k, v = (_host(x, wl.dtype).pin_memory() for x in wl.step_inputs(i))
        stepper.launch(q_host=q, k_host=k, v_host=v)
        stepper.stream.synchronize()
        counts.append(stepper.graph_count)
        assert np.array_equal(from_device(out_a), from_device(stepper.out_host)), f"step {i}"
    # Step 0 uploads the tables; steps 1 and 2 capture one graph per staging
    # half; every later step replays one, re-pointed, without recapturing.
    assert counts[2:] == [2] * (steps - 2), f"graphs dropped: counts per step {counts}"
    assert pk.pk_get_device_error()[0] == 0
    stepper.release()
    assert not stepper.buffers.state and stepper.graph_count == 0


def test_zero_copy_unpinned_inputs_are_exact_or_refused():
    """Zero-copy steps given ordinary (unpinned) host tensors: where the GPU
    reads host memory through the host's page tables they are used at their
    own addresses and the outputs equal the step-by-step path bit for bit;
    elsewhere the launch is refused with an invalid-argument status before any
    work. Never a wrong output."""
    wl = make_workload("gqa8b", num_seqs=16)
    wl.enable_memo()
    steps = 6
    a = DecodeState(wl, "cuda", extra_tokens=steps)
    b = DecodeState(wl, "cuda", extra_tokens=steps)
    stepper = pk.DecodeStepper(b.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, b.max_blocks,
                               b.k_cache, b.v_cache, zero_copy=True)
    ref_path = _Stepwise(a)
    counts = []
    for i in range(steps):
        q, k, v = (_host(x, wl.dtype) for x in wl.step_inputs(i))
        assert not q.is_pinned()
        try:
            stepper.launch(q_host=q, k_host=k, v_host=v)
        except pk.PagedKVError as e:
            assert i == 0 and e.status == pk.PK_ERR_INVALID_ARG
            stepper.release()
            pytest.skip("this GPU does not read host memory through the host's page tables")
        stepper.stream.synchronize()
        counts.append(stepper.graph_count)
        out_a = ref_path.step(i)
        assert np.array_equal(from_device(out_a), from_device(stepper.out_host)), f"step {i}"
    assert counts[2:] == [2] * (steps - 2), f"graphs dropped: counts per step {counts}"
    assert pk.pk_get_device_error()[0] == 0
    stepper.release()


@pytest.mark.parametrize("name,nseq,B", [("gqa8b", 24, None), ("prefix", 8, 32), ("mixed", 40, None)])
def test_zero_copy_steps_match_the_copying_steps(name, nseq, B):
    """Zero-copy mode (the kernels read q, k, v from and write out to pinned host
    memory) gives the copying mode's outputs and pools bit for bit, over full,
    resident and graph-replayed steps."""
    wl = make_workload(name, block_size=B, num_seqs=nseq)
    wl.enable_memo()
    steps = 10
    runs = []
    for zero_copy in (False, True):
        st = DecodeState(wl, "cuda", extra_tokens=steps)
        stepper = pk.DecodeStepper(st.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, st.max_blocks,
                                   st.k_cache, st.v_cache, zero_copy=zero_copy)
        outs = []
        for i in range(steps):
            q, k, v = wl.step_inputs(i)
            stepper.stream.synchronize()
            stepper.q_host.copy_(_host(q, wl.dtype))
            stepper.k_host.copy_(_host(k, wl.dtype))
            stepper.v_host.copy_(_host(v, wl.dtype))
            outs.append(from_device(stepper.step()).copy())
        assert pk.pk_get_device_error()[0] == 0
        runs.append((outs, from_device(st.k_cache), from_device(st.v_cache)))
        stepper.release()
    for a, b in zip(runs[0][0], runs[1][0]):
        assert np.array_equal(a, b)
    assert np.array_equal(runs[0][1], runs[1][1]) and np.array_equal(runs[0][2], runs[1][2])


@pytest.mark.parametrize("name,nseq,B,zero_copy", [("gqa8b", 24, None, True), ("prefix", 8, 8, False),
                                                   ("mixed", 40, None, True), ("long", 1, None, False)])
def test_pipelined_steps_match_the_stepwise_path(name, nseq, B, zero_copy):
    """The overlapped loop: the host half of step t+1 (prepare) runs right
    after step t is launched, while step t is on the GPU. Outputs and pools
    equal the step-by-step path's bit for bit over steps that cross block
    boundaries, start partitions and (prefix) copy on write."""
    wl = make_workload(name, block_size=B, num_seqs=nseq)
    wl.enable_memo()
    steps = 20
    a = DecodeState(wl, "cuda", extra_tokens=steps + 1)
    b = DecodeState(wl, "cuda", extra_tokens=steps + 1)
    stepper = pk.DecodeStepper(b.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, b.max_blocks,
                               b.k_cache, b.v_cache, zero_copy=zero_copy)
    ref_path = _Stepwise(a)
    stepper.prepare()
    for i in range(steps):
        out_a = ref_path.step(i)
        q, k, v = wl.step_inputs(i)
        stepper.q_host.copy_(_host(q, wl.dtype))
        stepper.k_host.copy_(_host(k, wl.dtype))
        stepper.v_host.copy_(_host(v, wl.dtype))
        stepper.launch_prepared()
        stepper.prepare()                  # step i + 1's host half while step i runs
        stepper.stream.synchronize()
        assert stepper.buffers.tables_resident == 0   # the prepared step is not launched yet
        assert np.array_equal(from_device(out_a), from_device(stepper.out_host)), f"step {i}"
    assert pk.pk_get_device_error()[0] == 0
    assert np.array_equal(from_device(a.k_cache), from_device(b.k_cache))
    assert np.array_equal(from_device(a.v_cache), from_device(b.v_cache))
    with pytest.raises(pk.PagedKVError):
        stepper.prepare()                  # one prepared step at a time
    stepper.release()


@pytest.mark.parametrize("name,nseq,B,part", [("gqa8b", 24, None, -1), ("gqa8b", 24, None, 256),
                                              ("prefix", 8, 8, -1), ("mixed", 40, None, -1),
                                              ("long", 1, None, 1024), ("tiny", None, None, -1)])
def test_advance_matches_append_then_attention(name, nseq, B, part):
    """pk_paged_attention_decode_advance (scatter, table bookkeeping and
    attention in one launch on resident tables, lengths alternating between
    two buffers) against pk_reshape_and_cache_append followed by the
    attention over the work list: outputs, pools, tables and lengths bit for
    bit over steps that open blocks, copy on write (prefix) and start
    partitions."""
    wl = make_workload(name, block_size=B, num_seqs=nseq)
    wl.enable_memo()
    steps = 12
    a = DecodeState(wl, "cuda", extra_tokens=steps)
    b = DecodeState(wl, "cuda", extra_tokens=steps)
    S, maxb = wl.num_seqs, a.max_blocks
    ta, la = (torch.from_numpy(x).cuda() for x in a.bm.export_tables(range(S), maxb))
    tb = ta.clone()
    lb = [la.clone(), torch.full_like(la, -7)]
    rp = None
    for i in range(steps):
        sa, sb = a.prepare_step(i), b.prepare_step(i)
        assert np.array_equal(sa.slots, sb.slots)
        da, db = a.upload(sa), b.upload(sb)
        if rp is None:
            rp, items = pk.pk_attention_plan(sa.ctx_lens, wl.num_q_heads, a.desc, part)
        else:
            items = pk.pk_attention_work_items(sa.ctx_lens, rp)
        items = torch.from_numpy(items).cuda()
        ws = a.alloc_workspace(sa.max_context_len, rp)
        if len(sa.pairs):
            pk.pk_copy_blocks(a.k_cache, a.v_cache, da["pairs"])
            pk.pk_copy_blocks(b.k_cache, b.v_cache, db["pairs"])
        out_a, out_b = a.new_out(), b.new_out()
        pk.pk_reshape_and_cache_append(da["k"], da["v"], da["slots"], a.k_cache, a.v_cache, ta, la)
        pk.pk_paged_attention_decode(out_a, da["q"], a.k_cache, a.v_cache, ta, la, wl.scale, sa.max_context_len,
                                     rp, ws, work_items=items)
        pk.pk_paged_attention_decode_advance(out_b, db["q"], db["k"], db["v"], db["slots"], b.k_cache, b.v_cache,
                                             tb, lb[i % 2], lb[(i + 1) % 2], wl.scale, sb.max_context_len, rp,
                                             items, ws)
        torch.cuda.synchronize()
        assert pk.pk_get_device_error()[0] == 0, f"step {i}"
        assert np.array_equal(from_device(out_a), from_device(out_b)), f"step {i}"
        assert np.array_equal(from_device(lb[(i + 1) % 2]), sa.ctx_lens), f"step {i}"
        assert np.array_equal(from_device(la), sa.ctx_lens)
        assert np.array_equal(from_device(tb), from_device(ta)), f"step {i}"
        assert np.array_equal(from_device(tb), sa.tables), f"step {i}"
    assert np.array_equal(from_device(a.k_cache), from_device(b.k_cache))
    assert np.array_equal(from_device(a.v_cache), from_device(b.v_cache))


def test_advance_records_a_slot_out_of_step():
    """A slot that is not at offset len mod B of its block: recorded, and the
    row's length is carried over unchanged."""
    wl = make_workload("gqa8b", num_seqs=4)
    st = DecodeState(wl, "cuda", extra_tokens=2)
    S, maxb = wl.num_seqs, st.max_blocks
    t, l_in = (torch.from_numpy(x).cuda() for x in st.bm.export_tables(range(S), maxb))
    si = st.prepare_step(0)
    d = st.upload(si)
    rp, items = pk.pk_attention_plan(si.ctx_lens, wl.num_q_heads, st.desc, 0)
    bad = d["slots"].clone()
    bad[1] += 1
    l_out = torch.full_like(l_in, -7)
    pk.pk_get_device_error()
    pk.pk_paged_attention_decode_advance(st.new_out(), d["q"], d["k"], d["v"], bad, st.k_cache, st.v_cache, t,
                                         l_in, l_out, wl.scale, si.max_context_len, rp,
                                         torch.from_numpy(items).cuda(), None)
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "context" and idx == 1
    got = from_device(l_out)
    assert got[1] == from_device(l_in)[1] and got[0] == si.ctx_lens[0]


@pytest.mark.parametrize("G,d,B", [(1, 64, 8), (8, 128, 32), (4, 64, 16), (2, 128, 8)])
def test_advance_shapes_against_the_oracle(G, d, B):
    """The one-launch resident step over head sizes, group sizes and block
    sizes, with lengths at the edges (a fresh sequence, block and stage
    boundaries, a partition boundary): every step equals append + attention
    bit for bit, and the last step matches the oracle's attention over the
    block manager's tables."""
    from workloads import Workload
    lens = np.array([1, B - 1, B, 63, 64, 200, 511, 1200], dtype=np.int64)
    N = int(sum(-(-int(c + 8) // B) for c in lens) + 16)
    wl = Workload(f"adv{G}_{d}_{B}", len(lens), 2 * G, 2, d, B, "bf16", N, lens, seed=G * 11 + d + B)
    wl.enable_memo()
    steps = 6
    a = DecodeState(wl, "cuda", extra_tokens=steps)
    b = DecodeState(wl, "cuda", extra_tokens=steps)
    S, maxb = wl.num_seqs, a.max_blocks
    ta, la = (torch.from_numpy(x).cuda() for x in a.bm.export_tables(range(S), maxb))
    tb, lb = ta.clone(), [la.clone(), torch.full_like(la, -7)]
    for i in range(steps):
        sa, sb = a.prepare_step(i), b.prepare_step(i)
        da, db = a.upload(sa), b.upload(sb)
        part = 64 if i % 2 else 0
        items = torch.from_numpy(pk.pk_attention_work_items(sa.ctx_lens, part)).cuda()
        ws = a.alloc_workspace(sa.max_context_len, part)
        out_a, out_b = a.new_out(), b.new_out()
        pk.pk_reshape_and_cache_append(da["k"], da["v"], da["slots"], a.k_cache, a.v_cache, ta, la)
        pk.pk_paged_attention_decode(out_a, da["q"], a.k_cache, a.v_cache, ta, la, wl.scale, sa.max_context_len,
                                     part, ws, work_items=items)
        pk.pk_paged_attention_decode_advance(out_b, db["q"], db["k"], db["v"], db["slots"], b.k_cache, b.v_cache,
                                             tb, lb[i % 2], lb[(i + 1) % 2], wl.scale, sb.max_context_len, part,
                                             items, ws)
        torch.cuda.synchronize()
        assert pk.pk_get_device_error()[0] == 0, f"step {i}"
        assert np.array_equal(from_device(out_a), from_device(out_b)), f"step {i}"
        assert np.array_equal(from_device(tb), sa.tables) and np.array_equal(from_device(lb[(i + 1) % 2]), sa.ctx_lens)
    ref = oracle.paged_attention(from_device(db["q"]), from_device(b.k_cache), from_device(b.v_cache), sb.tables,
                                 sb.ctx_lens, wl.scale, wl.dtype)
    assert_close(from_device(out_b), ref, wl.dtype, f"advance G={G} d={d} B={B}")
