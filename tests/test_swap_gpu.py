"""Preemption by swapping on the GPU: pk_bm_swap_out / pk_swap_blocks /
pk_bm_swap_in move a sequence's blocks to a pinned host pool and back.
Checked against the oracle (host pool and device pool bit for bit) and by
a round trip: after swapping out, letting another sequence overwrite the
freed blocks and swapping back in, attention is bit-identical."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from paged_kv_cache_113_gb300.harness import DecodeState, from_device, to_device
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.build()


def _host_pool(H, st):
    shape = (H,) + tuple(st.k_cache.shape[1:])
    return (torch.zeros(shape, dtype=st.k_cache.dtype).pin_memory(),
            torch.zeros(shape, dtype=st.k_cache.dtype).pin_memory())


@pytest.mark.parametrize("name,nseq,B", [("gqa8b", 16, None), ("prefix", 8, 32), ("mha7b", 6, None)])
def test_swap_round_trip_on_gpu(name, nseq, B):
    wl = make_workload(name, block_size=B, num_seqs=nseq)
    wl.enable_memo()
    st = DecodeState(wl, "cuda")
    pk.pk_get_device_error()
    d = st.upload(st.prepare_step(0))
    ws = st.alloc_workspace(d["max_context_len"], -1)
    before = st.new_out()
    st.run_step(d, before, ws)
    torch.cuda.synchronize()

    # Mirror on the oracle: same block-manager operations, numpy pools.
    ref = oracle.run_workload(wl, attention=False)
    rbm = ref["bm"]
    H = 2 * wl.num_blocks // 3
    horder = np.random.default_rng(5).permutation(H).astype(np.int32)
    st.bm.set_swap_space(H, horder)
    rbm.set_swap_space(H, horder)
    hk, hv = _host_pool(H, st)
    rhk = np.zeros((H,) + ref["k_cache"].shape[1:], ref["k_cache"].dtype)
    rhv = np.zeros_like(rhk)

    victims = [1, wl.num_seqs // 2, wl.num_seqs - 1]
    for s in victims:
        pairs = st.bm.swap_out(s)
        rpairs = rbm.swap_out(s)
        assert np.array_equal(pairs, rpairs)
        pk.pk_swap_blocks(st.k_cache, st.v_cache, hk, hv, torch.from_numpy(pairs).cuda(), pk.PK_SWAP_OUT)
        oracle.swap_copy(rhk, rhv, ref["k_cache"], ref["v_cache"], rpairs)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error()[0] == 0
    assert np.array_equal(from_device(hk), rhk) and np.array_equal(from_device(hv), rhv)

    # Another sequence takes the freed blocks and overwrites them.
    nfree = st.bm.num_free()
    st.bm.add_seq(10_000)
    slots, _ = st.bm.append(10_000, nfree * wl.block_size)
    junk = np.full((len(slots), wl.num_kv_heads, wl.head_dim), 0x7FC0, np.uint16)   # NaN
    pk.pk_reshape_and_cache(to_device(junk, "bf16", "cuda"), to_device(junk, "bf16", "cuda"),
                            torch.from_numpy(slots).cuda(), st.k_cache, st.v_cache)
    st.bm.free_seq(10_000)
    rbm.add_seq(10_000)
    rbm.append(10_000, nfree * wl.block_size)
    rbm.free_seq(10_000)

    for s in victims:
        pairs = st.bm.swap_in(s)
        rpairs = rbm.swap_in(s)
        assert np.array_equal(pairs, rpairs)
        pk.pk_swap_blocks(st.k_cache, st.v_cache, hk, hv, torch.from_numpy(pairs).cuda(), pk.PK_SWAP_IN)
        oracle.swap_copy(ref["k_cache"], ref["v_cache"], rhk, rhv, rpairs)
    st.bm.check_invariants()
    tables, lens = st.bm.export_tables(range(wl.num_seqs), st.max_blocks)
    assert np.array_equal(tables, rbm.export_tables(range(wl.num_seqs), st.max_blocks))
    d2 = dict(d, tables=torch.from_numpy(tables).cuda())
    after = st.new_out()
    st.attention(d2, after, ws)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error()[0] == 0
    assert np.array_equal(from_device(before), from_device(after))
    # Every block the sequences name holds the oracle's bits.
    named = np.unique(tables[tables >= 0])
    assert np.array_equal(from_device(st.k_cache)[named], ref["k_cache"][named])
    assert np.array_equal(from_device(st.v_cache)[named], ref["v_cache"][named])


def test_swap_blocks_rejects_bad_inputs():
    wl = make_workload("gqa8b", num_seqs=2)
    st = DecodeState(wl, "cuda")
    pk.pk_get_device_error()
    hk, hv = _host_pool(4, st)
    bad = torch.tensor([[0, 4]], dtype=torch.int64, device="cuda")          # host block 4 of 4
    pk.pk_swap_blocks(st.k_cache, st.v_cache, hk, hv, bad, pk.PK_SWAP_OUT)
    kind, idx = pk.pk_get_device_error()
    assert pk.DEVERR_NAMES[kind] == "pair" and idx == 0
    assert not hk.any() and not hv.any()
    with pytest.raises(ValueError):                                          # pageable host pool
        pk.pk_swap_blocks(st.k_cache, st.v_cache, torch.zeros_like(hk, device="cpu"), hv, bad, pk.PK_SWAP_OUT)
