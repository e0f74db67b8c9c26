"""Randomised GPU parity: seeded random shapes (group size, head size, block
size, KV heads, batch, lengths with edge values) through every attention form
-- the tensor-core kernel on the grid and on a planned work list, with the
scatter fused in, in advance mode on resident tables, and the CUDA-core
kernel -- each against the fp64 oracle; pools bit-exact."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from paged_kv_cache_113_gb300.harness import DecodeState, from_device
from parity_util import assert_close
from workloads import Workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.build()


def _random_workload(seed):
    rng = np.random.default_rng(9000 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    Hk = int(rng.choice([1, 2, 4]))
    d = int(rng.choice([64, 128]))
    B = int(rng.choice([8, 16, 32]))
    S = int(rng.integers(1, 13))
    edges = [1, B, B + 1, 63, 64, 65, 512, 513, 1024]
    lens = np.where(rng.random(S) < 0.4, rng.choice(edges, size=S), rng.integers(1, 1600, size=S)).astype(np.int64)
    N = int(sum(-(-int(c + 2) // B) for c in lens) + 8)
    return Workload(f"fuzz{seed}", S, G * Hk, Hk, d, B, "bf16", N, lens, seed=100 + seed)


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_every_attention_form(seed):
    wl = _random_workload(seed)
    wl.enable_memo()
    ref = oracle.run_workload(wl)
    rng = np.random.default_rng(seed)
    part = int(rng.choice([0, -1, wl.block_size * int(rng.integers(1, 40))]))
    # Separate scatter, then the grid and the planned work list, both kernels.
    st = DecodeState(wl, "cuda")
    si = st.prepare_step(0)
    assert np.array_equal(si.slots, ref["slots"]) and np.array_equal(si.tables, ref["tables"])
    d = st.upload(si)
    rp = st.resolve_partition(d["max_context_len"], part)
    items = torch.from_numpy(pk.pk_attention_work_items(si.ctx_lens, rp)).cuda()
    ws = st.alloc_workspace(d["max_context_len"], part)
    outs = {}
    first = True
    for impl in ("mma", "simt"):
        for dd in (d, dict(d, items=items, partition=rp)):
            out = st.new_out()
            if first:
                st.run_step(dd, out, ws, part, impl)
                first = False
            else:
                st.attention(dd, out, ws, part, impl)
            torch.cuda.synchronize()
            outs[(impl, "items" in dd)] = from_device(out)
    assert pk.pk_get_device_error()[0] == 0
    assert np.array_equal(from_device(st.k_cache), ref["k_cache"])
    assert np.array_equal(from_device(st.v_cache), ref["v_cache"])
    assert np.array_equal(outs[("mma", False)], outs[("mma", True)])
    for key, o in outs.items():
        assert_close(o, ref["out"], wl.dtype, f"{wl.name} {key} part={part}")
    # The scatter fused into the attention launch.
    st2 = DecodeState(wl, "cuda")
    d2 = st2.upload(st2.prepare_step(0))
    out = st2.new_out()
    pk.pk_paged_attention_decode_append(out, d2["q"], d2["k"], d2["v"], d2["slots"], st2.k_cache, st2.v_cache,
                                        d2["tables"], d2["ctx_lens"], wl.scale, d2["max_context_len"], rp, items, ws)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error()[0] == 0
    assert np.array_equal(from_device(out), outs[("mma", True)])
    assert np.array_equal(from_device(st2.k_cache), ref["k_cache"])
    # Advance mode on resident tables (lengths before the token in, after out).
    st3 = DecodeState(wl, "cuda")
    S, maxb = wl.num_seqs, st3.max_blocks
    t, l_in = (torch.from_numpy(x).cuda() for x in st3.bm.export_tables(range(S), maxb))
    d3 = st3.upload(st3.prepare_step(0))
    l_out = torch.full_like(l_in, -1)
    out = st3.new_out()
    pk.pk_paged_attention_decode_advance(out, d3["q"], d3["k"], d3["v"], d3["slots"], st3.k_cache, st3.v_cache, t,
                                         l_in, l_out, wl.scale, d3["max_context_len"], rp, items, ws)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error()[0] == 0
    assert np.array_equal(from_device(out), outs[("mma", True)])
    assert np.array_equal(from_device(l_out), si.ctx_lens) and np.array_equal(from_device(t), si.tables)
    assert np.array_equal(from_device(st3.v_cache), ref["v_cache"])
