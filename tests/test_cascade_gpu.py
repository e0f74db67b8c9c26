"""Cascade (shared-prefix) attention against the oracle.

The oracle computes plain attention per sequence; cascade attention reads
each group's shared prefix once and merges it with each member's own tokens,
so results agree within the bf16 tolerance (not bit for bit: the sums are
associated differently)."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from paged_kv_cache_113_gb300.harness import DecodeState, from_device
from parity_util import assert_close
from workloads import Workload, make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.build()


def _run(wl, parts=(-1, 0, 256), max_group=None, init_value=0.0, min_blocks=1):
    wl.enable_memo()
    ref = oracle.run_workload(wl)
    st = DecodeState(wl, "cuda", init_value=init_value)
    si = st.prepare_step(0)
    d = st.upload(si)
    st.run_step(d, st.new_out(), st.alloc_workspace(d["max_context_len"], -1))   # scatter the step token
    groups = st.cascade_groups(min_blocks, max_group)
    assert groups["num_groups"] > 0
    for part in parts:
        out = st.new_out()
        ws = st.alloc_cascade_workspace(d["max_context_len"], groups, part)
        st.attention_cascade(d, out, groups, ws, part)
        torch.cuda.synchronize()
        kind, idx = pk.pk_get_device_error()
        assert kind == 0, (pk.DEVERR_NAMES.get(kind), idx)
        assert_close(from_device(out), ref["out"], wl.dtype, f"{wl.name} cascade part={part}")
    return groups


@pytest.mark.parametrize("B", [8, 16, 32])
def test_cascade_prefix_workload_reduced(B):
    _run(make_workload("prefix", block_size=B, num_seqs=8))


@pytest.mark.slow
@pytest.mark.parametrize("B", [8, 16, 32])
def test_cascade_prefix_workload_full(B):
    g = _run(make_workload("prefix", block_size=B), parts=(-1,))
    assert g["num_groups"] == 32


def test_cascade_mixed_grouped_and_single():
    # Groups of at most 3: each family of 4 gives a group of 3 and one
    # sequence attended on its own.
    g = _run(make_workload("prefix", block_size=16, num_seqs=16), max_group=3)
    assert g["num_groups"] == 4 and int((g["seq_prefix_len"] > 0).sum().item()) == 12


@pytest.mark.parametrize("G,n", [(1, 16), (2, 8), (8, 2), (4, 3)])
def test_cascade_group_shapes(G, n):
    lens = np.concatenate([300 + np.arange(1, n + 1) * 7, 300 + np.arange(1, n + 1) * 13]).astype(np.int64)
    Hk = 2
    wl = Workload(f"casc{G}_{n}", 2 * n, Hk * G, Hk, 128, 16, "bf16", 2 * int(sum(-(-c // 16) for c in lens)),
                  lens, seed=40 + G, prefix_groups=2, prefix_n=n, prefix_len=300)
    _run(wl, parts=(-1, 0, 64, 16))


def test_cascade_nan_pool_and_ragged_prefix():
    # A prefix that ends mid-block: only its full blocks are shared, the
    # rest is each member's own; unwritten slots are NaN.
    lens = np.array([150, 161, 170, 190], dtype=np.int64)
    wl = Workload("casc_nan", 4, 32, 8, 128, 16, "bf16", 64, lens, seed=9, prefix_groups=1, prefix_n=4,
                  prefix_len=133)
    g = _run(wl, parts=(-1, 0, 32), init_value=float("nan"))
    assert int(g["prefix_len"][0].item()) == 128


def test_cascade_without_groups_is_regular_attention():
    wl = make_workload("gqa8b", num_seqs=8)
    wl.enable_memo()
    ref = oracle.run_workload(wl)
    st = DecodeState(wl, "cuda")
    d = st.upload(st.prepare_step(0))
    st.run_step(d, st.new_out(), st.alloc_workspace(d["max_context_len"], -1))
    groups = st.cascade_groups()
    assert groups["num_groups"] == 0
    out = st.new_out()
    st.attention_cascade(d, out, groups, st.alloc_workspace(d["max_context_len"], -1))
    torch.cuda.synchronize()
    assert_close(from_device(out), ref["out"], "bf16", "no groups")


@pytest.mark.parametrize("nseq", [16, 128])
def test_cascade_chat_requests_sharing_cached_system_prompts(nseq):
    """Requests that share a cached system prompt (not forks) form cascade groups."""
    wl = make_workload("chat", num_seqs=nseq)
    groups = _run(wl, parts=(-1,) if nseq > 16 else (-1, 0, 256))
    assert groups["max_prefix_len"] >= 512
