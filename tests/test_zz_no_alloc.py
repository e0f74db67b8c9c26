"""pk_paged_attention_decode_static: decode attention that allocates nothing.

Some callers cannot allocate device memory: a serving engine whose memory
planner already gave nearly all HBM to the KV pool, a host framework's
operator hook that hands over only input and output buffers, or a loop that
cannot pay for cudaMalloc/cudaFree and their implicit synchronisation. This
entry point keeps its split-K scratch in a static device array that the
library holds on every GPU that loads it.

The test calls it through the C ABI three times in a row, on workloads that
all split, and shapes the calls so that leftovers matter: the first call
fills the most scratch, and the second and third (smaller, other shapes)
then find the earlier calls' partials everywhere they write. Each output
must equal, bit for bit, pk_paged_attention_decode run with a
caller-allocated workspace (the same kernels, partitioning and merge order)
and match the oracle within the bf16 tolerance the parity tests use. It
also checks that a request larger than the static array is refused before
any launch. This file is collected last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from paged_kv_cache_113_gb300.harness import DecodeState, from_device
from parity_util import assert_close
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_static(st, d, out, partition):
    """The allocation-free entry point, called through the C ABI."""
    L = pk.lib()
    return L.pk_paged_attention_decode_static(
        _p(out), _p(d["q"]), _p(st.k_cache), _p(st.v_cache), _p(d["tables"]), _p(d["ctx_lens"]),
        ctypes.c_float(st.wl.scale), st.wl.block_size, st.wl.num_seqs, st.wl.num_q_heads,
        int(d["tables"].shape[1]), d["max_context_len"], partition, ctypes.byref(st.desc),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.build()


def test_static_scratch_matches_caller_workspace_three_calls():
    # (workload, sequences, partition): the first call writes the most
    # partials; the second and third, smaller and shaped differently, write
    # over them.
    cases = [("gqa8b", 24, 128), ("long", 1, 512), ("mixed", 6, 256)]
    written = 0
    for name, nseq, part in cases:
        wl = make_workload(name, num_seqs=nseq)
        wl.enable_memo()
        ref = oracle.run_workload(wl)
        st = DecodeState(wl, "cuda")
        d = st.upload(st.prepare_step(0))
        need = st.workspace_bytes(d["max_context_len"], part)
        assert 0 < need <= pk.PK_STATIC_WORKSPACE_BYTES      # it splits, and fits the array
        if written:
            assert need < written                               # all of it on scratch an earlier call wrote
        written = max(written, need)
        want = st.new_out()
        st.run_step(d, want, st.alloc_workspace(d["max_context_len"], part), part)
        got = torch.full_like(want, float("nan"))
        assert _call_static(st, d, got, part) == 0
        torch.cuda.synchronize()
        assert pk.pk_get_device_error()[0] == 0
        g = from_device(got)
        assert np.array_equal(g, from_device(want)), f"{name}: static scratch differs from a caller workspace"
        assert_close(g, ref["out"], wl.dtype, f"{name} static scratch, partition {part}")
        del st
        torch.cuda.empty_cache()


def test_static_scratch_refuses_oversized_requests():
    wl = make_workload("gqa8b", num_seqs=4)
    st = DecodeState(wl, "cuda")
    d = st.upload(st.prepare_step(0))
    out = st.new_out()
    # 64 sequences x 32 heads of 65536 tokens in 16-token partitions need
    # far more than the static array holds: refused before any launch.
    L = pk.lib()
    rc = L.pk_paged_attention_decode_static(
        _p(out), _p(d["q"]), _p(st.k_cache), _p(st.v_cache), _p(d["tables"]), _p(d["ctx_lens"]),
        ctypes.c_float(wl.scale), wl.block_size, 64, 32, int(d["tables"].shape[1]), 65536, 16,
        ctypes.byref(st.desc), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pk.PK_ERR_WORKSPACE
    assert pk.pk_get_device_error()[0] == 0
