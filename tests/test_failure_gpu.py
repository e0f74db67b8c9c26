"""Failure detection on the GPU without a fault: a pipeline wait that can
never complete ends after its poll limit, records a timeout in the device
error word and returns, and the context stays usable."""
import time

import numpy as np
import pytest

import oracle
import paged_kv_cache_113_gb300 as pk
from paged_kv_cache_113_gb300.harness import DecodeState, from_device
from parity_util import assert_close
from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.build()


def test_stuck_wait_times_out_reports_and_leaves_the_context_usable():
    pk.pk_get_device_error()
    times = {}
    for polls in (1 << 12, 0):            # a short limit, then the kernels' own limit
        t0 = time.perf_counter()
        assert pk.lib().pk_selftest_wait_timeout(polls, None) == pk.PK_OK
        torch.cuda.synchronize()
        times[polls] = time.perf_counter() - t0
        kind, idx = pk.pk_get_device_error()
        assert pk.DEVERR_NAMES[kind] == "timeout" and idx == 0, polls
    print(f"bounded wait: {times[1 << 12] * 1e3:.2f} ms at 4096 polls, {times[0]:.3f} s at the kernels' limit")
    assert times[0] < 5.0, "a stuck stage must end within about a second"
    # The context is intact: a normal step right after still matches the oracle.
    wl = make_workload("gqa8b", num_seqs=6)
    wl.enable_memo()
    ref = oracle.run_workload(wl)
    st = DecodeState(wl, "cuda")
    d = st.upload(st.prepare_step(0))
    out = st.new_out()
    st.run_step(d, out, st.alloc_workspace(d["max_context_len"], -1), -1)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error()[0] == 0
    assert_close(from_device(out), ref["out"], wl.dtype, "after the timeout")


def test_read_stream_reference_runs_and_leaves_its_sink():
    x = torch.zeros(1 << 24, dtype=torch.float32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    import ctypes
    for nbytes in (x.numel() * 4, 16, 16 * 1000 + 16):
        assert pk.lib().pk_read_stream(ctypes.c_void_p(x.data_ptr()), nbytes, ctypes.c_void_p(sink.data_ptr()),
                                       None) == pk.PK_OK
    torch.cuda.synchronize()
    assert int(sink.item()) == 0
