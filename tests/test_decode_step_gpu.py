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
from parity_util import assert_close
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
    for i in range(steps):
        si = a.prepare_step(i)
        d = a.upload(si)
        out_a = a.new_out()
        a.run_step(d, out_a, a.alloc_workspace(d["max_context_len"], -1))
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
