"""Pins of the allocator policy simulator ("The KV Cache Is an Allocator
Problem", sections "One request, two kinds of waste" and "The experiment").

Fixed by the page or by hand, not by the oracle: the (repaired) 80-slot
example, a hand-traced 10-slot trace under each policy and failure rule,
closed forms for a request that runs alone, and the page's structural
claims checked on random traces: exact contiguous growth never holds
reserved-but-unused slots, maximum reservation never fails to grow, paging
never fails while capacity is free, and paged waste stays below one block
per request.
"""
import numpy as np
import pytest

from oracle import allocator_sim as sim


def req(arrival, prompt, max_new, gen, completion):
    return dict(arrival=arrival, prompt=prompt, max_new=max_new, gen=gen, completion=completion)


def test_eighty_slot_example_contiguous_fails_paged_succeeds():
    """24 + 16 + 16 + 16 slots reserved in an 80-slot cache, the second request
    finishes, then a 20-slot request arrives: free capacity is 24 but the
    largest interval is 16, so contiguous placement rejects it; 4-slot blocks
    admit it."""
    trace = [req(0, 24, 0, 0, 10), req(0, 16, 0, 0, 2), req(0, 16, 0, 0, 10), req(0, 16, 0, 0, 10),
             req(3, 20, 0, 0, 5)]
    for policy in ("max_reservation", "exact_contiguous"):
        r = sim.simulate(trace, 80, policy)
        s = r["summary"]
        assert (s["admitted"], s["rejected"], s["rejected_despite_free"]) == (4, 1, 1)
        assert r["samples"][2]["free"] == 24 and r["samples"][2]["largest_free"] == 16
        assert s["peak_reserved"] == 72
    r = sim.simulate(trace, 80, "paged", 4)
    assert (r["summary"]["admitted"], r["summary"]["rejected"]) == (5, 0)
    assert r["samples"][3]["reserved"] == 24 + 16 + 16 + 20


def test_hand_traced_growth_trace():
    """10 slots. A: prompt 4, generates 3, leaves at step 3. B: prompt 2,
    generates 2, leaves at step 2. Both arrive at step 0."""
    trace = [req(0, 4, 4, 3, 3), req(0, 2, 2, 2, 2)]
    # max reservation: A holds [0, 8); B needs 4 contiguous, only 2 left.
    r = sim.simulate(trace, 10, "max_reservation")
    assert r["summary"]["rejected"] == 1 and r["summary"]["rejected_despite_free"] == 0
    assert [x["waste"] for x in r["samples"]] == [4, 3, 2, 0]
    assert r["summary"]["peak_waste"] == 4 and r["summary"]["peak_reserved"] == 8
    # exact contiguous, drop: A = [0, 4), B = [4, 6); at step 1 A cannot extend
    # (slot 4 is B's) although 4 slots are free, and is dropped.
    r = sim.simulate(trace, 10, "exact_contiguous", on_growth_failure="drop")
    s = r["summary"]
    assert (s["growth_failures"], s["growth_failures_despite_free"], s["dropped"], s["completed"]) == (1, 1, 1, 1)
    assert [(x["live"], x["largest_free"]) for x in r["samples"]] == [(6, 4), (3, 4), (0, 10), (0, 10)]
    # exact contiguous, stall: A fails at steps 1 and 2 (B still holds slot 4
    # during step 2's growth), extends at step 3, then leaves.
    r = sim.simulate(trace, 10, "exact_contiguous", on_growth_failure="stall")
    s = r["summary"]
    assert (s["growth_failures"], s["dropped"], s["completed"]) == (2, 0, 2)
    assert s["peak_live"] == 8                       # step 2, after B's second token
    assert [x["live"] for x in r["samples"]] == [6, 7, 4, 0]
    # paged B = 2 (5 blocks): A = {0, 1}, B = {2}; step 1 both open a block.
    r = sim.simulate(trace, 10, "paged", 2)
    assert [(x["reserved"], x["live"], x["largest_free"]) for x in r["samples"]] == \
        [(6, 6, 4), (10, 8, 0), (6, 6, 2), (0, 0, 10)]
    assert r["summary"]["peak_live"] == 10 and r["summary"]["peak_waste"] == 2


def test_contiguous_placement_is_first_fit():
    """20 slots: three 4-slot prompts at [0, 4), [4, 8), [8, 12); the first and
    third leave; a new 4-slot prompt goes to the lowest hole [0, 4), so it
    cannot grow (slot 4 is taken) although slots 8..19 are free."""
    trace = [req(0, 4, 0, 0, 2), req(0, 4, 0, 0, 9), req(0, 4, 0, 0, 2), req(3, 4, 2, 2, 8)]
    r = sim.simulate(trace, 20, "exact_contiguous")
    s = r["summary"]
    assert (s["growth_failures"], s["growth_failures_despite_free"], s["dropped"]) == (1, 1, 1)
    assert r["samples"][3]["largest_free"] == 12


def test_paged_capacity_is_whole_blocks():
    r = sim.simulate([req(0, 8, 0, 0, 2), req(0, 2, 0, 0, 2)], 10, "paged", 4)
    assert r["summary"]["rejected"] == 1 and r["summary"]["rejected_despite_free"] == 0
    assert r["samples"][0]["free"] == 0


@pytest.mark.parametrize("p,m,g,B", [(5, 20, 13, 4), (16, 16, 16, 16), (1, 40, 39, 8), (7, 3, 0, 4)])
def test_single_request_closed_forms(p, m, g, B):
    trace = [req(0, p, m, g, g + 2)]
    C = 4 * (p + m) + 16
    for t, x in enumerate(sim.simulate(trace, C, "max_reservation")["samples"][: g + 2]):
        live = p + min(t, g)
        assert (x["live"], x["reserved"], x["waste"]) == (live, p + m, p + m - live)
    for t, x in enumerate(sim.simulate(trace, C, "exact_contiguous")["samples"][: g + 2]):
        assert x["reserved"] == x["live"] == p + min(t, g)
    r = sim.simulate(trace, C, "paged", B)
    for t, x in enumerate(r["samples"][: g + 2]):
        live = p + min(t, g)
        assert x["reserved"] == B * -(-live // B) and x["waste"] == B * -(-live // B) - live
    assert r["summary"]["peak_waste"] == max(B * -(-(p + k) // B) - (p + k) for k in range(g + 1))


def _random_trace(rng, n, C):
    out = []
    for _ in range(n):
        a = int(rng.integers(0, 3 * n))
        p = int(rng.integers(1, C // 4))
        m = int(rng.integers(0, C // 3))
        g = int(rng.integers(0, m + 1))
        out.append(req(a, p, m, g, a + g + int(rng.integers(1, 4))))
    return out


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("rule", ["drop", "stall"])
def test_structural_claims_on_random_traces(seed, rule):
    rng = np.random.default_rng(seed)
    C = int(rng.choice([40, 80, 96]))
    trace = _random_trace(rng, int(rng.integers(5, 25)), C)
    n = len(trace)
    runs = {"max_reservation": sim.simulate(trace, C, "max_reservation", on_growth_failure=rule),
            "exact_contiguous": sim.simulate(trace, C, "exact_contiguous", on_growth_failure=rule)}
    for B in (1, 4, 8):
        runs[f"paged{B}"] = sim.simulate(trace, C, "paged", B, on_growth_failure=rule)
    for name, r in runs.items():
        s = r["summary"]
        assert s["admitted"] + s["rejected"] == n
        if rule == "drop":
            assert s["completed"] + s["dropped"] == s["admitted"]
            assert s["dropped"] == s["growth_failures"]
        cap = C if not name.startswith("paged") else (C // int(name[5:])) * int(name[5:])
        for x in r["samples"]:
            assert 0 <= x["live"] <= x["reserved"] <= cap
            assert x["free"] == cap - x["reserved"] and 0 <= x["largest_free"] <= x["free"]
            assert x["waste"] == x["reserved"] - x["live"]
        assert s["peak_reserved"] >= max(x["reserved"] for x in r["samples"])
    assert runs["max_reservation"]["summary"]["growth_failures"] == 0
    assert runs["exact_contiguous"]["summary"]["peak_waste"] == 0
    for B in (1, 4, 8):
        r = runs[f"paged{B}"]
        assert r["summary"]["rejected_despite_free"] == 0
        assert r["summary"]["growth_failures_despite_free"] == 0
        for x in r["samples"]:
            assert x["waste"] <= (B - 1) * x["active"] and x["reserved"] % B == 0
    # With one-slot blocks nothing is ever stranded: a request is rejected or
    # fails to grow only when the cache is full.
    assert runs["paged1"]["summary"]["peak_waste"] == 0
