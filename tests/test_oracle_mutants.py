"""The oracle pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of ``oracle/oracle.c`` (a
wrong head mapping, a wrong slot offset, a missing refcount update, a dropped
softmax step, ...), builds it with gcc, and runs the pin suites against that
build in a child process. Every mutant must make at least one pin fail. The
committed oracle itself is never modified.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_block_manager.py", "tests/test_oracle_prefix_cache.py",
        "tests/test_oracle_allocator_sim.py"]

MUTANTS = {
    "gqa_head_mapping": ("const int kvh = h / G;", "const int kvh = h % Hk;"),
    "key_slot_offset": ("size_t kbase = (((size_t)phys * B + (size_t)(t % B))",
                        "size_t kbase = (((size_t)phys * B + (size_t)((t + 1) % B))"),
    "value_from_key_pool": ("o[e] += w * element(v_cache,", "o[e] += w * element(k_cache,"),
    "missing_scale": ("x[t] = scale * dot;", "x[t] = dot;"),
    "missing_normalisation": ("double w = x[t] / z;", "double w = x[t];"),
    "missing_max_subtraction": ("x[t] = exp(x[t] - m);", "x[t] = exp(x[t]);"),
    "free_list_order": ("int b = alloc_order ? alloc_order[num_blocks - 1 - i] : num_blocks - 1 - i;",
                        "int b = alloc_order ? alloc_order[i] : i;"),
    "slot_offset": ("long long slot = (long long)s->table[t / B] * B + t % B;",
                    "long long slot = (long long)s->table[t / B] * B + (t + 1) % B;"),
    "cow_keeps_source_count": ("bm->refcount[tail] -= 1;", ";"),
    "cow_on_private_block": ("if (bm->refcount[tail] > 1) {", "if (bm->refcount[tail] >= 1) {"),
    "fork_without_increment": ("bm->refcount[p->table[j]] += 1;", ";"),
    "free_ignores_refcount": ("    bm->refcount[b] -= 1;\n    if (bm->refcount[b] == 0) {",
                              "    bm->refcount[b] = 0;\n    if (bm->refcount[b] == 0) {"),
    "swap_out_keeps_reference": ("        release(bm, d);\n        s->table[j] = h;", "        s->table[j] = h;"),
    "swap_in_shares_host_block": ("        bm->host_stack[bm->host_top++] = h;\n        s->table[j] = d;",
                                  "        s->table[j] = d;"),
    "cache_key_is_block_only": ("memcmp(bm->key[b], tokens, sizeof(int) * (size_t)len) == 0",
                                "memcmp(bm->key[b] + len - bm->block_size, tokens + len - bm->block_size,"
                                " sizeof(int) * (size_t)bm->block_size) == 0"),
    "evict_most_recent": ("bm->released[b] < bm->released[best]", "bm->released[b] > bm->released[best]"),
    "evict_shallowest_first": ("bm->key_len[b] > bm->key_len[best]", "bm->key_len[b] < bm->key_len[best]"),
    "no_retention": ("        if (bm->cached[b])\n            bm->released[b] = bm->clock;",
                     "        if (0)\n            bm->released[b] = bm->clock;"),
    "hit_without_reference": ("        bm->refcount[b] += 1;\n        bm->cache_hits += 1;",
                              "        bm->cache_hits += 1;"),
    "commit_partial_block": ("(long long)(j + 1) * B <= n; j++) {\n        int b = s->table[j];",
                             "(long long)j * B < n; j++) {\n        int b = s->table[j];"),
    "evictable_not_available": ("        if (bm->cached[b] && bm->refcount[b] == 0) n++;", ""),
    "evict_keeps_key": ("    uncache(bm, best);\n", ""),
    "copy_blocks_swapped": ("memcpy((char *)k_cache + (size_t)dst * blk_bytes, (char *)k_cache + (size_t)src * blk_bytes",
                            "memcpy((char *)k_cache + (size_t)src * blk_bytes, (char *)k_cache + (size_t)dst * blk_bytes"),
}


# Mistakes planted in the Python parts of the oracle: (module, old, new).
PY_MUTANTS = {
    "last_fit_placement": ("contiguous", "for start, length in self.holes():",
                           "for start, length in reversed(self.holes()):"),
    "grow_into_neighbour": ("contiguous", "if other != rid and s2 <= end < s2 + n2:",
                            "if other != rid and s2 < end < s2 + n2:"),
    "reserve_prompt_only": ("allocator_sim", 'return req["prompt"] + (req["max_new"] if self.reserve_max else 0)',
                            'return req["prompt"]'),
    "failed_growth_not_dropped": ("allocator_sim", "            if drop:\n", "            if False:\n"),
    "peaks_only_at_admission": ("allocator_sim", "                generated[i] += 1\n                note_peaks()\n",
                                "                generated[i] += 1\n"),
    "despite_free_misread": ("allocator_sim", "if alloc.capacity - alloc.reserved() >= 1:",
                             "if alloc.reserved() >= 1:"),
    "paged_need_rounds_down": ("allocator_sim", 'need = -(-req["prompt"] // self.B)', 'need = req["prompt"] // self.B'),
    "free_run_ignores_gaps": ("allocator_sim", "run = run + 1 if prev is not None and b == prev + 1 else 1",
                              "run = run + 1"),
    "paged_capacity_in_slots": ("allocator_sim", "self.capacity = self.N * B", "self.capacity = capacity"),
}

PY_PINS = ["tests/test_oracle_allocator_sim.py", "tests/test_oracle_block_manager.py"]

_BOOT = """
import importlib.util, sys
sys.path.insert(0, {root!r})
import oracle
spec = importlib.util.spec_from_file_location("oracle.{mod}", {path!r})
mod = importlib.util.module_from_spec(spec)
sys.modules["oracle.{mod}"] = mod
setattr(oracle, "{mod}", mod)
spec.loader.exec_module(mod)
import pytest
sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider", *{pins!r}]))
"""


def _run_py_mutant(name, tmpdir):
    module, old, new = PY_MUTANTS[name]
    text = open(os.path.join(ROOT, "oracle", module + ".py")).read()
    assert text.count(old) == 1, f"{name}: pattern must occur exactly once"
    path = os.path.join(tmpdir, f"{name}_{module}.py")
    with open(path, "w") as f:
        f.write(text.replace(old, new))
    boot = _BOOT.format(root=ROOT, mod=module, path=path, pins=PY_PINS)
    r = subprocess.run([sys.executable, "-c", boot], cwd=ROOT, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_python_mutant_is_caught(tmp_path):
    names = sorted(PY_MUTANTS)
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = dict(ex.map(lambda n: _run_py_mutant(n, str(tmp_path)), names))
    survivors = [n for n, rc in results.items() if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"
    assert all(rc == 1 for rc in results.values()), results


def _run_mutant(name, tmpdir):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"{name}: pattern must occur exactly once"
    c = os.path.join(tmpdir, f"{name}.c")
    so = os.path.join(tmpdir, f"{name}.so")
    with open(c, "w") as f:
        f.write(text.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so, c, "-lm"], check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_mutant_is_caught(tmp_path):
    names = sorted(MUTANTS)
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = dict(ex.map(lambda n: _run_mutant(n, str(tmp_path)), names))
    survivors = [n for n, rc in results.items() if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"
    # rc 1 = a test failed; anything else (crash, collection error) is not a pin.
    assert all(rc == 1 for rc in results.values()), results
