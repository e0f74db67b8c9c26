"""Pins for the oracle's scatter, block copy and paged attention.

Nothing here retypes the oracle's loops. Each test checks the oracle against
something the pages or mathematics fix independently:

* paged attention equals dense contiguous attention ("PagedAttention",
  llminference.xinbetween.com S06, section "Run it locally": the script
  asserts paged attention is numerically identical to contiguous attention).
  The dense side is PyTorch's own scaled_dot_product_attention in float64 on
  contiguous K/V, a library routine;
* closed forms of softmax attention (one token, equal keys, two tokens, the
  hard-max limit);
* invariance under any permutation of the physical blocks ("paged attention
  deep", aicassindra.com, section "The block table": the physical blocks are
  scattered arbitrarily, the logical view is contiguous).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def _build_pool(seqs_kv, B, N, Hk, d, order, dtype):
    """Drive the oracle block manager + scatter over contiguous per-seq K/V."""
    bm = oracle.BlockManager(N, B, order)
    npdt = np.float32 if dtype == "f32" else np.uint16
    kc = np.zeros((N, B, Hk, d), npdt)
    vc = np.zeros((N, B, Hk, d), npdt)
    for s, (k, v) in enumerate(seqs_kv):
        bm.add_seq(s)
        slots, cow = bm.append(s, len(k))
        assert cow is None
        oracle.reshape_and_cache(kc, vc, k, v, slots, N, B)
    ctx = np.array([len(k) for k, _ in seqs_kv], np.int64)
    maxb = int(-(-ctx.max() // B))
    return bm, kc, vc, bm.export_tables(range(len(seqs_kv)), maxb), ctx


def _as_f64(x, dtype):
    return (x.astype(np.float64) if dtype == "f32" else bf16_bits_to_f32(x).astype(np.float64))


def _sdpa_dense(q, ks, vs, scale, dtype):
    """float64 contiguous attention per sequence with torch's SDPA."""
    outs = []
    for s, (k, v) in enumerate(zip(ks, vs)):
        qt = torch.from_numpy(_as_f64(q[s], dtype))[:, None, :]         # [Hq, 1, d]
        kt = torch.from_numpy(_as_f64(k, dtype)).permute(1, 0, 2)       # [Hk, n, d]
        vt = torch.from_numpy(_as_f64(v, dtype)).permute(1, 0, 2)
        G = qt.shape[0] // kt.shape[0]
        kt = kt.repeat_interleave(G, dim=0)
        vt = vt.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        outs.append(o[:, 0, :].numpy())
    return np.stack(outs)


def _rand(rng, shape, dtype):
    x = rng.standard_normal(shape).astype(np.float32)
    return x if dtype == "f32" else f32_to_bf16_bits(x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_paged_equals_dense(dtype, B, G):
    rng = np.random.default_rng([7, B, G, dtype == "bf16"])
    S, Hk, d = 4, 2, 16
    Hq = Hk * G
    lens = rng.integers(1, 101, size=S)
    lens[0] = 1
    N = int(sum(-(-n // B) for n in lens)) + 5
    kv = [(_rand(rng, (n, Hk, d), dtype), _rand(rng, (n, Hk, d), dtype)) for n in lens]
    q = _rand(rng, (S, Hq, d), dtype)
    order = rng.permutation(N).astype(np.int32)
    _, kc, vc, tables, ctx = _build_pool(kv, B, N, Hk, d, order, dtype)
    scale = 1.0 / math.sqrt(d)
    got = oracle.paged_attention(q, kc, vc, tables, ctx, scale, dtype)
    want = _sdpa_dense(q, [k for k, _ in kv], [v for _, v in kv], scale, dtype)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_permutation_invariance_exact():
    rng = np.random.default_rng(11)
    B, Hk, d, G = 4, 2, 8, 2
    lens = [3, 9, 17, 40]
    N = 40
    kv = [(_rand(rng, (n, Hk, d), "bf16"), _rand(rng, (n, Hk, d), "bf16")) for n in lens]
    q = _rand(rng, (4, Hk * G, d), "bf16")
    outs = []
    for seed in (1, 2, 3):
        order = np.random.default_rng(seed).permutation(N).astype(np.int32)
        _, kc, vc, tables, ctx = _build_pool(kv, B, N, Hk, d, order, "bf16")
        outs.append(oracle.paged_attention(q, kc, vc, tables, ctx, 0.3, "bf16"))
    # Blocks differ, logical order does not: the double-precision sums match bit for bit.
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_single_token_returns_its_value():
    rng = np.random.default_rng(3)
    Hk, d = 2, 8
    kv = [(_rand(rng, (1, Hk, d), "f32"), _rand(rng, (1, Hk, d), "f32"))]
    q = _rand(rng, (1, 4, d), "f32")
    _, kc, vc, tables, ctx = _build_pool(kv, 4, 4, Hk, d, None, "f32")
    out = oracle.paged_attention(q, kc, vc, tables, ctx, 1.0, "f32")
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], kv[0][1][0, h // 2].astype(np.float64))


def test_equal_keys_average_the_values():
    rng = np.random.default_rng(4)
    n, Hk, d = 37, 1, 8
    k = np.repeat(_rand(rng, (1, Hk, d), "f32"), n, axis=0)
    v = _rand(rng, (n, Hk, d), "f32")
    q = _rand(rng, (1, 1, d), "f32")
    _, kc, vc, tables, ctx = _build_pool([(k, v)], 8, 8, Hk, d, np.arange(8, dtype=np.int32)[::-1].copy(), "f32")
    out = oracle.paged_attention(q, kc, vc, tables, ctx, 0.7, "f32")
    np.testing.assert_allclose(out[0, 0], v[:, 0, :].astype(np.float64).mean(axis=0), rtol=0, atol=1e-14)


def test_two_tokens_logistic_weight():
    # Two tokens with scores x0, x1: weight of token 0 is 1 / (1 + exp(x1 - x0)).
    d = 4
    q = np.array([[[1.0, 0.0, 0.0, 0.0]]], np.float32)
    k = np.array([[[0.5, 0, 0, 0]], [[-1.25, 0, 0, 0]]], np.float32)
    v = np.array([[[1.0, 2.0, 3.0, 4.0]], [[-1.0, 0.0, 5.0, 8.0]]], np.float32)
    _, kc, vc, tables, ctx = _build_pool([(k, v)], 2, 2, 1, d, np.array([1, 0], np.int32), "f32")
    scale = 0.9
    out = oracle.paged_attention(q, kc, vc, tables, ctx, scale, "f32")[0, 0]
    w0 = 1.0 / (1.0 + math.exp(scale * (-1.25 - 0.5)))
    want = w0 * v[0, 0].astype(np.float64) + (1 - w0) * v[1, 0].astype(np.float64)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-15)


def test_hard_max_limit_selects_argmax_value():
    rng = np.random.default_rng(5)
    n, d = 50, 16
    k = _rand(rng, (n, 1, d), "f32")
    v = _rand(rng, (n, 1, d), "f32")
    q = _rand(rng, (1, 1, d), "f32")
    _, kc, vc, tables, ctx = _build_pool([(k, v)], 16, 4, 1, d, None, "f32")
    scores = k[:, 0, :].astype(np.float64) @ q[0, 0].astype(np.float64)
    top = int(np.argmax(scores))
    gap = np.sort(scores)[-1] - np.sort(scores)[-2]
    out = oracle.paged_attention(q, kc, vc, tables, ctx, 800.0 / gap, "f32")
    np.testing.assert_allclose(out[0, 0], v[top, 0].astype(np.float64), rtol=0, atol=1e-12)


def test_select_matches_full():
    rng = np.random.default_rng(6)
    kv = [(_rand(rng, (n, 2, 8), "bf16"), _rand(rng, (n, 2, 8), "bf16")) for n in (5, 33)]
    q = _rand(rng, (2, 4, 8), "bf16")
    _, kc, vc, tables, ctx = _build_pool(kv, 8, 10, 2, 8, None, "bf16")
    full = oracle.paged_attention(q, kc, vc, tables, ctx, 0.5, "bf16")
    sel = np.array([[1, 3], [0, 0]], np.int32)
    part = oracle.paged_attention(q, kc, vc, tables, ctx, 0.5, "bf16", select=sel)
    assert np.array_equal(part[1, 3], full[1, 3]) and np.array_equal(part[0, 0], full[0, 0])
    assert np.isnan(part[0, 1]).all()


def test_scatter_then_logical_read_back():
    # The pool, read back in each sequence's logical order through its table,
    # is exactly the sequence of tokens that was appended ("paged attention
    # deep", section "The block table").
    rng = np.random.default_rng(8)
    B, N, Hk, d = 4, 30, 3, 8
    kv = [(_rand(rng, (n, Hk, d), "bf16"), _rand(rng, (n, Hk, d), "bf16")) for n in (1, 4, 5, 23)]
    order = rng.permutation(N).astype(np.int32)
    bm, kc, vc, tables, ctx = _build_pool(kv, B, N, Hk, d, order, "bf16")
    for s, (k, v) in enumerate(kv):
        blocks = tables[s][tables[s] >= 0]
        flat_k = kc[blocks].reshape(-1, Hk, d)[: len(k)]
        flat_v = vc[blocks].reshape(-1, Hk, d)[: len(v)]
        assert np.array_equal(flat_k, k) and np.array_equal(flat_v, v)
    # Slots that no sequence owns were never written.
    used = np.zeros(N * B, bool)
    for s, (k, _) in enumerate(kv):
        blocks = tables[s][tables[s] >= 0]
        for t in range(len(k)):
            used[blocks[t // B] * B + t % B] = True
    assert not kc.reshape(N * B, -1)[~used].any()


def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(9)
    N, B, Hk, d = 6, 4, 2, 8
    kc = _rand(rng, (N, B, Hk, d), "bf16")
    vc = _rand(rng, (N, B, Hk, d), "bf16")
    k0, v0 = kc.copy(), vc.copy()
    oracle.copy_blocks(kc, vc, np.array([[1, 4], [2, 0]]))
    for b, src in ((4, 1), (0, 2)):
        assert np.array_equal(kc[b], k0[src]) and np.array_equal(vc[b], v0[src])
    for b in (1, 2, 3, 5):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])


def test_out_of_range_inputs_are_rejected():
    kc = np.zeros((2, 4, 1, 4), np.float32)
    vc = np.zeros_like(kc)
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(kc, vc, np.zeros((1, 1, 4), np.float32), np.zeros((1, 1, 4), np.float32),
                                 np.array([8]), 2, 4)
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kc, vc, np.array([[0, 2]]))
