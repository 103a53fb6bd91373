"""Pins for the oracle: each check ties it to something other than itself --
values the pages print, closed forms, a library routine (numpy / scipy), or
invariants -- so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails here.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# exact 16-bit conversions: every bit pattern against numpy's own decoding
# --------------------------------------------------------------------------
def test_half_conversion_all_patterns():
    lib = oracle._load()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.fdo_half_to_double(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_conversion_all_patterns():
    lib = oracle._load()
    bits = np.arange(65536, dtype=np.uint32)
    # bf16 is the upper half of an IEEE binary32 pattern
    with np.errstate(invalid="ignore"):
        want = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([lib.fdo_bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# --------------------------------------------------------------------------
# the pages' worked values
# --------------------------------------------------------------------------
def test_dkv_worked_example_full_output(golden_dir):
    g = _load(golden_dir, "dkv_worked_example.json")
    s = np.array([0.0, math.log(2), math.log(3), math.log(4)])
    V = np.array(g["values"], dtype=np.float64).reshape(4, 1)
    # a 1-d "head" with q = 1 and keys equal to the scores, scale 1
    o, lse = oracle.attend([1.0], s.reshape(4, 1), V, 1.0)
    assert o[0] == pytest.approx(g["full_output"], abs=1e-14)
    num, den = g["full_output_fraction"]
    assert o[0] == pytest.approx(num / den, abs=1e-14)
    assert lse == pytest.approx(math.log(10.0), abs=1e-14)


def test_dkv_worked_example_states_and_merge(golden_dir):
    g = _load(golden_dir, "dkv_worked_example.json")
    s = np.array([0.0, math.log(2), math.log(3), math.log(4)]).reshape(4, 1)
    V = np.array(g["values"], dtype=np.float64).reshape(4, 1)
    mA, lA, uA = oracle.segment_state([1.0], s[:2], V[:2], 1.0)
    mB, lB, uB = oracle.segment_state([1.0], s[2:], V[2:], 1.0)
    assert mA == pytest.approx(math.log(2), abs=1e-15)
    assert lA == pytest.approx(g["block_A"]["ell"], abs=1e-14)
    assert uA[0] == pytest.approx(g["block_A"]["u"], abs=1e-14)
    assert mB == pytest.approx(math.log(4), abs=1e-15)
    assert lB == pytest.approx(g["block_B"]["ell"], abs=1e-14)
    assert uB[0] == pytest.approx(g["block_B"]["u"], abs=1e-14)
    # local outputs u/ell are 5/3 and 44/7
    a, b = g["block_A"]["local_output_fraction"], g["block_B"]["local_output_fraction"]
    assert uA[0] / lA == pytest.approx(a[0] / a[1], abs=1e-14)
    assert uB[0] / lB == pytest.approx(b[0] / b[1], abs=1e-14)
    m, ell, u = oracle.merge([mA, mB], [lA, lB], np.stack([uA, uB]))
    assert m == pytest.approx(math.log(4), abs=1e-15)
    assert ell == pytest.approx(g["merged"]["ell"], abs=1e-14)
    assert u[0] == pytest.approx(g["merged"]["u"], abs=1e-14)
    o, lse = oracle.finalize(m, ell, u)
    assert o[0] == pytest.approx(g["merged"]["output"], abs=1e-14)
    assert lse == pytest.approx(math.log(10.0), abs=1e-14)
    # the naive average of local outputs is the wrong answer the page warns of
    naive = 0.5 * (a[0] / a[1] + b[0] / b[1])
    assert naive == pytest.approx(g["naive_average"], abs=1e-3)
    assert abs(naive - o[0]) > 0.9


def test_fd_merge_trap(golden_dir):
    g = _load(golden_dir, "fd_merge_trap.json")
    lse = np.array(g["lse"])
    o = np.array(g["o"])
    # a normalised state (o_i, lse_i) is the (m, ell, u) state (lse_i, 1, o_i)
    m, ell, u = oracle.merge(lse, np.ones(3), o)
    out, L = oracle.finalize(m, ell, u)
    # the page printed float32 values to 8 significant digits
    np.testing.assert_allclose(out, g["printed_stable_merge"], rtol=0, atol=1e-7)
    assert L == pytest.approx(g["printed_merged_lse"], abs=1e-5)
    # the printed weights are float32 shortest-repr strings (5-8 significant digits)
    w = np.exp(lse - m)
    np.testing.assert_allclose(w, g["printed_stable_weights"], rtol=0, atol=5e-8)


def test_merge_all_empty_and_some_empty():
    D = 3
    m, ell, u = oracle.merge([-np.inf, -np.inf], [0.0, 0.0], np.zeros((2, D)))
    assert m == -np.inf and ell == 0.0 and np.all(u == 0.0)
    o, lse = oracle.finalize(m, ell, u)
    assert lse == -np.inf and np.all(o == 0.0)
    # an empty state must not change a non-empty one (weight e^{-inf} = 0, no NaN)
    u1 = np.array([1.0, -2.0, 3.0])
    m2, l2, uu = oracle.merge([-np.inf, 0.7, -np.inf], [0.0, 2.0, 0.0],
                              np.stack([np.zeros(D), u1, np.zeros(D)]))
    assert m2 == 0.7 and l2 == 2.0 and np.array_equal(uu, u1)


# --------------------------------------------------------------------------
# attention against scipy (softmax / logsumexp) on tiny inputs
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(12))
def test_attend_matches_scipy(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 65))
    D = int(rng.integers(1, 9))
    gain = [1.0, 10.0, 60.0][seed % 3]
    q = rng.standard_normal(D) * gain
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    scale = 1.0 / math.sqrt(D)
    s = (K @ q) * scale
    want_o = scipy.special.softmax(s) @ V
    want_lse = scipy.special.logsumexp(s)
    o, lse = oracle.attend(q, K, V, scale)
    np.testing.assert_allclose(o, want_o, rtol=1e-12, atol=1e-13)
    assert lse == pytest.approx(want_lse, rel=1e-13, abs=1e-13)


def test_attend_closed_forms():
    rng = np.random.default_rng(7)
    D = 5
    # one key: output is that value, LSE is its score
    q, k, v = rng.standard_normal(D), rng.standard_normal((1, D)), rng.standard_normal((1, D))
    o, lse = oracle.attend(q, k, v, 0.5)
    np.testing.assert_allclose(o, v[0], rtol=0, atol=1e-15)
    assert lse == pytest.approx(0.5 * float(q @ k[0]), abs=1e-14)
    # q = 0: equal scores, output is the mean of V, LSE = log L
    L = 37
    V = rng.standard_normal((L, D))
    o, lse = oracle.attend(np.zeros(D), rng.standard_normal((L, D)), V, 1.0)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-13, atol=1e-14)
    assert lse == pytest.approx(math.log(L), abs=1e-14)
    # one dominant score (+80 against scores near 0): output is that value
    K = np.zeros((L, D))
    K[11, 0] = 80.0
    o, lse = oracle.attend(np.eye(D)[0], K, V, 1.0)
    np.testing.assert_allclose(o, V[11], rtol=0, atol=1e-30 + 1e-12)
    assert lse == pytest.approx(80.0 + math.log1p((L - 1) * math.exp(-80.0)), abs=1e-12)
    # empty key set: zero output, LSE = -inf
    o, lse = oracle.attend(np.ones(D), np.zeros((0, D)), np.zeros((0, D)), 1.0)
    assert lse == -np.inf and np.all(o == 0.0)


@pytest.mark.parametrize("seed", range(6))
def test_split_invariance(seed):
    """Attend over splits then merge (in any order, or as a tree) equals one pass
    ("Flash-Decoding ..." §2 claim and §3 check)."""
    rng = np.random.default_rng(100 + seed)
    L, D = 300, 6
    q = rng.standard_normal(D) * 4
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    scale = 1 / math.sqrt(D)
    o_full, lse_full = oracle.attend(q, K, V, scale)
    cuts = np.sort(rng.integers(0, L + 1, size=9))
    bounds = [0, *cuts.tolist(), L]                      # uneven, some empty
    states = [oracle.segment_state(q, K[a:b], V[a:b], scale) for a, b in zip(bounds[:-1], bounds[1:])]
    order = rng.permutation(len(states))
    m = [states[i][0] for i in order]
    ell = [states[i][1] for i in order]
    u = np.stack([states[i][2] for i in order])
    o, lse = oracle.finalize(*oracle.merge(m, ell, u))
    np.testing.assert_allclose(o, o_full, rtol=1e-12, atol=1e-13)
    assert lse == pytest.approx(lse_full, abs=1e-12)
    h = len(states) // 2
    left = oracle.merge(m[:h], ell[:h], u[:h])
    right = oracle.merge(m[h:], ell[h:], u[h:])
    tree = oracle.merge([left[0], right[0]], [left[1], right[1]], np.stack([left[2], right[2]]))
    o2, lse2 = oracle.finalize(*tree)
    np.testing.assert_allclose(o2, o_full, rtol=1e-12, atol=1e-13)
    assert lse2 == pytest.approx(lse_full, abs=1e-12)


# --------------------------------------------------------------------------
# batched decode: conversions, GQA map, strides, paging, lengths
# --------------------------------------------------------------------------
def _rand16(rng, shape, dtype):
    x = rng.standard_normal(shape).astype(np.float32)
    if dtype == "f16":
        return x.astype(np.float16)
    # bf16 by truncating the low half of the f32 pattern: any bf16 values do
    return ((x.view(np.uint32) >> 16).astype(np.uint16))


def _as_f64(a, dtype):
    if dtype == "f16":
        return a.astype(np.float64)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_rows_match_attend(dtype):
    rng = np.random.default_rng(3)
    B, Hq, Hkv, T, D = 2, 6, 3, 50, 16
    q = _rand16(rng, (B, Hq, D), dtype)
    k = _rand16(rng, (B, Hkv, T, D), dtype)
    v = _rand16(rng, (B, Hkv, T, D), dtype)
    seqlens = np.array([50, 17], dtype=np.int32)
    out, lse = oracle.decode(q, k, v, seqlens, dtype=dtype, n_kv_heads=Hkv)
    G = Hq // Hkv
    qd, kd, vd = _as_f64(q, dtype), _as_f64(k, dtype), _as_f64(v, dtype)
    for b in range(B):
        for h in range(Hq):
            L = seqlens[b]
            s = kd[b, h // G, :L] @ qd[b, h] / math.sqrt(D)
            want = scipy.special.softmax(s) @ vd[b, h // G, :L]
            np.testing.assert_allclose(out[b * Hq + h], want, rtol=1e-12, atol=1e-13)
            assert lse[b * Hq + h] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


def test_decode_gqa_head_map():
    """Query head h must read KV head h // G: give each KV head a constant V."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, T, D = 2, 8, 2, 9, 4
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, T, D)).astype(np.float16)
    consts = np.array([[1.5, -3.0], [0.25, 7.0]], dtype=np.float16)   # [b, kv head]
    v = np.broadcast_to(consts[:, :, None, None], (B, Hkv, T, D)).astype(np.float16).copy()
    out, _ = oracle.decode(q, k, v, [T, T], dtype="f16", n_kv_heads=Hkv)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(out[b * Hq + h], float(consts[b, h // 4]), rtol=1e-14)


def test_decode_strided_views_equal_contiguous():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, T, D = 2, 4, 2, 33, 8
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k_bthd = rng.standard_normal((B, T, Hkv, D)).astype(np.float16)   # token-major storage
    v_bthd = rng.standard_normal((B, T, Hkv, D)).astype(np.float16)
    k_view = k_bthd.transpose(0, 2, 1, 3)                             # [B, Hkv, T, D] view
    v_view = v_bthd.transpose(0, 2, 1, 3)
    sl = [33, 20]
    o1, l1 = oracle.decode(q, k_view, v_view, sl, dtype="f16", n_kv_heads=Hkv)
    o2, l2 = oracle.decode(q, np.ascontiguousarray(k_view), np.ascontiguousarray(v_view), sl,
                           dtype="f16", n_kv_heads=Hkv)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_decode_paged_equals_gathered(page_size):
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D = 3, 4, 2, 8
    sl = np.array([45, 1, 0], dtype=np.int32)
    max_pages = -(-45 // page_size)
    n_pages = B * max_pages + 5
    pool_k = rng.standard_normal((n_pages, Hkv, page_size, D)).astype(np.float16)
    pool_v = rng.standard_normal((n_pages, Hkv, page_size, D)).astype(np.float16)
    bt = rng.permutation(n_pages)[: B * max_pages].reshape(B, max_pages).astype(np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    # gather the logical cache with numpy fancy indexing: [B, max_pages, Hkv, ps, D]
    gk = pool_k[bt].transpose(0, 2, 1, 3, 4).reshape(B, Hkv, max_pages * page_size, D)
    gv = pool_v[bt].transpose(0, 2, 1, 3, 4).reshape(B, Hkv, max_pages * page_size, D)
    o1, l1 = oracle.decode(q, pool_k, pool_v, sl, dtype="f16", n_kv_heads=Hkv,
                           page_size=page_size, block_table=bt)
    o2, l2 = oracle.decode(q, gk, gv, sl, dtype="f16", n_kv_heads=Hkv)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # the empty sequence: zero output and LSE = -inf
    assert np.all(o1[2 * Hq:] == 0.0) and np.all(l1[2 * Hq:] == -np.inf)


def test_decode_ignores_tokens_past_length_and_rows_subset():
    rng = np.random.default_rng(8)
    B, Hq, Hkv, T, D = 2, 4, 4, 40, 8
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, T, D)).astype(np.float16)
    v = rng.standard_normal((B, Hkv, T, D)).astype(np.float16)
    sl = [25, 40]
    o1, l1 = oracle.decode(q, k, v, sl, dtype="f16", n_kv_heads=Hkv)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 25:] = np.float16(np.inf)
    v2[0, :, 25:] = np.float16(np.nan)
    o2, l2 = oracle.decode(q, k2, v2, sl, dtype="f16", n_kv_heads=Hkv)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    rows = [7, 0, 5]
    o3, l3 = oracle.decode(q, k, v, sl, dtype="f16", n_kv_heads=Hkv, rows=rows)
    assert np.array_equal(o3, o1[rows]) and np.array_equal(l3, l1[rows])


# --------------------------------------------------------------------------
# split-count heuristic: the pages' printed table and efficiency values
# --------------------------------------------------------------------------
def test_plan_table_132sm(golden_dir):
    g = _load(golden_dir, "fd_split_table_132sm.json")
    for batch, heads, ctx, work, splits, ctas in g["rows"]:
        assert batch * heads == work
        nb = -(-ctx // g["block_n"])
        assert oracle.plan(work, g["slots"], nb, g["max_splits"]) == splits
        assert oracle.num_splits_ref(work, g["slots"], nb, g["max_splits"]) == splits
        assert work * splits == ctas


def test_plan_efficiency_comment(golden_dir):
    g = _load(golden_dir, "fa3_efficiency_comment.json")
    for s, e in g["efficiency_printed_2dp"].items():
        assert round(oracle.efficiency_ref(g["work_items"], g["slots"], int(s)), 2) == e
    # C statement reports the same efficiencies for eligible counts
    _, eff = oracle.plan(g["work_items"], g["slots"], 1000, 128, return_eff=True)
    assert round(eff[2], 2) == 0.89 and round(eff[3], 2) == 0.67


def test_plan_edge_cases():
    assert oracle.plan(8, 264, 0) == 1                 # no KV blocks
    assert oracle.num_splits_ref(8, 264, 0) == 1
    assert oracle.plan(212, 264, 5000) == 1            # work >= 0.8 * slots
    assert oracle.plan(1, 264, 1) == 1                 # one block cannot split


def test_plan_c_and_python_statements_agree():
    rng = np.random.default_rng(11)
    for slots in (216, 264, 296, 304):
        for work in list(range(1, 70)) + [96, 128, 200, 240, 300]:
            for nb in (0, 1, 2, 3, 7, 8, 31, 32, 33, 63, 64, 100, 127, 128, 129, 250,
                       256, 257, 1000, 1024, 2048, 2100, 4096):
                assert oracle.plan(work, slots, nb) == oracle.num_splits_ref(work, slots, nb), \
                    (work, slots, nb)
    for _ in range(3000):
        work = int(rng.integers(1, 400))
        slots = int(rng.integers(8, 400))
        nb = int(rng.integers(0, 2200))
        ms = int(rng.integers(1, 160))
        assert oracle.plan(work, slots, nb, ms) == oracle.num_splits_ref(work, slots, nb, ms)


# --------------------------------------------------------------------------
# short query blocks: position i of q_len sees the first L - q_len + 1 + i keys
# --------------------------------------------------------------------------
@pytest.mark.parametrize("q_len", [2, 4, 8])
def test_query_block_reduces_to_single_queries_on_prefixes(q_len):
    rng = np.random.default_rng(40 + q_len)
    B, Hq, Hkv, T, D = 3, 8, 2, 70, 16
    q = rng.standard_normal((B, q_len, Hq, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, T, D)).astype(np.float16)
    v = rng.standard_normal((B, Hkv, T, D)).astype(np.float16)
    sl = np.array([70, 9, 3], dtype=np.int32)
    out, lse = oracle.decode(q, k, v, sl, dtype="f16", n_kv_heads=Hkv)
    out = out.reshape(B, q_len, Hq, D)
    lse = lse.reshape(B, q_len, Hq)
    for i in range(q_len):
        prefix = np.maximum(sl - q_len + 1 + i, 0).astype(np.int32)
        o1, l1 = oracle.decode(np.ascontiguousarray(q[:, i]), k, v, prefix, dtype="f16", n_kv_heads=Hkv)
        assert np.array_equal(out[:, i].reshape(-1, D), o1)
        assert np.array_equal(lse[:, i].reshape(-1), l1)
    # sequence 2 holds 3 tokens: with q_len > 3 its first positions see nothing
    for i in range(q_len):
        if 3 - q_len + 1 + i <= 0:
            assert np.all(out[2, i] == 0.0) and np.all(np.isneginf(lse[2, i]))


def test_query_block_against_scipy():
    rng = np.random.default_rng(77)
    q_len, Hq, D, L = 4, 2, 8, 11
    q = rng.standard_normal((1, q_len, Hq, D)).astype(np.float16)
    k = rng.standard_normal((1, 1, L, D)).astype(np.float16)
    v = rng.standard_normal((1, 1, L, D)).astype(np.float16)
    out, lse = oracle.decode(q, k, v, [L], dtype="f16", n_kv_heads=1)
    kd, vd, qd = k[0, 0].astype(np.float64), v[0, 0].astype(np.float64), q[0].astype(np.float64)
    for i in range(q_len):
        n = L - q_len + 1 + i
        for h in range(Hq):
            s = kd[:n] @ qd[i, h] / math.sqrt(D)
            r = i * Hq + h
            np.testing.assert_allclose(out[r], scipy.special.softmax(s) @ vd[:n], rtol=1e-12, atol=1e-13)
            assert lse[r] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


# --------------------------------------------------------------------------
# fp8 e4m3 caches with one scale per tensor
# --------------------------------------------------------------------------
def test_e4m3_conversion_all_patterns():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    bits = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = bits.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(b)) for b in range(256)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], want[~nan])
    assert np.nanmax(got) == 448.0


def test_e4m3_conversion_closed_form():
    """The E4M3 'fn' definition written out: sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 is subnormal (2^-6 x m/8); S.1111.111
    is NaN and there are no infinities, so S.1111.110 = 448 is the largest."""
    for b in range(256):
        sgn = -1.0 if b & 0x80 else 1.0
        e, m = (b >> 3) & 0xF, b & 0x7
        got = oracle.e4m3_to_double(b)
        if e == 0xF and m == 0x7:
            assert math.isnan(got), b
            continue
        want = sgn * (2.0 ** -6) * (m / 8.0) if e == 0 else sgn * 2.0 ** (e - 7) * (1.0 + m / 8.0)
        assert got == want, (b, got, want)
    assert oracle.e4m3_to_double(0x7E) == 448.0 and oracle.e4m3_to_double(0x01) == 2.0 ** -9


def test_e4m3_cache_with_scales_against_scipy():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(91)
    B, Hq, Hkv, T, D = 2, 4, 2, 40, 16
    ks, vs = 0.037, 2.5
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k8 = torch.from_numpy(rng.standard_normal((B, Hkv, T, D)) * 20).to(torch.float8_e4m3fn)
    v8 = torch.from_numpy(rng.standard_normal((B, Hkv, T, D))).to(torch.float8_e4m3fn)
    sl = np.array([40, 13], dtype=np.int32)
    out, lse = oracle.decode(q, k8, v8, sl, dtype="f16", n_kv_heads=Hkv, kv_dtype="e4m3",
                             k_scale=ks, v_scale=vs)
    kd = k8.to(torch.float64).numpy() * ks
    vd = v8.to(torch.float64).numpy() * vs
    qd = q.astype(np.float64)
    for b in range(B):
        for h in range(Hq):
            L = sl[b]
            s = kd[b, h // 2, :L] @ qd[b, h] / math.sqrt(D)
            np.testing.assert_allclose(out[b * Hq + h], scipy.special.softmax(s) @ vd[b, h // 2, :L],
                                       rtol=1e-12, atol=1e-13)
            assert lse[b * Hq + h] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)
