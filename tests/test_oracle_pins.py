"""Pins of the CPU oracle against values fixed by the pages and by mathematics.

Each test checks an oracle function against something other than itself:
hand-worked cases (tests/golden), closed forms, brute-force enumeration,
invariants, exhaustive nearest-value search, or a library routine the step
reduces to in a special case. CPU only.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# FP8 e4m3
# ---------------------------------------------------------------------------
def e4m3_value_from_format(code: int) -> float:
    """OCP e4m3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent
    field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_decode_matches_format_and_torch():
    table = oracle.e4m3_decode_table()
    ref = np.array([e4m3_value_from_format(c) for c in range(256)])
    assert np.array_equal(np.isnan(table), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(table[ok], ref[ok])
    # library cross-check: torch's float8_e4m3fn decoding of every code
    tq = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(tq), np.isnan(ref))
    assert np.array_equal(tq[ok], ref[ok])
    assert table[0x7E] == 448.0 and table[0x01] == 2.0 ** -9 and table[0x08] == 2.0 ** -6


def _nearest_even_reference(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code by search over the sorted positive code values,
    ties to the even code, saturation at 448, sign carried separately."""
    pos_codes = np.arange(0, 0x7F)  # 0x00..0x7E: finite, increasing values
    pos_vals = np.array([e4m3_value_from_format(int(c)) for c in pos_codes])
    a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << 7
    hi = np.searchsorted(pos_vals, a, side="left")  # first value >= a
    hi = np.clip(hi, 0, len(pos_vals) - 1)
    lo = np.clip(hi - 1, 0, None)
    d_hi = pos_vals[hi] - a
    d_lo = a - pos_vals[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (pos_codes[lo] % 2 == 0))
    exact = pos_vals[hi] == a
    code = np.where(exact, pos_codes[hi], np.where(pick_lo, pos_codes[lo], pos_codes[hi]))
    code = np.where(a >= 448.0, 0x7E, code)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def test_e4m3_encode_exhaustive_nearest_even():
    # every fp32 bit pattern with magnitude in [2^-12, 2^9] (everything below
    # rounds to zero, everything above saturates), both signs, in chunks
    lo_bits = np.float32(2.0 ** -12).view(np.uint32)
    hi_bits = np.float32(2.0 ** 9).view(np.uint32)
    step = 1 << 22
    for start in range(int(lo_bits), int(hi_bits) + 1, step):
        bits = np.arange(start, min(start + step, int(hi_bits) + 1), dtype=np.uint32)
        x = bits.view(np.float32)
        for xs in (x, -x):
            got = oracle.e4m3_encode(xs)
            ref = _nearest_even_reference(xs)
            bad = np.nonzero(got != ref)[0]
            assert bad.size == 0, (xs[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_specials_and_torch():
    x = np.array([0.0, -0.0, 1e-30, -1e-30, 448.0, 449.0, 463.99, 464.0, 1e6, -1e6,
                  2.0 ** -10, 2.0 ** -10 * 1.0000001, 3 * 2.0 ** -10], np.float32)
    q = oracle.e4m3_encode(x)
    assert list(q) == [0x00, 0x80, 0x00, 0x80, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE,
                       0x00, 0x01, 0x02]
    # torch's e4m3fn cast is round-to-nearest-even without saturation: agree
    # on every finite value inside the range
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(200_000) * rng.choice([1e-3, 1e-1, 1, 30, 300], 200_000)).astype(np.float32)
    v = np.clip(v, -448, 448)
    tq = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), tq)


# ---------------------------------------------------------------------------
# fp32 exp / sigmoid
# ---------------------------------------------------------------------------
def _ulp32(x):
    x = np.abs(x.astype(np.float32))
    return (np.nextafter(x, np.float32(np.inf)) - x).astype(np.float64)


def test_exp32_within_two_ulp():
    x = np.concatenate([np.linspace(-87.0, 88.5, 2_000_003, dtype=np.float32),
                        np.linspace(-1, 1, 1_000_001, dtype=np.float32)])
    y = oracle.exp32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    err = np.abs(y - ref) / _ulp32(ref.astype(np.float32))
    assert err.max() <= 2.0, err.max()
    assert oracle.exp32(np.array([0.0], np.float32))[0] == 1.0
    assert np.isinf(oracle.exp32(np.array([89.0], np.float32))[0])
    assert oracle.exp32(np.array([-110.0], np.float32))[0] == 0.0


def test_sigmoid32_within_three_ulp():
    x = np.linspace(-30, 30, 1_000_001, dtype=np.float32)
    y = oracle.sigmoid32(x).astype(np.float64)
    xd = x.astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-xd))
    err = np.abs(y - ref) / _ulp32(ref.astype(np.float32))
    assert err.max() <= 3.0, err.max()
    assert oracle.sigmoid32(np.array([0.0], np.float32))[0] == 0.5


# ---------------------------------------------------------------------------
# Gate
# ---------------------------------------------------------------------------
def _load_gate_cases():
    with open(os.path.join(GOLDEN, "gate_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_gate_cases(), ids=lambda c: c["name"])
def test_gate_handworked(case):
    scoring = oracle.SIGMOID if case["scoring"] == "sigmoid" else oracle.SOFTMAX
    logits = np.array(case["logits"], np.float32)
    bias = None if case["bias"] is None else np.array(case["bias"], np.float32)
    ids, w = oracle.gate(logits, bias, case["num_groups"], case["topk_group"], case["top_k"],
                         scoring, case["renormalize"], case["rsf"])
    assert ids.tolist() == case["ids"]
    tol = case.get("w_tol_rel", 0.0)
    np.testing.assert_allclose(w, np.array(case["w"]), rtol=tol, atol=0)


def _gate_problem(rng, T, E, G, scale_bias=0.3):
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * scale_bias).astype(np.float32)
    # plant exact ties: copy some logits within rows
    logits[:, 1] = logits[:, 0]
    return logits, bias


def _check_selection(keys, gsz, TG, K, ids):
    """Brute force: the kept groups are a best TG-subset of all C(G, TG) subsets
    under (score desc, index asc); the picks are the K best keys of the kept
    groups under (key desc, index asc), in that order."""
    E = keys.size
    G = E // gsz
    gscore = []
    for g in range(G):
        v = np.sort(keys[g * gsz:(g + 1) * gsz])[::-1]
        gscore.append(np.float32(v[0] + v[1]) if gsz >= 2 else v[0])
    rank = sorted(range(G), key=lambda g: (-float(gscore[g]), g))
    best = None
    for sub in itertools.combinations(range(G), TG):
        key = sorted((rank.index(g) for g in sub))
        if best is None or key < best[0]:
            best = (key, set(sub))
    kept = best[1]
    allowed = [e for e in range(E) if e // gsz in kept]
    want = sorted(allowed, key=lambda e: (-float(keys[e]), e))[:K]
    assert list(ids) == want


@pytest.mark.parametrize("E,G,TG,K", [(8, 4, 2, 2), (16, 4, 2, 3), (12, 3, 2, 4), (16, 8, 3, 5),
                                      (16, 16, 4, 4), (16, 2, 1, 8), (6, 1, 1, 3)])
def test_gate_bruteforce_enumeration(E, G, TG, K):
    rng = np.random.default_rng(E * 100 + G * 10 + K)
    T = 200
    logits, bias = _gate_problem(rng, T, E, G)
    ids, w = oracle.gate(logits, bias, G, TG, K, oracle.SIGMOID, True, 2.5)
    s = oracle.sigmoid32(logits)
    keys = (s + bias[None, :]).astype(np.float32)  # fp32 add, as the gate does
    for t in range(T):
        _check_selection(keys[t], E // G, TG, K, ids[t])


def test_gate_weight_sum_is_rsf_and_linear():
    rng = np.random.default_rng(7)
    logits, bias = _gate_problem(rng, 500, 64, 8)
    for rsf in (1.0, 2.5):
        ids, w = oracle.gate(logits, bias, 8, 4, 8, oracle.SIGMOID, True, rsf)
        ulp = float(np.spacing(np.float32(rsf)))
        assert np.abs(w.astype(np.float64).sum(1) - rsf).max() <= 8 * ulp
        # all ids distinct within a token
        assert all(len(set(r)) == 8 for r in ids.tolist())
    ids1, w1 = oracle.gate(logits, bias, 8, 4, 8, oracle.SIGMOID, True, 1.0)
    ids2, w2 = oracle.gate(logits, bias, 8, 4, 8, oracle.SIGMOID, True, 2.0)
    assert np.array_equal(ids1, ids2)
    assert np.array_equal(w2, w1 * 2)  # scaling by 2 is exact
    # softmax: closed form for K=2 (renormalised pair)
    lg = rng.standard_normal((300, 8)).astype(np.float32)
    ids, w = oracle.gate(lg, None, 1, 1, 2, oracle.SOFTMAX, True, 1.0)
    top = np.argsort(-lg, axis=1, kind="stable")[:, :2]
    assert np.array_equal(ids, top)
    l0 = np.take_along_axis(lg, top[:, :1], 1)[:, 0].astype(np.float64)
    l1 = np.take_along_axis(lg, top[:, 1:2], 1)[:, 0].astype(np.float64)
    np.testing.assert_allclose(w[:, 0], 1.0 / (1.0 + np.exp(l1 - l0)), rtol=1e-6)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-6)


def test_gate_no_renormalise():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((50, 16)).astype(np.float32)
    ids, w = oracle.gate(lg, None, 1, 1, 4, oracle.SIGMOID, False, 2.5)
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(lg, ids, 1).astype(np.float64)))
    np.testing.assert_allclose(w, s * 2.5, rtol=1e-6)
    ids, w = oracle.gate(lg, None, 1, 1, 4, oracle.SOFTMAX, False, 1.0)
    p = np.exp(lg - lg.max(1, keepdims=True))
    p = p / p.sum(1, keepdims=True)
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-6)


def test_gate_rejects_bad_arguments():
    lg = np.zeros((2, 8), np.float32)
    for args in [(3, 1, 2), (4, 5, 2), (4, 2, 5), (4, 0, 1)]:
        with pytest.raises(ValueError):
            oracle.gate(lg, None, *args, oracle.SIGMOID, True, 1.0)
    with pytest.raises(ValueError):  # softmax takes no correction bias
        oracle.gate(lg, np.zeros(8, np.float32), 1, 1, 2, oracle.SOFTMAX, True, 1.0)


# ---------------------------------------------------------------------------
# Routing / pre-reorder
# ---------------------------------------------------------------------------
def _ids(rng, T, E, K, skew=False):
    if skew:
        p = np.zeros(E)
        p[: max(K, E // 4)] = 1.0
        p /= p.sum()
        return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,K,skew", [(37, 8, 2, False), (300, 64, 8, True), (1, 4, 4, False),
                                        (0, 8, 2, False)])
def test_route_invariants(T, E, K, skew):
    rng = np.random.default_rng(T + E)
    ids = _ids(rng, T, E, K, skew) if T else np.zeros((0, K), np.int32)
    off, s2d = oracle.route(ids, E)
    hist = np.bincount(ids.ravel(), minlength=E)
    assert off[0] == 0 and np.array_equal(np.diff(off), hist)
    assert np.array_equal(np.sort(s2d), np.arange(T * K))  # bijection onto [0, M)
    flat = ids.ravel()
    for e in range(E):
        seg = np.nonzero(flat == e)[0]  # flattened (t,k) indices, ascending
        dst = s2d[seg]
        assert np.array_equal(dst, np.arange(off[e], off[e + 1]))  # in segment, ascending t


def test_permute_then_unpermute_is_identity():
    rng = np.random.default_rng(11)
    T, H, E, K = 50, 64, 16, 4
    ids = _ids(rng, T, E, K)
    x = rng.standard_normal((T, H))
    off, s2d = oracle.route(ids, E)
    perm = np.zeros((T * K, H))
    perm[s2d] = np.repeat(x, K, axis=0)
    w = np.zeros((T, K), np.float32)
    w[:, 0] = 1.0
    out = oracle.unpermute_sum(perm, s2d, w)
    assert np.array_equal(out, x)
    # and with weights: sum of K equal rows times weights
    w = rng.random((T, K)).astype(np.float32)
    out = oracle.unpermute_sum(perm, s2d, w)
    np.testing.assert_allclose(out, x * w.astype(np.float64).sum(1, keepdims=True), rtol=1e-12)


def _bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_row_quant_closed_form():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((40, 96)) * (10.0 ** rng.uniform(-3, 3, (40, 1)))
    x[3] = 0.0  # an all-zero row
    xb = _bf16_bits(x)
    xv = oracle.bf16_to_f64(xb)
    q, s = oracle.row_quant(xb)
    amax = np.abs(xv).max(1).astype(np.float32)
    exp_s = (np.maximum(amax, np.float32(1e-10)) / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(s, exp_s)
    dec = oracle.e4m3_decode(q)
    # each code is the nearest-even e4m3 of x / scale (pinned above), so
    # |dec - x/s| <= half an e4m3 step: relative 2^-4 for normal values
    r = xv / s[:, None].astype(np.float64)
    assert np.all(np.abs(dec - r) <= np.maximum(np.abs(r) * 2.0 ** -4, 2.0 ** -10) + 1e-12)
    # the row maximum lands on +-448 (code 0x7E / 0xFE)
    nz = amax > 0
    am = np.argmax(np.abs(xv), 1)
    assert np.all(np.abs(dec[np.arange(40), am])[nz] == 448.0)
    assert np.all(q[3] == 0)


def test_permute_quant_scatter():
    rng = np.random.default_rng(9)
    T, H, E, K = 33, 64, 8, 2
    ids = _ids(rng, T, E, K)
    xb = _bf16_bits(rng.standard_normal((T, H)))
    a_q, sa, s2d, off = oracle.permute_quant(xb, ids, E)
    q, s = oracle.row_quant(xb)
    off2, s2d2 = oracle.route(ids, E)
    assert np.array_equal(off, off2) and np.array_equal(s2d, s2d2)
    for t in range(T):
        for k in range(K):
            d = s2d[t * K + k]
            assert np.array_equal(a_q[d], q[t]) and sa[d] == s[t]


# ---------------------------------------------------------------------------
# Grouped GEMM
# ---------------------------------------------------------------------------
def _codes_of(vals):
    """e4m3 codes of exactly representable values."""
    return oracle.e4m3_encode(np.asarray(vals, np.float32))


def test_grouped_gemm_exact_integers():
    rng = np.random.default_rng(1)
    E, N, Kd = 3, 24, 64
    counts = [5, 0, 9]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    Av = rng.integers(-4, 5, (M, Kd)).astype(np.float32)
    Bv = rng.integers(-3, 4, (E, N, Kd)).astype(np.float32)
    A, B = _codes_of(Av), _codes_of(Bv)
    C = oracle.grouped_gemm(A, np.ones(M, np.float32), B, np.ones((E, N), np.float32), off)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        ref = Av[r0:r1].astype(np.int64) @ Bv[e].astype(np.int64).T
        assert np.array_equal(C[r0:r1], ref.astype(np.float64))


def test_grouped_gemm_scales_per_row_and_channel():
    """scale_a applies per ROW of the permuted activations, not per expert
    (the bug fixed in sglang #6772 indexed it by expert id)."""
    rng = np.random.default_rng(2)
    E, N, Kd = 2, 16, 32
    off = np.array([0, 4, 10], np.int32)
    M = 10
    A = rng.integers(0, 256, (M, Kd)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0  # no NaN codes
    B = rng.integers(0, 256, (E, N, Kd)).astype(np.uint8)
    B[(B & 0x7F) == 0x7F] = 0
    sa = (10.0 ** rng.uniform(-3, 3, M)).astype(np.float32)
    sb = rng.uniform(0.5, 2, (E, N)).astype(np.float32)
    C = oracle.grouped_gemm(A, sa, B, sb, off)
    Ad = oracle.e4m3_decode(A)
    Bd = oracle.e4m3_decode(B)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        ref = (Ad[r0:r1] @ Bd[e].T) * sa[r0:r1, None].astype(np.float64) * sb[e][None, :].astype(np.float64)
        np.testing.assert_allclose(C[r0:r1], ref, rtol=1e-13, atol=1e-300)
    # a per-expert scale (first row's scale for the whole segment) differs
    wrong = (Ad[4:10] @ Bd[1].T) * np.float64(sa[4]) * sb[1][None, :].astype(np.float64)
    assert not np.allclose(C[4:10], wrong, rtol=1e-3)


def test_silu_mul_closed_forms():
    from scipy.special import expit
    g = np.array([0.0, 30.0, -30.0, 1.0, -2.5, 100.0])
    u = np.array([1.0, 2.0, 3.0, -1.0, 0.5, 1.0])
    C = np.concatenate([g, u])[None, :]
    h = oracle.silu_mul(C)[0]
    assert h[0] == 0.0
    np.testing.assert_allclose(h[1], 60.0, rtol=1e-12)
    np.testing.assert_allclose(h[5], 100.0, rtol=1e-15)
    np.testing.assert_allclose(h, g * expit(g) * u, rtol=1e-14)


def test_bf16_round_single_rounding():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 2 ** -8 + 2 ** -40, 1.0 + 3 * 2 ** -8, -1.5,
                  1.0 + 2 ** -8 - 2 ** -40, 3.0e38, 0.0])
    got = oracle.bf16_round(v)
    # torch rounds fp32 -> bf16 correctly; build the expected values from
    # the cases where fp64 -> fp32 is exact, and the tie-breaking ones by hand
    assert got[0] == 0x3F80
    assert got[1] == 0x3F80          # exact tie -> even
    assert got[2] == 0x3F81          # above the tie -> up (double rounding would give even)
    assert got[3] == 0x3F82          # tie -> even (up)
    assert got[4] == 0xBFC0
    assert got[5] == 0x3F80          # below the tie -> down
    assert got[7] == 0x0000
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100_000).astype(np.float32)
    tb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(x.astype(np.float64)), tb)


# ---------------------------------------------------------------------------
# Whole layer
# ---------------------------------------------------------------------------
def _random_layer(rng, T, H, I, E):
    from moe_expert_layer_grouped_gb300 import synth
    x = _bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w13, s13 = synth.quantize_weight_rows(torch.from_numpy(rng.standard_normal((E, 2 * I, H)) * 0.02).float())
    w2, s2 = synth.quantize_weight_rows(torch.from_numpy(rng.standard_normal((E, H, I)) * 0.02).float())
    return x, logits, w13.numpy(), s13.numpy(), w2.numpy(), s2.numpy()


def _dense_fp8_mlp(x, w13e, s13e, w2e, s2e):
    """One expert applied to every token, with numpy matmuls: per-token FP8
    input, w13 with both scales, silu(gate)*up rounded to bf16, per-token
    requantisation, w2 with both scales."""
    I = w2e.shape[1]
    q, sa = oracle.row_quant(x)
    C = (oracle.e4m3_decode(q) @ oracle.e4m3_decode(w13e).T) * sa[:, None].astype(np.float64) \
        * s13e[None, :].astype(np.float64)
    g, u = C[:, :I], C[:, I:]
    h = g / (1 + np.exp(-g)) * u
    hb = oracle.bf16_round(h)
    q2, sa2 = oracle.row_quant(hb)
    return (oracle.e4m3_decode(q2) @ oracle.e4m3_decode(w2e).T) * sa2[:, None].astype(np.float64) \
        * s2e[None, :].astype(np.float64)


def test_layer_single_expert_is_dense_fp8_mlp():
    """E=1, K=1, rsf=1: routing is the identity and the layer is a dense FP8
    MLP, computed here with numpy matmuls."""
    rng = np.random.default_rng(4)
    T, H, I = 6, 64, 32
    x, logits, w13, s13, w2, s2 = _random_layer(rng, T, H, I, 1)
    out, ids, w = oracle.forward_tokens(x, logits, None, w13, s13, w2, s2, 1, 1, 1,
                                        oracle.SOFTMAX, True, 1.0)
    assert np.all(ids == 0) and np.all(w == 1.0)
    ref = _dense_fp8_mlp(x, w13[0], s13[0], w2[0], s2[0])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("n_shared", [1, 2])
def test_layer_shared_experts_add_dense_mlps(n_shared):
    """Shared experts (stored after the E routed ones) add each one's dense
    FP8 MLP with weight 1, whatever routed_scaling_factor is: the layer with
    them minus the layer without them is the sum of those MLPs (numpy)."""
    rng = np.random.default_rng(40 + n_shared)
    T, H, I, E = 12, 64, 32, 8
    x, logits, w13, s13, w2, s2 = _random_layer(rng, T, H, I, E + n_shared)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    args = (4, 2, 3, oracle.SIGMOID, True, 2.5)
    base, ids0, w0 = oracle.forward_tokens(x, logits[:, :E], bias, w13[:E], s13[:E], w2[:E],
                                           s2[:E], *args)
    out, ids, w = oracle.forward_tokens(x, logits[:, :E], bias, w13, s13, w2, s2, *args,
                                        n_shared=n_shared)
    assert np.array_equal(ids, ids0) and np.array_equal(w, w0)  # the gate sees E experts
    ref = sum(_dense_fp8_mlp(x, w13[E + j], s13[E + j], w2[E + j], s2[E + j])
              for j in range(n_shared))
    np.testing.assert_allclose(out - base, ref, rtol=1e-9, atol=1e-12 * np.abs(out).max())
    # the step-by-step path (shared experts as extra slots of every token) agrees
    steps = oracle.forward_steps(x, logits[:, :E], bias, w13, s13, w2, s2, *args,
                                 n_shared=n_shared)
    assert np.array_equal(steps["ids"][:, 3:], np.tile(np.arange(E, E + n_shared), (T, 1)))
    assert np.all(steps["w"][:, 3:] == 1.0)
    np.testing.assert_allclose(out, steps["out"], rtol=1e-12, atol=1e-12 * np.abs(out).max())


def test_layer_token_path_equals_step_path_and_is_linear_in_rsf():
    rng = np.random.default_rng(6)
    T, H, I, E = 24, 64, 32, 8
    x, logits, w13, s13, w2, s2 = _random_layer(rng, T, H, I, E)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    steps = oracle.forward_steps(x, logits, bias, w13, s13, w2, s2, 4, 2, 3, oracle.SIGMOID,
                                 True, 2.5)
    out, ids, w = oracle.forward_tokens(x, logits, bias, w13, s13, w2, s2, 4, 2, 3,
                                        oracle.SIGMOID, True, 2.5)
    assert np.array_equal(ids, steps["ids"]) and np.array_equal(w, steps["w"])
    np.testing.assert_allclose(out, steps["out"], rtol=1e-12, atol=1e-12 * np.abs(out).max())
    out1, _, _ = oracle.forward_tokens(x, logits, bias, w13, s13, w2, s2, 4, 2, 3,
                                       oracle.SIGMOID, True, 1.25)
    np.testing.assert_allclose(out, 2 * out1, rtol=1e-6, atol=1e-9)
    # a subset of tokens gives the same rows
    sub = np.array([5, 0, 23], np.int64)
    outs, _, _ = oracle.forward_tokens(x, logits, bias, w13, s13, w2, s2, 4, 2, 3,
                                       oracle.SIGMOID, True, 2.5, tokens=sub)
    assert np.array_equal(outs, out[sub])


# ---------------------------------------------------------------------------
# Block-quantised FP8 (128-channel activation blocks, 128 x 128 weight blocks)
# ---------------------------------------------------------------------------
def test_block_quant_is_row_quant_per_block():
    """Each 128-block of a row is quantised exactly as a row of its own by
    the (exhaustively pinned) per-token rule; a block's scale depends only on
    that block (scaling one block by 4 scales only its scale)."""
    rng = np.random.default_rng(50)
    R, nb = 9, 5
    x = rng.standard_normal((R, nb * 128)) * (10.0 ** rng.uniform(-3, 3, (R, nb)))[:, :, None].repeat(128, 2).reshape(R, -1)
    xb = _bf16_bits(x)
    q, s = oracle.block_quant(xb)
    q1, s1 = oracle.row_quant(xb.reshape(R * nb, 128))
    assert np.array_equal(q.reshape(R * nb, 128), q1)
    assert np.array_equal(s.reshape(-1).view(np.uint32), s1.view(np.uint32))
    x2 = x.copy()
    x2[:, 128:256] *= 4.0
    q2, s2 = oracle.block_quant(_bf16_bits(x2))
    assert np.array_equal(q2, q)
    assert np.array_equal(s2[:, 1], s[:, 1] * 4) and np.array_equal(s2[:, [0, 2, 3, 4]], s[:, [0, 2, 3, 4]])


def test_grouped_gemm_block_exact_with_power_of_two_scales():
    """Small integer codes and power-of-two block scales: every term is exact,
    so the result equals sum over K blocks of 2^(u+v) x (integer block dot
    product), computed here with numpy integer matmuls per block. A swapped
    or transposed scale index changes the powers and fails."""
    rng = np.random.default_rng(51)
    counts, N, Kd = [70, 0, 33], 384, 512
    E, KB, NB = len(counts), Kd // 128, N // 128
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    Ai = rng.integers(-3, 4, (M, Kd))
    Bi = rng.integers(-2, 3, (E, N, Kd))
    A = _codes_of(Ai.astype(np.float32))
    B = _codes_of(Bi.astype(np.float32))
    u = rng.integers(-6, 7, (M, KB))
    v = rng.integers(-6, 7, (E, NB, KB))
    C = oracle.grouped_gemm_block(A, (2.0 ** u).astype(np.float32), B,
                                  (2.0 ** v).astype(np.float32), off)
    ref = np.zeros((M, N))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        for kb in range(KB):
            ks = slice(kb * 128, (kb + 1) * 128)
            part = Ai[rows, ks] @ Bi[e, :, ks].T                       # exact integers
            ref[rows] += part * 2.0 ** (u[rows, kb][:, None] + np.repeat(v[e, :, kb], 128)[None, :])
    assert np.array_equal(C, ref)


def test_grouped_gemm_block_with_uniform_scales_is_per_token_gemm():
    """Scales constant along K (one per row, one per 128-row weight block)
    reduce block FP8 to the per-row x per-channel GEMM."""
    rng = np.random.default_rng(52)
    counts, N, Kd = [40, 17], 256, 384
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    A = _codes_of(rng.standard_normal((M, Kd)).astype(np.float32))
    B = _codes_of(rng.standard_normal((E, N, Kd)).astype(np.float32))
    ra = (10.0 ** rng.uniform(-2, 1, M)).astype(np.float32)
    rb = (10.0 ** rng.uniform(-3, -1, (E, N // 128))).astype(np.float32)
    C = oracle.grouped_gemm_block(A, np.repeat(ra[:, None], Kd // 128, 1), B,
                                  np.repeat(rb[:, :, None], Kd // 128, 2), off)
    ref = oracle.grouped_gemm(A, ra, B, np.repeat(rb, 128, 1), off)
    np.testing.assert_allclose(C, ref, rtol=1e-12, atol=0)


def _random_block_layer(rng, T, H, I, E):
    from moe_expert_layer_grouped_gb300 import synth
    x = _bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w13, s13 = synth.quantize_weight_blocks(
        torch.from_numpy(rng.standard_normal((E, 2 * I, H)) * 0.02).float())
    w2, s2 = synth.quantize_weight_blocks(
        torch.from_numpy(rng.standard_normal((E, H, I)) * 0.02).float())
    return x, logits, w13.numpy(), s13.numpy(), w2.numpy(), s2.numpy()


def _dense_block_mlp(x, w13e, s13e, w2e, s2e):
    """One expert on every token in block FP8 with numpy: dequantise the
    codes block by block, multiply in fp64."""
    I = w2e.shape[1]

    def deq_act(bits):
        q, s = oracle.block_quant(bits)
        return oracle.e4m3_decode(q) * np.repeat(s.astype(np.float64), 128, 1)

    def deq_w(q, s):
        return oracle.e4m3_decode(q) * np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)

    C = deq_act(x) @ deq_w(w13e, s13e).T
    g, u = C[:, :I], C[:, I:]
    hb = oracle.bf16_round(g / (1 + np.exp(-g)) * u)
    return deq_act(hb) @ deq_w(w2e, s2e).T


def test_layer_block_single_expert_is_dense_block_mlp():
    # H and I both span two 128-channel blocks, so a scale carried from one
    # block to the next (activations, h or weights) changes the result
    rng = np.random.default_rng(53)
    T, H, I = 6, 256, 256
    x, logits, w13, s13, w2, s2 = _random_block_layer(rng, T, H, I, 1)
    out, ids, w = oracle.forward_tokens_block(x, logits, None, w13, s13, w2, s2, 1, 1, 1,
                                              oracle.SOFTMAX, True, 1.0)
    assert np.all(ids == 0) and np.all(w == 1.0)
    ref = _dense_block_mlp(x, w13[0], s13[0], w2[0], s2[0])
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def test_layer_block_token_path_equals_step_path_with_shared_expert():
    rng = np.random.default_rng(54)
    T, H, I, E, S = 20, 256, 256, 8, 1
    x, logits, w13, s13, w2, s2 = _random_block_layer(rng, T, H, I, E + S)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    args = (4, 2, 3, oracle.SIGMOID, True, 2.5)
    steps = oracle.forward_steps_block(x, logits[:, :E], bias, w13, s13, w2, s2, *args,
                                       n_shared=S)
    out, ids, w = oracle.forward_tokens_block(x, logits[:, :E], bias, w13, s13, w2, s2, *args,
                                              n_shared=S)
    assert np.array_equal(ids, steps["ids"][:, :3]) and np.array_equal(w, steps["w"][:, :3])
    np.testing.assert_allclose(out, steps["out"], rtol=1e-12, atol=1e-12 * np.abs(out).max())
    # the shared expert adds its dense block MLP with weight 1
    base, _, _ = oracle.forward_tokens_block(x, logits[:, :E], bias, w13[:E], s13[:E], w2[:E],
                                             s2[:E], *args)
    ref = _dense_block_mlp(x, w13[E], s13[E], w2[E], s2[E])
    np.testing.assert_allclose(out - base, ref, rtol=1e-9, atol=1e-12 * np.abs(out).max())


# ---------------------------------------------------------------------------
# NVFP4 (E2M1 elements, an E4M3 scale per 16 elements, an fp32 global scale)
# ---------------------------------------------------------------------------
# the eight E2M1 magnitudes of the published format, codes 0..7 in order;
# codes 8..15 are their negatives
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_nearest_even(v):
    """Brute force: the code of the nearest E2M1 magnitude to |v| (ties to the
    even code, beyond 6 the largest), with the sign of v in bit 3."""
    mag = np.asarray(E2M1_MAGNITUDES)
    a = np.minimum(np.abs(v.astype(np.float64)), 6.0)
    d = np.abs(a[:, None] - mag[None, :])
    best = d.min(1, keepdims=True)
    tied = d == best
    # among the nearest codes take the even one (there are at most two)
    code = np.where(tied[:, ::2].any(1), np.argmax(tied & (np.arange(8) % 2 == 0), 1),
                    np.argmax(tied, 1))
    return (code | (np.signbit(v) << 3)).astype(np.uint8)


def test_e2m1_decode_matches_the_format():
    t = oracle.e2m1_decode_table()
    assert t[:8].tolist() == E2M1_MAGNITUDES
    assert t[8:].tolist() == [-m for m in E2M1_MAGNITUDES]
    assert np.signbit(t[8])  # code 8 is -0


def test_e2m1_encode_exhaustive_nearest_even():
    # every fp32 in [2^-4, 2^4): all rounding boundaries, the subnormal 0.5
    # and saturation from 6 up
    bits = np.arange(np.float32(2.0 ** -4).view(np.uint32), np.float32(16.0).view(np.uint32),
                     dtype=np.uint32)
    x = bits.view(np.float32)
    got = oracle.e2m1_encode(x)
    for lo in range(0, x.size, 1 << 22):
        sl = slice(lo, lo + (1 << 22))
        assert np.array_equal(got[sl], _e2m1_nearest_even(x[sl]))
    # negatives, zeros, tiny values, infinities
    rng = np.random.default_rng(11)
    y = np.concatenate([-x[rng.integers(0, x.size, 1 << 16)],
                        np.array([0.0, -0.0, 1e-30, -1e-30, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5,
                                  5.0, -5.0, 6.0, 7.0, 1e30, np.inf, -np.inf], np.float32)])
    assert np.array_equal(oracle.e2m1_encode(y), _e2m1_nearest_even(y))


def test_nvfp4_quant_closed_form():
    rng = np.random.default_rng(12)
    R, C = 24, 128
    x = rng.standard_normal((R, C)) * (10.0 ** rng.uniform(-2, 2, (R, 1)))
    x[2, 16:32] = 0.0       # an all-zero block
    xb = _bf16_bits(x)
    xv = oracle.bf16_to_f64(xb)
    for g in (np.float32(2.0 ** -3), np.float32(0.0137)):
        q, sb = oracle.nvfp4_quant(xb, g)
        blocks = np.abs(xv.reshape(R, C // 16, 16)).max(2).astype(np.float32)
        # block scale: the E4M3 code of (amax / 6) / g in fp32
        assert np.array_equal(sb, oracle.e4m3_encode((blocks / np.float32(6.0)) / g))
        step = (oracle.e4m3_decode(sb).astype(np.float32) * g).astype(np.float32)
        stepx = np.repeat(step, 16, 1)
        r = np.where(stepx > 0, xv.astype(np.float32) / np.where(stepx > 0, stepx, 1), 0)
        exp_q = np.where(stepx > 0, _e2m1_nearest_even(r.ravel().astype(np.float32))
                         .reshape(R, C), 0)
        assert np.array_equal(q, exp_q)
        # the block maximum lands on +-6 (its scale is within 2^-4 of amax/6)
        am = np.abs(xv.reshape(R, C // 16, 16)).argmax(2)
        qb = q.reshape(R, C // 16, 16)
        top = np.take_along_axis(qb, am[..., None], 2)[..., 0] & 0x7
        assert np.all(top[blocks > 0] == 7)
        assert np.all(sb[2, 1] == 0) and np.all(q[2, 16:32] == 0)


def _nvfp4_problem(rng, counts, N, Kd):
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    A = rng.integers(0, 16, (M, Kd)).astype(np.uint8)
    B = rng.integers(0, 16, (E, N, Kd)).astype(np.uint8)
    return off, M, A, B


def test_grouped_gemm_nvfp4_exact_with_power_of_two_scales():
    """Power-of-two block and global scales: every term is exact, so the
    result equals a numpy sum over 16-element blocks of (decoded dot product)
    x 2^(u+v) x ga x gb[e]. A transposed or shifted block index changes the
    powers and fails."""
    rng = np.random.default_rng(13)
    counts, N, Kd = [9, 0, 20], 48, 96
    off, M, A, B = _nvfp4_problem(rng, counts, N, Kd)
    E, KB = len(counts), Kd // 16
    u = rng.integers(-5, 6, (M, KB))
    v = rng.integers(-5, 6, (E, N, KB))
    sa = oracle.e4m3_encode((2.0 ** u).astype(np.float32))
    sb = oracle.e4m3_encode((2.0 ** v).astype(np.float32))
    ga = np.float32(0.25)
    gb = np.array([2.0, 0.5, 8.0], np.float32)
    C = oracle.grouped_gemm_nvfp4(A, sa, ga, B, sb, gb, off)
    tab = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
    Av, Bv = tab[A], tab[B]
    ref = np.zeros((M, N))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        for kb in range(KB):
            ks = slice(kb * 16, (kb + 1) * 16)
            part = Av[rows, ks] @ Bv[e, :, ks].T
            ref[rows] += part * 2.0 ** (u[rows, kb][:, None] + v[e, :, kb][None, :])
        ref[rows] *= float(ga) * float(gb[e])
    assert np.array_equal(C, ref)


def test_grouped_gemm_nvfp4_uniform_scales_is_a_plain_product():
    rng = np.random.default_rng(14)
    counts, N, Kd = [7, 5], 32, 64
    off, M, A, B = _nvfp4_problem(rng, counts, N, Kd)
    one = oracle.e4m3_encode(np.float32(1.0))
    sa = np.full((M, Kd // 16), one, np.uint8)
    sb = np.full((2, N, Kd // 16), one, np.uint8)
    C = oracle.grouped_gemm_nvfp4(A, sa, 1.0, B, sb, np.ones(2, np.float32), off)
    tab = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
    for e in range(2):
        rows = slice(off[e], off[e + 1])
        assert np.array_equal(C[rows], tab[A[rows]] @ tab[B[e]].T)


def _random_nvfp4_layer(rng, T, H, I, E):
    x = _bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)

    def weights(rows, cols):
        codes = rng.integers(0, 16, (E, rows, cols)).astype(np.uint8)
        scales = oracle.e4m3_encode((2.0 ** rng.uniform(-7, -3, (E, rows, cols // 16)))
                                    .astype(np.float32))
        g = rng.uniform(0.5, 2.0, E).astype(np.float32)
        return codes, scales, g

    w13, s13, g13 = weights(2 * I, H)
    w2, s2, g2 = weights(H, I)
    return x, logits, w13, s13, g13, w2, s2, g2


def _dense_nvfp4_mlp(x, w13e, s13e, g13e, w2e, s2e, g2e, ga1, ga2):
    """One expert on every token in NVFP4 with numpy: dequantise codes times
    block scales times global scales, multiply in fp64."""
    tab = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
    I = w2e.shape[1]

    def deq_act(bits, g):
        q, sb = oracle.nvfp4_quant(bits, g)
        return tab[q] * np.repeat(oracle.e4m3_decode(sb), 16, 1) * float(g)

    def deq_w(q, s, g):
        return tab[q] * np.repeat(oracle.e4m3_decode(s), 16, 1) * float(g)

    C = deq_act(x, ga1) @ deq_w(w13e, s13e, g13e).T
    g, u = C[:, :I], C[:, I:]
    hb = oracle.bf16_round(g / (1 + np.exp(-g)) * u)
    return deq_act(hb, ga2) @ deq_w(w2e, s2e, g2e).T


def test_layer_nvfp4_single_expert_is_dense_nvfp4_mlp():
    # H and I span several 16-element blocks, and the two activation global
    # scales differ, so a scale taken from the wrong block or tensor shows
    rng = np.random.default_rng(61)
    T, H, I = 6, 64, 48
    x, logits, w13, s13, g13, w2, s2, g2 = _random_nvfp4_layer(rng, T, H, I, 1)
    ga1, ga2 = np.float32(0.0125), np.float32(0.0031)
    out, ids, w = oracle.forward_tokens_nvfp4(x, logits, None, w13, s13, g13, w2, s2, g2, ga1,
                                              ga2, 1, 1, 1, oracle.SOFTMAX, True, 1.0)
    assert np.all(ids == 0) and np.all(w == 1.0)
    ref = _dense_nvfp4_mlp(x, w13[0], s13[0], g13[0], w2[0], s2[0], g2[0], ga1, ga2)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def test_layer_nvfp4_token_path_equals_step_path_with_shared_expert():
    rng = np.random.default_rng(62)
    T, H, I, E, S = 20, 64, 48, 8, 1
    x, logits, w13, s13, g13, w2, s2, g2 = _random_nvfp4_layer(rng, T, H, I, E + S)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    ga1, ga2 = np.float32(0.0125), np.float32(0.0031)
    args = (4, 2, 3, oracle.SIGMOID, True, 2.5)
    steps = oracle.forward_steps_nvfp4(x, logits[:, :E], bias, w13, s13, g13, w2, s2, g2, ga1,
                                       ga2, *args, n_shared=S)
    out, ids, w = oracle.forward_tokens_nvfp4(x, logits[:, :E], bias, w13, s13, g13, w2, s2, g2,
                                              ga1, ga2, *args, n_shared=S)
    assert np.array_equal(ids, steps["ids"][:, :3]) and np.array_equal(w, steps["w"][:, :3])
    np.testing.assert_allclose(out, steps["out"], rtol=1e-12, atol=1e-12 * np.abs(out).max())
    # the shared expert adds its dense NVFP4 MLP with weight 1
    base, _, _ = oracle.forward_tokens_nvfp4(x, logits[:, :E], bias, w13[:E], s13[:E], g13[:E],
                                             w2[:E], s2[:E], g2[:E], ga1, ga2, *args)
    ref = _dense_nvfp4_mlp(x, w13[E], s13[E], g13[E], w2[E], s2[E], g2[E], ga1, ga2)
    np.testing.assert_allclose(out - base, ref, rtol=1e-9, atol=1e-12 * np.abs(out).max())
