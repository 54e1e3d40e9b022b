"""Per-step parity of the CUDA kernels (through the C ABI) against the CPU
oracle: bit-exact for the gate, routing, FP8 codes and scales; within the
layer tolerance for the GEMMs and the post-reorder."""
import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
import oracle
from moe_expert_layer_grouped_gb300 import synth

from gpu_util import (assert_parity, bf16_bits, bf16_np, np_bf16_to_torch, ragged_offsets,
                      random_e4m3)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert moe.moe_device_status() == 0


# ---------------------------------------------------------------------------
# gate
# ---------------------------------------------------------------------------
GATE_CASES = [
    # (T, E, G, TG, K, scoring, renorm, rsf, bias kind)
    (8, 8, 1, 1, 2, synth.SOFTMAX, True, 1.0, "none"),
    (128, 256, 8, 4, 8, synth.SIGMOID, True, 2.5, "normal"),
    (8192, 256, 8, 4, 8, synth.SIGMOID, True, 2.5, "zero"),
    (16384, 256, 8, 4, 8, synth.SIGMOID, True, 2.5, "skewed"),
    (4096, 8, 1, 1, 2, synth.SOFTMAX, True, 1.0, "none"),
    (333, 72, 6, 2, 5, synth.SIGMOID, True, 1.7, "normal"),
    (257, 1024, 64, 3, 32, synth.SIGMOID, True, 2.5, "normal"),
    (100, 64, 1, 1, 6, synth.SIGMOID, False, 2.5, "normal"),
    (100, 20, 1, 1, 3, synth.SOFTMAX, False, 1.0, "none"),
    (64, 16, 16, 4, 4, synth.SIGMOID, True, 1.0, "normal"),
]


@pytest.mark.parametrize("case", GATE_CASES, ids=lambda c: f"T{c[0]}E{c[1]}G{c[2]}K{c[4]}")
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gate_bit_exact(case, seed):
    T, E, G, TG, K, scoring, renorm, rsf, bias_kind = case
    if seed and T > 1000:
        pytest.skip("large cases run on seed 0")
    logits = synth.normal((T, E), 1.0, seed, "logits")
    wl = synth.Workload("g", T, 128, 64, E, G, TG, K, scoring, renorm, rsf, bias_kind)
    bias = synth.router_bias(wl, seed)
    # exact ties inside rows
    logits[:, 1] = logits[:, 0]
    ids, w = moe.moe_gate(logits.to(DEV), None if bias is None else bias.to(DEV), G, TG, K,
                          scoring, renorm, rsf)
    rids, rw = oracle.gate(logits.numpy(), None if bias is None else bias.numpy(), G, TG, K,
                           scoring, renorm, rsf)
    gi, gw = ids.cpu().numpy(), w.cpu().numpy()
    bad = np.nonzero((gi != rids).any(1))[0]
    assert bad.size == 0, f"{bad.size} tokens differ, first {bad[:3]}: {gi[bad[:3]]} vs {rids[bad[:3]]}"
    assert np.array_equal(gw.view(np.uint32), rw.view(np.uint32))


def test_gate_sigmoid_sweep_bit_exact():
    """E=1, K=1, no renormalisation, rsf=1: the weight is the fp32 sigmoid
    itself, so a sweep of logits exposes the kernel's exp/sigmoid bit for bit."""
    x = np.concatenate([
        np.linspace(-110, 110, 1 << 22, dtype=np.float32),
        np.random.default_rng(0).standard_normal(1 << 20).astype(np.float32) * 4,
        np.array([0.0, -0.0, 88.7, -88.7, 103.9, -103.9, 16.6, 17.0], np.float32),
    ]).reshape(-1, 1)
    ids, w = moe.moe_gate(torch.from_numpy(x).to(DEV), None, 1, 1, 1, synth.SIGMOID, False, 1.0)
    ref = oracle.sigmoid32(x[:, 0])
    got = w.cpu().numpy()[:, 0]
    bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
    assert bad.size == 0, (x[bad[:5], 0], got[bad[:5]], ref[bad[:5]])


def _oracle_in_threads(fn, x, pool, parts=16):
    """fn over slices of x on a thread pool (the oracle's C calls run without
    the interpreter lock, so the slices run on separate cores)."""
    out = np.empty_like(x)
    cut = np.linspace(0, x.size, parts + 1).astype(np.int64)

    def job(i):
        out[cut[i]:cut[i + 1]] = fn(x[cut[i]:cut[i + 1]])

    list(pool.map(job, range(parts)))
    return out


def test_sigmoid_bit_exact_on_every_fp32_up_to_88():
    """Every fp32 x with |x| <= 88 (2.24e9 values of both signs, zeros and
    subnormals included), the range where exp(-x) stays finite: the gate's
    weight for E=1, K=1, no renormalisation and rsf=1 is the fp32 sigmoid,
    and it equals the oracle's bit for bit."""
    from concurrent.futures import ThreadPoolExecutor
    chunk = 1 << 27
    top = 0x42B00000  # bit pattern of 88.0f
    with ThreadPoolExecutor(max_workers=16) as pool:
        for sign in (0, 0x80000000):
            for start in range(0, top + 1, chunk):
                bits = np.arange(start, min(start + chunk, top + 1), dtype=np.uint32)
                x = (bits | np.uint32(sign)).view(np.float32)
                _, w = moe.moe_gate(torch.from_numpy(x).view(-1, 1).to(DEV), None, 1, 1, 1,
                                    synth.SIGMOID, False, 1.0)
                got = w.view(-1).cpu().numpy().view(np.uint32)
                ref = _oracle_in_threads(oracle.sigmoid32, x, pool).view(np.uint32)
                bad = np.nonzero(got != ref)[0]
                assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


# ---------------------------------------------------------------------------
# pre-reorder + quantisation
# ---------------------------------------------------------------------------
def _ids(rng, T, E, K, hot=None):
    if hot is not None:
        p = np.full(E, 1e-3)
        p[:hot] = 1.0
        p /= p.sum()
        return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,H,E,K,hot", [(1, 32, 4, 1, None), (37, 128, 8, 2, None),
                                         (300, 7168, 256, 8, None), (1000, 4096, 8, 2, None),
                                         (2049, 256, 64, 6, 10), (70, 16384, 3, 3, None),
                                         # the one-launch path ends at T*K = 4096
                                         (512, 512, 1024, 8, 40), (513, 512, 1024, 8, 40),
                                         (128, 7168, 256, 8, 60), (4096, 256, 16, 1, None)])
def test_permute_quant_bit_exact(T, H, E, K, hot):
    rng = np.random.default_rng(T + H)
    ids = _ids(rng, T, E, K, hot)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)
                         * 10.0 ** rng.uniform(-3, 3, (T, 1)).astype(np.float32)).to(torch.bfloat16)
    x[0, :] = 0  # an all-zero token
    a_q, sa, s2d, off = moe.moe_permute_quant(x.to(DEV), torch.from_numpy(ids).to(DEV), E)
    r_aq, r_sa, r_s2d, r_off = oracle.permute_quant(bf16_bits(x), ids, E)
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(s2d.cpu().numpy(), r_s2d)
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), r_sa.view(np.uint32))
    assert np.array_equal(a_q.cpu().numpy(), r_aq)


def test_permute_empty_and_bad_ids():
    E = 8
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros((0, 2), dtype=torch.int32, device=DEV)
    a_q, sa, s2d, off = moe.moe_permute_quant(x, ids, E)
    assert off.cpu().tolist() == [0] * (E + 1)
    assert moe.moe_device_status() == 0
    # an expert id out of range is caught on the device and skipped
    x = torch.ones((4, 64), dtype=torch.bfloat16, device=DEV)
    bad = torch.tensor([[0, 1], [2, 99], [3, 4], [5, -1]], dtype=torch.int32, device=DEV)
    moe.moe_permute_quant(x, bad, E)
    assert moe.moe_device_status() == 1
    assert moe.moe_device_status() == 0  # cleared


@pytest.mark.parametrize("T", [64, 1200])   # the one-launch and the three-launch routing
def test_permute_bad_ids_same_on_both_paths(T):
    """Out-of-range ids get destination -1, an id repeated within a token
    counts once and shares its first occurrence's row, both raise the device
    error; the rest is the stable counting sort (checked against a plain
    numpy restatement of that rule)."""
    rng = np.random.default_rng(T)
    E, K, H = 16, 4, 128
    ids = _ids(rng, T, E, K)
    ids[3, 2] = 99            # out of range
    ids[5, 3] = ids[5, 1]     # repeat within the token
    ids[T - 1, 0] = -7
    x = torch.randn((T, H), dtype=torch.bfloat16, device=DEV)
    a_q, sa, s2d, off = moe.moe_permute_quant(x, torch.from_numpy(ids).to(DEV), E)
    assert moe.moe_device_status() == 1
    cnt = np.zeros(E, np.int64)
    first = np.full((T, K), -1)
    for t in range(T):
        for k in range(K):
            e = ids[t, k]
            if 0 <= e < E and e not in ids[t, :k]:
                first[t, k] = e
    for e in first[first >= 0]:
        cnt[e] += 1
    ref_off = np.concatenate([[0], np.cumsum(cnt)])
    assert np.array_equal(off.cpu().numpy(), ref_off)
    seen = np.zeros(E, np.int64)
    ref = np.full((T, K), -1)
    for t in range(T):
        for k in range(K):
            e = ids[t, k]
            if 0 <= e < E:
                ref[t, k] = ref_off[e] + seen[e]
        for e in set(first[t][first[t] >= 0]):
            seen[e] += 1
    assert np.array_equal(s2d.cpu().numpy().reshape(T, K), ref)


def test_fp8_encoder_matches_oracle_on_every_bf16():
    """Rows whose amax is exactly 448 have scale 1, so the codes are the
    encoder applied to every finite bf16 value."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = (bits.astype(np.uint32) << 16).view(np.float32)
    bits = bits[np.isfinite(v) & (np.abs(v) <= 448.0)]
    n = bits.size
    cols = 256
    rows = (n + cols - 2) // (cols - 1)
    pad = np.full(rows * (cols - 1) - n, bits[0], np.uint16)
    body = np.concatenate([bits, pad]).reshape(rows, cols - 1)
    m448 = np.full((rows, 1), 0x43E0, np.uint16)  # bf16 448.0
    h_bits = np.concatenate([body, m448], axis=1)
    q, s = moe.moe_act_quant(np_bf16_to_torch(h_bits, DEV))
    assert np.all(s.cpu().numpy() == 1.0)
    ref = oracle.e4m3_encode(oracle.bf16_to_f64(h_bits).astype(np.float32))
    got = q.cpu().numpy()
    bad = np.nonzero(got != ref)
    assert bad[0].size == 0, (h_bits[bad][:5], got[bad][:5], ref[bad][:5])


@pytest.mark.parametrize("amax", [448.0 * (1 + 2.0 ** -21), 448.0 * (1 - 2.0 ** -22),
                                  448.0 * (1 + 2.0 ** -19), 336.0 * (1 + 2.0 ** -21)])
def test_fp8_encoder_near_rounding_boundaries(amax):
    """Scales a few fp32 ulps from 1 (or 0.75) put the quotients of the bf16
    values that are e4m3 midpoints within 2^-20 of a rounding boundary, on
    either side of it: the codes are the encoder applied to the IEEE fp32
    quotient x / scale, scale = amax / 448 as the kernel forms it."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = (bits.astype(np.uint32) << 16).view(np.float32)
    bits = bits[np.isfinite(v) & (np.abs(v) <= 448.0)]
    cols = 256
    rows = -(-bits.size // cols)
    h_bits = np.concatenate([bits, np.zeros(rows * cols - bits.size, np.uint16)]).reshape(rows, cols)
    a32 = np.float32(amax)
    q, s = moe.moe_act_quant(np_bf16_to_torch(h_bits, DEV),
                             row_amax=torch.full((rows,), float(a32), device=DEV))
    sc = a32 / np.float32(448.0)
    assert np.all(s.cpu().numpy() == sc)
    x = oracle.bf16_to_f64(h_bits).astype(np.float32)
    ref = oracle.e4m3_encode((x / sc).astype(np.float32))
    got = q.cpu().numpy()
    bad = np.nonzero(got != ref)
    assert bad[0].size == 0, (h_bits[bad][:5], got[bad][:5], ref[bad][:5])


@pytest.mark.parametrize("M,I", [(1, 32), (513, 2048), (4099, 14336), (64, 96), (37, 512),
                                 (300, 1024), (70, 4096), (33, 7168), (17, 12288), (5, 20480)])
def test_act_quant_bit_exact(M, I):
    """Every launch shape of the requant: a warp per row (up to 512
    channels), a CTA of 64 threads holding 2 or 4 vectors each (up to 2048),
    of 256 threads holding 2 to 8 (up to 16384), two passes beyond."""
    rng = np.random.default_rng(M)
    h = torch.from_numpy(rng.standard_normal((M, I)).astype(np.float32)
                         * 10.0 ** rng.uniform(-4, 2, (M, 1)).astype(np.float32)).to(torch.bfloat16)
    q, s = moe.moe_act_quant(h.to(DEV))
    rq, rs = oracle.row_quant(bf16_bits(h))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)
    # with a supplied row amax (what the w13 epilogue can produce)
    amax = h.float().abs().amax(1).to(DEV)
    q2, s2 = moe.moe_act_quant(h.to(DEV), row_amax=amax)
    assert torch.equal(q2, q) and torch.equal(s2, s)


# ---------------------------------------------------------------------------
# grouped GEMM
# ---------------------------------------------------------------------------
def _gemm_problem(rng, counts, N, Kd, integer=False):
    E = len(counts)
    off = ragged_offsets(counts)
    M = int(off[-1])
    if integer:
        # small integers: every partial sum stays below 2^14, so the result
        # is exact whatever the accumulator's internal alignment
        A = oracle.e4m3_encode(rng.integers(-2, 3, (M, Kd)).astype(np.float32))
        B = oracle.e4m3_encode(rng.integers(-1, 2, (E, N, Kd)).astype(np.float32))
        sa = np.ones(M, np.float32)
        sb = np.ones((E, N), np.float32)
    else:
        A = random_e4m3(rng, (M, Kd))
        B = random_e4m3(rng, (E, N, Kd))
        sa = (10.0 ** rng.uniform(-3, 1, M)).astype(np.float32)
        sb = (10.0 ** rng.uniform(-4, -2, (E, N))).astype(np.float32)
    return A, sa, B, sb, off


def _run_gemm(A, sa, B, sb, off, epi, row_amax=False):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    ra = None
    if row_amax:
        ra = torch.zeros(A.shape[0], dtype=torch.float32, device=DEV)
    C = moe.moe_grouped_gemm(t(A), t(sa), t(B), t(sb), t(off), epi, row_amax=ra)
    return C, ra


GEMM_SHAPES = [
    # counts per expert, N, Kd
    ([5, 0, 9], 256, 128),
    ([130, 1, 0, 257, 128], 512, 256),
    ([300], 768, 384),
    ([17, 64, 200, 3], 320, 96),
    ([400, 260], 512, 224),      # CTA pairs with K not a multiple of 128
    ([129, 127], 256, 7168),
    # few rows per expert overall (small token tiles) but one expert with
    # several token chunks
    ([150, 0, 3, 40, 0, 0, 7, 0, 0, 0, 0, 0, 0, 0, 0, 1], 256, 512),
]


@pytest.mark.parametrize("counts,N,Kd", GEMM_SHAPES)
def test_grouped_gemm_exact_integers(counts, N, Kd):
    rng = np.random.default_rng(sum(counts) + N)
    A, sa, B, sb, off = _gemm_problem(rng, counts, N, Kd, integer=True)
    C, _ = _run_gemm(A, sa, B, sb, off, moe.EPI_BF16)
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    exp = torch.from_numpy(ref).to(torch.bfloat16).float().numpy()  # exact ints, one rounding
    got = bf16_np(C)
    bad = np.argwhere(got != exp)
    assert bad.shape[0] == 0, f"{bad.shape[0]} mismatches, first {bad[:5].tolist()}"


@pytest.mark.parametrize("counts,N,Kd", GEMM_SHAPES)
def test_grouped_gemm_bf16_epilogue(counts, N, Kd):
    rng = np.random.default_rng(7 * sum(counts) + Kd)
    A, sa, B, sb, off = _gemm_problem(rng, counts, N, Kd)
    C, _ = _run_gemm(A, sa, B, sb, off, moe.EPI_BF16)
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    got = bf16_np(C)
    # per element: fp32 accumulation + one bf16 rounding
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max())
    assert_parity(got, ref, "grouped gemm bf16")


@pytest.mark.parametrize("counts,N,Kd", GEMM_SHAPES)
def test_grouped_gemm_silu_epilogue(counts, N, Kd):
    rng = np.random.default_rng(11 * sum(counts) + N)
    A, sa, B, sb, off = _gemm_problem(rng, counts, N, Kd)
    C, ra = _run_gemm(A, sa, B, sb, off, moe.EPI_SILU_MUL, row_amax=True)
    ref = oracle.silu_mul(oracle.grouped_gemm(A, sa, B, sb, off))
    got = bf16_np(C)
    assert_parity(got, ref, "grouped gemm silu")
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-4 * np.abs(ref).max())
    # the row amax is the max |h| of the stored bf16 row
    assert np.array_equal(ra.cpu().numpy(), np.abs(got).max(1).astype(np.float32))


def test_grouped_gemm_scale_a_is_per_row():
    """Rows of one expert with scales 1e-3..1e3: each output row must carry
    its own row's scale (the per-expert indexing bug fixed in sglang #6772
    would use one scale for the whole segment)."""
    rng = np.random.default_rng(3)
    A, _, B, sb, off = _gemm_problem(rng, [200], 256, 256)
    sa = (10.0 ** np.linspace(-3, 3, 200)).astype(np.float32)
    C, _ = _run_gemm(A, sa, B, sb, off, moe.EPI_BF16)
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    got = bf16_np(C)
    row_err = np.abs(got - ref).max(1) / np.abs(ref).max(1)
    assert row_err.max() <= 2.0 ** -7


def test_grouped_gemm_rows_outside_segments_untouched():
    rng = np.random.default_rng(5)
    A, sa, B, sb, off = _gemm_problem(rng, [40, 0, 30], 256, 128)
    M = A.shape[0]
    # the segments cover only the first 50 of the M rows
    off = np.array([0, 20, 20, 50], np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    C = torch.full((M, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm(t(A), t(sa), t(B), t(sb), t(off), moe.EPI_BF16, C=C)
    assert torch.all(C[50:] == 7.0)
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    assert_parity(bf16_np(C[:50]), ref[:50])


def test_grouped_gemm_empty():
    t = torch.zeros
    A = t((0, 128), dtype=torch.uint8, device=DEV)
    B = t((4, 256, 128), dtype=torch.uint8, device=DEV)
    C = moe.moe_grouped_gemm(A, t(0, device=DEV), B, t((4, 256), device=DEV),
                             t(5, dtype=torch.int32, device=DEV))
    assert C.shape == (0, 256)


# ---------------------------------------------------------------------------
# post-reorder
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,K,H", [(1, 1, 8), (50, 8, 7168), (33, 2, 4096), (7, 32, 64)])
def test_unpermute_sum(T, K, H):
    rng = np.random.default_rng(T * K)
    M = T * K
    s2d = rng.permutation(M).astype(np.int32)
    down = torch.from_numpy(rng.standard_normal((M, H)).astype(np.float32)).to(torch.bfloat16)
    w = rng.random((T, K)).astype(np.float32) * 2.5
    out = moe.moe_unpermute_sum(down.to(DEV), torch.from_numpy(s2d).to(DEV),
                                torch.from_numpy(w).to(DEV))
    ref = oracle.unpermute_sum(bf16_np(down), s2d, w)
    got = bf16_np(out)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * K)
    # one-hot weights give back the permuted rows exactly
    w1 = np.zeros((T, K), np.float32)
    w1[:, 0] = 1.0
    out1 = moe.moe_unpermute_sum(down.to(DEV), torch.from_numpy(s2d).to(DEV),
                                 torch.from_numpy(w1).to(DEV))
    assert torch.equal(out1.cpu(), down[torch.from_numpy(s2d[::K].astype(np.int64))])


def test_permute_then_unpermute_identity_on_gpu():
    rng = np.random.default_rng(1)
    T, H, E, K = 300, 512, 16, 4
    ids = torch.from_numpy(_ids(rng, T, E, K)).to(DEV)
    x = torch.randn((T, H), dtype=torch.bfloat16, device=DEV)
    a_q, sa, s2d, off = moe.moe_permute_quant(x, ids, E)
    # move bf16 rows with the same permutation, then sum back with one-hot w
    perm = torch.empty((T * K, H), dtype=torch.bfloat16, device=DEV)
    perm[s2d.long()] = x.repeat_interleave(K, 0)
    w = torch.zeros((T, K), dtype=torch.float32, device=DEV)
    w[:, 0] = 1
    back = moe.moe_unpermute_sum(perm, s2d, w)
    assert torch.equal(back, x)
