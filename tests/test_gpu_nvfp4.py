"""NVFP4 path on the GPU through the C ABI, against the oracle's NVFP4
functions: the E2M1 conversion on every bf16 value in [-6, 6] (the
quantiser with a unit step), the requant and the pre-reorder bit for bit,
the block-scaled grouped GEMM on one tile first and then on ragged shapes
of both epilogues, and the whole layer (every token of the small and decode
layers, a token of every GEMM tile of the prefill layer)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
import oracle
from moe_expert_layer_grouped_gb300 import synth

from gpu_util import assert_parity, bf16_np, ragged_offsets, tile_cover_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert moe.moe_device_status() == 0


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _unpack(t):
    return synth.unpack_e2m1(t.cpu()).numpy()


def _bf16_bits(a32):
    return torch.from_numpy(np.ascontiguousarray(a32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("g", [1.0, 1 + 2.0 ** -22, 1 - 2.0 ** -23, 1 + 2.0 ** -19])
def test_e2m1_conversion_of_every_bf16_in_range(g):
    """Blocks of one 6.0 and 15 test values: with g = 1 the block scale is
    e4m3(6/6/1) = 1.0 exactly, so the codes are e2m1(v) of each bf16 v. A g
    a few fp32 ulps from 1 keeps the scale code at 1.0 and moves the
    quotients v / g of the bf16 values at e2m1 midpoints just to one side of
    the boundary (within 2^-20 of it, or just outside for 2^-19)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 6.0)
    v = vals[keep]
    n = -(-v.size // 15) * 15
    v = np.concatenate([v, np.zeros(n - v.size, np.float32)]).reshape(-1, 15)
    blocks = np.concatenate([np.full((v.shape[0], 1), 6.0, np.float32), v], axis=1)
    rows = blocks.reshape(-1, 256) if blocks.size % 256 == 0 else \
        np.concatenate([blocks.ravel(), np.zeros(256 - blocks.size % 256, np.float32)]).reshape(-1, 256)
    h = _bf16_bits(rows)
    g32 = float(np.float32(g))
    q, sf = moe.moe_act_quant_nvfp4(_t(h).view(torch.bfloat16), g32)
    torch.cuda.synchronize()
    oq, osf = oracle.nvfp4_quant(h, g32)
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.all(osf[:, 0] == 0x38)                 # e4m3 1.0 in every block
    got = _unpack(q)
    exp = oracle.e2m1_encode((rows.astype(np.float32) / np.float32(g32)).astype(np.float32))
    assert np.array_equal(oq, exp)                   # the oracle's quantiser agrees
    bad = np.argwhere(got != exp)
    assert bad.shape[0] == 0, (bad.shape[0], bad[:5].tolist())


@pytest.mark.parametrize("g", [1.0, 0.37, 5.0 / (6 * 448)])
def test_act_quant_nvfp4_matches_oracle(g):
    rng = np.random.default_rng(7)
    M, I = 257, 512
    x = rng.standard_normal((M, I)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-4, 3, (M, 1))).astype(np.float32)   # rows of every size
    x[3] = 0.0                                                       # all-zero row
    x[5, 16:32] = 0.0                                                # an all-zero block
    x[9, :16] = 1e-30                                                # scale below e4m3
    h = _bf16_bits(x)
    q, sf = moe.moe_act_quant_nvfp4(_t(h).view(torch.bfloat16), g)
    torch.cuda.synchronize()
    oq, osf = oracle.nvfp4_quant(h, g)
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(_unpack(q), oq)


@pytest.mark.parametrize("M,I", [(70, 256), (33, 2048), (20, 4096), (9, 8192), (7, 12288),
                                 (5, 14336), (3, 20480), (41, 96), (6, 2080)])
def test_act_quant_nvfp4_every_launch_shape(M, I):
    """A CTA per row of 64 threads holding 2 or 4 vectors each, of 256 threads
    holding 2 to 8 (I % 256 == 0), and a warp per row beyond 16384 channels
    or when I is not a multiple of 256."""
    rng = np.random.default_rng(M + I)
    x = rng.standard_normal((M, I)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-3, 2, (M, 1))).astype(np.float32)
    x[0, 32:48] = 0.0
    h = _bf16_bits(x)
    g = 5.0 / (6 * 448)
    q, sf = moe.moe_act_quant_nvfp4(_t(h).view(torch.bfloat16), g)
    torch.cuda.synchronize()
    oq, osf = oracle.nvfp4_quant(h, g)
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(_unpack(q), oq)


@pytest.mark.parametrize("T,H,E,K", [(8, 256, 8, 2), (300, 512, 24, 6), (4099, 256, 64, 6),
                                     # scale bytes one by one (H % 256 != 0), both routings
                                     (37, 224, 16, 4), (600, 224, 16, 4),
                                     # DeepSeek-V3's H on both routings
                                     (40, 7168, 32, 8), (1030, 7168, 64, 8)])
def test_permute_quant_nvfp4_matches_oracle(T, H, E, K):
    rng = np.random.default_rng(T + H)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    x_bits = x.view(torch.int16).numpy().view(np.uint16).copy()
    g = 5.0 / (6 * 448)
    a_q, sf, s2d, off = moe.moe_permute_quant_nvfp4(x.to(DEV), _t(ids), E, g)
    torch.cuda.synchronize()
    o_aq, o_sf, o_s2d, o_off = oracle.permute_quant_nvfp4(x_bits, ids, E, g)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(s2d.cpu().numpy(), o_s2d)
    assert np.array_equal(sf.cpu().numpy(), o_sf)
    assert np.array_equal(_unpack(a_q), o_aq)


def _fp4_problem(rng, counts, N, Kd):
    E = len(counts)
    off = ragged_offsets(counts)
    M = int(off[-1])
    A = rng.integers(0, 16, (M, Kd)).astype(np.uint8)
    B = rng.integers(0, 16, (E, N, Kd)).astype(np.uint8)
    sa = rng.integers(0x20, 0x40, (M, Kd // 16)).astype(np.uint8)    # 2^-3 .. 2^0 area
    sb = rng.integers(0x20, 0x40, (E, N, Kd // 16)).astype(np.uint8)
    gb = (10.0 ** rng.uniform(-3, -1, E)).astype(np.float32)
    return A, sa, B, sb, gb, off


def _run_fp4(A, sa, ga, B, sb, gb, off, epi):
    pa = synth.pack_e2m1(torch.from_numpy(A))
    pb = synth.pack_e2m1(torch.from_numpy(B))
    sba = moe.moe_nvfp4_arrange_scales(_t(sb), epi)
    return moe.moe_grouped_gemm_nvfp4(pa.to(DEV), _t(sa), ga, pb.to(DEV), sba, _t(gb),
                                      _t(off), epi)


@pytest.mark.parametrize("silu", [False, True])
def test_arranged_scales_follow_their_definition(silu):
    """Every scale byte lands where the header says (the copy order of the
    GEMM): block (e, nb, c, j), byte 16*(m%32) + 4*(m/32) + b."""
    rng = np.random.default_rng(2)
    E, N, Kd = 3, 256, 512
    sb = rng.integers(0, 256, (E, N, Kd // 16)).astype(np.uint8)
    epi = moe.EPI_SILU_MUL if silu else moe.EPI_BF16
    got = moe.moe_nvfp4_arrange_scales(_t(sb), epi).cpu().numpy().reshape(-1)
    I, KB = N // 2, Kd // 256
    NB = I // 64 if silu else N // 128
    exp = np.empty_like(got)
    for e in range(E):
        for nb in range(NB):
            for m in range(128):
                row = (64 * nb + m if m < 64 else I + 64 * nb + m - 64) if silu else 128 * nb + m
                for c in range(KB):
                    base = ((e * NB + nb) * KB + c) * 2048
                    for j in range(4):
                        for b in range(4):
                            exp[base + 512 * j + 16 * (m % 32) + 4 * (m // 32) + b] = \
                                sb[e, row, 16 * c + 4 * j + b]
    assert np.array_equal(got, exp)


def test_nvfp4_gemm_one_tile():
    """One expert, 64 tokens, one 128-row weight block, one K chunk."""
    rng = np.random.default_rng(1)
    A, sa, B, sb, gb, off = _fp4_problem(rng, [64], 128, 256)
    C = _run_fp4(A, sa, 0.5, B, sb, gb, off, moe.EPI_BF16)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    ref = oracle.grouped_gemm_nvfp4(A, sa, 0.5, B, sb, gb, off)
    got = bf16_np(C)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max())
    assert_parity(got, ref, "nvfp4 gemm, one tile")


FP4_SHAPES = [
    # counts per expert, N, Kd
    ([5, 0, 9], 256, 256),
    ([130, 1, 0, 257, 128], 256, 512),
    ([300], 384, 768),
    ([17, 64, 200, 3], 128, 256),
    ([129, 127], 256, 7168),
    ([150, 0, 3, 40, 0, 0, 7, 0, 0, 0, 0, 0, 0, 0, 0, 1], 256, 512),
    # few rows per expert: two K chunks per stage (even chunk count, the ring
    # wrapping within a tile), and one per stage (odd chunk count)
    ([3, 0, 9, 1, 5, 2, 0, 7], 256, 2048),
    ([3, 9, 1, 5], 256, 768),
    # many rows per expert with 256-row weight tiles (SiLU: I % 128 == 0,
    # bf16: N % 256 == 0): the two-accumulator kernel. Three 256-row tiles,
    # five K chunks on a three-stage ring (it wraps inside a tile), experts of
    # 0, 1 and 511 tokens (four 128-token chunks); one K chunk per tile.
    ([260, 0, 129, 511, 1, 40], 768, 1280),
    ([1000, 300], 512, 256),
    # 480 experts: the tile table leaves room for three stages only
    ([33 + (7 * e) % 29 for e in range(480)], 256, 512),
]


@pytest.mark.parametrize("counts,N,Kd", FP4_SHAPES)
def test_nvfp4_gemm_bf16_epilogue(counts, N, Kd):
    rng = np.random.default_rng(sum(counts) + N + Kd)
    A, sa, B, sb, gb, off = _fp4_problem(rng, counts, N, Kd)
    C = _run_fp4(A, sa, 0.25, B, sb, gb, off, moe.EPI_BF16)
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm_nvfp4(A, sa, 0.25, B, sb, gb, off)
    got = bf16_np(C)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max())
    assert_parity(got, ref, "nvfp4 gemm bf16")


@pytest.mark.parametrize("counts,N,Kd", FP4_SHAPES)
def test_nvfp4_gemm_silu_epilogue(counts, N, Kd):
    rng = np.random.default_rng(3 * sum(counts) + N + Kd)
    A, sa, B, sb, gb, off = _fp4_problem(rng, counts, N, Kd)
    C = _run_fp4(A, sa, 0.25, B, sb, gb, off, moe.EPI_SILU_MUL)
    torch.cuda.synchronize()
    ref = oracle.silu_mul(oracle.grouped_gemm_nvfp4(A, sa, 0.25, B, sb, gb, off))
    got = bf16_np(C)
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-4 * np.abs(ref).max())
    assert_parity(got, ref, "nvfp4 gemm silu")


def _layer_nvfp4(wl, d):
    return moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                        wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                        n_shared=wl.n_shared, quant="nvfp4",
                        nvfp4=dict(g13=d["g13"], g2=d["g2"], ga1=wl.ga1, ga2=wl.ga2))


def _check_nvfp4_layer(wl, seed, sample=False):
    d = synth.make_inputs(wl, seed=seed, device=DEV)
    layer = _layer_nvfp4(wl, d)
    out = layer(d["x"], d["logits"])
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    n = synth.to_numpy_inputs({k: d[k] for k in ("x", "logits", "bias", "s13", "g13", "s2",
                                                  "g2")})
    w13, w2 = _unpack(d["w13"]), _unpack(d["w2"])
    if sample:
        ids, _ = oracle.gate(n["logits"], n["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                             wl.scoring, wl.renormalize, wl.rsf)
        tokens, _ = tile_cover_tokens(ids, wl.E, quant="nvfp4", seed=seed)
    else:
        tokens = np.arange(wl.T, dtype=np.int64)
    ref, _, _ = oracle.forward_tokens_nvfp4(n["x"], n["logits"], n["bias"], w13, n["s13"],
                                            n["g13"], w2, n["s2"], n["g2"], wl.ga1, wl.ga2,
                                            wl.num_groups, wl.topk_group, wl.top_k, wl.scoring,
                                            wl.renormalize, wl.rsf, tokens=tokens,
                                            n_shared=wl.n_shared)
    assert_parity(bf16_np(out[torch.from_numpy(tokens).to(DEV)]), ref, wl.name)
    return layer, d, out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_nvfp4_tiny(seed):
    _check_nvfp4_layer(synth.WORKLOADS["tiny_nvfp4"], seed)


def test_forward_nvfp4_dsv3_decode_t128():
    _check_nvfp4_layer(synth.WORKLOADS["dsv3_decode_t128_nvfp4"], 0)


def test_forward_nvfp4_dsv3_prefill_every_tile():
    _check_nvfp4_layer(synth.WORKLOADS["dsv3_prefill_t8192_nvfp4"], 0, sample=True)


def test_forward_nvfp4_shared_expert_ragged_and_host_buffers():
    """A shared expert (every token's weight-1 slot) on the NVFP4 path, every
    token against the oracle; ~84 rows per expert, so both GEMMs take the
    two-accumulator kernel, the shared expert's 300 rows in three token
    chunks. The host-buffer entry point gives the same bytes."""
    wl = synth.Workload("nvfp4_shared", 300, 512, 256, 24, 4, 2, 6, synth.SIGMOID, True, 2.5,
                        "normal", n_shared=1, quant="nvfp4")
    layer, d, out = _check_nvfp4_layer(wl, 3)
    xh, lh = d["x"].cpu().pin_memory(), d["logits"].cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, lh, oh)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert torch.equal(oh.view(torch.int16), out.cpu().view(torch.int16))
