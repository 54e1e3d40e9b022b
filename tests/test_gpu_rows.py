"""The token-order path of the layer through the C ABI: the pre-reorder that
stores each token's codes once (moe_permute_quant_rows) and the grouped GEMM
that gathers a tile's token rows through row_token (moe_grouped_gemm_rows).

The pre-reorder is checked bit for bit against the oracle (codes, scales,
src2dst, offsets) and row_token against its definition; the gathering GEMM
must give bit for bit what moe_grouped_gemm gives on the same rows stored in
permuted order (A[r] = A_tok[row_token[r]]), on ragged shapes of every
launch configuration, and match the oracle within the GEMM tolerance.
(moe_forward keeps the K-fold copies: the gathering GEMM measured slower.)"""
import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
import oracle

from gpu_util import assert_parity, bf16_bits, bf16_np, ragged_offsets, random_e4m3

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


@pytest.mark.parametrize("T,H,E,K", [(8, 128, 8, 2), (300, 384, 24, 6), (4099, 256, 64, 6),
                                     (1024, 7168, 256, 8)])
def test_permute_quant_rows_matches_oracle(T, H, E, K):
    rng = np.random.default_rng(T + H)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    x_bits = x.view(torch.int16).numpy().view(np.uint16).copy()
    a_tok, sa, s2d, rt, off = moe.moe_permute_quant_rows(x.to(DEV), _t(ids), E)
    torch.cuda.synchronize()
    o_aq, o_sa, o_s2d, o_off = oracle.permute_quant(x_bits, ids, E)
    q, _ = oracle.row_quant(x_bits)          # each token's codes, once
    assert np.array_equal(a_tok.cpu().numpy(), q)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(s2d.cpu().numpy(), o_s2d)
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), o_sa.view(np.uint32))
    rt = rt.cpu().numpy()
    assert np.array_equal(rt[o_s2d], np.repeat(np.arange(T, dtype=np.int32), K))
    # the permuted codes are the token rows the GEMM will gather
    assert np.array_equal(q[rt], o_aq)
    assert moe.moe_device_status() == 0


GATHER_SHAPES = [
    # counts per expert, N, Kd: few rows per expert (64-token tiles) and many
    # (256-token CTA-pair tiles), ragged chunks, K not a multiple of 128
    ([5, 0, 9], 256, 128),
    ([130, 1, 0, 257, 128], 512, 256),
    ([300], 768, 384),
    ([400, 260], 512, 224),
    ([129, 127], 256, 7168),
    ([150, 0, 3, 40, 0, 0, 7, 0, 0, 0, 0, 0, 0, 0, 0, 1], 256, 512),
    ([1000, 1040, 990, 1010], 1024, 1024),
]


def _gather_problem(rng, counts, N, Kd):
    E = len(counts)
    off = ragged_offsets(counts)
    M = int(off[-1])
    T = max(1, M // 3 + 5)
    A_tok = random_e4m3(rng, (T, Kd))
    row_token = rng.integers(0, T, M).astype(np.int32)   # any token may fill any row
    B = random_e4m3(rng, (E, N, Kd))
    sa = (10.0 ** rng.uniform(-3, 1, M)).astype(np.float32)
    sb = (10.0 ** rng.uniform(-4, -2, (E, N))).astype(np.float32)
    return A_tok, row_token, sa, B, sb, off


@pytest.mark.parametrize("epi", ["bf16", "silu"])
@pytest.mark.parametrize("counts,N,Kd", GATHER_SHAPES)
def test_gather_gemm_equals_permuted_gemm(counts, N, Kd, epi):
    rng = np.random.default_rng(sum(counts) * 3 + N + Kd)
    A_tok, rt, sa, B, sb, off = _gather_problem(rng, counts, N, Kd)
    e = moe.EPI_SILU_MUL if epi == "silu" else moe.EPI_BF16
    M = int(off[-1])
    ra_g = torch.zeros(M, dtype=torch.float32, device=DEV) if epi == "silu" else None
    ra_p = torch.zeros(M, dtype=torch.float32, device=DEV) if epi == "silu" else None
    Cg = moe.moe_grouped_gemm_rows(_t(A_tok), _t(rt), _t(sa), _t(B), _t(sb), _t(off), e,
                                   row_amax=ra_g)
    A = A_tok[rt]
    Cp = moe.moe_grouped_gemm(_t(A), _t(sa), _t(B), _t(sb), _t(off), e, row_amax=ra_p)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert np.array_equal(bf16_bits(Cg), bf16_bits(Cp))
    if ra_g is not None:
        assert torch.equal(ra_g, ra_p)
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    if epi == "silu":
        ref = oracle.silu_mul(ref)
    assert_parity(bf16_np(Cg), ref, f"gather gemm {epi}")


def test_gather_gemm_reads_rows_outside_the_tensor_as_zero():
    rng = np.random.default_rng(5)
    A_tok, rt, sa, B, sb, off = _gather_problem(rng, [300, 40], 256, 256)
    T = A_tok.shape[0]
    rt[::7] = T                                   # past the end of A_tok
    Cg = moe.moe_grouped_gemm_rows(_t(A_tok), _t(rt), _t(sa), _t(B), _t(sb), _t(off),
                                   moe.EPI_BF16)
    torch.cuda.synchronize()
    A = np.concatenate([A_tok, np.zeros((1, A_tok.shape[1]), np.uint8)])[rt]
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    got = bf16_np(Cg)
    assert np.all(got[::7] == 0)
    assert_parity(got, ref, "gather gemm, rows outside")
