"""The per-token GEMM's configuration for long K with many rows per expert:
CTA pairs holding 256 weight rows per CTA in two accumulators (gemm_wide.cu).
moe_grouped_gemm takes it by itself for K >= 32 blocks of 128 and many rows
per expert (SiLU: I % 256 == 0, bf16: N % 512 == 0). It is checked here
against the oracle on every element, on ragged shapes of that configuration,
and against the CTA-pair kernel with one accumulator per CTA. That kernel
still runs when a row amax (SiLU) or a row gather is asked for, on the same
rows and with the same K order of the same MMA shape, so the two must agree
bit for bit."""
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


WIDE_SHAPES = [
    # counts per expert (M > 32 E), N, Kd
    ([300, 0, 257, 1, 256, 40], 512, 4096),        # SiLU I=256: one pair tile of 512 rows
    ([513, 129, 255], 1024, 4096),                 # SiLU I=512 / bf16 N=1024: two pair tiles
    ([700, 90], 512, 7168),                        # 56 K blocks
    ([64] * 4 + [1000], 1536, 4096),               # three pair tiles, a long expert
]


def _problem(rng, counts, N, Kd):
    E = len(counts)
    off = ragged_offsets(counts)
    M = int(off[-1])
    A = random_e4m3(rng, (M, Kd))
    B = random_e4m3(rng, (E, N, Kd))
    sa = (10.0 ** rng.uniform(-3, 1, M)).astype(np.float32)
    sb = (10.0 ** rng.uniform(-4, -2, (E, N))).astype(np.float32)
    return A, sa, B, sb, off


@pytest.mark.parametrize("counts,N,Kd", WIDE_SHAPES)
def test_wide_silu_matches_oracle_and_the_one_accumulator_kernel(counts, N, Kd):
    rng = np.random.default_rng(sum(counts) + N + Kd)
    A, sa, B, sb, off = _problem(rng, counts, N, Kd)
    M = int(off[-1])
    assert M > 32 * len(counts)
    h = moe.moe_grouped_gemm(_t(A), _t(sa), _t(B), _t(sb), _t(off), moe.EPI_SILU_MUL)
    ra = torch.zeros(M, dtype=torch.float32, device=DEV)
    h1 = moe.moe_grouped_gemm(_t(A), _t(sa), _t(B), _t(sb), _t(off), moe.EPI_SILU_MUL,
                              row_amax=ra)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    ref = oracle.silu_mul(oracle.grouped_gemm(A, sa, B, sb, off))
    got = bf16_np(h)
    assert_parity(got, ref, "wide silu")
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-4 * np.abs(ref).max())
    assert np.array_equal(bf16_bits(h), bf16_bits(h1))


@pytest.mark.parametrize("counts,N,Kd", [(c, n * (2 if n % 512 else 1), k)
                                         for c, n, k in WIDE_SHAPES])
def test_wide_bf16_matches_oracle_and_the_one_accumulator_kernel(counts, N, Kd):
    rng = np.random.default_rng(3 * sum(counts) + N + Kd)
    A, sa, B, sb, off = _problem(rng, counts, N, Kd)
    M = int(off[-1])
    C = moe.moe_grouped_gemm(_t(A), _t(sa), _t(B), _t(sb), _t(off), moe.EPI_BF16)
    # the same rows gathered through an identity row map: the one-accumulator
    # pair kernel
    C1 = moe.moe_grouped_gemm_rows(_t(A), _t(np.arange(M, dtype=np.int32)), _t(sa), _t(B),
                                   _t(sb), _t(off), moe.EPI_BF16)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    got = bf16_np(C)
    assert_parity(got, ref, "wide bf16")
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max())
    assert np.array_equal(bf16_bits(C), bf16_bits(C1))


def test_wide_guard_bands_untouched():
    """Rows of the output outside the experts' segments and the bytes after
    the buffer stay as they were (no tile writes past its chunk)."""
    rng = np.random.default_rng(11)
    counts, N, Kd = [300, 257], 512, 4096
    A, sa, B, sb, off = _problem(rng, counts, N, Kd)
    M = int(off[-1])
    big = torch.full((M + 64, N // 2), -7.0, dtype=torch.bfloat16, device=DEV)
    h = big[:M]
    moe.moe_grouped_gemm(_t(A), _t(sa), _t(B), _t(sb), _t(off), moe.EPI_SILU_MUL, C=h)
    torch.cuda.synchronize()
    assert torch.all(big[M:] == -7.0)
