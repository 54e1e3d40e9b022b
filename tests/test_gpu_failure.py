"""Failure detection on the GPU without a fault: a GEMM pipeline wait that
can never complete (one stage's bytes are never loaded) must give up after
its bound, report MOE_DEV_PIPE_TIMEOUT through the device error word and
leave the context usable for the next call."""
import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
import oracle

from gpu_util import assert_parity, bf16_np, ragged_offsets, random_e4m3

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert moe.moe_device_status() == moe.DEV_OK
    yield


def _problem(epi, counts=(20, 3, 0, 17, 9, 30, 1, 12), N=256, Kd=1024):
    rng = np.random.default_rng(77 + epi + len(counts) + Kd)
    # K = 1024 gives every tile several pipeline stages whatever their depth
    # in K
    off = ragged_offsets(list(counts))
    M = int(off[-1])
    A = random_e4m3(rng, (M, Kd))
    B = random_e4m3(rng, (len(counts), N, Kd))
    sa = (10.0 ** rng.uniform(-3, 1, M)).astype(np.float32)
    sb = (10.0 ** rng.uniform(-4, -2, (len(counts), N))).astype(np.float32)
    return A, sa, B, sb, off


@pytest.mark.parametrize("epi", [moe.EPI_BF16, moe.EPI_SILU_MUL])
@pytest.mark.parametrize("counts,N,Kd", [
    ((20, 3, 0, 17, 9, 30, 1, 12), 256, 1024),  # few rows: single CTAs
    ((300, 0, 129, 211), 256, 1024),            # many: CTA pairs
    ((300, 0, 129, 211), 512, 4096)])           # many, 32 K blocks: the two-accumulator pairs
def test_gemm_wait_timeout_is_reported_and_context_survives(epi, counts, N, Kd):
    """The decode-shaped problem runs single CTAs; the others (more than 32
    rows per expert) CTA pairs with one or two accumulators per CTA, where the
    stalled CTA's peer gives up on its own bounded waits and both meet at the
    teardown's cluster barrier."""
    A, sa, B, sb, off = _problem(epi, counts, N, Kd)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    N = B.shape[1]
    cols = N // 2 if epi == moe.EPI_SILU_MUL else N
    C = torch.zeros((A.shape[0], cols), dtype=torch.bfloat16, device=DEV)
    moe.moe_test_gemm_timeout(t(A), t(sa), t(B), t(sb), t(off), epi, C, stall_stage=1)
    assert moe.moe_device_status() == moe.DEV_PIPE_TIMEOUT
    assert moe.moe_device_status() == moe.DEV_OK        # reading clears it
    # the same GEMM right after, on the same context, is correct
    C2 = moe.moe_grouped_gemm(t(A), t(sa), t(B), t(sb), t(off), epi)
    assert moe.moe_device_status() == moe.DEV_OK
    ref = oracle.grouped_gemm(A, sa, B, sb, off)
    if epi == moe.EPI_SILU_MUL:
        ref = oracle.silu_mul(ref)
    assert_parity(bf16_np(C2), ref, "gemm after a timeout")


def _fp4_problem(counts, N, Kd, seed):
    rng = np.random.default_rng(seed)
    E = len(counts)
    off = ragged_offsets(counts)
    M = int(off[-1])
    A = rng.integers(0, 16, (M, Kd)).astype(np.uint8)
    B = rng.integers(0, 16, (E, N, Kd)).astype(np.uint8)
    sa = rng.integers(0x20, 0x40, (M, Kd // 16)).astype(np.uint8)
    sb = rng.integers(0x20, 0x40, (E, N, Kd // 16)).astype(np.uint8)
    gb = (10.0 ** rng.uniform(-3, -1, E)).astype(np.float32)
    return A, sa, B, sb, gb, off


@pytest.mark.parametrize("epi", [moe.EPI_BF16, moe.EPI_SILU_MUL])
@pytest.mark.parametrize("counts", [[20, 3, 0, 17, 9, 30, 1, 12],   # few rows: 128-row tiles
                                    [300, 0, 129, 211]])             # many: 256-row tiles
def test_nvfp4_gemm_wait_timeout_is_reported_and_context_survives(epi, counts):
    """Both NVFP4 kernels: the decode-shaped problem takes the 128-row-tile
    kernel, the other (more than 32 rows per expert, 256-row weight tiles)
    the two-accumulator kernel."""
    from moe_expert_layer_grouped_gb300 import synth
    N, Kd = 512, 1024
    A, sa, B, sb, gb, off = _fp4_problem(counts, N, Kd, 5 + epi + len(counts))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    pa = synth.pack_e2m1(torch.from_numpy(A)).to(DEV)
    pb = synth.pack_e2m1(torch.from_numpy(B)).to(DEV)
    sba = moe.moe_nvfp4_arrange_scales(t(sb), epi)
    cols = N // 2 if epi == moe.EPI_SILU_MUL else N
    C = torch.zeros((A.shape[0], cols), dtype=torch.bfloat16, device=DEV)
    moe.moe_test_gemm_nvfp4_timeout(pa, t(sa), 0.5, pb, sba, t(gb), t(off), epi, C,
                                    stall_stage=1)
    assert moe.moe_device_status() == moe.DEV_PIPE_TIMEOUT
    assert moe.moe_device_status() == moe.DEV_OK
    C2 = moe.moe_grouped_gemm_nvfp4(pa, t(sa), 0.5, pb, sba, t(gb), t(off), epi)
    assert moe.moe_device_status() == moe.DEV_OK
    ref = oracle.grouped_gemm_nvfp4(A, sa, 0.5, B, sb, gb, off)
    if epi == moe.EPI_SILU_MUL:
        ref = oracle.silu_mul(ref)
    assert_parity(bf16_np(C2), ref, "nvfp4 gemm after a timeout")
