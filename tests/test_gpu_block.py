"""Block-quantised FP8 (128-channel activation scales, 128 x 128 weight
scales) on the GPU, through the C ABI, against the CPU oracle: the block
permute-quant and requant bit-exact; the block GEMMs and the whole layer
within the layer tolerance."""
import time

import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
import oracle
from moe_expert_layer_grouped_gb300 import synth

from gpu_util import (assert_parity, bf16_bits, bf16_np, np_bf16_to_torch, ragged_offsets,
                      random_e4m3, tile_cover_tokens)

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


def _blocky_bf16(rng, R, C):
    """bf16 rows whose 128-blocks span magnitudes 1e-4..1e3 (and one all-zero block)."""
    mag = 10.0 ** rng.uniform(-4, 3, (R, C // 128))
    x = rng.standard_normal((R, C)) * np.repeat(mag, 128, 1)
    x[0, :128] = 0.0
    return torch.from_numpy(x).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# block quantisation steps (bit-exact)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,I", [(1, 128), (37, 384), (300, 2048), (5, 7168)])
def test_act_quant_block_bit_exact(M, I):
    rng = np.random.default_rng(M + I)
    h = _blocky_bf16(rng, M, I)
    q, s = moe.moe_act_quant_block(h.to(DEV))
    rq, rs = oracle.block_quant(bf16_bits(h))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("T,H,E,K", [(1, 128, 4, 2), (129, 384, 16, 4), (64, 7168, 256, 8),
                                     (513, 1024, 8, 2)])
def test_permute_quant_block_bit_exact(T, H, E, K):
    rng = np.random.default_rng(T * 7 + H)
    x = _blocky_bf16(rng, T, H)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    a_q, sa, s2d, off = moe.moe_permute_quant_block(x.to(DEV), _t(ids), E)
    ra, rsa, rs2d, roff = oracle.permute_quant_block(bf16_bits(x), ids, E)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(s2d.cpu().numpy(), rs2d)
    assert np.array_equal(a_q.cpu().numpy(), ra)
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), rsa.view(np.uint32))


# ---------------------------------------------------------------------------
# block GEMM (tolerance)
# ---------------------------------------------------------------------------
def _block_problem(rng, counts, N, Kd):
    E = len(counts)
    off = ragged_offsets(counts)
    M = int(off[-1])
    A = random_e4m3(rng, (M, Kd))
    B = random_e4m3(rng, (E, N, Kd))
    sa = (10.0 ** rng.uniform(-3, 1, (M, Kd // 128))).astype(np.float32)
    sb = (10.0 ** rng.uniform(-4, -2, (E, N // 128, Kd // 128))).astype(np.float32)
    return A, sa, B, sb, off


BLOCK_SHAPES = [
    # counts per expert, N, Kd
    ([5, 0, 9], 256, 128),
    ([130, 1, 0, 257, 128], 512, 256),      # several 128-token chunks per expert
    ([300], 768, 384),
    ([17, 64, 200, 3], 256, 384),
    ([129, 127], 256, 7168),                # long K: 56 blocks of scales
    # few rows per expert overall (64-token tiles) with one multi-chunk expert
    ([150, 0, 3, 40, 0, 0, 7, 0, 0, 0, 0, 0, 0, 0, 0, 1], 256, 512),
]


@pytest.mark.parametrize("counts,N,Kd", BLOCK_SHAPES)
def test_grouped_gemm_block_bf16(counts, N, Kd):
    rng = np.random.default_rng(3 * sum(counts) + Kd)
    A, sa, B, sb, off = _block_problem(rng, counts, N, Kd)
    C = moe.moe_grouped_gemm_block(_t(A), _t(sa), _t(B), _t(sb), _t(off), moe.EPI_BF16)
    ref = oracle.grouped_gemm_block(A, sa, B, sb, off)
    got = bf16_np(C)
    # per element: fp32 accumulation of the scaled block partials + one bf16 rounding
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max())
    assert_parity(got, ref, "block gemm bf16")


@pytest.mark.parametrize("counts,N,Kd", BLOCK_SHAPES)
def test_grouped_gemm_block_silu(counts, N, Kd):
    rng = np.random.default_rng(5 * sum(counts) + N)
    A, sa, B, sb, off = _block_problem(rng, counts, N, Kd)
    C = moe.moe_grouped_gemm_block(_t(A), _t(sa), _t(B), _t(sb), _t(off), moe.EPI_SILU_MUL)
    ref = oracle.silu_mul(oracle.grouped_gemm_block(A, sa, B, sb, off))
    got = bf16_np(C)
    assert_parity(got, ref, "block gemm silu")
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-4 * np.abs(ref).max())


def test_grouped_gemm_block_scales_per_block():
    """Each K block carries its own scale (1e-3..1e3 across the blocks of a
    row, and across the weight blocks): a kernel that applied one scale per
    row or per tile would be off by orders of magnitude."""
    rng = np.random.default_rng(9)
    A, _, B, _, off = _block_problem(rng, [200, 60], 256, 1024)
    M, KB = A.shape[0], 8
    sa = (10.0 ** rng.uniform(-3, 3, (M, KB))).astype(np.float32)
    sb = (10.0 ** rng.uniform(-3, 3, (2, 2, KB))).astype(np.float32)
    C = moe.moe_grouped_gemm_block(_t(A), _t(sa), _t(B), _t(sb), _t(off), moe.EPI_BF16)
    ref = oracle.grouped_gemm_block(A, sa, B, sb, off)
    got = bf16_np(C)
    row_err = np.abs(got - ref).max(1) / np.abs(ref).max(1)
    assert row_err.max() <= 2.0 ** -7


# ---------------------------------------------------------------------------
# whole layer
# ---------------------------------------------------------------------------
def _check_block_layer(wl, seed, n_sample=None):
    dev_gen = wl.T > 64
    d = synth.make_inputs(wl, seed=seed, device=DEV if dev_gen else "cpu")
    d = {k: (None if v is None else v.to(DEV)) for k, v in d.items()}
    layer = moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                         wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                         n_shared=wl.n_shared, quant="block")
    out = layer(d["x"], d["logits"])
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    n = synth.to_numpy_inputs(d)
    if n_sample is None:
        tokens = np.arange(wl.T, dtype=np.int64)
    else:  # a token of every tile of both block GEMMs, the tile edges, 40 random ones
        ids, _ = oracle.gate(n["logits"], n["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                             wl.scoring, wl.renormalize, wl.rsf)
        if wl.n_shared:
            shared = np.arange(wl.E, wl.E + wl.n_shared, dtype=np.int32)
            ids = np.concatenate([ids, np.broadcast_to(shared, (wl.T, wl.n_shared))], axis=1)
        tokens, ntiles = tile_cover_tokens(ids, wl.E + wl.n_shared, quant="block", seed=seed)
    t0 = time.time()
    ref, _, _ = oracle.forward_tokens_block(n["x"], n["logits"], n["bias"], n["w13"], n["s13"],
                                            n["w2"], n["s2"], wl.num_groups, wl.topk_group,
                                            wl.top_k, wl.scoring, wl.renormalize, wl.rsf,
                                            tokens=tokens, n_shared=wl.n_shared)
    if n_sample is not None:
        print(f"{wl.name}: {tokens.size} tokens cover {ntiles} tiles; "
              f"oracle {time.time() - t0:.1f} s")
    got = bf16_np(out[torch.from_numpy(tokens).to(DEV)])
    assert_parity(got, ref, wl.name)
    return layer, d, out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_block_tiny(seed):
    _check_block_layer(synth.WORKLOADS["tiny_block"], seed)


def test_forward_block_dsv3_decode_t128():
    _check_block_layer(synth.WORKLOADS["dsv3_decode_t128_block"], 0)


@pytest.mark.parametrize("name", ["dsv3_prefill_t8192_block", "mixtral_t4096_block"])
def test_forward_block_large_every_tile(name):
    _check_block_layer(synth.WORKLOADS[name], 0, n_sample="tiles")


def test_forward_block_shared_expert_ragged_and_host_buffers():
    wl = synth.Workload("block_shared", 300, 384, 256, 24, 4, 2, 6, synth.SIGMOID, True, 2.5,
                        "normal", n_shared=1, quant="block")
    layer, d, out = _check_block_layer(wl, 3)
    xh, lh = d["x"].cpu().pin_memory(), d["logits"].cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, lh, oh)
    torch.cuda.synchronize()
    assert torch.equal(oh.view(torch.int16), out.cpu().view(torch.int16))
