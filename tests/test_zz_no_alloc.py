"""The allocation-free pre-reorder entry point, moe_permute_quant_noalloc.

Some callers cannot allocate device memory or hand the library a workspace:
a plug-in running inside another runtime that owns all device memory and
gives it only its input and output buffers, or a latency-critical loop that
must not allocate. For them the library offers moe_permute_quant_noalloc,
which uses a fixed scratch array in the library's own device memory instead
of a caller workspace. These tests call it through the C ABI, twice in a
row, and check every output bit for bit against moe_permute_quant (which
takes the caller's workspace) and against the CPU oracle. Both calls are
large enough to take the three-kernel path, the one that uses the scratch,
and the first uses more of it than the second, so the second call would
read the first call's leftovers if any of them were read at all.

This file is collected after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe

MOE_OK = 0
MOE_ERR_WORKSPACE = -3
SCRATCH_BYTES = 4 << 20  # MOE_PERMUTE_NOALLOC_SCRATCH_BYTES


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    return moe.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls():
    import oracle
    lib = _lib()
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # both calls have more than 512 tokens, so both take the three-kernel path
    # (per-block expert bitmasks and bases in the scratch); the first covers
    # 256 blocks of 32 tokens x 256 experts, the second 32 x 256
    cases = [(8192, 256, 256, 8), (1024, 7168, 256, 8)]
    for T, H, E, K in cases:
        assert T > 512 and lib.moe_permute_workspace_size(T, E, K) <= SCRATCH_BYTES
    need = [lib.moe_permute_workspace_size(T, E, K) for T, _, E, K in cases]
    assert need[0] > need[1]
    for call, (T, H, E, K) in enumerate(cases):
        rng = np.random.default_rng(100 + call)
        ids_np = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
        ids = torch.from_numpy(ids_np).to(dev)
        x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
        x_bits = x.view(torch.int16).numpy().view(np.uint16).copy()
        x = x.to(dev)
        ref_aq, ref_sa, ref_s2d, ref_off = moe.moe_permute_quant(x, ids, E)
        M = T * K
        a_q = torch.empty((M, H), dtype=torch.uint8, device=dev)
        sa = torch.empty(M, dtype=torch.float32, device=dev)
        s2d = torch.empty(M, dtype=torch.int32, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        st = lib.moe_permute_quant_noalloc(_p(x), _p(ids), T, H, E, K, _p(a_q), _p(sa),
                                           _p(s2d), _p(off), stream)
        assert st == MOE_OK
        torch.cuda.synchronize()
        # the same bits as the workspace entry point
        assert torch.equal(off, ref_off), f"call {call}: offsets"
        assert torch.equal(s2d, ref_s2d), f"call {call}: src2dst"
        assert torch.equal(sa.view(torch.int32), ref_sa.view(torch.int32)), f"call {call}: scales"
        assert torch.equal(a_q, ref_aq), f"call {call}: codes"
        # and the oracle's
        o_aq, o_sa, o_s2d, o_off = oracle.permute_quant(x_bits, ids_np, E)
        assert np.array_equal(off.cpu().numpy(), o_off), f"call {call}: offsets vs oracle"
        assert np.array_equal(s2d.cpu().numpy(), o_s2d), f"call {call}: src2dst vs oracle"
        assert np.array_equal(sa.cpu().numpy().view(np.uint32), o_sa.view(np.uint32)), \
            f"call {call}: scales vs oracle"
        assert np.array_equal(a_q.cpu().numpy(), o_aq), f"call {call}: codes vs oracle"
    assert moe.moe_device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Sizes whose scratch would exceed the fixed array are refused before
    anything touches the device."""
    lib = _lib()
    E, K = 256, 8
    assert lib.moe_permute_workspace_size(65536, E, K) <= SCRATCH_BYTES
    T = 65536 + 32
    assert lib.moe_permute_workspace_size(T, E, K) > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x100000)  # aligned, never dereferenced
    st = lib.moe_permute_quant_noalloc(fake, fake, T, 64, E, K, fake, fake, fake, fake, None)
    assert st == MOE_ERR_WORKSPACE
