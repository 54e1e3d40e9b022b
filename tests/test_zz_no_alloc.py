"""The allocation-free pre-reorder entry point, moe_permute_quant_noalloc.

Some callers cannot allocate device memory or hand the library a workspace:
a plug-in running inside another runtime that owns all device memory and
gives it only its input and output buffers, or a latency-critical loop that
must not allocate. For them the library offers moe_permute_quant_noalloc,
which uses a fixed scratch array in the library's own device memory instead
of a caller workspace. These tests call it through the C ABI and check that
it returns exactly what moe_permute_quant (which takes the caller's
workspace) returns, on two calls in a row, so the second call must not be
disturbed by what the first left in the shared scratch.

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
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = _lib()
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the first call uses more scratch (more 32-token blocks x experts) than
    # the second, so stale entries would be visible if any were read
    for call, (T, H, E, K) in enumerate([(4099, 256, 64, 6), (300, 7168, 256, 8)]):
        rng = np.random.default_rng(100 + call)
        ids = torch.from_numpy(
            np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)).to(dev)
        x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
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
        assert torch.equal(off, ref_off), f"call {call}: offsets"
        assert torch.equal(s2d, ref_s2d), f"call {call}: src2dst"
        assert torch.equal(sa.view(torch.int32), ref_sa.view(torch.int32)), f"call {call}: scales"
        assert torch.equal(a_q, ref_aq), f"call {call}: codes"
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
