"""The pipelined host entry point (moe_forward_host_pipelined) on the GPU:
n batches from pinned host memory, with copies on the library's copy streams
overlapping the forwards, give for every batch exactly what the device
entry point gives for that batch alone. That holds bit for bit, for every
quantisation mode and with shared experts. The layer itself is checked
against the oracle elsewhere; here the comparison is with the device
forward, whose parity tests cover it."""
import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
from moe_expert_layer_grouped_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert moe.moe_device_status() == 0


def _layer(wl, seed=0):
    d = synth.make_inputs(wl, seed=seed, device=DEV)
    fp4 = dict(g13=d["g13"], g2=d["g2"], ga1=wl.ga1, ga2=wl.ga2) if wl.quant == "nvfp4" else None
    return moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                        wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                        n_shared=wl.n_shared, quant=wl.quant, nvfp4=fp4)


def _batches(wl, n, seed=1):
    out = []
    for b in range(n):
        d = synth.make_inputs(wl, seed=seed * 100 + b, device="cpu", weights=False)
        out.append((d["x"].pin_memory(), d["logits"].pin_memory()))
    return out


def _bits(t):
    return t.view(torch.int16).numpy().copy()


@pytest.mark.parametrize("name,n", [("tiny", 1), ("tiny", 2), ("tiny", 5), ("tiny_shared", 4),
                                    ("tiny_block", 5), ("tiny_nvfp4", 5),
                                    ("dsv3_decode_t128", 3), ("dsv3_decode_t128_block", 3),
                                    ("dsv3_decode_t128_nvfp4", 3)])
def test_pipelined_batches_equal_the_device_forward(name, n):
    wl = synth.WORKLOADS[name]
    layer = _layer(wl)
    bs = _batches(wl, n)
    outs = [torch.empty((wl.T, layer.H), dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    layer.forward_host_pipelined([b[0] for b in bs], [b[1] for b in bs], outs)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    for i, (x, lg) in enumerate(bs):
        ref = layer(x.to(DEV), lg.to(DEV))
        torch.cuda.synchronize()
        assert np.array_equal(_bits(outs[i]), _bits(ref.cpu())), (name, i)


def test_pipelined_reuses_host_buffers_across_batches():
    """The same x / logits buffers in several batches (as a serving loop that
    cycles a few staging buffers would pass them), and the same output buffer
    for batches i and i+2: the last batch written there wins."""
    wl = synth.WORKLOADS["tiny"]
    layer = _layer(wl)
    bs = _batches(wl, 2)
    xs = [bs[i % 2][0] for i in range(6)]
    ls = [bs[i % 2][1] for i in range(6)]
    o = [torch.empty((wl.T, layer.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    outs = [o[i % 2] for i in range(6)]
    layer.forward_host_pipelined(xs, ls, outs)
    torch.cuda.synchronize()
    for j in range(2):
        ref = layer(bs[j][0].to(DEV), bs[j][1].to(DEV)).cpu()
        assert np.array_equal(_bits(o[j]), _bits(ref))


def test_pipelined_then_stream_order():
    """Work queued on the caller's stream after the call sees every output:
    a device copy of an output made on the stream right after the call."""
    wl = synth.WORKLOADS["tiny_block"]
    layer = _layer(wl)
    bs = _batches(wl, 3, seed=7)
    outs = [torch.empty((wl.T, layer.H), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    layer.forward_host_pipelined([b[0] for b in bs], [b[1] for b in bs], outs)
    dev_copy = outs[2].to(DEV, non_blocking=True)  # queued on the same stream
    torch.cuda.synchronize()
    ref = layer(bs[2][0].to(DEV), bs[2][1].to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(dev_copy.view(torch.int16), ref.view(torch.int16))
