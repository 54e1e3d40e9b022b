"""Expert-parallel steps on the GPU through the C ABI: the receive-side
merge and the gather back (bit-exact against their definitions), the layer
on one rank holding every expert (equal to moe_forward bit for bit), and 2
and 4 ranks emulated on one GPU: each rank's launches run in turn, the
exchanges are device copies, and no kernel waits on another rank. Every
rank's output rows are the one-GPU layer's, bit for bit, and the oracle's
within the layer tolerance."""
import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
import oracle
from moe_expert_layer_grouped_gb300 import ep, synth

from gpu_util import assert_parity, bf16_np
from test_ep_gloo import recv_merge

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert moe.moe_device_status() == 0


def test_recv_reorder_and_return_gather_match_their_definitions():
    rng = np.random.default_rng(11)
    R, EPR, H = 3, 5, 256
    cnt = rng.integers(0, 40, (R, EPR)).astype(np.int32)
    cnt[1, 2] = 0
    cnt[2, :] = 0                                   # a source that sends nothing
    Mr = int(cnt.sum())
    rows = rng.integers(0, 256, (Mr, H)).astype(np.uint8)
    sc = rng.standard_normal(Mr).astype(np.float32)
    r_rows, r_sc, r_off, r_a2r = recv_merge(rows, sc, cnt)
    a_q, sa, off, a2r = moe.moe_ep_recv_reorder(torch.from_numpy(rows).to(DEV),
                                                torch.from_numpy(sc).to(DEV),
                                                torch.from_numpy(cnt).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(a2r.cpu().numpy(), r_a2r)
    assert np.array_equal(a_q.cpu().numpy(), r_rows)
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), r_sc.view(np.uint32))
    down = torch.randn((Mr, H), device=DEV).to(torch.bfloat16)
    back = moe.moe_ep_return_gather(down, a2r)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), down[a2r.long()].view(torch.int16))
    assert moe.moe_device_status() == 0


def test_recv_reorder_rejects_counts_that_do_not_add_up():
    cnt = torch.tensor([[3, 2]], dtype=torch.int32, device=DEV)        # 5 rows announced
    rows = torch.zeros((4, 64), dtype=torch.uint8, device=DEV)        # 4 arrive
    sc = torch.ones(4, dtype=torch.float32, device=DEV)
    _, _, off, _ = moe.moe_ep_recv_reorder(rows, sc, cnt)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.DEV_BAD_OFFSETS
    assert off.cpu().tolist() == [0, 0, 0]


def _problem(T, H, I, E, G, TG, K, seed=4):
    wl = synth.Workload("ep", T, H, I, E, G, TG, K, synth.SIGMOID, True, 2.5, "normal")
    d = synth.make_inputs(wl, seed=seed, device=DEV)
    return wl, d


def _one_gpu(wl, d):
    return moe.moe_forward(d["x"], d["logits"], d["bias"], d["w13"], d["s13"], d["w2"],
                           d["s2"], wl.num_groups, wl.topk_group, wl.top_k, wl.scoring,
                           wl.renormalize, wl.rsf)


@pytest.mark.parametrize("shape", [(128, 1024, 512, 32, 8, 4, 8),     # few rows per expert
                                   (2048, 1024, 512, 16, 4, 2, 4)])   # CTA-pair GEMMs
def test_one_rank_with_every_expert_equals_moe_forward(shape):
    wl, d = _problem(*shape)
    layer = moe.EPMoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.E,
                           wl.num_groups, wl.topk_group, wl.top_k, wl.scoring, wl.renormalize,
                           wl.rsf, ep.LoopbackExchange())
    out = layer(d["x"], d["logits"])
    ref = _one_gpu(wl, d)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert moe.moe_device_status() == 0


def _emulated(wl, d, R):
    """R ranks on one GPU: rank r holds experts [r*E/R, (r+1)*E/R) and tokens
    [r*T/R, (r+1)*T/R); each step runs for every rank in turn and the
    all-to-alls are device copies in source-rank order."""
    E, EPR, Tr = wl.E, wl.E // R, wl.T // R
    src = []
    for s in range(R):
        x, lg = d["x"][s * Tr:(s + 1) * Tr], d["logits"][s * Tr:(s + 1) * Tr]
        ids, w = moe.moe_gate(lg, d["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                              wl.scoring, wl.renormalize, wl.rsf)
        a_q, sa, s2d, off, cnt = moe.moe_ep_dispatch(x, ids, E, R)
        src.append(dict(w=w, a_q=a_q, sa=sa, s2d=s2d, off=off.cpu().tolist(), cnt=cnt))
    backs = []
    for r in range(R):
        lo, hi = r * EPR, (r + 1) * EPR
        counts = torch.stack([s["cnt"][lo:hi] for s in src]).contiguous()
        rows = torch.cat([s["a_q"][s["off"][lo]:s["off"][hi]] for s in src]).contiguous()
        scales = torch.cat([s["sa"][s["off"][lo]:s["off"][hi]] for s in src]).contiguous()
        back = moe.moe_ep_expert_forward(rows, scales, counts, d["w13"][lo:hi].contiguous(),
                                         d["s13"][lo:hi].contiguous(),
                                         d["w2"][lo:hi].contiguous(),
                                         d["s2"][lo:hi].contiguous())
        sizes = [s["off"][hi] - s["off"][lo] for s in src]
        backs.append(torch.split(back, sizes))
    outs = []
    for s_i, s in enumerate(src):
        ret = torch.cat([backs[r][s_i] for r in range(R)]).contiguous()
        outs.append(moe.moe_ep_combine(ret, s["s2d"], s["w"]))
    return torch.cat(outs)


@pytest.mark.parametrize("R", [2, 4])
@pytest.mark.parametrize("shape", [(128, 1024, 512, 32, 8, 4, 8),
                                   (2048, 1024, 512, 16, 4, 2, 4)])
def test_emulated_ranks_equal_the_one_gpu_layer_and_the_oracle(R, shape):
    wl, d = _problem(*shape)
    out = _emulated(wl, d, R)
    ref = _one_gpu(wl, d)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    tokens = np.arange(0, wl.T, max(1, wl.T // 64))
    n = synth.to_numpy_inputs(d)
    o, _, _ = oracle.forward_tokens(n["x"], n["logits"], n["bias"], n["w13"], n["s13"], n["w2"],
                                    n["s2"], wl.num_groups, wl.topk_group, wl.top_k, wl.scoring,
                                    wl.renormalize, wl.rsf, tokens=tokens)
    assert_parity(bf16_np(out[torch.from_numpy(tokens).to(DEV)]), o, f"ep R={R}")
