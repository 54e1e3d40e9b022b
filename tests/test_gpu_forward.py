"""Whole-layer parity of moe_forward (C ABI, CUDA kernels) against the CPU
oracle on the five workloads: every token on the small ones, a fixed sample of
tokens on the large ones (a token's output depends on that token alone), run
through the same MoELayer call the benchmark times. Plus edge cases: the
per-row scale regression, guard bands around every output, empty and one-token
batches, the host-buffer entry point. Shared experts (moe_forward_shared)
are checked the same way on layers that add one or two of them."""
import time

import numpy as np
import pytest
import torch

import moe_expert_layer_grouped_gb300 as moe
import oracle
from moe_expert_layer_grouped_gb300 import synth

from gpu_util import assert_parity, bf16_bits, bf16_np, tile_cover_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert moe.moe_device_status() == 0


def _layer(wl, d):
    return moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                        wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                        n_shared=wl.n_shared)


def _oracle_tokens(wl, d, tokens):
    n = {k: (None if v is None else v) for k, v in synth.to_numpy_inputs(d).items()}
    return oracle.forward_tokens(n["x"], n["logits"], n["bias"], n["w13"], n["s13"], n["w2"],
                                 n["s2"], wl.num_groups, wl.topk_group, wl.top_k, wl.scoring,
                                 wl.renormalize, wl.rsf, tokens=tokens, n_shared=wl.n_shared)


def _cover_tokens(wl, d, seed, quant="token"):
    """Tokens that reach every tile of both GEMMs at the launch the forward
    uses (from the oracle's routing), plus 40 random ones and the ends."""
    n = synth.to_numpy_inputs({"logits": d["logits"], "bias": d["bias"]})
    ids, _ = oracle.gate(n["logits"], n["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                         wl.scoring, wl.renormalize, wl.rsf)
    S = wl.n_shared
    if S:
        shared = np.broadcast_to(np.arange(wl.E, wl.E + S, dtype=np.int32), (wl.T, S))
        ids = np.concatenate([ids, shared], axis=1)
    return tile_cover_tokens(ids, wl.E + S, quant=quant, seed=seed)


def _check_workload(wl, seed, device_gen, n_sample=None):
    """n_sample None: every token; "tiles": a token of every GEMM tile (and
    the tile edges) plus 40 random ones; an int: that many random ones."""
    d = synth.make_inputs(wl, seed=seed, device=DEV if device_gen else "cpu")
    d = {k: (None if v is None else v.to(DEV)) for k, v in d.items()}
    layer = _layer(wl, d)
    out = layer(d["x"], d["logits"])
    ids, w = moe.moe_gate(d["logits"], d["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                          wl.scoring, wl.renormalize, wl.rsf)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    ntiles = None
    if n_sample is None:
        tokens = np.arange(wl.T, dtype=np.int64)
    elif n_sample == "tiles":
        tokens, ntiles = _cover_tokens(wl, d, seed)
    else:
        rng = np.random.default_rng(seed)
        tokens = np.unique(np.concatenate([[0, wl.T - 1],
                                           rng.choice(wl.T, n_sample, replace=False)]))
    t0 = time.time()
    ref, rids, rw = _oracle_tokens(wl, d, tokens)
    dt = time.time() - t0
    if ntiles is not None:
        print(f"{wl.name}: {tokens.size} tokens cover {ntiles} tiles; oracle {dt:.1f} s")
    sel = torch.from_numpy(tokens).to(DEV)
    assert np.array_equal(ids[sel].cpu().numpy(), rids)
    assert np.array_equal(w[sel].cpu().numpy(), rw)
    got = bf16_np(out[sel])
    return assert_parity(got, ref, wl.name)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_tiny(seed):
    _check_workload(synth.WORKLOADS["tiny"], seed, device_gen=False)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_dsv3_decode_t128(seed):
    _check_workload(synth.WORKLOADS["dsv3_decode_t128"], seed, device_gen=True,
                    n_sample=None if seed == 0 else 32)


@pytest.mark.parametrize("name", ["dsv3_prefill_t8192", "mixtral_t4096", "dsv3_skewed_t16384",
                                  "dsv3_skewed_half_t16384"])
def test_forward_large_every_tile(name):
    _check_workload(synth.WORKLOADS[name], 0, device_gen=True, n_sample="tiles")


def test_skewed_half_device_inputs_split_about_half():
    # the benchmark draws its inputs on the device (another generator than
    # the CPU's): the hot experts still take about half of the assignments
    wl = synth.WORKLOADS["dsv3_skewed_half_t16384"]
    for seed in (0, 1):
        d = synth.make_inputs(wl, seed=seed, device=DEV, weights=False)
        ids, _ = moe.moe_gate(d["logits"], d["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                              wl.scoring, wl.renormalize, wl.rsf)
        ids = ids.cpu().numpy()
        share = np.mean(ids % 10 == 0)
        assert 0.40 <= share <= 0.60, (seed, share)
        assert not np.any(ids % 8 == 7)


@pytest.mark.parametrize("T,H,I,E,G,TG,K,scoring,rsf", [
    (1, 256, 128, 16, 4, 2, 4, synth.SIGMOID, 2.5),      # one token
    (5, 128, 64, 1, 1, 1, 1, synth.SOFTMAX, 1.0),        # dense: E=1, K=1
    (300, 384, 192, 24, 4, 2, 6, synth.SIGMOID, 2.5),    # ragged tiles
    (129, 512, 256, 3, 1, 1, 3, synth.SIGMOID, 1.0),     # every expert takes every token
])
def test_forward_shapes(T, H, I, E, G, TG, K, scoring, rsf):
    bias = "none" if scoring == synth.SOFTMAX else "normal"
    wl = synth.Workload("shape", T, H, I, E, G, TG, K, scoring, True, rsf, bias)
    _check_workload(wl, 3, device_gen=False)


@pytest.mark.parametrize("name,seed,n_sample", [
    ("tiny_shared", 0, None), ("tiny_shared", 1, None), ("tiny_shared", 2, None),
    ("dsv3_decode_t128_shared", 0, None), ("dsv3_prefill_t8192_shared", 0, "tiles"),
])
def test_forward_shared_expert(name, seed, n_sample):
    wl = synth.WORKLOADS[name]
    _check_workload(wl, seed, device_gen=wl.T > 8, n_sample=n_sample)


def test_forward_two_shared_experts_ragged():
    wl = synth.Workload("two_shared", 100, 256, 128, 16, 4, 2, 4, synth.SIGMOID, True, 2.5,
                        "normal", n_shared=2)
    _check_workload(wl, 7, device_gen=False)


def test_forward_shared_zero_and_host_buffers():
    """n_shared = 0 is moe_forward bit for bit; the host-buffer entry point
    gives the device one's output bit for bit."""
    wl = synth.WORKLOADS["tiny_shared"].with_tokens(40)
    d = {k: (None if v is None else v.to(DEV)) for k, v in synth.make_inputs(wl, 9).items()}
    E = wl.E
    cfg = (wl.num_groups, wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf)
    routed = (d["w13"][:E], d["s13"][:E], d["w2"][:E], d["s2"][:E])
    a = moe.moe_forward(d["x"], d["logits"], d["bias"], *routed, *cfg)
    b = moe.moe_forward_shared(d["x"], d["logits"], d["bias"], *routed, 0, *cfg)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    layer = _layer(wl, d)
    dev_out = layer(d["x"], d["logits"])
    xh, lh = d["x"].cpu().pin_memory(), d["logits"].cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, lh, oh)
    torch.cuda.synchronize()
    assert torch.equal(oh.view(torch.int16), dev_out.cpu().view(torch.int16))
    # the shared expert contributes: the layer differs from the routed-only one
    assert not torch.equal(dev_out, a)


@pytest.mark.parametrize("T,quant", [(48, "token"), (48, "block"), (1, "token")])
def test_forward_maximum_sizes(T, quant):
    """The largest arguments the library takes: E = 1024 experts, top-32 of
    them (4 of 8 groups kept), hidden size 16384; every token against the oracle."""
    wl = synth.Workload(f"max_{quant}", T, 16384, 128, 1024, 8, 4, 32, synth.SIGMOID, True, 2.5,
                        "normal", quant=quant)
    d = synth.make_inputs(wl, seed=11, device=DEV)
    layer = moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                         wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                         quant=quant)
    out = layer(d["x"], d["logits"])
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    n = synth.to_numpy_inputs(d)
    fwd = oracle.forward_tokens_block if quant == "block" else oracle.forward_tokens
    ref, _, _ = fwd(n["x"], n["logits"], n["bias"], n["w13"], n["s13"], n["w2"], n["s2"],
                    wl.num_groups, wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf)
    assert_parity(bf16_np(out), ref, wl.name)


@pytest.mark.parametrize("name", ["dsv3_decode_t128", "dsv3_decode_t128_block",
                                  "dsv3_decode_t128_shared"])
def test_forward_cuda_graph_replay(name):
    """A forward recorded into a CUDA graph, replayed on new inputs written
    into the same buffers, gives the eager forward's output bit for bit."""
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, seed=0, device=DEV)
    layer = moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                         wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                         n_shared=wl.n_shared, quant=wl.quant)
    x, logits = d["x"].clone(), d["logits"].clone()
    out = torch.empty_like(x)
    g = layer.capture(x, logits, out)
    for seed in (1, 2):
        b = synth.make_inputs(wl, seed=seed, device=DEV, weights=False)
        x.copy_(b["x"])
        logits.copy_(b["logits"])
        g.replay()
        eager = layer(b["x"], b["logits"])
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert moe.moe_device_status() == 0


def test_forward_rsf_linear_and_empty_batch():
    wl = synth.Workload("lin", 64, 256, 128, 16, 4, 2, 4, synth.SIGMOID, True, 1.0, "normal")
    d = {k: (None if v is None else v.to(DEV)) for k, v in synth.make_inputs(wl, 4).items()}
    args = (d["w13"], d["s13"], d["w2"], d["s2"], 4, 2, 4, synth.SIGMOID, True)
    o1 = moe.moe_forward(d["x"], d["logits"], d["bias"], *args[:4], *args[4:], 1.0)
    o2 = moe.moe_forward(d["x"], d["logits"], d["bias"], *args[:4], *args[4:], 2.0)
    # rsf scales the weights exactly by 2; only the final bf16 rounding differs
    assert torch.equal(o2, (o1.float() * 2).to(torch.bfloat16))
    empty = moe.moe_forward(d["x"][:0], d["logits"][:0], d["bias"], *args[:4], *args[4:], 1.0)
    assert empty.shape == (0, 256)


def test_row_scale_regression():
    """Tokens routed to the same experts with magnitudes 1e-3..1e3: each
    token's output must be right relative to its own size, which only a
    per-row scale_a gives (sglang #6772: scale_a indexed by expert id made
    EPMoE wrong without block quantisation)."""
    wl = synth.Workload("rows", 64, 256, 128, 4, 1, 1, 2, synth.SIGMOID, True, 1.0, "none")
    d = synth.make_inputs(wl, 5)
    d["x"] = (d["x"].float() * (10.0 ** torch.linspace(-3, 3, 64)).unsqueeze(1)).to(torch.bfloat16)
    d["logits"][:, :2] += 10.0  # everyone picks experts 0 and 1
    dd = {k: (None if v is None else v.to(DEV)) for k, v in d.items()}
    out = _layer(wl, dd)(dd["x"], dd["logits"])
    ref, _, _ = _oracle_tokens(wl, d, np.arange(64))
    got = bf16_np(out)
    per_token = np.abs(got - ref).max(1) / np.abs(ref).max(1)
    assert per_token.max() <= 2e-2, per_token.max()


def test_guard_bands_around_every_output():
    """Outputs written into the middle of larger buffers filled with a
    sentinel: nothing outside the documented extents changes."""
    T, H, I, E, K = 70, 256, 128, 8, 2
    wl = synth.Workload("guard", T, H, I, E, 1, 1, K, synth.SOFTMAX, True, 1.0, "none")
    d = {k: (None if v is None else v.to(DEV)) for k, v in synth.make_inputs(wl, 6).items()}
    G = 4096  # guard bytes on each side

    def guarded(nbytes):
        buf = torch.full((nbytes + 2 * G,), 0xA5, dtype=torch.uint8, device=DEV)
        return buf, buf[G:G + nbytes]

    def intact(buf, nbytes):
        return bool((buf[:G] == 0xA5).all() and (buf[G + nbytes:] == 0xA5).all())

    M = T * K
    b_ids, ids = guarded(M * 4)
    b_w, w = guarded(M * 4)
    moe.moe_gate(d["logits"], None, 1, 1, K, synth.SOFTMAX, True, 1.0,
                 topk_ids=ids.view(torch.int32).view(T, K), topk_w=w.view(torch.float32).view(T, K))
    ids_t, w_t = ids.view(torch.int32).view(T, K), w.view(torch.float32).view(T, K)
    b_aq, aq = guarded(M * H)
    b_sa, sa = guarded(M * 4)
    b_sd, sd = guarded(M * 4)
    b_off, off = guarded((E + 1) * 4)
    moe.moe_permute_quant(d["x"], ids_t, E, a_q=aq.view(M, H), scale_a=sa.view(torch.float32),
                          src2dst=sd.view(torch.int32), offsets=off.view(torch.int32))
    b_h, h = guarded(M * I * 2)
    moe.moe_grouped_gemm(aq.view(M, H), sa.view(torch.float32), d["w13"], d["s13"],
                         off.view(torch.int32), moe.EPI_SILU_MUL,
                         C=h.view(torch.bfloat16).view(M, I))
    b_q2, q2 = guarded(M * I)
    b_s2, s2 = guarded(M * 4)
    moe.moe_act_quant(h.view(torch.bfloat16).view(M, I), q=q2.view(M, I),
                      scale=s2.view(torch.float32))
    b_dn, dn = guarded(M * H * 2)
    moe.moe_grouped_gemm(q2.view(M, I), s2.view(torch.float32), d["w2"], d["s2"],
                         off.view(torch.int32), moe.EPI_BF16, C=dn.view(torch.bfloat16).view(M, H))
    b_out, out = guarded(T * H * 2)
    moe.moe_unpermute_sum(dn.view(torch.bfloat16).view(M, H), sd.view(torch.int32), w_t,
                          out=out.view(torch.bfloat16).view(T, H))
    torch.cuda.synchronize()
    for buf, n in [(b_ids, M * 4), (b_w, M * 4), (b_aq, M * H), (b_sa, M * 4), (b_sd, M * 4),
                   (b_off, (E + 1) * 4), (b_h, M * I * 2), (b_q2, M * I), (b_s2, M * 4),
                   (b_dn, M * H * 2), (b_out, T * H * 2)]:
        assert intact(buf, n)
    # and the step-by-step chain equals moe_forward
    full = moe.moe_forward(d["x"], d["logits"], None, d["w13"], d["s13"], d["w2"], d["s2"], 1, 1,
                           K, synth.SOFTMAX, True, 1.0)
    assert torch.equal(full, out.view(torch.bfloat16).view(T, H))


def test_forward_host_buffers_match_device_call():
    wl = synth.Workload("host", 32, 1024, 512, 32, 4, 2, 4, synth.SIGMOID, True, 2.5, "normal")
    d = {k: (None if v is None else v.to(DEV)) for k, v in synth.make_inputs(wl, 7, DEV).items()}
    layer = _layer(wl, d)
    ref = layer(d["x"], d["logits"]).cpu()
    xh = d["x"].cpu().pin_memory()
    lh = d["logits"].cpu().pin_memory()
    oh = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, lh, oh)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh, ref)
    # pinned buffers are read and written in place by the kernels; pageable
    # ones (and a mix) go through staging copies: the same result every way
    for pinned in [(False, False, False), (True, False, True), (False, True, True)]:
        xs = d["x"].cpu().pin_memory() if pinned[0] else d["x"].cpu().clone()
        ls = d["logits"].cpu().pin_memory() if pinned[1] else d["logits"].cpu().clone()
        os_ = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16)
        if pinned[2]:
            os_ = os_.pin_memory()
        layer.forward_host(xs, ls, os_)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(os_, ref), pinned
    assert moe.moe_device_status() == 0


def test_repeated_calls_are_deterministic():
    wl = synth.WORKLOADS["dsv3_decode_t128"]
    d = {k: (None if v is None else v.to(DEV)) for k, v in synth.make_inputs(wl, 0, DEV).items()}
    layer = _layer(wl, d)
    a = layer(d["x"], d["logits"]).clone()
    for _ in range(3):
        assert torch.equal(layer(d["x"], d["logits"]), a)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode_t128", "dsv3_prefill_t8192",
                                  "dsv3_decode_t128_block"])
def test_back_to_back_steps_share_the_workspace(name):
    """Forwards issued back to back on one stream (no host synchronisation,
    one workspace; the kernels of a step are chained to each other) give,
    batch by batch, the output of the same batch run on its own."""
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, seed=0, device=DEV)
    layer = moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                         wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                         n_shared=wl.n_shared, quant=wl.quant)
    batches = [synth.make_inputs(wl, seed=s, device=DEV, weights=False) for s in (1, 2, 3, 4)]
    alone = []
    for b in batches:
        alone.append(layer(b["x"], b["logits"]).clone())
        torch.cuda.synchronize()
    outs = [torch.empty_like(b["x"]) for b in batches]
    for _ in range(2):
        for b, o in zip(batches, outs):
            layer(b["x"], b["logits"], out=o)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    for a, o in zip(alone, outs):
        assert torch.equal(o.view(torch.int16), a.view(torch.int16))
