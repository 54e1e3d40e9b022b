"""Benchmark of the MoE layer forward on GB300.

One step = one moe_forward over one batch of synthetic tokens (gate,
pre-reorder + FP8 quant, w13 GEMM + SiLU*mul, requant, w2 GEMM, weighted
post-reorder). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-secondary] [--no-cpu-baseline]

Default workload: DeepSeek-V3-shaped decode, T=128 tokens, H=7168, I=2048,
E=256 experts (8 groups, 4 kept, top-8), sigmoid + correction bias, rsf 2.5;
FP8 e4m3 per-channel weights resident in HBM. A second object in the same
line ("secondary") reports the T=8192 prefill shape of the same layer.
Multi-GPU (torchrun): every rank runs an independent replica on its own
batch (weak scaling; the data path has no collective); the barrier and the
max-over-ranks time use NCCL only for timing.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "dsv3_decode_t128"
SECONDARY_WORKLOAD = "dsv3_prefill_t8192"
# earlier GB300 measurements, used only without the measured peaks file:
# a copy at 6.8 TB/s, cuBLAS bf16 at 1.9 PFLOP/s in a burst and ~1.7 sustained
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
FP8_PER_BF16 = 2.0  # nominal dense FP8 : bf16 tensor throughput
FP4_PER_BF16 = 6.0  # nominal dense FP4 : bf16 on GB300 (13.5 : 2.25 PFLOP/s)


def launches_per_forward(wl):
    """Kernels one forward launches: gate, pre-reorder (one launch for T <= 512
    and T*K <= 4096 slots, else three), w13 GEMM, requant, w2 GEMM, post-reorder."""
    k = wl.top_k + wl.n_shared
    pre = 1 if (wl.T <= 512 and wl.T * k <= 4096) else 3
    return 5 + pre
N_BATCHES = 4  # distinct token batches cycled through the timed steps


DTYPES = {"token": "fp8_e4m3 x fp8_e4m3 -> fp32 (bf16 io)",
          "block": "fp8_e4m3 x fp8_e4m3, 128-blocks -> fp32 (bf16 io)",
          "nvfp4": "e2m1 x e2m1, e4m3 scale per 16 -> fp32 (bf16 io)"}
DATA = {"token": "synthetic (seeded; weights ~N(0,0.02) quantised to e4m3 per channel)",
        "block": "synthetic (seeded; weights ~N(0,0.02) quantised to e4m3 per 128x128 block)",
        "nvfp4": "synthetic (seeded; NVFP4 weights drawn in the format, std ~0.02)"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    sm_max=float(p.get("sm_max_mhz", 0)), source="measured")
    except Exception:
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS,
                    bf16_sustained=FALLBACK_BF16_TFLOPS_SUSTAINED, sm_max=2070.0,
                    source="fallback")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = [l for (t, l) in self.lines if t0 <= t <= t1] or [l for (_, l) in self.lines[-3:]]
        for l in rows:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# algorithmic work of one step
# ---------------------------------------------------------------------------
def step_work(wl, offsets_list):
    """Algorithmic bytes / flops per forward, averaged over the batches.
    Weights count once per expert that received at least one token. Shared
    experts count as experts every token visits (E + n_shared experts,
    top_k + n_shared slots); the logits cover the E routed experts."""
    T, H, I, E, K = wl.T, wl.H, wl.I, wl.E + wl.n_shared, wl.top_k + wl.n_shared
    M = T * K
    res = []
    for off in offsets_list:
        cnt = off[1:] - off[:-1]
        active = int((cnt > 0).sum())
        if wl.quant == "nvfp4":  # half-byte codes, a scale byte per 16, a global scale
            w13 = active * (2 * I * H // 2 + 2 * I * H // 16 + 4)
            w2 = active * (H * I // 2 + H * I // 16 + 4)
            sa, sa2 = M * H // 16, M * I // 16
            gemm13_bytes = w13 + M * H // 2 + sa + M * I * 2 + (E + 1) * 4
            gemm2_bytes = w2 + M * I // 2 + sa2 + M * H * 2 + (E + 1) * 4
            flops13 = 2.0 * M * 2 * I * H
            flops2 = 2.0 * M * H * I
            layer_bytes = w13 + w2 + T * H * 2 + T * wl.E * 4 + T * H * 2
            res.append(dict(active=active, gemm13_bytes=gemm13_bytes, gemm2_bytes=gemm2_bytes,
                            flops13=flops13, flops2=flops2, layer_bytes=layer_bytes,
                            layer_flops=flops13 + flops2))
            continue
        if wl.quant == "block":  # scales per 128 x 128 weight block / 128 channels
            w13 = active * (2 * I * H + (2 * I // 128) * (H // 128) * 4)
            w2 = active * (H * I + (H // 128) * (I // 128) * 4)
            sa, sa2 = M * (H // 128) * 4, M * (I // 128) * 4
        else:
            w13 = active * (2 * I * H + 2 * I * 4)
            w2 = active * (H * I + H * 4)
            sa, sa2 = M * 4, M * 4
        gemm13_bytes = w13 + M * H + sa + M * I * 2 + (E + 1) * 4
        gemm2_bytes = w2 + M * I + sa2 + M * H * 2 + (E + 1) * 4
        flops13 = 2.0 * M * 2 * I * H
        flops2 = 2.0 * M * H * I
        layer_bytes = w13 + w2 + T * H * 2 + T * wl.E * 4 + T * H * 2
        res.append(dict(active=active, gemm13_bytes=gemm13_bytes, gemm2_bytes=gemm2_bytes,
                        flops13=flops13, flops2=flops2, layer_bytes=layer_bytes,
                        layer_flops=flops13 + flops2))
    avg = {k: sum(r[k] for r in res) / len(res) for k in res[0]}
    return avg


def max_over_ranks(value, dist, device):
    """The slowest rank's value (timing is taken as the max over ranks)."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms_per_step):
    """Whole-job throughput: every rank processes its own batch each step."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def rank_seed(seed, rank):
    """Each replica draws its own token batches (weights are per-rank copies)."""
    return seed + rank


def _strip_comments(src):
    """C++ source without comments and blank lines (the hash below follows
    the code, not its comments)."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            i = src.find("\n", i)
            if i < 0:
                break
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] == '"':  # string literal (inline PTX): copied as is
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return "\n".join(l.rstrip() for l in "".join(out).splitlines() if l.strip())


def kernel_source_hash():
    """Identifies the code of the grouped GEMM (comments and blank lines
    ignored), to tell whether a recorded ncu capture was taken on it."""
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_common.cuh", "ptx.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "moe_expert_layer_grouped_gb300", "csrc", f)) as fh:
            h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """dram bytes per launch of the w13 GEMM from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_w13_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def make_batches(wl, seed, dev, synth):
    batches = []
    for b in range(N_BATCHES):
        d = synth.make_inputs(wl, seed=seed * 100 + b, device=dev, weights=False)
        batches.append((d["x"], d["logits"]))
    return batches


def align(torch, barrier):
    """Every rank's work done and, with several ranks, all ranks at the same
    point: taken on both sides of a timed region."""
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
        torch.cuda.synchronize()


def time_forward(layer, batches, steps, warmup, torch, out, barrier=None):
    for i in range(warmup):
        x, l = batches[i % len(batches)]
        layer(x, l, out=out)
    align(torch, barrier)
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(steps):
        x, l = batches[i % len(batches)]
        layer(x, l, out=out)
    e1.record(st)
    align(torch, barrier)
    return e0.elapsed_time(e1)


def time_breakdown(moe, layer, wl, batches, steps, torch):
    """The same launches as moe_forward, issued step by step through the C ABI
    with events between them, to time each kernel inside a running step.
    With shared experts the gate's K routed slots are widened to K + n_shared
    by a torch copy between the gate's and the permute's events (moe_forward
    does this inside its gate kernel), so it is not part of any kernel time."""
    dev = batches[0][0].device
    S = wl.n_shared
    T, H, I, E, K = wl.T, wl.H, wl.I, wl.E + S, wl.top_k + S
    M = T * K
    ids_r = torch.empty((T, wl.top_k), dtype=torch.int32, device=dev)
    w_r = torch.empty((T, wl.top_k), dtype=torch.float32, device=dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    if S:
        ids[:, wl.top_k:] = torch.arange(wl.E, E, dtype=torch.int32, device=dev)
        w[:, wl.top_k:] = 1.0
    block = wl.quant == "block"
    fp4 = wl.quant == "nvfp4"
    a_q = torch.empty((M, H), dtype=torch.uint8, device=dev)
    sa = torch.empty((M, H // 128) if block else M, dtype=torch.float32, device=dev)
    s2d = torch.empty(M, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    pws = torch.empty(max(moe.moe_permute_workspace_size(T, E, K), 256), dtype=torch.uint8,
                      device=dev)
    h = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
    q2 = torch.empty((M, I), dtype=torch.uint8, device=dev)
    sa2 = torch.empty((M, I // 128) if block else M, dtype=torch.float32, device=dev)
    down = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if fp4:  # NVFP4 codes and E4M3 block scales, preallocated like the FP8 buffers
        fa = torch.empty((M, H // 2), dtype=torch.uint8, device=dev)
        fsa = torch.empty((M, H // 16), dtype=torch.uint8, device=dev)
        fq = torch.empty((M, I // 2), dtype=torch.uint8, device=dev)
        fsf = torch.empty((M, I // 16), dtype=torch.uint8, device=dev)
    names = ["gate", "permute_quant", "grouped_gemm_w13", "act_quant", "grouped_gemm_w2",
             "unpermute_sum"]
    st = torch.cuda.current_stream()

    def one(i, ev):
        x, l = batches[i % len(batches)]
        if ev: ev[0].record(st)
        moe.moe_gate(l, layer.bias, wl.num_groups, wl.topk_group, wl.top_k, wl.scoring,
                     wl.renormalize, wl.rsf, topk_ids=ids if not S else ids_r,
                     topk_w=w if not S else w_r)
        if ev: ev[1].record(st)
        if S:
            ids[:, :wl.top_k] = ids_r
            w[:, :wl.top_k] = w_r
        if ev: ev[7].record(st)
        if fp4:  # (the layer holds the arranged weight scales)
            moe.moe_permute_quant_nvfp4(x, ids, E, layer.ga1, workspace=pws, a_q=fa, sf=fsa,
                                        src2dst=s2d, offsets=off)
            if ev: ev[2].record(st)
            moe.moe_grouped_gemm_nvfp4(fa, fsa, layer.ga1, layer.w13, layer.s13, layer.g13,
                                       off, moe.EPI_SILU_MUL, C=h)
            if ev: ev[3].record(st)
            moe.moe_act_quant_nvfp4(h, layer.ga2, q=fq, sf=fsf)
            if ev: ev[4].record(st)
            moe.moe_grouped_gemm_nvfp4(fq, fsf, layer.ga2, layer.w2, layer.s2, layer.g2,
                                       off, moe.EPI_BF16, C=down)
            if ev: ev[5].record(st)
            moe.moe_unpermute_sum(down, s2d, w, out=out)
            if ev: ev[6].record(st)
            return
        if block:
            moe.moe_permute_quant_block(x, ids, E, a_q=a_q, scale_a=sa, src2dst=s2d,
                                        offsets=off, workspace=pws)
        else:
            moe.moe_permute_quant(x, ids, E, a_q=a_q, scale_a=sa, src2dst=s2d, offsets=off,
                                  workspace=pws)
        if ev: ev[2].record(st)
        if block:
            moe.moe_grouped_gemm_block(a_q, sa, layer.w13, layer.s13, off, moe.EPI_SILU_MUL, C=h)
        else:
            moe.moe_grouped_gemm(a_q, sa, layer.w13, layer.s13, off, moe.EPI_SILU_MUL, C=h)
        if ev: ev[3].record(st)
        if block:
            moe.moe_act_quant_block(h, q=q2, scale=sa2)
        else:
            moe.moe_act_quant(h, q=q2, scale=sa2)
        if ev: ev[4].record(st)
        if block:
            moe.moe_grouped_gemm_block(q2, sa2, layer.w2, layer.s2, off, moe.EPI_BF16, C=down)
        else:
            moe.moe_grouped_gemm(q2, sa2, layer.w2, layer.s2, off, moe.EPI_BF16, C=down)
        if ev: ev[5].record(st)
        moe.moe_unpermute_sum(down, s2d, w, out=out)
        if ev: ev[6].record(st)

    for i in range(3):
        one(i, None)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(steps)]
    for i in range(steps):
        one(i, evs[i])
    torch.cuda.synchronize()
    tot = {n: 0.0 for n in names}
    for ev in evs:
        for j, n in enumerate(names):
            tot[n] += (ev[7] if j == 1 else ev[j]).elapsed_time(ev[j + 1])
    offs = []
    for b in range(len(batches)):
        one(b, None)
        torch.cuda.synchronize()
        offs.append(off.cpu().numpy().copy())
    return {n: tot[n] / steps for n in names}, offs


def time_graph(layer, batches, steps, warmup, torch):
    """Per-step time of graph replays of the forward (device time of the
    replays only; each batch is copied into the graph's buffers first)."""
    x = batches[0][0].clone()
    lg = batches[0][1].clone()
    out = torch.empty_like(x)
    g = layer.capture(x, lg, out)
    st = torch.cuda.current_stream()
    for i in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    total = 0.0
    for i in range(steps):
        xb, lb = batches[i % len(batches)]
        x.copy_(xb)
        lg.copy_(lb)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        g.replay()
        e1.record(st)
        e1.synchronize()
        total += e0.elapsed_time(e1)
    return total / steps


def time_e2e(layer, batches, steps, warmup, torch, barrier=None):
    """End to end through the public host-buffer API: every step copies its
    inputs from pinned host memory and its output back. The headline runs
    the steps through one moe_forward_host_pipelined call (MoELayer.
    forward_host_pipelined), where batch i+1's inputs and batch i-1's output
    cross the host link while batch i computes. The second figure calls
    moe_forward_host once per step, one batch at a time. Returns
    (pipelined ms/step, one-call-per-step ms/step, H2D bytes, D2H bytes)."""
    xs = [b[0].cpu().pin_memory() for b in batches]
    ls = [b[1].cpu().pin_memory() for b in batches]
    T, H = batches[0][0].shape
    outs = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in batches]
    st = torch.cuda.current_stream()

    def pick(n):
        idx = [i % len(batches) for i in range(n)]
        return [xs[j] for j in idx], [ls[j] for j in idx], [outs[j] for j in idx]

    layer.forward_host_pipelined(*pick(max(warmup, 3)))
    align(torch, barrier)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    args = pick(steps)
    e0.record(st)
    layer.forward_host_pipelined(*args)
    e1.record(st)
    align(torch, barrier)
    piped = e0.elapsed_time(e1) / steps

    for i in range(warmup):
        j = i % len(batches)
        layer.forward_host(xs[j], ls[j], outs[j])
    align(torch, barrier)
    e0.record(st)
    for i in range(steps):
        j = i % len(batches)
        layer.forward_host(xs[j], ls[j], outs[j])
    e1.record(st)
    align(torch, barrier)
    single = e0.elapsed_time(e1) / steps
    h2d = xs[0].numel() * 2 + ls[0].numel() * 4
    d2h = outs[0].numel() * 2
    return piped, single, h2d, d2h


def make_layer(moe, wl, d):
    fp4 = dict(g13=d["g13"], g2=d["g2"], ga1=wl.ga1, ga2=wl.ga2) if wl.quant == "nvfp4" else None
    return moe.MoELayer(d["w13"], d["s13"], d["w2"], d["s2"], d["bias"], wl.num_groups,
                        wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf, wl.T,
                        n_shared=wl.n_shared, quant=wl.quant, nvfp4=fp4)


def run_workload(moe, synth, torch, wl, seed, steps, warmup, dev, pk, want_clocks,
                 barrier=None):
    d = synth.make_inputs(wl, seed=seed, device=dev, weights=True)
    layer = make_layer(moe, wl, d)
    batches = make_batches(wl, seed, dev, synth)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
    clocks = ClockSampler(dev.index) if want_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    t0 = time.time()
    ms_total = time_forward(layer, batches, steps, warmup, torch, out, barrier)
    t1 = time.time()
    if clocks:
        clocks.stop()
    if moe.moe_device_status() != 0:
        raise RuntimeError("device error during the timed region")
    ms = ms_total / steps
    kern, offs = time_breakdown(moe, layer, wl, batches, max(10, min(steps, 200)), torch)
    work = step_work(wl, offs)
    return dict(layer=layer, batches=batches, ms=ms, ms_total=ms_total, kern=kern, work=work,
                clocks=clocks.summary(t0, t1) if clocks else None, t0=t0, t1=t1)


def roofline_decode(r, pk, workload):
    k = r["kern"]["grouped_gemm_w13"]
    bytes_ = r["work"]["gemm13_bytes"]
    achieved = bytes_ / (k * 1e-3) / 1e9
    tr = recorded_traffic(workload)
    return {"kernel": "grouped_gemm_w13", "bound": "hbm", "achieved": round(achieved, 1),
            "peak": pk["hbm"], "unit": "GB/s", "frac": round(achieved / pk["hbm"], 4),
            "traffic": tr, "algorithmic_bytes_per_launch": int(bytes_),
            "launch_ms": round(k, 4), "peak_source": f"{pk['source']} hbm_gbs"}


def tensor_ratio(wl):
    """Nominal dense tensor throughput of the workload's operand type over bf16."""
    return FP4_PER_BF16 if wl.quant == "nvfp4" else FP8_PER_BF16


def roofline_prefill(r, pk, clocks=None, ratio=FP8_PER_BF16):
    """Tensor roofline of the w13 GEMM. The GEMM is timed in a loop of a
    fraction of a second at full clock, a burst, so the denominator is the
    burst bf16 figure x the FP8:bf16 ratio; the sustained-derived fraction
    and a clock-normalised figure (the launch time scaled by the median SM
    clock over the maximum, i.e. the rate at the maximum clock) stand beside
    it."""
    k = r["kern"]["grouped_gemm_w13"]
    fl = r["work"]["flops13"]
    achieved = fl / (k * 1e-3) / 1e12
    peak = pk["bf16"] * ratio
    peak_sus = pk["bf16_sustained"] * ratio
    kind = "fp4" if ratio == FP4_PER_BF16 else "fp8"
    out = {"kernel": "grouped_gemm_w13", "bound": "tensor", "achieved": round(achieved, 1),
           "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
           "traffic": None, "algorithmic_flops_per_launch": fl, "launch_ms": round(k, 4),
           "peak_source": f"{pk['source']} bf16_tflops (burst) x {ratio} ({kind}/bf16)",
           "frac_of_sustained_peak": round(achieved / peak_sus, 4),
           "sustained_peak": round(peak_sus, 1)}
    norm = clock_normalised(achieved, clocks, pk)
    if norm is not None:
        out["clock_normalised"] = {"achieved": round(norm[0], 1), "frac": round(norm[0] / peak, 4),
                                   "sm_mhz": norm[1], "to_mhz": norm[2]}
    return out


def clock_normalised(rate, clocks, pk):
    """The rate the same work would reach at the maximum SM clock: time x
    median SM MHz / max MHz. None without a clock record."""
    if not clocks or not clocks.get("sm_mhz"):
        return None
    mx = clocks.get("sm_max_mhz") or pk.get("sm_max") or 2070.0
    med = float(clocks["sm_mhz"])
    if med <= 0 or mx <= 0:
        return None
    return rate * mx / med, med, mx


def layer_fracs(r, pk, clocks=None, ratio=FP8_PER_BF16):
    """The layer's tensor fraction (whole step) for its operand type (FP8, or
    FP4 with ratio FP4_PER_BF16): burst denominator, the sustained one, and
    clock-normalised."""
    kind = "fp4" if ratio == FP4_PER_BF16 else "fp8"
    tf = r["work"]["layer_flops"] / (r["ms"] * 1e-3) / 1e12
    out = {f"layer_{kind}_tensor_frac": round(tf / (pk["bf16"] * ratio), 4),
           f"layer_{kind}_tensor_frac_of_sustained": round(tf / (pk["bf16_sustained"] * ratio),
                                                           4)}
    norm = clock_normalised(tf, clocks, pk)
    if norm is not None:
        out[f"layer_{kind}_tensor_frac_clock_normalised"] = round(norm[0] / (pk["bf16"] * ratio),
                                                                  4)
    return out


def layer_bound(r, pk, ratio=FP8_PER_BF16):
    """The layer's own roofline: the larger of its tensor time (all GEMM
    FLOPs at the burst peak of its operand type) and its HBM time (the bytes
    no implementation can avoid: the active experts' weights and scales, x,
    logits and out, at the measured copy rate), and the step time's
    fraction of it. Intermediates (permuted rows, h, down) are not counted:
    they are this implementation's choice."""
    t_ms = r["work"]["layer_flops"] / (pk["bf16"] * ratio * 1e12) * 1e3
    h_ms = r["work"]["layer_bytes"] / (pk["hbm"] * 1e9) * 1e3
    bound = max(t_ms, h_ms)
    return {"bound": "tensor" if t_ms >= h_ms else "hbm", "tensor_ms": round(t_ms, 4),
            "hbm_ms": round(h_ms, 4), "frac": round(bound / r["ms"], 4)}


def workload_config(wl, world):
    """The `config` object of both arms' JSON lines: the workload and its
    shapes, nothing measured."""
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
            "num_groups": wl.num_groups, "topk_group": wl.topk_group, "top_k": wl.top_k,
            "scoring": "sigmoid" if wl.scoring == 0 else "softmax", "rsf": wl.rsf,
            "n_shared": wl.n_shared, "quant": wl.quant, "batches_cycled": N_BATCHES,
            "l2": "no flush: each step streams the active experts' weights (GBs, see "
                  "layer_bytes_gb) through the 129 MB L2",
            "parallelism": f"replicas x{world} (no collective on the data path)"}


def oracle_forward(oracle, synth, wl, n):
    """The oracle's whole-layer function for the workload's format, as
    f(tokens) -> (out, ids, w); n: the inputs as numpy arrays."""
    if wl.quant == "nvfp4":
        import torch
        w13 = synth.unpack_e2m1(torch.from_numpy(n["w13"])).numpy()
        w2 = synth.unpack_e2m1(torch.from_numpy(n["w2"])).numpy()
        return lambda tokens: oracle.forward_tokens_nvfp4(
            n["x"], n["logits"], n["bias"], w13, n["s13"], n["g13"], w2, n["s2"], n["g2"],
            wl.ga1, wl.ga2, wl.num_groups, wl.topk_group, wl.top_k, wl.scoring, wl.renormalize,
            wl.rsf, tokens=tokens, n_shared=wl.n_shared)
    fwd = oracle.forward_tokens_block if wl.quant == "block" else oracle.forward_tokens
    return lambda tokens: fwd(n["x"], n["logits"], n["bias"], n["w13"], n["s13"], n["w2"],
                              n["s2"], wl.num_groups, wl.topk_group, wl.top_k, wl.scoring,
                              wl.renormalize, wl.rsf, tokens=tokens, n_shared=wl.n_shared)


def cpu_baseline(synth, torch, wl, seed, r, budget_s=15.0):
    """The oracle, as it stands, on a bounded sample of tokens of the first
    timed batch; weights copied from the device."""
    import numpy as np
    import oracle
    L = r["layer"]
    d = {"w13": L.w13, "s13": L.s13, "w2": L.w2, "s2": L.s2, "bias": L.bias,
         "x": r["batches"][0][0], "logits": r["batches"][0][1]}
    if wl.quant == "nvfp4":  # the row-major block scales (the layer's are arranged)
        d.update(s13=L.s13_rows, s2=L.s2_rows, g13=L.g13, g2=L.g2)
    fwd = oracle_forward(oracle, synth, wl, synth.to_numpy_inputs(d))
    threads = oracle.get_threads()
    t = time.time()
    fwd(np.arange(min(threads, wl.T), dtype=np.int64))
    per_tok = (time.time() - t) / min(threads, wl.T)
    ntok = int(max(1, min(wl.T, budget_s / max(per_tok, 1e-6))))
    reps = max(1, int(budget_s / max(per_tok * ntok, 1e-6)))
    toks = np.tile(np.arange(ntok, dtype=np.int64), reps)
    t = time.time()
    fwd(toks)
    dt = time.time() - t
    return {"value": round(toks.size / dt, 3), "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{ntok} of the {wl.T} tokens of one {wl.name} batch, x{reps}, whole layer "
                      f"(gate..post-reorder), {dt:.1f} s"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import moe_expert_layer_grouped_gb300 as moe
    from moe_expert_layer_grouped_gb300 import synth
    import __graft_entry__
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist.barrier()
        if rank != 0:
            __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    wl = synth.WORKLOADS[args.workload]
    steps = args.steps if args.steps is not None else max(20, int(4000 * 128 / wl.T))
    warmup = max(3, args.warmup)
    seed = rank_seed(args.seed, rank)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    barrier = dist.barrier if world > 1 else None
    r = run_workload(moe, synth, torch, wl, seed, steps, warmup, dev, pk, want_clocks=True,
                     barrier=barrier)
    ms_total = max_over_ranks(r["ms_total"], dist if world > 1 else None, dev)
    ms = ms_total / steps
    value = job_tokens_per_s(wl.T, world, ms)

    # the clocks of the host-buffer runs too: they run right after the device-timed
    # region, and a power cap reached there shows up only in them
    e2e_clocks = ClockSampler(dev.index)
    e2e_clocks.start()
    time.sleep(0.3)
    te0 = time.time()
    e2e_ms, e2e1_ms, h2d, d2h = time_e2e(r["layer"], r["batches"], steps, warmup, torch,
                                         barrier)
    te1 = time.time()
    e2e_clocks.stop()
    graph_ms = time_graph(r["layer"], r["batches"], steps, warmup, torch)
    e2e_ms = max_over_ranks(e2e_ms, dist if world > 1 else None, dev)
    e2e1_ms = max_over_ranks(e2e1_ms, dist if world > 1 else None, dev)

    line = {
        "metric": "MoE-layer tokens/s + % of FP8/HBM roofline, DeepSeek-V3 shape T=128/8192",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPES[wl.quant],
        "data": DATA[wl.quant],
        "config": workload_config(wl, world),
        "layer_bytes_gb": round(r["work"]["layer_bytes"] / 1e9, 3),
        "tflops": round(r["work"]["layer_flops"] / (r["ms"] * 1e-3) / 1e12, 2),
        "layer_hbm_gbs": round(r["work"]["layer_bytes"] / (r["ms"] * 1e-3) / 1e9, 1),
        **(layer_fracs(r, pk, r["clocks"], tensor_ratio(wl)) if wl.T > 512 else {}),
        "layer_bound": layer_bound(r, pk, tensor_ratio(wl)),
        "active_experts": r["work"]["active"],
        "kernels_ms": {k: round(v, 4) for k, v in r["kern"].items()},
        "roofline": (roofline_decode(r, pk, wl.name) if wl.T <= 512
                     else roofline_prefill(r, pk, r["clocks"], tensor_ratio(wl))),
        "e2e": {"value": round(job_tokens_per_s(wl.T, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5),
                "clocks": e2e_clocks.summary(te0, te1),
                "api": "MoELayer.forward_host_pipelined -> moe_forward_host_pipelined: every "
                       "step's x and logits copied in from pinned host memory and its output "
                       "copied back, batch i+1's inputs and batch i-1's output in flight "
                       "while batch i computes",
                "one_call_per_step": {
                    "value": round(job_tokens_per_s(wl.T, world, e2e1_ms), 1),
                    "ms_per_step": round(e2e1_ms, 5),
                    "api": "MoELayer.forward_host -> moe_forward_host, one batch per call"}},
        "graph": {"ms_per_step": round(graph_ms, 5),
                  "note": "the same forward replayed from a CUDA graph (MoELayer.capture), "
                          "inputs copied into its fixed buffers between steps, copies untimed"},
        "gpu_launches": steps * launches_per_forward(wl),
        "clocks": r["clocks"],
    }
    if not args.no_secondary and rank == 0 and world == 1:
        wl2 = synth.WORKLOADS[SECONDARY_WORKLOAD]
        del r
        torch.cuda.empty_cache()
        s_steps = max(50, steps // 10)
        r2 = run_workload(moe, synth, torch, wl2, seed, s_steps, warmup, dev, pk,
                          want_clocks=True)
        line["secondary"] = {
            "workload": wl2.name, "T": wl2.T, "value": round(wl2.T / (r2["ms"] * 1e-3), 1),
            "unit": "tokens/s", "ms_per_step": round(r2["ms"], 4), "steps": s_steps,
            "tflops": round(r2["work"]["layer_flops"] / (r2["ms"] * 1e-3) / 1e12, 2),
            **layer_fracs(r2, pk, r2["clocks"]),
            "kernels_ms": {k: round(v, 4) for k, v in r2["kern"].items()},
            "roofline": roofline_prefill(r2, pk, r2["clocks"]), "clocks": r2["clocks"]}
        r = None
        del r2
        torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        d = synth.make_inputs(wl, seed=seed, device=dev, weights=True)
        layer = make_layer(moe, wl, d)
        line["cpu_baseline"] = cpu_baseline(synth, torch, wl, seed,
                                            {"layer": layer, "batches": make_batches(
                                                wl, seed, dev, synth)})
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, timed on the host cores
    on a bounded sample of the same workload (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from moe_expert_layer_grouped_gb300 import synth
    from oracle import build as oracle_build
    oracle_build.build()
    wl = synth.WORKLOADS[args.workload]
    steps = args.steps if args.steps is not None else 3
    warmup = max(0, args.warmup)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = synth.make_inputs(wl, seed=args.seed, device=dev, weights=True)
    n = synth.to_numpy_inputs(d)
    del d
    fwd = oracle_forward(oracle, synth, wl, n)
    threads = oracle.get_threads()
    t = time.time()
    fwd(np.arange(min(threads, wl.T), dtype=np.int64))
    per_tok = (time.time() - t) / min(threads, wl.T)
    # about 90 s for the whole run (warm-up included), at least one token per
    # oracle thread per step
    budget = 90.0 / max(1, steps + warmup)
    ntok = int(max(min(threads, wl.T), min(wl.T, budget / max(per_tok, 1e-6))))
    toks = np.arange(ntok, dtype=np.int64)
    for _ in range(warmup):
        fwd(toks)
    t = time.time()
    for _ in range(steps):
        fwd(toks)
    dt = (time.time() - t) / steps
    value = ntok / dt
    sample = (f"{ntok} of the {wl.T} tokens of one {wl.name} batch per step, whole layer "
              f"(gate..post-reorder) in fp64")
    line = {
        "impl": "reference",
        "metric": "MoE-layer tokens/s + % of FP8/HBM roofline, DeepSeek-V3 shape T=128/8192",
        "value": round(value, 3), "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
        "warmup": warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (codes decoded exactly)",
        "data": "synthetic (seeded)",
        "config": workload_config(wl, args.gpus),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
