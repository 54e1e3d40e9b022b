"""Seeded synthetic inputs for the MoE layer forward.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds none of the layer's arithmetic: it only draws
tensors with torch's seeded generators and converts the expert weights to the
FP8 e4m3 storage format the layer consumes (per-output-channel scale =
row amax / 448, codes from torch's own e4m3fn cast), which is input
preparation, not a step of the forward.

Workloads (the shapes, value distributions and routing structure of a
DeepSeek-V3-style and a Mixtral-style MoE layer):
  tiny               T=8     H=128  I=64    E=8   G=1 TG=1 K=2 softmax rsf 1.0
  dsv3_decode_t128   T=128   H=7168 I=2048  E=256 G=8 TG=4 K=8 sigmoid rsf 2.5
                     bias ~N(0, 0.1)
  dsv3_prefill_t8192 T=8192  same layer, bias 0
  mixtral_t4096      T=4096  H=4096 I=14336 E=8   G=1 TG=1 K=2 softmax rsf 1.0
  dsv3_skewed_t16384 T=16384 same layer as decode; bias +3.0 on the 26
                     experts with e % 10 == 0, -10 on the 32 with e % 8 == 7,
                     the rest ~N(0, 0.1)
  dsv3_skewed_half_t16384 the same with +0.225 on the 26 hot experts: the
                     gate sends them about half of the token-expert
                     assignments (49.8 % with seed 0, 47-52 % over seeds;
                     ~185 experts active, up to 3400-5000 rows each) instead
                     of all of them
  dsv3_decode_t128_e32 / dsv3_prefill_t2048_e32: the DeepSeek-V3 layer with
                     32 experts, small cases for profiling
  *_shared           the same layers plus n_shared shared experts (DeepSeek-V3
                     has one, of the routed experts' size), stored after the
                     routed experts in w13/w2 and drawn after them from the
                     same streams, so the routed weights are unchanged
  *_block            the same layers with block-quantised FP8 weights
                     (DeepSeek-V3's checkpoint format: one scale per 128 x 128
                     block, s13 [E, 2I/128, H/128], s2 [E, H/128, I/128]) drawn
                     from the same fp32 values; tiny_block has I = 128
Hidden states and router logits ~N(0, 1); weights ~N(0, 0.02).
"""
from dataclasses import dataclass, replace
from typing import Optional

import torch

SIGMOID = 0
SOFTMAX = 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    num_groups: int
    topk_group: int
    top_k: int
    scoring: int
    renormalize: bool
    rsf: float
    bias: str  # "none" | "normal" | "zero" | "skewed"
    n_shared: int = 0  # shared experts, stored as experts E .. E+n_shared-1
    # "token": per-channel weight scales; "block": 128 x 128 blocks; "nvfp4":
    # E2M1 weights with an E4M3 scale per 16 along K and a global scale
    quant: str = "token"
    hot_bias: float = 3.0  # "skewed": the bias of the experts with e % 10 == 0
    # NVFP4 activations' global scales (calibrated input scales: about the
    # largest |x| and |h| over 6 x 448, so block scales use the E4M3 range)
    ga1: float = 5.0 / (6 * 448)
    ga2: float = 2.0 / (6 * 448)

    @property
    def M(self):
        return self.T * self.top_k

    def with_tokens(self, T):
        return replace(self, T=T, name=f"{self.name}@T{T}")


WORKLOADS = {
    "tiny": Workload("tiny", 8, 128, 64, 8, 1, 1, 2, SOFTMAX, True, 1.0, "none"),
    "dsv3_decode_t128": Workload("dsv3_decode_t128", 128, 7168, 2048, 256, 8, 4, 8,
                                 SIGMOID, True, 2.5, "normal"),
    "dsv3_prefill_t8192": Workload("dsv3_prefill_t8192", 8192, 7168, 2048, 256, 8, 4, 8,
                                   SIGMOID, True, 2.5, "zero"),
    "mixtral_t4096": Workload("mixtral_t4096", 4096, 4096, 14336, 8, 1, 1, 2, SOFTMAX,
                              True, 1.0, "none"),
    "dsv3_skewed_t16384": Workload("dsv3_skewed_t16384", 16384, 7168, 2048, 256, 8, 4, 8,
                                   SIGMOID, True, 2.5, "skewed"),
    # about half of the assignments to the 26 hot experts: with +3.0 every
    # token takes 8 of them (each group holds at least three, and 4 groups
    # are kept), so the hot bias is lowered until the gate splits ~50 / 50
    "dsv3_skewed_half_t16384": Workload("dsv3_skewed_half_t16384", 16384, 7168, 2048, 256, 8,
                                        4, 8, SIGMOID, True, 2.5, "skewed", hot_bias=0.225),
    # the same layer with 32 experts (1.4 GB of weights): small cases for
    # profiling the decode (weight-streaming) and prefill (tensor) GEMMs
    "dsv3_decode_t128_e32": Workload("dsv3_decode_t128_e32", 128, 7168, 2048, 32, 8, 4, 8,
                                     SIGMOID, True, 2.5, "normal"),
    "dsv3_prefill_t2048_e32": Workload("dsv3_prefill_t2048_e32", 2048, 7168, 2048, 32, 8, 4, 8,
                                       SIGMOID, True, 2.5, "zero"),
}
for _name, _S in [("tiny", 1), ("dsv3_decode_t128", 1), ("dsv3_prefill_t8192", 1)]:
    WORKLOADS[f"{_name}_shared"] = replace(WORKLOADS[_name], name=f"{_name}_shared",
                                           n_shared=_S)
WORKLOADS["tiny_block"] = replace(WORKLOADS["tiny"], name="tiny_block", I=128, quant="block")
for _name in ["dsv3_decode_t128", "dsv3_prefill_t8192", "mixtral_t4096", "dsv3_decode_t128_e32",
              "dsv3_prefill_t2048_e32"]:
    WORKLOADS[f"{_name}_block"] = replace(WORKLOADS[_name], name=f"{_name}_block",
                                          quant="block")

WORKLOADS["tiny_nvfp4"] = replace(WORKLOADS["tiny"], name="tiny_nvfp4", H=256, I=256,
                                  quant="nvfp4")
for _name in ["dsv3_decode_t128", "dsv3_prefill_t8192", "mixtral_t4096", "dsv3_decode_t128_e32",
              "dsv3_prefill_t2048_e32"]:
    WORKLOADS[f"{_name}_nvfp4"] = replace(WORKLOADS[_name], name=f"{_name}_nvfp4",
                                          quant="nvfp4")

# tensor ids: each tensor draws from its own generator stream
_TID = {"x": 0, "logits": 1, "bias": 2, "w13": 3, "w2": 4}


def _gen(seed: int, tensor: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + _TID[tensor] * 7919 + 17) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal(shape, std, seed, tensor, device="cpu", dtype=torch.float32):
    g = _gen(seed, tensor, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std).to(dtype)


def quantize_weight_rows(w: torch.Tensor):
    """fp32 weights [..., rows, cols] -> (e4m3 codes as uint8, fp32 scale per row)."""
    amax = w.abs().amax(dim=-1)
    scale = torch.clamp(amax, min=1e-12) / 448.0
    q = (w / scale.unsqueeze(-1)).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale.to(torch.float32)


def quantize_weight_blocks(w: torch.Tensor, blk: int = 128):
    """fp32 weights [..., rows, cols] -> (e4m3 codes as uint8, fp32 scale per
    blk x blk block [..., rows/blk, cols/blk])."""
    *lead, R, C = w.shape
    wb = w.reshape(*lead, R // blk, blk, C // blk, blk)
    amax = wb.abs().amax(dim=(-3, -1))
    scale = torch.clamp(amax, min=1e-12) / 448.0
    q = (wb / scale[..., :, None, :, None]).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.reshape(*lead, R, C).view(torch.uint8), scale.to(torch.float32)


def expert_weights(E, rows, cols, seed, tensor, device="cpu", std=0.02, quant="token"):
    """[E, rows, cols] FP8 codes + scales ([E, rows] per channel, or
    [E, rows/128, cols/128] per block), drawn expert by expert."""
    q = torch.empty((E, rows, cols), dtype=torch.uint8, device=device)
    if quant == "block":
        s = torch.empty((E, rows // 128, cols // 128), dtype=torch.float32, device=device)
    else:
        s = torch.empty((E, rows), dtype=torch.float32, device=device)
    g = _gen(seed, tensor, device)
    for e in range(E):
        w = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).mul_(std)
        q[e], s[e] = quantize_weight_blocks(w) if quant == "block" else quantize_weight_rows(w)
    return q, s


# NVFP4 weights are drawn directly in their format (no quantiser): E2M1
# magnitude codes 0..7 with these probabilities (a half-normal folded onto
# 0, 0.5, 1, 1.5, 2, 3, 4, 6), a random sign, E4M3 block-scale codes uniform
# in [0x28, 0x38] (0.25 .. 1.0), and a global scale so that values have a
# standard deviation near 0.02.
E2M1_MAG_PROBS = [0.10, 0.19, 0.19, 0.16, 0.13, 0.12, 0.07, 0.04]
NVFP4_WEIGHT_G = 0.02 / 1.6


def pack_e2m1(codes: torch.Tensor) -> torch.Tensor:
    """E2M1 codes [..., 2n] (uint8, 0..15) -> bytes [..., n], element 2j in
    the low nibble of byte j."""
    c = codes.to(torch.uint8)
    return c[..., 0::2] | (c[..., 1::2] << 4)


def unpack_e2m1(packed: torch.Tensor) -> torch.Tensor:
    """bytes [..., n] -> E2M1 codes [..., 2n] (the inverse of pack_e2m1)."""
    p = packed.to(torch.uint8)
    return torch.stack([p & 0xF, p >> 4], dim=-1).reshape(*p.shape[:-1], 2 * p.shape[-1])


def expert_weights_nvfp4(E, rows, cols, seed, tensor, device="cpu"):
    """[E, rows, cols] NVFP4 weights: packed codes [E, rows, cols/2], E4M3
    block scales [E, rows, cols/16] (uint8), global scales [E] f32."""
    q = torch.empty((E, rows, cols // 2), dtype=torch.uint8, device=device)
    sb = torch.empty((E, rows, cols // 16), dtype=torch.uint8, device=device)
    g = _gen(seed, tensor, device)
    cdf = torch.cumsum(torch.tensor(E2M1_MAG_PROBS, dtype=torch.float32, device=device), 0)
    for e in range(E):
        u = torch.rand((rows, cols), generator=g, device=device)
        mag = torch.bucketize(u, cdf[:-1], right=True).to(torch.uint8)
        sign = (torch.rand((rows, cols), generator=g, device=device) < 0.5).to(torch.uint8) << 3
        q[e] = pack_e2m1(mag | sign)
        sb[e] = torch.randint(0x28, 0x39, (rows, cols // 16), generator=g, device=device,
                              dtype=torch.int32).to(torch.uint8)
    gs = torch.full((E,), NVFP4_WEIGHT_G, dtype=torch.float32, device=device)
    return q, sb, gs


def router_bias(wl: Workload, seed, device="cpu") -> Optional[torch.Tensor]:
    if wl.bias == "none":
        return None
    if wl.bias == "zero":
        return torch.zeros(wl.E, dtype=torch.float32, device=device)
    b = normal((wl.E,), 0.1, seed, "bias", device)
    if wl.bias == "skewed":
        e = torch.arange(wl.E, device=device)
        b = torch.where(e % 10 == 0, torch.full_like(b, wl.hot_bias), b)
        b = torch.where(e % 8 == 7, torch.full_like(b, -10.0), b)
    return b


def make_inputs(wl: Workload, seed=0, device="cpu", weights=True):
    """All inputs of one forward, on `device`.

    x: bf16 [T,H]; logits: f32 [T,E]; bias: f32 [E] or None;
    w13: u8 [E,2I,H] (rows 0..I-1 gate, I..2I-1 up) with s13 f32 [E,2I];
    w2: u8 [E,H,I] with s2 f32 [E,H]; with n_shared shared experts the
    leading dimension is E + n_shared. Block workloads: s13 [E, 2I/128, H/128],
    s2 [E, H/128, I/128]. NVFP4 workloads: w13 [E,2I,H/2] and w2 [E,H,I/2]
    packed E2M1 codes, s13 [E,2I,H/16] and s2 [E,H,I/16] E4M3 block scales
    (uint8), g13 and g2 [E] f32 global scales.
    """
    d = dict(
        x=normal((wl.T, wl.H), 1.0, seed, "x", device, torch.bfloat16),
        logits=normal((wl.T, wl.E), 1.0, seed, "logits", device),
        bias=router_bias(wl, seed, device),
    )
    if weights:
        n = wl.E + wl.n_shared
        if wl.quant == "nvfp4":
            d["w13"], d["s13"], d["g13"] = expert_weights_nvfp4(n, 2 * wl.I, wl.H, seed, "w13",
                                                                device)
            d["w2"], d["s2"], d["g2"] = expert_weights_nvfp4(n, wl.H, wl.I, seed, "w2", device)
            return d
        d["w13"], d["s13"] = expert_weights(n, 2 * wl.I, wl.H, seed, "w13", device,
                                            quant=wl.quant)
        d["w2"], d["s2"] = expert_weights(n, wl.H, wl.I, seed, "w2", device, quant=wl.quant)
    return d


def to_numpy_inputs(d):
    """torch inputs -> numpy arrays in the oracle's formats (bf16 as uint16)."""
    out = {}
    for k, v in d.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.detach().cpu().view(torch.int16).numpy().view("uint16")
        else:
            out[k] = v.detach().cpu().numpy()
    return out
