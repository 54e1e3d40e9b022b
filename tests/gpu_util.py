"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

# Layer and GEMM outputs: max |err| <= 2e-2 * max |ref| and
# sum |err| / sum |ref| <= 5e-3 (fp32 accumulation against exact fp64).
MAX_REL = 2e-2
MEAN_REL = 5e-3


def tol_report(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    max_rel = err.max() / scale if scale > 0 else err.max()
    mean_rel = err.sum() / np.abs(ref).sum() if np.abs(ref).sum() > 0 else err.sum()
    return max_rel, mean_rel


def assert_parity(got, ref, what=""):
    max_rel, mean_rel = tol_report(got, ref)
    assert max_rel <= MAX_REL and mean_rel <= MEAN_REL, \
        f"{what}: max|err|/max|ref|={max_rel:.3e} sum|err|/sum|ref|={mean_rel:.3e}"
    return max_rel, mean_rel


def bf16_np(t):
    """bf16 torch tensor -> float64 numpy."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_bf16_to_torch(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def ragged_offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def random_e4m3(rng, shape):
    """Random FP8 codes without the NaN patterns 0x7F / 0xFF (as uint8)."""
    q = rng.integers(0, 256, shape).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] &= 0xFE
    return q
