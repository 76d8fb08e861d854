"""Helpers shared by the GPU parity tests (host-side comparison only)."""
import numpy as np
import torch

from synth import f32_from_bf16_bits


def bf64(bits):
    return f32_from_bf16_bits(bits).astype(np.float64)


def tokens64(x):
    return bf64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(got, ref) -> float:
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(np.asarray(got, np.float64) - ref) / max(np.linalg.norm(ref), 1e-300))


# Output tolerance: bf16 operands and outputs with fp32 accumulation.  The relative
# L2 bound is the contract; the element-wise bound (2e-2 relative plus 2e-2 of the
# tensor's RMS) catches localised errors that an L2 norm would average away.
REL_L2 = 2e-2


def assert_close_bf16(got, ref, what="", elem_rms=2e-2):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    r = rel_l2(got, ref)
    assert r <= REL_L2, f"{what}: rel L2 {r:.3e}"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bad = np.abs(got - ref) > 2e-2 * np.abs(ref) + elem_rms * rms
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, first at {np.argwhere(bad)[0]}"
    return r


# Weight gradients sum, per element, over the tokens of one expert (16 on average in
# the 512-token cases): a single product can dominate an element, and the bf16
# rounding of the recomputed pre-activations and of their gradients (about 2^-8
# relative per product) is then not averaged away.  Element-wise bound 6e-2 of the
# RMS (a misplaced or missing tile is off by the RMS itself); rel L2 stays 2e-2.
GRAD_ELEM_RMS = 6e-2


def assert_close_grad(got, ref, what=""):
    return assert_close_bf16(got, ref, what, elem_rms=GRAD_ELEM_RMS)
