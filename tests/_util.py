"""Helpers shared by the GPU parity tests: device transfer of bf16 bit
patterns and the tolerance check of the attention outputs."""
import numpy as np

import workloads as wl

# Tolerances for the attention outputs (bf16 out, fp32 accumulation) against
# the fp64 oracle, over the whole output tensor: max-abs 1e-2 and
# relative-L2 5e-3.
MAX_ABS = 1e-2
REL_L2 = 5e-3


def to_dev(a, device="cuda"):
    import torch

    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def bits(t):
    """Device bf16 tensor -> numpy uint16 bit patterns."""
    import torch

    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t):
    return wl.bf16_to_f64(bits(t))


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = got - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d) / nref) if nref > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values in the output"
    max_abs, rel = errors(got, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {max_abs:.3e} (<= {MAX_ABS}), rel-L2 {rel:.3e} (<= {REL_L2})"
    return max_abs, rel
