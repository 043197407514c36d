"""Helpers shared by the GPU parity tests: device transfer of bf16 bit
patterns, the tolerance check of the attention outputs and the rounding
check of the decode append's bf16 results."""
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


def pair_scale(x, gain):
    """|y_i| + |y_{i+D/2}| for every element, y the normalised vector (the
    oracle at position 0, where the rotation is the identity)."""
    import oracle

    y = np.abs(oracle.qk_norm_rope(x, np.zeros(x.shape[0], np.int32), gain, eps=wl.RMS_EPS, theta=wl.ROPE_THETA))
    h = y.shape[-1] // 2
    s = y[..., :h] + y[..., h:]
    return np.concatenate([s, s], axis=-1)


def assert_rounded_match(got_bits, ref, scale, what):
    """bf16 results of fp32 arithmetic against the oracle's fp64 values: each element
    must be the bf16 rounding of some value within e of the oracle's fp64 value
    v: rounding is monotone, so it must lie between the roundings of v - e and
    v + e.  Almost everywhere those two coincide and the check is bit-exact
    equality with the oracle's own rounding; near a rounding boundary, or where
    the rotation cancels to a value far below its inputs, the fp32 evaluation
    error may land on several bf16 values.  e = 2^-18 (|y_i| + |y_{i+D/2}|),
    y the normalised pair before the rotation -- about 16 times the fp32 error
    of the products, the rotation and the fp32 sin/cos of an angle reduced in
    fp64.
    """
    ref_bits = wl.bf16_bits(ref.astype(np.float32))
    e = 2.0 ** -18 * scale
    lo = wl.bf16_to_f64(wl.bf16_bits((ref - e).astype(np.float32)))
    hi = wl.bf16_to_f64(wl.bf16_bits((ref + e).astype(np.float32)))
    got = wl.bf16_to_f64(got_bits)
    exact = got_bits == ref_bits
    bad = ~exact & ~((lo <= got) & (got <= hi))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements are not a rounding of a value within "
                           f"the fp32 error of the oracle's; first at {np.argwhere(bad)[0]}")
    # almost all elements are bit-exact
    assert (~exact).sum() <= max(4, exact.size // 200), f"{what}: {int((~exact).sum())} inexact elements"
    return int((~exact).sum())
