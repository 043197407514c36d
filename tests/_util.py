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


def assert_close_bf16(got, ref, what="", rtol=2.0 ** -8, atol=1e-3, rel_l2=REL_L2):
    """bf16 results of operators whose outputs are not bounded by 1 (the
    encoder layer: LayerNorm outputs, residual streams): every element within
    rtol |ref| + atol of the oracle -- rtol = 2^-8 is one bf16 ulp relative,
    twice the final rounding's half ulp, the rest of the budget covering
    fp32-vs-fp64 evaluation inside the operators and the rare intermediate
    rounding that lands on the other side of a bf16 boundary -- and the
    relative L2 error over the whole tensor within rel_l2 (5e-3)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values in the output"
    d = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol
    bad = d > bound
    _, rel = errors(got, ref)
    worst = int(np.argmax(d / bound))
    assert not bad.any() and rel <= rel_l2, (
        f"{what}: {int(bad.sum())} of {d.size} elements outside {rtol:.3g} |ref| + {atol:g} (worst at flat index "
        f"{worst}: got {got.flat[worst]:.6g}, ref {ref.flat[worst]:.6g}); rel-L2 {rel:.3e} (<= {rel_l2})")
    return float(d.max()), rel


def assert_close_rows(got, ref, what="", rtol_row=2.0 ** -7, atol=1e-3, rel_l2=REL_L2):
    """The encoder layer's output against the oracle.  The layer rounds its
    residual stream h to bf16 between operators (the oracle at the same
    boundaries); where the fp32 and fp64 evaluations of h fall on opposite
    sides of a bf16 rounding boundary the two sides carry h values one ulp
    apart, and that ulp (2^-8 of |h|) reaches the output y = h + mlp(h)
    whatever the size of y itself.  So each row is bounded by the scale of
    the row: max |got - ref| <= 2^-7 (two ulps) * max |ref| of the row +
    atol; and the relative L2 error over the whole tensor stays within 5e-3."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values in the output"
    g2 = got.reshape(got.shape[0], -1)
    r2 = ref.reshape(ref.shape[0], -1)
    d = np.abs(g2 - r2).max(axis=1)
    bound = rtol_row * np.abs(r2).max(axis=1) + atol
    _, rel = errors(got, ref)
    worst = int(np.argmax(d / bound))
    assert (d <= bound).all() and rel <= rel_l2, (
        f"{what}: {int((d > bound).sum())} of {len(d)} rows over {rtol_row:.3g} max|ref row| + {atol:g} (worst row "
        f"{worst}: max err {d[worst]:.4g}, bound {bound[worst]:.4g}); rel-L2 {rel:.3e} (<= {rel_l2}); elements "
        f"outside 2^-8|ref|+1e-3: {int((np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + 1e-3).sum())} of {got.size}")
    return float(d.max()), rel
