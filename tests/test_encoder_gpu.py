"""GPU parity of the AuT encoder layer (qa_encoder_layer) and its pieces
(qa_layer_norm, qa_linear on the tensor cores) against the fp64 oracle,
through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close_bf16, assert_close_rows, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def _bf16(rng, shape, scale=1.0):
    return wl.bf16_bits(rng.standard_normal(size=shape).astype(np.float32) * np.float32(scale))


@pytest.mark.parametrize("T,d", [(333, 896), (1, 896), (64, 128), (40, 2048)])
def test_layer_norm_matches_oracle(T, d):
    rng = np.random.default_rng(T + d)
    x = _bf16(rng, (T, d), 2.0)
    g = wl.bf16_bits(rng.uniform(0.5, 1.5, d).astype(np.float32))
    b = _bf16(rng, d, 0.1)
    out = qa.qa_layer_norm(to_dev(x), to_dev(g), to_dev(b), eps=1e-5, debug_checks=True)
    torch.cuda.synchronize()
    assert_close_bf16(f64(out), oracle.layer_norm(x, g, b, eps=1e-5), f"layer norm T={T} d={d}")


@pytest.mark.parametrize("M,K,N,bias,gelu,res", [
    (300, 896, 2688, True, False, False),   # the q|k|v projection's shape, ragged M
    (257, 896, 3584, True, True, False),    # fc1: bias and gelu
    (129, 3584, 896, True, False, True),    # fc2: bias and residual
    (128, 896, 896, False, False, False),   # one exact M tile, no epilogue extras
    (1, 136, 200, True, True, True),        # a single row, K not a multiple of 64, N not of 224
    (700, 64, 520, True, False, True),      # several M tiles, a ragged N tile, one K block
    (4096, 896, 2688, True, False, True),   # 192 tiles: several per pair of SMs (both accumulators reused)
    (5000, 512, 1040, True, True, False),   # 100 tiles of the 256-wide N tile, the last one ragged
])
def test_linear_matches_oracle(M, K, N, bias, gelu, res):
    rng = np.random.default_rng(M * 7 + K + N)
    x = _bf16(rng, (M, K))
    w = _bf16(rng, (N, K), K ** -0.5)
    b = _bf16(rng, N, 0.1) if bias else None
    r = _bf16(rng, (M, N)) if res else None
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    qa.qa_linear(to_dev(x), to_dev(w), None if b is None else to_dev(b), out, gelu=gelu,
                 residual=None if r is None else to_dev(r), debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.linear(x, w, b, gelu=gelu, residual=r)
    assert_close_bf16(f64(out), ref, f"linear {M}x{K}x{N} bias={bias} gelu={gelu} res={res}")


def _layer_inputs(w):
    dev = {k: to_dev(v) for k, v in w["weights"].items()}
    return to_dev(w["x"]), dev


def _run_layer(w, cu, weights=None):
    x, dw = _layer_inputs(w)
    if weights is not None:
        dw = weights
    out = torch.full_like(x, float("nan"))
    qa.qa_encoder_layer(x, to_dev(cu), dw, out, n_heads=w["n_heads"], ln_eps=w["eps"], debug_checks=True)
    torch.cuda.synchronize()
    return out


def test_encoder_layer_matches_oracle():
    counts = (130, 13, 250)
    w = wl.encoder_layer_workload(61, counts)
    cu = oracle.window_plan(counts)
    got = f64(_run_layer(w, cu))
    ref = oracle.encoder_layer(w["x"], cu, w["weights"], n_heads=w["n_heads"], eps=w["eps"])
    assert_close_rows(got, ref, "encoder layer, 393 tokens in 6 windows")


def test_encoder_attention_block_matches_oracle():
    # with fc2's weight and bias zero the layer returns h, the attention
    # block's output, rounded to bf16
    counts = (104, 57)
    w = wl.encoder_layer_workload(62, counts)
    cu = oracle.window_plan(counts)
    x, dw = _layer_inputs(w)
    dw["w_fc2"] = torch.zeros_like(dw["w_fc2"])
    dw["b_fc2"] = torch.zeros_like(dw["b_fc2"])
    got = f64(_run_layer(w, cu, dw))
    ref = oracle.encoder_layer(w["x"], cu, w["weights"], n_heads=w["n_heads"], eps=w["eps"], blocks=1)
    assert_close_rows(got, ref, "attention block")


def test_encoder_layer_is_window_local_bit_exact():
    counts = (250, 77)
    w = wl.encoder_layer_workload(63, counts)
    cu = oracle.window_plan(counts)
    whole = bits(_run_layer(w, cu))
    for i in (0, 2, len(cu) - 2):
        a, b = int(cu[i]), int(cu[i + 1])
        one = dict(w, x=w["x"][a:b])
        np.testing.assert_array_equal(bits(_run_layer(one, np.array([0, b - a], np.int32))), whole[a:b])


def test_workload_aut_encoder_layer_sampled_windows():
    # the AuT workload (70 220 tokens, 680 windows) through one 0.6B layer;
    # the oracle checks whole windows spread over the sequence (the layer is
    # window-local, so a window's rows are the layer of that window alone),
    # every row of each
    w = wl.encoder_layer_aut()
    cu = qa.qa_window_plan(w["token_counts"])
    got = f64(_run_layer(w, cu))
    assert np.isfinite(got).all()
    picks = sorted(set(np.linspace(0, len(cu) - 2, 24).astype(int).tolist()))
    for i in picks:
        a, b = int(cu[i]), int(cu[i + 1])
        ref = oracle.encoder_layer(w["x"][a:b], np.array([0, b - a], np.int32), w["weights"], n_heads=w["n_heads"],
                                   eps=w["eps"])
        assert_close_rows(got[a:b], ref, f"AuT encoder layer, window {i} (rows {a}..{b})")


def test_encoder_layer_rejects_bad_arguments():
    w = wl.encoder_layer_workload(64, (20,))
    x, dw = _layer_inputs(w)
    cu = to_dev(np.array([0, 20], np.int32))
    with pytest.raises(qa.QAError) as e:
        qa.qa_encoder_layer(x, cu, dw, n_heads=5, ln_eps=1e-5)  # 896 / 5 is not a head size
    assert e.value.status == -1 and "n_heads" in str(e.value)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qa.QAError) as e:
        qa.qa_encoder_layer(x, cu, dw, n_heads=14, ln_eps=1e-5, workspace=small)
    assert e.value.status == -1 and "workspace" in str(e.value)


def test_encoder_layer_1p7b_shape_matches_oracle():
    # the 1.7B tower's layer ("GGUF layout": d_model 1024, 16 heads of 64,
    # FFN 4096): its widths (3072, 1024, 4096) take the 256-wide N tiles
    counts = (200, 104, 31)
    w = wl.encoder_layer_workload(65, counts, d=1024, h=16, d_ffn=4096)
    cu = oracle.window_plan(counts)
    got = f64(_run_layer(w, cu))
    ref = oracle.encoder_layer(w["x"], cu, w["weights"], n_heads=w["n_heads"], eps=w["eps"])
    assert_close_rows(got, ref, "encoder layer 1.7B shape, 335 tokens")


def test_gelu_is_exact_to_the_rounding():
    # every bf16 value in [-8, 8] through qa_linear with an identity weight
    # (x W^T = x exactly): each output must be a correct bf16 rounding of a
    # number within 4e-7 (1 + |x|) of the exact u / 2 (1 + erf(u / sqrt 2)),
    # computed here in fp64 -- the erf approximation's own bound is 1.5e-7
    import math
    mag = np.arange(0x3A80, 0x4101, dtype=np.uint16)  # 2^-10 .. 8 (bf16 bit patterns)
    vals = np.concatenate([[0], mag, mag | 0x8000]).astype(np.uint16)
    n = 128
    rows = -(-len(vals) // n)
    xb = np.zeros(rows * n, np.uint16)
    xb[:len(vals)] = vals
    x = xb.reshape(rows, n)
    w = np.zeros((n, n), np.uint16)
    w[np.arange(n), np.arange(n)] = 0x3F80  # 1.0
    out = qa.qa_linear(to_dev(x), to_dev(w), gelu=True, debug_checks=True)
    torch.cuda.synchronize()
    got = f64(out).reshape(-1)
    xf = (x.reshape(-1).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = np.array([u * 0.5 * (1.0 + math.erf(u / math.sqrt(2.0))) for u in xf])
    ulp = np.where(exact != 0, 2.0 ** (np.floor(np.log2(np.abs(exact) + 1e-300)) - 7), 0.0)
    bound = 0.5 * ulp + 4e-7 * (1.0 + np.abs(xf))
    bad = np.abs(got - exact) > bound
    assert not bad.any(), f"{bad.sum()} outputs, first at x={xf[bad][0]}: got {got[bad][0]} exact {exact[bad][0]}"
