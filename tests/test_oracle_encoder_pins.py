"""Pins of the oracle's encoder-layer functions (LayerNorm, Linear with bias,
exact gelu and residual, the whole pre-norm AuT layer) to things other than
the oracle itself (CPU only):

* a library special case: torch float64 ``layer_norm`` and ``gelu``;
* numpy float64 matrix products (the oracle multiplies in plain C loops);
* closed forms: a constant row normalises to the LayerNorm bias, a row of
  two alternating values to +-1 / sqrt(1 + eps / var); gelu(0) = 0,
  gelu(u) - gelu(-u) = u;
* an independent numpy statement of the whole layer with an explicit
  block-diagonal mask over the packed sequence, bf16 at the same operator
  boundaries;
* window locality: the rows of one window come out the same when the window
  is run alone.

The last tests plant plausible mistakes in copies of the oracle's C source
(unbiased variance, LayerNorm bias dropped, tanh gelu, projection bias
dropped, attention residual dropped, k and v swapped, FFN residual taken from
the layer input), compile each copy and check that a pin catches it.
"""
import math
import subprocess

import numpy as np
import pytest

import oracle
import workloads as wl

torch = pytest.importorskip("torch")


def f64(a):
    return wl.bf16_to_f64(a)


def bf16_round(v):
    """float64 -> bf16 bits, through binary32, round to nearest even."""
    return wl.bf16_bits(np.asarray(v, np.float64).astype(np.float32))


def small_layer(seed=11, counts=(30, 13), d=64, h=4, d_ffn=128):
    w = wl.encoder_layer_workload(seed, counts, d=d, h=h, d_ffn=d_ffn)
    w["cu"] = oracle.window_plan(counts, 13)
    return w


# ------------------------------------------------------------ LayerNorm
def test_layer_norm_matches_torch_float64():
    rng = np.random.default_rng(1)
    x = wl.bf16_bits(rng.standard_normal((37, 96)).astype(np.float32) * 3 + 1)
    g = wl.bf16_bits(rng.uniform(0.5, 1.5, 96).astype(np.float32))
    b = wl.bf16_bits(rng.standard_normal(96).astype(np.float32))
    got = oracle.layer_norm(x, g, b, eps=1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(f64(x)), (96,), torch.from_numpy(f64(g)),
                                         torch.from_numpy(f64(b)), eps=1e-5).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_layer_norm_closed_forms():
    d = 64
    g = wl.bf16_bits(np.full(d, 2.0, np.float32))
    b = wl.bf16_bits(np.linspace(-1, 1, d).astype(np.float32))
    const = wl.bf16_bits(np.full((3, d), 1.5, np.float32))
    np.testing.assert_array_equal(oracle.layer_norm(const, g, b, eps=1e-5), np.tile(f64(b), (3, 1)))
    # alternating a, c: mean (a + c) / 2, variance ((a - c) / 2)^2
    a, c, eps = 3.0, -1.0, 1e-5
    row = wl.bf16_bits(np.where(np.arange(d) % 2 == 0, a, c).astype(np.float32))[None, :]
    var = ((a - c) / 2) ** 2
    z = 1.0 / math.sqrt(1.0 + eps / var)
    ref = np.where(np.arange(d) % 2 == 0, z, -z) * 2.0 + f64(b)
    np.testing.assert_allclose(oracle.layer_norm(row, g, b, eps=eps)[0], ref, rtol=0, atol=1e-13)


# ------------------------------------------------------- Linear and gelu
def test_linear_matches_numpy_and_torch_gelu():
    rng = np.random.default_rng(2)
    T, K, N = 23, 80, 48
    x = wl.bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    w = wl.bf16_bits(rng.standard_normal((N, K)).astype(np.float32) / 9)
    bias = wl.bf16_bits(rng.standard_normal(N).astype(np.float32))
    res = wl.bf16_bits(rng.standard_normal((T, N)).astype(np.float32))
    lin = f64(x) @ f64(w).T + f64(bias)
    np.testing.assert_allclose(oracle.linear(x, w, bias), lin, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.linear(x, w), f64(x) @ f64(w).T, rtol=0, atol=1e-12)
    gelu = torch.nn.functional.gelu(torch.from_numpy(lin), approximate="none").numpy()
    np.testing.assert_allclose(oracle.linear(x, w, bias, gelu=True), gelu, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.linear(x, w, bias, residual=res), lin + f64(res), rtol=0, atol=1e-12)


def test_gelu_closed_forms():
    # x W^T with W = identity rows picks single inputs: gelu(0) = 0,
    # gelu(u) - gelu(-u) = u, and gelu(u) -> u for large u
    vals = np.array([0.0, 0.5, -0.5, 2.0, -2.0, 8.0], np.float32)
    x = wl.bf16_bits(vals[:, None])
    w = wl.bf16_bits(np.ones((1, 1), np.float32))
    g = oracle.linear(x, w, gelu=True)[:, 0]
    assert g[0] == 0.0
    assert abs((g[1] - g[2]) - 0.5) < 1e-15 and abs((g[3] - g[4]) - 2.0) < 1e-15
    assert abs(g[5] - 8.0) < 1e-13
    assert abs(g[1] - 0.5 * 0.5 * (1 + math.erf(0.5 / math.sqrt(2)))) < 1e-16


# ------------------------------------------------------- the whole layer
def brute_layer(w, blocks=2):
    """The layer written out with numpy: dense scores over the whole packed
    sequence and a boolean block-diagonal mask; bf16 (through binary32) after
    every operator, the last one returned unrounded."""
    x = w["x"]
    W = {k: f64(v) for k, v in w["weights"].items()}
    T, d = x.shape
    H = w["n_heads"]
    Dh = d // H
    cu = np.asarray(w["cu"])
    win = np.searchsorted(cu, np.arange(T), side="right") - 1
    mask = win[:, None] == win[None, :]

    def ln(v, g, b):
        mu = v.mean(axis=1, keepdims=True)
        var = ((v - mu) ** 2).mean(axis=1, keepdims=True)
        return (v - mu) / np.sqrt(var + w["eps"]) * g + b

    xf = f64(x)
    a = f64(bf16_round(ln(xf, W["ln1_g"], W["ln1_b"])))
    qkv = f64(bf16_round(a @ W["w_qkv"].T + W["b_qkv"]))
    q, k, v = qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:]
    o = np.zeros((T, d))
    for hh in range(H):
        sl = slice(hh * Dh, (hh + 1) * Dh)
        S = q[:, sl] @ k[:, sl].T / math.sqrt(Dh)
        S = np.where(mask, S, -np.inf)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        o[:, sl] = P @ v[:, sl]
    o = f64(bf16_round(o))
    h = xf + (o @ W["w_o"].T + W["b_o"])
    if blocks == 1:
        return h
    h = f64(bf16_round(h))
    a2 = f64(bf16_round(ln(h, W["ln2_g"], W["ln2_b"])))
    u = a2 @ W["w_fc1"].T + W["b_fc1"]
    from scipy.special import erf

    f = f64(bf16_round(0.5 * u * (1 + erf(u / math.sqrt(2)))))
    return h + (f @ W["w_fc2"].T + W["b_fc2"])


def _layer(w, blocks=2):
    return oracle.encoder_layer(w["x"], w["cu"], w["weights"], n_heads=w["n_heads"], eps=w["eps"], blocks=blocks)


@pytest.mark.parametrize("blocks", [1, 2])
def test_encoder_layer_matches_numpy_brute_force(blocks):
    w = small_layer()
    np.testing.assert_allclose(_layer(w, blocks), brute_layer(w, blocks), rtol=0, atol=1e-9)


def test_encoder_layer_is_window_local():
    w = small_layer(seed=12, counts=(40, 9, 26))
    whole = _layer(w)
    cu = w["cu"]
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        one = dict(w, x=w["x"][a:b], cu=np.array([0, b - a], np.int32))
        np.testing.assert_array_equal(_layer(one), whole[a:b])


# ----------------------------------------- planted mistakes are caught by pins
MUTATIONS = {
    "ln_unbiased_variance": ("    var /= c->d;\n", "    var /= (c->d - 1);\n"),
    "ln_bias_dropped": ("* inv * bf16_to_double(c->g[i]) + bf16_to_double(c->b[i]);", "* inv * bf16_to_double(c->g[i]);"),
    "gelu_tanh": ("return 0.5 * u * (1.0 + erf(u / sqrt(2.0)));",
                  "return 0.5 * u * (1.0 + tanh(0.7978845608028654 * (u + 0.044715 * u * u * u)));"),
    "projection_bias_dropped": ("            acc += bf16_to_double(c->bias[n]);", "            acc += 0.0;"),
    "attention_residual_dropped": ("oracle_linear(o, T, d, w_o, d, b_o, 0, x, tmp, n_threads);",
                                   "oracle_linear(o, T, d, w_o, d, b_o, 0, NULL, tmp, n_threads);"),
    "k_v_swapped": ("k[(size_t)t * d + i] = qkv[(size_t)t * 3 * d + d + i];\n"
                    "            v[(size_t)t * d + i] = qkv[(size_t)t * 3 * d + 2 * d + i];",
                    "k[(size_t)t * d + i] = qkv[(size_t)t * 3 * d + 2 * d + i];\n"
                    "            v[(size_t)t * d + i] = qkv[(size_t)t * 3 * d + d + i];"),
    "ffn_residual_from_input": ("oracle_linear(f, T, d_ffn, w_fc2, d, b_fc2, 0, h, y, n_threads);",
                                "oracle_linear(f, T, d_ffn, w_fc2, d, b_fc2, 0, x, y, n_threads);"),
}


def _pins_pass():
    ok = True
    rng = np.random.default_rng(3)
    x = wl.bf16_bits(rng.standard_normal((9, 64)).astype(np.float32) * 2 + 0.5)
    g = wl.bf16_bits(rng.uniform(0.5, 1.5, 64).astype(np.float32))
    b = wl.bf16_bits(rng.standard_normal(64).astype(np.float32))
    ref = torch.nn.functional.layer_norm(torch.from_numpy(f64(x)), (64,), torch.from_numpy(f64(g)),
                                         torch.from_numpy(f64(b)), eps=1e-5).numpy()
    ok &= np.allclose(oracle.layer_norm(x, g, b, eps=1e-5), ref, atol=1e-9)
    w = small_layer()
    for blocks in (1, 2):
        ok &= np.allclose(_layer(w, blocks), brute_layer(w, blocks), atol=1e-9)
    return bool(ok)


def test_unmutated_oracle_passes_the_encoder_pins(oracle_lib):
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_encoder_pins_catch_planted_mistakes(oracle_lib, name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                    "-o", str(so), str(mutant_c), "-lm", "-lpthread"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.bind_library(str(so)))
    with np.errstate(all="ignore"):
        try:
            caught = not _pins_pass()
        except ValueError:
            caught = True
    assert caught, f"planted mistake '{name}' went unnoticed by every pin"
