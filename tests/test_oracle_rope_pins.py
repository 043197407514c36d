"""Pins of the oracle's per-head QK-norm, NEOX RoPE and decode KV append
(CPU only).

Each pin is independent of ``oracle/oracle.c``:

* a library special case: at position 0 the rotation is the identity, so the
  result must equal torch's float64 ``rms_norm`` with the [head_dim] gain,
  including inputs small enough for the epsilon to matter;
* closed forms: a unit vector e_i rotates in the plane (i, i + 64) by
  pos * 1e6^(-2 i / 128); for i = 0, 16 and 32 that frequency is 1, 10^(-3/2)
  and 10^(-3), so e_0 at position 1, e_16 at position 1 and e_32 at position
  1000 land on cos/sin of 1, 1/sqrt(1000) and 1, in the rotate-half layout
  (not interleaved) and with the standard sign (e_64 goes to -sin, cos);
* rotation invariants: pair norms are kept, and q.k after rotation depends
  only on the position difference;
* the append: a numpy scatter of the rotated, bf16-rounded k row and the
  untouched v row into slot (seq_len - 1) % 16 of page
  page_table[b][(seq_len - 1) // 16], nothing else changed.

The last tests plant plausible mistakes in copies of the oracle's C source
and check that some pin catches each one.
"""
import math
import subprocess

import numpy as np
import pytest

import oracle
import workloads as wl

torch = pytest.importorskip("torch")

EPS, THETA, D = wl.RMS_EPS, wl.ROPE_THETA, 128


def _unit(i, a=1.0):
    x = np.zeros((1, 1, D), np.float32)
    x[0, 0, i] = a
    return wl.bf16_bits(x)


def _rms_norm_torch(x_bits, gain):
    x = torch.from_numpy(wl.bf16_to_f64(x_bits))
    g = torch.from_numpy(np.asarray(gain, np.float64))
    return torch.nn.functional.rms_norm(x, (D,), weight=g, eps=EPS).numpy()


def _gains(seed):
    return wl.append_inputs(wl.rng_for(seed), 1)["q_gain"]


def _rope(x, pos, gain):
    return oracle.qk_norm_rope(x, np.asarray(pos, np.int32), gain, eps=EPS, theta=THETA)


# ------------------------------------------------------------- the norm alone
@pytest.mark.parametrize("x_scale", [1.0, 1e-3, 40.0])
def test_position_zero_is_torch_rms_norm(oracle_lib, x_scale):
    rng = wl.rng_for(21)
    x = wl.bf16_bits(rng.standard_normal((6, 3, D), dtype=np.float32) * np.float32(x_scale))
    g = _gains(22)
    got = _rope(x, np.zeros(6), g)
    ref = _rms_norm_torch(x, g)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_epsilon_matters_for_small_inputs(oracle_lib):
    # mean square 1e-6 = eps: the norm is 1/sqrt(2e-6), not 1/sqrt(1e-6)
    x = np.full((1, 1, D), 1e-3, np.float32)
    xb = wl.bf16_bits(x)
    xv = wl.bf16_to_f64(xb)[0, 0, 0]
    got = _rope(xb, [0], np.ones(D, np.float32))[0, 0]
    np.testing.assert_allclose(got, xv / math.sqrt(xv * xv + EPS), rtol=1e-12)


# ------------------------------------------------------- closed-form rotations
def _unit_norm():
    return 1.0 / math.sqrt(1.0 / D + EPS)  # RMSNorm of a unit basis vector


@pytest.mark.parametrize("i,pos,angle", [(0, 1, 1.0), (16, 1, 1.0 / math.sqrt(1000.0)), (32, 1000, 1.0),
                                         (0, 3, 3.0), (32, 4000, 4.0)])
def test_first_half_unit_vector_rotates_into_second_half(oracle_lib, i, pos, angle):
    z = _rope(_unit(i), [pos], np.ones(D, np.float32))[0, 0]
    y = _unit_norm()
    expect = np.zeros(D)
    expect[i] = y * math.cos(angle)
    expect[i + 64] = y * math.sin(angle)
    np.testing.assert_allclose(z, expect, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("i,pos,angle", [(0, 1, 1.0), (32, 1000, 1.0)])
def test_second_half_unit_vector_rotates_back(oracle_lib, i, pos, angle):
    z = _rope(_unit(i + 64), [pos], np.ones(D, np.float32))[0, 0]
    y = _unit_norm()
    expect = np.zeros(D)
    expect[i] = -y * math.sin(angle)
    expect[i + 64] = y * math.cos(angle)
    np.testing.assert_allclose(z, expect, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- rotation invariants
def test_pair_norms_are_kept(oracle_lib):
    rng = wl.rng_for(23)
    x = wl.normal_bf16(rng, (5, 4, D))
    g = _gains(24)
    pos = np.array([0, 1, 999, 16383, 65535], np.int32)
    z = _rope(x, pos, g)
    y = _rms_norm_torch(x, g)
    np.testing.assert_allclose(z[..., :64] ** 2 + z[..., 64:] ** 2, y[..., :64] ** 2 + y[..., 64:] ** 2,
                               rtol=1e-10, atol=1e-12)


def test_scores_depend_only_on_position_difference(oracle_lib):
    rng = wl.rng_for(25)
    q = wl.normal_bf16(rng, (1, 1, D))
    k = wl.normal_bf16(rng, (1, 1, D))
    gq, gk = _gains(26), _gains(27)
    dots = []
    for m, n in [(7, 3), (107, 103), (20007, 20003), (60004, 60000)]:
        dots.append(float(_rope(q, [m], gq)[0, 0] @ _rope(k, [n], gk)[0, 0]))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)
    far = float(_rope(q, [8], gq)[0, 0] @ _rope(k, [3], gk)[0, 0])
    assert abs(far - dots[0]) > 1e-6  # and the difference itself matters


# --------------------------------------------------------------- the append
def small_append():
    # lengths not multiples of 16, so a position off by one stays in the same page
    return wl.decode_append_workload(31, (1, 17, 40, 203), num_pages=32, max_pages=16)


def _expected_append(w):
    pos = w["seq_lens"] - 1
    q_rot = _rope(w["q_new"], pos, w["q_gain"])
    k_rot = _rope(w["k_new"], pos, w["k_gain"])
    kp, vp = w["k_pages"].copy(), w["v_pages"].copy()
    for b, p in enumerate(pos):
        page = w["page_table"][b, p // 16]
        kp[page, p % 16] = wl.bf16_bits(k_rot[b].astype(np.float32))
        vp[page, p % 16] = w["v_new"][b]
    return q_rot, k_rot, wl.bf16_bits(q_rot.astype(np.float32)), kp, vp


def _run_append(w):
    return oracle.decode_append(w["q_new"], w["k_new"], w["v_new"], w["q_gain"], w["k_gain"], w["page_table"],
                                w["seq_lens"], w["k_pages"], w["v_pages"], eps=EPS, theta=THETA)


def test_append_matches_numpy_scatter(oracle_lib):
    w = small_append()
    r = _run_append(w)
    q_rot, k_rot, q_bits, kp, vp = _expected_append(w)
    np.testing.assert_array_equal(r["q_rot"], q_rot)
    np.testing.assert_array_equal(r["k_rot"], k_rot)
    np.testing.assert_array_equal(r["q"], q_bits)
    np.testing.assert_array_equal(r["k_pages"], kp)
    np.testing.assert_array_equal(r["v_pages"], vp)


def test_append_rejects_a_bad_page_and_an_empty_request(oracle_lib):
    w = small_append()
    w["page_table"] = w["page_table"].copy()
    w["page_table"][2, 2] = 99
    with pytest.raises(ValueError):
        _run_append(w)
    w = small_append()
    w["seq_lens"] = w["seq_lens"].copy()
    w["seq_lens"][0] = 0
    with pytest.raises(ValueError):
        _run_append(w)


def test_decode_after_append_attends_to_the_new_token(oracle_lib):
    # a request of length 1 attends only to its own appended token: out = v
    w = small_append()
    r = _run_append(w)
    out = oracle.decode(r["q"], r["k_pages"], r["v_pages"], w["page_table"], w["seq_lens"])
    np.testing.assert_array_equal(out[0], np.repeat(wl.bf16_to_f64(w["v_new"][0]), 2, axis=0))


# ----------------------------------------- planted mistakes are caught by pins
MUTATIONS = {
    "rope_sign": ("z[i] = y0 * ca - y1 * sa;", "z[i] = y0 * ca + y1 * sa;"),
    "rope_exponent": ("pow(theta, -2.0 * i / D)", "pow(theta, -1.0 * i / D)"),
    "rope_pair_layout": ("double y1 = bf16_to_double(x[i + half]) * r * (double)gain[i + half];",
                         "double y1 = bf16_to_double(x[i ^ 1]) * r * (double)gain[i ^ 1];"),
    "norm_eps_outside": ("double r = 1.0 / sqrt(ms + eps);", "double r = 1.0 / (sqrt(ms) + eps);"),
    "norm_sum_not_mean": ("    ms /= D;\n", "    ms /= 1;\n"),
    "norm_gain_dropped": ("double y0 = bf16_to_double(x[i]) * r * (double)gain[i];",
                          "double y0 = bf16_to_double(x[i]) * r;"),
    "append_position": ("int cur = seq_lens[b] - 1; /* the new token's position */",
                        "int cur = seq_lens[b]; /* the new token's position */"),
    "append_slot": ("int slot = cur % page_size;", "int slot = (cur + 1) % page_size;"),
}


def _pins_pass():
    ok = True
    g = _gains(22)
    rng = wl.rng_for(21)
    x = wl.bf16_bits(rng.standard_normal((4, 2, D), dtype=np.float32) * np.float32(1e-3))
    ok &= np.allclose(_rope(x, np.zeros(4), g), _rms_norm_torch(x, g), rtol=1e-9, atol=1e-12)
    x = wl.normal_bf16(rng, (4, 2, D))
    ok &= np.allclose(_rope(x, np.zeros(4), g), _rms_norm_torch(x, g), rtol=1e-9, atol=1e-12)
    y = _unit_norm()
    for i, pos, a in [(0, 1, 1.0), (16, 1, 1.0 / math.sqrt(1000.0)), (32, 1000, 1.0)]:
        z = _rope(_unit(i), [pos], np.ones(D, np.float32))[0, 0]
        ok &= math.isclose(z[i], y * math.cos(a), rel_tol=1e-9) and math.isclose(z[i + 64], y * math.sin(a),
                                                                                   rel_tol=1e-9)
    z = _rope(_unit(64), [1], np.ones(D, np.float32))[0, 0]
    ok &= math.isclose(z[0], -y * math.sin(1.0), rel_tol=1e-9) and math.isclose(z[64], y * math.cos(1.0),
                                                                                 rel_tol=1e-9)
    w = small_append()
    r = _run_append(w)
    _, _, q_bits, kp, vp = _expected_append(w)
    ok &= np.array_equal(r["q"], q_bits) and np.array_equal(r["k_pages"], kp) and np.array_equal(r["v_pages"], vp)
    return bool(ok)


def test_unmutated_oracle_passes_the_rope_pins(oracle_lib):
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_rope_pins_catch_planted_mistakes(oracle_lib, name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
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
