"""Pins of the fp64 oracle to things other than itself (CPU only).

Each pin is independent of ``oracle/oracle.c``:

* brute force: dense numpy score matrices with an explicit boolean mask,
  written here from the definition of attention;
* a library special case: torch's float64 CPU ``scaled_dot_product_attention``
  with the KV heads repeated for GQA;
* mpmath at 50 digits for single rows;
* closed forms (q = 0 gives the mean of the visible values, one key returns
  its value, constant values come back unchanged, probabilities sum to one);
* structural invariants (permuted page table, window split, GQA vs repeated
  MHA, decode of a prefill's last query, attending through written pages);
* printed values from the pages under ``tests/golden/``.

The last tests plant plausible mistakes in copies of the oracle's C source
(dropped scale, missing normalisation, interleaved GQA grouping, causal off by
one, head-major pool indexing, a causal window, a wrong page-write slot),
compile each copy on the CPU and check that some pin catches it.
"""
import math
import os

import numpy as np
import pytest

import oracle
import workloads as wl

TOL = 1e-12
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- brute force
def _softmax_rows(S, mask):
    S = np.where(mask, S, -np.inf)
    m = S.max(axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    E = np.where(mask, np.exp(S - m), 0.0)
    Z = E.sum(axis=-1, keepdims=True)
    return np.divide(E, Z, out=np.zeros_like(E), where=Z > 0)


def brute_decode(q, kp, vp, table, lens, scale=None):
    q = wl.bf16_to_f64(q)
    B, Hq, D = q.shape
    Hkv = kp.shape[2]
    scale = 1 / math.sqrt(D) if scale is None else scale
    Lmax = max(int(lens.max()), 1)
    pos = np.arange(Lmax)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        # dense K/V over all positions up to Lmax; invalid ones are masked
        pages = np.where(pos < lens[b], table[b, np.minimum(pos // 16, table.shape[1] - 1)], 0)
        K = wl.bf16_to_f64(kp[pages, pos % 16])  # [Lmax, Hkv, D]
        V = wl.bf16_to_f64(vp[pages, pos % 16])
        mask = pos < lens[b]
        K = np.where(mask[:, None, None], K, 0.0)
        V = np.where(mask[:, None, None], V, 0.0)
        grp = Hq // Hkv
        Kq = np.repeat(K, grp, axis=1)  # [Lmax, Hq, D]
        Vq = np.repeat(V, grp, axis=1)
        S = np.einsum("hd,jhd->hj", q[b], Kq) * scale
        P = _softmax_rows(S, np.broadcast_to(mask, S.shape))
        out[b] = np.einsum("hj,jhd->hd", P, Vq)
    return out


def brute_prefill(q, k, v, cu, scale=None):
    q, k, v = wl.bf16_to_f64(q), wl.bf16_to_f64(k), wl.bf16_to_f64(v)
    T, Hq, D = q.shape
    grp = Hq // k.shape[1]
    scale = 1 / math.sqrt(D) if scale is None else scale
    req = np.searchsorted(cu, np.arange(T), side="right") - 1
    t = np.arange(T)
    mask = (req[:, None] == req[None, :]) & (t[None, :] <= t[:, None])
    Kq, Vq = np.repeat(k, grp, axis=1), np.repeat(v, grp, axis=1)
    S = np.einsum("ihd,jhd->hij", q, Kq) * scale
    P = _softmax_rows(S, np.broadcast_to(mask, S.shape))
    return np.einsum("hij,jhd->ihd", P, Vq)


def brute_window(q, k, v, cu, scale=None):
    q, k, v = wl.bf16_to_f64(q), wl.bf16_to_f64(k), wl.bf16_to_f64(v)
    T, H, D = q.shape
    scale = 1 / math.sqrt(D) if scale is None else scale
    win = np.searchsorted(cu, np.arange(T), side="right") - 1
    mask = win[:, None] == win[None, :]
    S = np.einsum("ihd,jhd->hij", q, k) * scale
    P = _softmax_rows(S, np.broadcast_to(mask, S.shape))
    return np.einsum("hij,jhd->ihd", P, v)


# ------------------------------------------------------------ small inputs
def small_decode(seed=11, lengths=(37, 1, 16, 0, 29), num_pages=16, max_pages=3, hq=4, hkv=2, d=8):
    return wl.decode_workload(seed, lengths, num_pages, max_pages, hq, hkv, d)


def small_prefill(seed=12, lengths=(9, 1, 17, 6), num_pages=8, max_pages=2, hq=4, hkv=2, d=8):
    return wl.prefill_workload(seed, lengths, num_pages, max_pages, hq, hkv, d)


def small_window(seed=13, counts=(11, 3, 7), h=3, d=8, window=4):
    w = wl.window_workload(seed, counts, h, d)
    w["cu_windows"] = oracle.window_plan(counts, window)
    return w


# -------------------------------------------------------------- brute force
def test_decode_matches_brute_force(oracle_lib):
    w = small_decode()
    got = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    ref = brute_decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, atol=TOL, rtol=0)


def test_decode_rows_subset(oracle_lib):
    w = small_decode()
    full = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    rows = np.array([0, 7, 13, 19], np.int32)
    sub = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"], rows=rows)
    np.testing.assert_array_equal(sub, full.reshape(-1, full.shape[-1])[rows])


def test_prefill_matches_brute_force(oracle_lib):
    w = small_prefill()
    got = oracle.prefill(w["q"], w["k"], w["v"], w["cu_seqlens"])
    ref = brute_prefill(w["q"], w["k"], w["v"], w["cu_seqlens"])
    np.testing.assert_allclose(got, ref, atol=TOL, rtol=0)


def test_window_matches_brute_force(oracle_lib):
    w = small_window()
    got = oracle.window(w["q"], w["k"], w["v"], w["cu_windows"])
    ref = brute_window(w["q"], w["k"], w["v"], w["cu_windows"])
    np.testing.assert_allclose(got, ref, atol=TOL, rtol=0)


def test_page_write_matches_numpy_scatter(oracle_lib):
    w = small_prefill()
    kp, vp = oracle.page_write(w["k"], w["v"], w["cu_seqlens"], w["page_table"], w["k_pages"], w["v_pages"])
    ek, ev = w["k_pages"].copy(), w["v_pages"].copy()
    cu = w["cu_seqlens"]
    touched = np.zeros(ek.shape[:2], bool)
    for r in range(len(cu) - 1):
        for i in range(cu[r + 1] - cu[r]):
            p, s = w["page_table"][r, i // 16], i % 16
            ek[p, s], ev[p, s] = w["k"][cu[r] + i], w["v"][cu[r] + i]
            touched[p, s] = True
    np.testing.assert_array_equal(kp, ek)
    np.testing.assert_array_equal(vp, ev)
    assert (kp[~touched] == wl.BF16_NAN).all() and (vp[~touched] == wl.BF16_NAN).all()


# ------------------------------------------------------ library special case
torch = pytest.importorskip("torch")


def _sdpa(q, k, v, mask, scale):
    # q [H, n, D], k/v [H, m, D], mask [n, m] bool (True = attend)
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask), scale=scale).numpy()


def test_prefill_matches_torch_sdpa(oracle_lib):
    w = small_prefill(seed=21, lengths=(13, 20))
    got = oracle.prefill(w["q"], w["k"], w["v"], w["cu_seqlens"])
    q, k, v = (wl.bf16_to_f64(w[x]) for x in ("q", "k", "v"))
    cu, D = w["cu_seqlens"], q.shape[-1]
    for r in range(len(cu) - 1):
        a, b = cu[r], cu[r + 1]
        qq = q[a:b].transpose(1, 0, 2)
        kk = np.repeat(k[a:b], 2, axis=1).transpose(1, 0, 2)
        vv = np.repeat(v[a:b], 2, axis=1).transpose(1, 0, 2)
        causal = np.tril(np.ones((b - a, b - a), bool))
        ref = _sdpa(qq, kk, vv, causal, 1 / math.sqrt(D)).transpose(1, 0, 2)
        np.testing.assert_allclose(got[a:b], ref, atol=TOL, rtol=0)


def test_window_matches_torch_sdpa(oracle_lib):
    w = small_window(seed=22, counts=(10, 5), window=4)
    got = oracle.window(w["q"], w["k"], w["v"], w["cu_windows"])
    q, k, v = (wl.bf16_to_f64(w[x]).transpose(1, 0, 2) for x in ("q", "k", "v"))
    cu = w["cu_windows"]
    T = q.shape[1]
    win = np.searchsorted(cu, np.arange(T), side="right") - 1
    ref = _sdpa(q, k, v, win[:, None] == win[None, :], 1 / math.sqrt(q.shape[-1]))
    np.testing.assert_allclose(got, ref.transpose(1, 0, 2), atol=TOL, rtol=0)


def test_decode_matches_torch_sdpa(oracle_lib):
    w = small_decode(seed=23, lengths=(40, 7))
    got = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    for b, L in enumerate(w["seq_lens"]):
        pos = np.arange(L)
        pages = w["page_table"][b, pos // 16]
        K = wl.bf16_to_f64(w["k_pages"][pages, pos % 16])  # [L, Hkv, D]
        V = wl.bf16_to_f64(w["v_pages"][pages, pos % 16])
        qq = wl.bf16_to_f64(w["q"][b])[:, None, :]  # [Hq, 1, D]
        kk = np.repeat(K, 2, axis=1).transpose(1, 0, 2)
        vv = np.repeat(V, 2, axis=1).transpose(1, 0, 2)
        ref = _sdpa(qq, kk, vv, np.ones((1, L), bool), 1 / math.sqrt(qq.shape[-1]))[:, 0]
        np.testing.assert_allclose(got[b], ref, atol=TOL, rtol=0)


# ---------------------------------------------------------------- mpmath
def test_attend_row_matches_mpmath(oracle_lib):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(5)
    n, D = 12, 16
    q, K, V = rng.normal(size=D) * 3, rng.normal(size=(n, D)), rng.normal(size=(n, D))
    scale = 1 / math.sqrt(D)
    out, p = oracle.attend_row(q, K, V, scale)
    s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[d]) * mpmath.mpf(K[j, d]) for d in range(D))
         for j in range(n)]
    e = [mpmath.exp(x) for x in s]
    z = mpmath.fsum(e)
    for j in range(n):
        assert abs(float(e[j] / z) - p[j]) < 1e-15
    for d in range(D):
        ref = mpmath.fsum(e[j] / z * mpmath.mpf(V[j, d]) for j in range(n))
        assert abs(float(ref) - out[d]) < 1e-14


# ------------------------------------------------------------ closed forms
def _zero_q(w, key="q"):
    w = dict(w)
    w[key] = np.zeros_like(w[key])
    return w


def test_zero_query_gives_mean_of_visible_values(oracle_lib):
    w = _zero_q(small_decode())
    got = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    for b, L in enumerate(w["seq_lens"]):
        pos = np.arange(L)
        V = wl.bf16_to_f64(w["v_pages"][w["page_table"][b, pos // 16], pos % 16])
        want = V.mean(axis=0) if L else np.zeros(V.shape[1:])
        np.testing.assert_allclose(got[b], np.repeat(want, 2, axis=0), atol=TOL, rtol=0)

    p = _zero_q(small_prefill())
    got = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    v = wl.bf16_to_f64(p["v"])
    cu = p["cu_seqlens"]
    for r in range(len(cu) - 1):
        seg = v[cu[r]:cu[r + 1]]
        prefix_mean = np.cumsum(seg, axis=0) / np.arange(1, len(seg) + 1)[:, None, None]
        np.testing.assert_allclose(got[cu[r]:cu[r + 1]], np.repeat(prefix_mean, 2, axis=1), atol=TOL, rtol=0)

    x = _zero_q(small_window())
    got = oracle.window(x["q"], x["k"], x["v"], x["cu_windows"])
    v = wl.bf16_to_f64(x["v"])
    cu = x["cu_windows"]
    for i in range(len(cu) - 1):
        np.testing.assert_allclose(got[cu[i]:cu[i + 1]], np.broadcast_to(v[cu[i]:cu[i + 1]].mean(0), got[cu[i]:cu[i + 1]].shape), atol=TOL, rtol=0)


def test_single_key_returns_its_value_exactly(oracle_lib):
    w = small_decode(lengths=(1, 1, 1))
    got = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    for b in range(3):
        v0 = wl.bf16_to_f64(w["v_pages"][w["page_table"][b, 0], 0])
        np.testing.assert_array_equal(got[b], np.repeat(v0, 2, axis=0))
    p = small_prefill()
    got = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    for start in p["cu_seqlens"][:-1]:
        np.testing.assert_array_equal(got[start], np.repeat(wl.bf16_to_f64(p["v"][start]), 2, axis=0))
    x = small_window(counts=(5,), window=1)
    got = oracle.window(x["q"], x["k"], x["v"], x["cu_windows"])
    np.testing.assert_array_equal(got, wl.bf16_to_f64(x["v"]))


def test_constant_values_come_back(oracle_lib):
    x = small_window()
    c = wl.bf16_bits(np.linspace(-2, 2, x["v"].shape[-1], dtype=np.float32))
    x["v"] = np.broadcast_to(c, x["v"].shape).copy()
    got = oracle.window(x["q"], x["k"], x["v"], x["cu_windows"])
    np.testing.assert_allclose(got, np.broadcast_to(wl.bf16_to_f64(c), got.shape), atol=TOL, rtol=0)


def test_probabilities_sum_to_one(oracle_lib):
    rng = np.random.default_rng(3)
    for n in (1, 2, 17, 300):
        _, p = oracle.attend_row(rng.normal(size=64) * 4, rng.normal(size=(n, 64)), rng.normal(size=(n, 64)), 0.125)
        assert abs(p.sum() - 1.0) < TOL and (p >= 0).all()


def test_empty_sequence_gives_zero_row(oracle_lib):
    w = small_decode(lengths=(0, 5))
    got = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert (got[0] == 0).all() and np.abs(got[1]).sum() > 0


# ------------------------------------------------------------- invariants
def test_permuted_page_table_equals_contiguous_layout(oracle_lib):
    w = small_decode(lengths=(37, 29, 16))
    B, Hkv, D = 3, w["k_pages"].shape[2], w["k_pages"].shape[3]
    ck = np.full_like(w["k_pages"], wl.BF16_NAN)
    cv = np.full_like(w["v_pages"], wl.BF16_NAN)
    table = np.full_like(w["page_table"], -1)
    nxt = 0
    for b, L in enumerate(w["seq_lens"]):
        for p in range(-(-int(L) // 16)):
            ck[nxt], cv[nxt] = w["k_pages"][w["page_table"][b, p]], w["v_pages"][w["page_table"][b, p]]
            table[b, p] = nxt
            nxt += 1
    a = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    c = oracle.decode(w["q"], ck, cv, table, w["seq_lens"])
    np.testing.assert_array_equal(a, c)


def test_window_split_equals_separate_calls(oracle_lib):
    x = small_window()
    whole = oracle.window(x["q"], x["k"], x["v"], x["cu_windows"])
    cu = x["cu_windows"]
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        one = oracle.window(x["q"][a:b], x["k"][a:b], x["v"][a:b], np.array([0, b - a], np.int32))
        np.testing.assert_array_equal(whole[a:b], one)


def test_gqa_equals_mha_with_repeated_kv(oracle_lib):
    w = small_decode()
    gqa = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    mha = oracle.decode(w["q"], np.repeat(w["k_pages"], 2, axis=2), np.repeat(w["v_pages"], 2, axis=2),
                        w["page_table"], w["seq_lens"])
    np.testing.assert_array_equal(gqa, mha)
    p = small_prefill()
    gqa = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    mha = oracle.prefill(p["q"], np.repeat(p["k"], 2, axis=1), np.repeat(p["v"], 2, axis=1), p["cu_seqlens"])
    np.testing.assert_array_equal(gqa, mha)


def test_decode_through_written_pages_equals_prefill(oracle_lib):
    p = small_prefill(lengths=(9, 1, 17, 6))
    kp, vp = oracle.page_write(p["k"], p["v"], p["cu_seqlens"], p["page_table"], p["k_pages"], p["v_pages"])
    pre = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    cu = p["cu_seqlens"]
    B = len(cu) - 1
    for i in range(17):  # every prefix length that some request reaches
        lens = np.array([min(i + 1, cu[r + 1] - cu[r]) for r in range(B)], np.int32)
        rows = np.array([cu[r] + lens[r] - 1 for r in range(B)])
        dec = oracle.decode(p["q"][rows], kp, vp, p["page_table"], lens)
        np.testing.assert_allclose(dec, pre[rows], atol=TOL, rtol=0)


def test_tiny_workload_cross_pin(oracle_lib):
    """Decode with the prefill's last query row equals the prefill's last row."""
    t = wl.tiny()
    kp, vp = oracle.page_write(t["k"], t["v"], t["cu_seqlens"], t["page_table"], t["k_pages"], t["v_pages"])
    pre = oracle.prefill(t["q"], t["k"], t["v"], t["cu_seqlens"])
    dec = oracle.decode(t["q"][63:64], kp, vp, t["page_table"], t["seq_lens"])
    np.testing.assert_allclose(dec[0], pre[63], atol=TOL, rtol=0)
    assert sorted(t["page_table"][0].tolist()) == [0, 1, 2, 3]


# ----------------------------------------------------- printed values (golden)
def _golden():
    rows = []
    with open(os.path.join(GOLDEN, "window_plan.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_golden_window_values(oracle_lib):
    seen = set()
    for key, *args in _golden():
        seen.add(key)
        if key == "after_cnn_len":
            assert oracle.after_cnn_len(int(args[0])) == int(args[1])
        elif key == "window_tokens":
            assert oracle.window_tokens() == int(args[0])
        elif key == "tokens_for_chunks":
            assert int(args[0]) * oracle.after_cnn_len(2 * oracle.N_WINDOW) == int(args[1])
        elif key == "plan":
            cu = oracle.window_plan([int(args[0])])
            assert np.diff(cu).tolist() == [int(x) for x in args[1].split(",")]
        elif key == "pages_for_audio_seconds":
            sec, prompt, page, pages = map(int, args)
            chunks = sec * 100 // (2 * oracle.N_WINDOW)
            tokens = chunks * oracle.after_cnn_len(2 * oracle.N_WINDOW) + prompt
            assert tokens // page == pages  # "about 122 pages"
    assert seen == {"after_cnn_len", "window_tokens", "tokens_for_chunks", "plan", "pages_for_audio_seconds"}


def test_after_cnn_len_is_ceil_div_8(oracle_lib):
    for r in range(1, 201):
        assert oracle.after_cnn_len(r) == -(-r // 8)


def test_window_plan_shapes(oracle_lib):
    assert oracle.window_plan([0, 104, 105, 208, 1]).tolist() == [0, 104, 208, 209, 313, 417, 418]
    counts = [wl.encoder_tokens_for_frames(n) for n in (1000, 1050, 99, 100 * 1200)]
    assert counts[:3] == [130, 130 + 7, 13]
    cu = oracle.window_plan(counts)
    sizes = np.diff(cu)
    assert sizes.max() == 104 and cu[-1] == sum(counts)


# ----------------------------------------- planted mistakes are caught by pins
# Each mutation plants one plausible mistake in a copy of the oracle's C
# source; the copy is compiled on the CPU and the brute-force / closed-form
# pins are run against it.  At least one pin must fail for every mutant.
MUTATIONS = {
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "no_normalisation": ("double p = s[j] / z;", "double p = s[j];"),
    "gqa_interleaved": ("int g = h / (c->Hq / c->Hkv);", "int g = h % c->Hkv;"),
    "causal_off_by_one": ("int n = t - first + 1; /* keys j <= i within the request */",
                          "int n = t - first; /* keys j < i */"),
    "pool_head_major": ("size_t base = (((size_t)page * c->page_size + slot) * c->Hkv + g) * c->D;",
                        "size_t base = (((size_t)page * c->Hkv + g) * c->page_size + slot) * c->D;"),
    "window_causal": ("int n = c->cu[w + 1] - first; /* every row of the window */",
                      "int n = t - first + 1;"),
    "page_write_slot": ("size_t dst = ((size_t)page * page_size + i % page_size) * row_elems;",
                        "size_t dst = ((size_t)page * page_size + (i / page_size) % page_size) * row_elems;"),
}


def _pins_pass():
    """Runs the brute-force pins on small inputs; True when all agree."""
    ok = True
    w = small_decode()
    got = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    ok &= np.allclose(got, brute_decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"]), atol=1e-9)
    p = small_prefill()
    got = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    ok &= np.allclose(got, brute_prefill(p["q"], p["k"], p["v"], p["cu_seqlens"]), atol=1e-9)
    x = small_window()
    got = oracle.window(x["q"], x["k"], x["v"], x["cu_windows"])
    ok &= np.allclose(got, brute_window(x["q"], x["k"], x["v"], x["cu_windows"]), atol=1e-9)
    kp, vp = oracle.page_write(p["k"], p["v"], p["cu_seqlens"], p["page_table"], p["k_pages"], p["v_pages"])
    pre = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    last = p["cu_seqlens"][1:] - 1
    dec = oracle.decode(p["q"][last], kp, vp, p["page_table"], np.diff(p["cu_seqlens"]))
    ok &= np.allclose(dec, pre[last], atol=1e-9)
    return bool(ok)


def test_unmutated_oracle_passes_the_pins(oracle_lib):
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(oracle_lib, name, tmp_path, monkeypatch):
    import subprocess

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
