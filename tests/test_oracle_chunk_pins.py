"""Pins of the oracle's chunked prefill and positioned page write (CPU only).

Each pin is independent of ``oracle/oracle.c``'s chunked code:

* brute force: a dense numpy score matrix over the cached positions (gathered
  through the page table here) and the new rows, with the explicit mask
  key j visible to new row i iff j <= n_past + i;
* with no cached positions the chunked prefill is the plain prefill;
* splitting a prompt: prefill of its first a rows, their page write, then the
  chunked prefill of the rest with n_past = a gives the one-shot prefill's
  rows (so the cached gather and the causal offset agree with prefill);
* a chunk of one row is a decode step over the pages with that row written;
* the positioned page write is a numpy scatter at positions n_past + i.

The last tests plant mistakes in copies of the C source and check that some
pin catches each one.
"""
import math
import subprocess

import numpy as np
import pytest

import oracle
import workloads as wl


def brute_chunk(w):
    q = wl.bf16_to_f64(w["q"])
    k, v = wl.bf16_to_f64(w["k"]), wl.bf16_to_f64(w["v"])
    kp, vp = wl.bf16_to_f64(w["k_pages"]), wl.bf16_to_f64(w["v_pages"])
    cu, past, table = w["cu_seqlens"], w["n_past"], w["page_table"]
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    out = np.zeros((T, Hq, D))
    for r in range(len(cu) - 1):
        a, b, P = int(cu[r]), int(cu[r + 1]), int(past[r])
        n = b - a
        if n == 0:
            continue
        pos = np.arange(P)
        Kc = kp[table[r, pos // 16], pos % 16] if P else np.zeros((0, Hkv, D))
        Vc = vp[table[r, pos // 16], pos % 16] if P else np.zeros((0, Hkv, D))
        K = np.concatenate([Kc, k[a:b]])  # [P + n, Hkv, D]
        V = np.concatenate([Vc, v[a:b]])
        mask = np.arange(P + n)[None, :] <= P + np.arange(n)[:, None]
        for h in range(Hq):
            g = h // (Hq // Hkv)
            S = q[a:b, h] @ K[:, g].T / math.sqrt(D)
            S = np.where(mask, S, -np.inf)
            E = np.exp(S - S.max(axis=1, keepdims=True))
            out[a:b, h] = (E / E.sum(axis=1, keepdims=True)) @ V[:, g]
    return out


def small_chunk(seed=41):
    return wl.chunk_workload(seed, (0, 20, 33, 16, 5), (7, 1, 40, 16, 0), num_pages=24, max_pages=6)


def _chunk(w, **kw):
    return oracle.prefill_chunk(w["q"], w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"],
                                w["k_pages"], w["v_pages"], **kw)


def test_matches_brute_force(oracle_lib):
    w = small_chunk()
    np.testing.assert_allclose(_chunk(w), brute_chunk(w), rtol=0, atol=1e-12)


def test_no_cached_positions_is_the_prefill(oracle_lib):
    w = wl.chunk_workload(42, (0, 0, 0), (9, 30, 1), num_pages=8, max_pages=2)
    np.testing.assert_array_equal(_chunk(w), oracle.prefill(w["q"], w["k"], w["v"], w["cu_seqlens"]))


@pytest.mark.parametrize("split", [1, 16, 17, 40])
def test_split_prompt_equals_one_shot(oracle_lib, split):
    L = 57
    p = wl.prefill_workload(43, (L,), num_pages=8, max_pages=4)
    one_shot = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    # first `split` rows: prefill + page write
    head = np.array([0, split], np.int32)
    kp, vp = oracle.page_write(p["k"][:split], p["v"][:split], head, p["page_table"], p["k_pages"], p["v_pages"])
    # the rest as a chunk after `split` cached positions
    tail = np.array([0, L - split], np.int32)
    got = oracle.prefill_chunk(p["q"][split:], p["k"][split:], p["v"][split:], tail, np.array([split], np.int32),
                               p["page_table"], kp, vp)
    np.testing.assert_allclose(got, one_shot[split:], rtol=0, atol=1e-12)


def test_one_row_chunk_is_a_decode_step(oracle_lib):
    w = wl.chunk_workload(44, (37, 1, 64), (1, 1, 1), num_pages=12, max_pages=5)
    got = _chunk(w)
    kp, vp = oracle.page_write_at(w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"], w["k_pages"],
                                  w["v_pages"])
    dec = oracle.decode(w["q"], kp, vp, w["page_table"], w["n_past"] + 1)
    np.testing.assert_allclose(got, dec, rtol=0, atol=1e-12)


def test_page_write_at_is_a_scatter(oracle_lib):
    w = small_chunk()
    kp, vp = oracle.page_write_at(w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"], w["k_pages"],
                                  w["v_pages"])
    ek, ev = w["k_pages"].copy(), w["v_pages"].copy()
    cu = w["cu_seqlens"]
    for r in range(len(cu) - 1):
        for i in range(int(cu[r + 1] - cu[r])):
            pos = int(w["n_past"][r]) + i
            page = w["page_table"][r, pos // 16]
            ek[page, pos % 16] = w["k"][cu[r] + i]
            ev[page, pos % 16] = w["v"][cu[r] + i]
    np.testing.assert_array_equal(kp, ek)
    np.testing.assert_array_equal(vp, ev)


def test_rejects_positions_past_the_page_table(oracle_lib):
    w = small_chunk()
    w["n_past"] = w["n_past"].copy()
    w["n_past"][2] = 6 * 16 - 39  # 33 + 40 rows would now end past 6 pages
    with pytest.raises(ValueError):
        _chunk(w)


MUTATIONS = {
    "chunk_causal_off_by_one": ("int n = past + i + 1;       /* keys: every cached position and new rows j <= i */",
                                "int n = past + i;           /* keys: every cached position and new rows j <= i */"),
    "chunk_cached_slot": ("size_t base = (((size_t)page * c->page_size + j % c->page_size) * c->Hkv + g) * c->D;",
                          "size_t base = (((size_t)page * c->page_size + (j / c->page_size) % c->page_size) * c->Hkv + g) * c->D;"),
    "write_at_position": ("int pos = n_past[r] + i; /* the new row's position */",
                          "int pos = i; /* the new row's position */"),
}


def _pins_pass():
    ok = True
    w = small_chunk()
    ok &= np.allclose(_chunk(w), brute_chunk(w), atol=1e-9)
    L, split = 57, 17
    p = wl.prefill_workload(43, (L,), num_pages=8, max_pages=4)
    one_shot = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    kp, vp = oracle.page_write(p["k"][:split], p["v"][:split], np.array([0, split], np.int32), p["page_table"],
                               p["k_pages"], p["v_pages"])
    got = oracle.prefill_chunk(p["q"][split:], p["k"][split:], p["v"][split:], np.array([0, L - split], np.int32),
                               np.array([split], np.int32), p["page_table"], kp, vp)
    ok &= np.allclose(got, one_shot[split:], atol=1e-9)
    kp, vp = oracle.page_write_at(w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"], w["k_pages"],
                                  w["v_pages"])
    cu = w["cu_seqlens"]
    r, i = 2, 5
    pos = int(w["n_past"][r]) + i
    ok &= bool(np.array_equal(kp[w["page_table"][r, pos // 16], pos % 16], w["k"][cu[r] + i]))
    return bool(ok)


def test_unmutated_oracle_passes_the_chunk_pins(oracle_lib):
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_chunk_pins_catch_planted_mistakes(oracle_lib, name, tmp_path, monkeypatch):
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
