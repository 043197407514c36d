"""GPU parity of the decode calls with qa_attn_params.stable_metadata = 1
(the kernel reads lengths and page table before the preceding kernel on the
stream has finished, everything else after) and 2 (it also streams its first
pool pages before) against the fp64 oracle, in the orders a decode step
launches them: after the append that writes q (level 1: the append writes
the pools), after a plain kernel that writes q, layers queued back to back
on one stream, the layers of one captured graph; and a caller of ABI 1,
whose struct has no such field, is not affected by the byte it leaves there.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402

EPS, THETA = wl.RMS_EPS, wl.ROPE_THETA
KEYS = ("q_new", "k_new", "v_new", "q_gain", "k_gain", "page_table", "seq_lens", "k_pages", "v_pages")


def _oracle_step(w):
    r = oracle.decode_append(w["q_new"], w["k_new"], w["v_new"], w["q_gain"], w["k_gain"], w["page_table"],
                             w["seq_lens"], w["k_pages"], w["v_pages"], eps=EPS, theta=THETA)
    return oracle.decode(r["q"], r["k_pages"], r["v_pages"], w["page_table"], w["seq_lens"])


def test_after_the_append_that_writes_q():
    w = wl.with_append(wl.decode_0p6b(), 3)
    ref = _oracle_step(w)
    d = {k: to_dev(w[k]) for k in KEYS}
    s = torch.cuda.Stream()
    q_rot = torch.empty_like(d["q_new"])
    out = torch.empty_like(d["q_new"])
    with torch.cuda.stream(s):
        qa.qa_decode_append(d["q_new"], d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"],
                            d["seq_lens"], d["k_pages"], d["v_pages"], q_out=q_rot, rms_eps=EPS, rope_theta=THETA,
                            stream=s)
        qa.qa_decode_attn(q_rot, d["k_pages"], d["v_pages"], d["page_table"], d["seq_lens"], out, stream=s,
                          stable_metadata=True)
    torch.cuda.synchronize()
    assert_close(f64(out), ref, "append then decode, stable metadata")
    assert qa.qa_device_status() == 0


@pytest.mark.parametrize("level", [1, 2])
def test_back_to_back_layers_on_one_stream(level):
    # three layers' calls queued without a host sync: each may start while
    # the one before it is finishing (level 2: streaming its pools early)
    base = wl.decode_0p6b()
    layers = [_layer(base, i) for i in range(3)]
    refs = [oracle.decode(c["q"], c["k_pages"], c["v_pages"], c["page_table"], c["seq_lens"]) for c in layers]
    pt, sl = to_dev(base["page_table"]), to_dev(base["seq_lens"])
    dev = [{k: to_dev(c[k]) for k in ("q", "k_pages", "v_pages")} for c in layers]
    B = len(base["seq_lens"])
    ws = torch.zeros(qa.qa_decode_workspace_size(B, 2000, num_pages=dev[0]["k_pages"].shape[0],
                                                 max_pages_per_seq=pt.shape[1]), dtype=torch.uint8, device="cuda")
    outs = [torch.empty_like(d["q"]) for d in dev]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for rep in range(3):
            for d, o in zip(dev, outs):
                qa.qa_decode_attn(d["q"], d["k_pages"], d["v_pages"], pt, sl, o, workspace=ws, stream=s,
                                  stable_metadata=level)
    torch.cuda.synchronize()
    for i, (o, r) in enumerate(zip(outs, refs)):
        assert_close(f64(o), r, f"level {level} layer {i}")
    assert qa.qa_device_status() == 0


def test_noalloc_layers_back_to_back_at_level_2():
    # the entry point without a workspace shares the library's scratch; calls
    # ordered on one stream may overlap their prologues at level 2
    base = wl.decode_0p6b()
    layers = [_layer(base, i) for i in range(3)]
    refs = [oracle.decode(c["q"], c["k_pages"], c["v_pages"], c["page_table"], c["seq_lens"]) for c in layers]
    pt, sl = to_dev(base["page_table"]), to_dev(base["seq_lens"])
    dev = [{k: to_dev(c[k]) for k in ("q", "k_pages", "v_pages")} for c in layers]
    outs = [torch.empty_like(d["q"]) for d in dev]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for rep in range(2):
            for d, o in zip(dev, outs):
                qa.qa_decode_attn_noalloc(d["q"], d["k_pages"], d["v_pages"], pt, sl, o, stream=s, stable_metadata=2)
    torch.cuda.synchronize()
    for i, (o, r) in enumerate(zip(outs, refs)):
        assert_close(f64(o), r, f"no-alloc layer {i}")
    assert qa.qa_device_status() == 0


@pytest.mark.parametrize("level", [1, 2])
def test_fused_step_after_a_kernel_that_writes_q(level):
    w = wl.with_append(wl.decode_0p6b(), 4)
    ref = _oracle_step(w)
    d = {k: to_dev(w[k]) for k in KEYS}
    src = d["q_new"].clone()
    d["q_new"].zero_()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d["q_new"].copy_(src)  # the q projection's stand-in, just before the step
        out = qa.qa_decode_step(d["q_new"], d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"],
                                d["seq_lens"], d["k_pages"], d["v_pages"], rms_eps=EPS, rope_theta=THETA, stream=s,
                                stable_metadata=level)
    torch.cuda.synchronize()
    assert_close(f64(out), ref, "fused step, stable metadata")
    assert qa.qa_device_status() == 0


def _layer(base, i):
    """Layer i over the same page table and lengths: a fresh query and the
    base keys scaled by 2^-i (exact in bf16); the values stay at N(0, 1),
    the scale the absolute tolerance is stated for."""
    c = dict(base)
    c["q"] = wl.normal_bf16(wl.rng_for(700 + i), base["q"].shape)
    c["k_pages"] = wl.bf16_bits((wl.bf16_to_f64(base["k_pages"]) * 2.0 ** -i).astype(np.float32))
    return c


def test_prefill_layers_back_to_back_at_level_1():
    # the prefill bucket's calls for three layers (own q, k, v and pools; one
    # cu_seqlens and page table) queued on one stream without a host sync
    base = wl.prefill_bucket()
    layers = []
    for i in range(3):
        c = dict(base)
        rng = wl.rng_for(800 + i)
        for key in ("q", "k", "v"):
            c[key] = wl.normal_bf16(rng, base[key].shape)
        layers.append(c)
    cu, pt = to_dev(base["cu_seqlens"]), to_dev(base["page_table"])
    dev = [{key: to_dev(c[key]) for key in ("q", "k", "v", "k_pages", "v_pages")} for c in layers]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        outs = [qa.qa_prefill_attn(d["q"], d["k"], d["v"], cu, pt, d["k_pages"], d["v_pages"], stream=s,
                                   stable_metadata=1) for d in dev]
    torch.cuda.synchronize()
    for i, (c, d, o) in enumerate(zip(layers, dev, outs)):
        assert_close(f64(o), oracle.prefill(c["q"], c["k"], c["v"], c["cu_seqlens"]), f"prefill layer {i}")
        ekp, evp = oracle.page_write(c["k"], c["v"], c["cu_seqlens"], c["page_table"], c["k_pages"], c["v_pages"])
        np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
        np.testing.assert_array_equal(bits(d["v_pages"]), evp)
    assert qa.qa_device_status() == 0


def test_chunked_prefill_twice_at_level_1():
    w = wl.chunk_reprefill()
    ref = oracle.prefill_chunk(w["q"], w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"], w["k_pages"],
                               w["v_pages"])
    d = {key: to_dev(w[key]) for key in ("q", "k", "v", "cu_seqlens", "n_past", "page_table", "k_pages", "v_pages")}
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        # the second call rewrites the same rows with the same values and
        # reads the same cached pages
        outs = [qa.qa_prefill_chunk_attn(d["q"], d["k"], d["v"], d["cu_seqlens"], d["n_past"], d["page_table"],
                                         d["k_pages"], d["v_pages"], stream=s, stable_metadata=1) for _ in range(2)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert_close(f64(o), ref, f"chunked prefill call {i}")
    ekp, evp = oracle.page_write_at(w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"], w["k_pages"],
                                    w["v_pages"])
    np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
    np.testing.assert_array_equal(bits(d["v_pages"]), evp)
    assert qa.qa_device_status() == 0


@pytest.mark.parametrize("level", [1, 2])
def test_chunked_prefill_layers_chained_through_q(level):
    # three layers of the re-prefill bucket queued on one stream, each with
    # its own k, v and pool buffers (one cu_seqlens, n_past and page table); layer
    # i's q is layer i - 1's output, written by the kernel right before it,
    # so q must be read only after the wait even where (level 2) the first
    # cached tile's K and V rows are requested before it
    base = wl.chunk_reprefill()
    layers = []
    for i in range(3):
        c = dict(base)
        rng = wl.rng_for(900 + i)
        for key in ("k", "v"):
            c[key] = wl.normal_bf16(rng, base[key].shape)
        layers.append(c)  # its pools: a device copy of its own (same cached rows)
    cu, npast, pt = to_dev(base["cu_seqlens"]), to_dev(base["n_past"]), to_dev(base["page_table"])
    dev = [{key: to_dev(c[key]) for key in ("k", "v", "k_pages", "v_pages")} for c in layers]
    q0 = to_dev(base["q"])
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    with torch.cuda.stream(s):
        q = q0
        for d in dev:
            q = qa.qa_prefill_chunk_attn(q, d["k"], d["v"], cu, npast, pt, d["k_pages"], d["v_pages"], stream=s,
                                         stable_metadata=level)
            outs.append(q)
    torch.cuda.synchronize()
    q_in = base["q"]
    for i, (c, d, o) in enumerate(zip(layers, dev, outs)):
        ref = oracle.prefill_chunk(q_in, c["k"], c["v"], c["cu_seqlens"], c["n_past"], c["page_table"],
                                   c["k_pages"], c["v_pages"])
        assert_close(f64(o), ref, f"chunked prefill layer {i}, level {level}")
        ekp, evp = oracle.page_write_at(c["k"], c["v"], c["cu_seqlens"], c["n_past"], c["page_table"],
                                        c["k_pages"], c["v_pages"])
        np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
        np.testing.assert_array_equal(bits(d["v_pages"]), evp)
        q_in = bits(o)
    assert qa.qa_device_status() == 0


def test_graph_of_layers_follows_refills():
    base = wl.decode_0p6b()
    layers = [_layer(base, i) for i in range(3)]
    refs = [oracle.decode(c["q"], c["k_pages"], c["v_pages"], c["page_table"], c["seq_lens"]) for c in layers]
    pt, sl = to_dev(base["page_table"]), to_dev(base["seq_lens"])
    qs = [to_dev(c["q"]) for c in layers]
    kp = [to_dev(c["k_pages"]) for c in layers]
    vp = [to_dev(c["v_pages"]) for c in layers]
    outs = [torch.empty_like(q) for q in qs]
    B = len(base["seq_lens"])
    ws = torch.zeros(qa.qa_decode_workspace_size(B, 2000, num_pages=kp[0].shape[0],
                                                 max_pages_per_seq=pt.shape[1]), dtype=torch.uint8, device="cuda")
    srcs = [q.clone() for q in qs]
    g = qa.qa_decode_graph_create(qs, kp, vp, pt, sl, outs, workspace=ws, stable_metadata=2)
    try:
        for rep in range(2):
            for q in qs:
                q.zero_()
            for o in outs:
                o.zero_()
            for q, src in zip(qs, srcs):
                q.copy_(src)  # refilled in place right before the replay
            g.launch()
            torch.cuda.synchronize()
            for i, (o, r) in enumerate(zip(outs, refs)):
                assert_close(f64(o), r, f"replay {rep} layer {i}")
    finally:
        g.close()
    assert qa.qa_device_status() == 0


def test_abi1_caller_ignores_the_field():
    w = wl.decode_0p6b()
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    d = {k: to_dev(w[k]) for k in ("q", "k_pages", "v_pages", "page_table", "seq_lens")}
    B = len(w["seq_lens"])
    out = torch.empty_like(d["q"])
    ws = torch.zeros(qa.qa_decode_workspace_size(B, 2000, num_pages=d["k_pages"].shape[0],
                                                 max_pages_per_seq=d["page_table"].shape[1]), dtype=torch.uint8,
                     device="cuda")
    p = qa._params(n_q_heads=16, n_kv_heads=8, head_dim=128, num_pages=d["k_pages"].shape[0],
                   max_pages_per_seq=d["page_table"].shape[1], workspace=ws, stable_metadata=True)
    p.abi_version = 1
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    for call in range(2):  # the second call reuses the workspace the first left
        out.zero_()
        st = qa._lib.qa_decode_attn(vp(d["q"]), vp(d["k_pages"]), vp(d["v_pages"]), vp(d["page_table"]),
                                    vp(d["seq_lens"]), B, vp(out), ctypes.byref(p))
        assert st == 0, qa.qa_last_error()
        torch.cuda.synchronize()
        assert_close(f64(out), ref, f"ABI 1 caller, call {call}")
    assert qa.qa_device_status() == 0
