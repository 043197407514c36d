"""Captured attention steps (qa_decode_graph_create / qa_prefill_graph_create
+ qa_graph_launch): a replay gives the same results as the eager calls, and a
replay after refilling the captured buffers in place reflects the new
contents; checked against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def _layer(base, i):
    """Layer i of a decode step over the same page table: a fresh query,
    the base pools scaled by 2^-i (K) and 2^i (V), exact in bf16 (sentinel
    NaNs stay NaN)."""
    w = dict(base)
    w["q"] = wl.normal_bf16(wl.rng_for(600 + i), base["q"].shape)
    w["k_pages"] = wl.bf16_bits((wl.bf16_to_f64(base["k_pages"]) * 2.0 ** -i).astype(np.float32))
    w["v_pages"] = wl.bf16_bits((wl.bf16_to_f64(base["v_pages"]) * 2.0 ** i).astype(np.float32))
    return w


def test_decode_step_graph_matches_eager_and_follows_refills():
    lengths = (40, 300, 1, 17)
    n_layers = 3
    base = wl.decode_workload(500, lengths, num_pages=40, max_pages=20)
    ws_layers = [_layer(base, i) for i in range(n_layers)]  # one page table and one set of lengths for all layers
    pt, sl = to_dev(base["page_table"]), to_dev(base["seq_lens"])
    qs = [to_dev(w["q"]) for w in ws_layers]
    kps = [to_dev(w["k_pages"]) for w in ws_layers]
    vps = [to_dev(w["v_pages"]) for w in ws_layers]
    outs = [torch.empty_like(q) for q in qs]
    ws = torch.zeros(qa.qa_decode_workspace_size(4, 300, num_pages=40, max_pages_per_seq=20), dtype=torch.uint8,
                     device="cuda")
    eager = [qa.qa_decode_attn(qs[i], kps[i], vps[i], pt, sl, workspace=ws) for i in range(n_layers)]
    g = qa.qa_decode_graph_create(qs, kps, vps, pt, sl, outs, workspace=ws)
    g.launch()
    torch.cuda.synchronize()
    for i in range(n_layers):
        assert torch.equal(outs[i], eager[i])
        ref = oracle.decode(ws_layers[i]["q"], ws_layers[i]["k_pages"], ws_layers[i]["v_pages"],
                            ws_layers[i]["page_table"], ws_layers[i]["seq_lens"])
        assert_close(f64(outs[i]), ref, f"graph layer {i}")
    # refill the captured query buffers in place and replay on another stream
    rng = wl.rng_for(510)
    new_q = [wl.normal_bf16(rng, (4, 16, 128)) for _ in range(n_layers)]
    for i in range(n_layers):
        qs[i].copy_(to_dev(new_q[i]))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g.launch(stream=s)
    s.synchronize()
    for i in range(n_layers):
        ref = oracle.decode(new_q[i], ws_layers[i]["k_pages"], ws_layers[i]["v_pages"], ws_layers[i]["page_table"],
                            ws_layers[i]["seq_lens"])
        assert_close(f64(outs[i]), ref, f"graph replay after refill, layer {i}")
    g.close()
    assert qa.qa_device_status() == 0


def test_prefill_bucket_graph_matches_eager():
    lengths = (100, 129, 7)
    n_layers = 2
    base = wl.prefill_workload(520, lengths, num_pages=32, max_pages=12)
    rng = wl.rng_for(521)
    ws_layers = []
    for i in range(n_layers):  # fresh q/k/v per layer, one page table and bucket
        w = dict(base)
        T = int(base["cu_seqlens"][-1])
        w["q"], w["k"], w["v"] = (wl.normal_bf16(rng, (T, 16, 128)), wl.normal_bf16(rng, (T, 8, 128)),
                                  wl.normal_bf16(rng, (T, 8, 128)))
        ws_layers.append(w)
    cu, pt = to_dev(ws_layers[0]["cu_seqlens"]), to_dev(ws_layers[0]["page_table"])
    qs = [to_dev(w["q"]) for w in ws_layers]
    ks = [to_dev(w["k"]) for w in ws_layers]
    vs = [to_dev(w["v"]) for w in ws_layers]
    kps = [to_dev(w["k_pages"]) for w in ws_layers]
    vps = [to_dev(w["v_pages"]) for w in ws_layers]
    outs = [torch.empty_like(q) for q in qs]
    g = qa.qa_prefill_graph_create(qs, ks, vs, cu, pt, kps, vps, outs)
    g.launch()
    torch.cuda.synchronize()
    for i, w in enumerate(ws_layers):
        ref = oracle.prefill(w["q"], w["k"], w["v"], w["cu_seqlens"])
        assert_close(f64(outs[i]), ref, f"prefill graph layer {i}")
        ekp, evp = oracle.page_write(w["k"], w["v"], w["cu_seqlens"], w["page_table"], w["k_pages"], w["v_pages"])
        np.testing.assert_array_equal(bits(kps[i]), ekp)
        np.testing.assert_array_equal(bits(vps[i]), evp)
    g.close()


def test_capture_reports_an_invalid_call():
    w = wl.decode_workload(530, (20,), num_pages=4, max_pages=2)
    q, kp, vp = to_dev(w["q"]), to_dev(w["k_pages"]), to_dev(w["v_pages"])
    pt, sl = to_dev(w["page_table"]), to_dev(w["seq_lens"])
    tiny_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")  # too small: the captured call is rejected
    with pytest.raises(qa.QAError) as e:
        qa.qa_decode_graph_create([q], [kp], [vp], pt, sl, [torch.empty_like(q)], workspace=tiny_ws)
    assert "workspace" in str(e.value)


def test_a_set_of_buckets_captured_side_by_side():
    # a serving loop keeps one captured step per decode batch size and per
    # packed prefill bucket (M* page, "Serving notes": graphs captured per
    # decode batch and per prefill bucket) and replays whichever the step
    # needs: two decode batches and two prefill buckets, captured up front,
    # replayed interleaved with refills in between, each against the oracle
    decode_sets = {}
    for B, lengths in ((2, (33, 700)), (5, (1, 16, 17, 250, 1999))):
        base = wl.decode_workload(540 + B, lengths, num_pages=220, max_pages=125)
        d = {k: to_dev(base[k]) for k in ("q", "k_pages", "v_pages", "page_table", "seq_lens")}
        ws = torch.zeros(qa.qa_decode_workspace_size(B, 2000, num_pages=220, max_pages_per_seq=125),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty_like(d["q"])
        g = qa.qa_decode_graph_create([d["q"]], [d["k_pages"]], [d["v_pages"]], d["page_table"], d["seq_lens"],
                                      [out], workspace=ws)
        decode_sets[B] = (base, d, out, g)
    prefill_sets = {}
    for name, lengths in (("small", (64, 9)), ("large", (300, 129, 77))):
        base = wl.prefill_workload(550 + len(lengths), lengths, num_pages=64, max_pages=20)
        d = {k: to_dev(base[k]) for k in ("q", "k", "v", "cu_seqlens", "page_table", "k_pages", "v_pages")}
        out = torch.empty_like(d["q"])
        g = qa.qa_prefill_graph_create([d["q"]], [d["k"]], [d["v"]], d["cu_seqlens"], d["page_table"],
                                       [d["k_pages"]], [d["v_pages"]], [out])
        prefill_sets[name] = (base, d, out, g)
    rng = wl.rng_for(560)
    for rnd in range(2):
        for B, (base, d, out, g) in decode_sets.items():
            q = wl.normal_bf16(rng, base["q"].shape)
            d["q"].copy_(to_dev(q))
            g.launch()
            torch.cuda.synchronize()
            ref = oracle.decode(q, base["k_pages"], base["v_pages"], base["page_table"], base["seq_lens"])
            assert_close(f64(out), ref, f"decode batch {B}, round {rnd}")
        for name, (base, d, out, g) in prefill_sets.items():
            T = int(base["cu_seqlens"][-1])
            q = wl.normal_bf16(rng, (T, 16, 128))
            d["q"].copy_(to_dev(q))
            g.launch()
            torch.cuda.synchronize()
            ref = oracle.prefill(q, base["k"], base["v"], base["cu_seqlens"])
            assert_close(f64(out), ref, f"prefill bucket {name}, round {rnd}")
            ekp, evp = oracle.page_write(base["k"], base["v"], base["cu_seqlens"], base["page_table"],
                                         base["k_pages"], base["v_pages"])
            np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
            np.testing.assert_array_equal(bits(d["v_pages"]), evp)
    for _, _, _, g in list(decode_sets.values()) + list(prefill_sets.values()):
        g.close()
    assert qa.qa_device_status() == 0
