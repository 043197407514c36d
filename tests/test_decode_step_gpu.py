"""GPU parity of qa_decode_step (the fused decode step: QK-norm + NEOX RoPE
+ KV append of the new token and the paged GQA decode in one launch) against
the fp64 oracle's append followed by its decode, through the C ABI.

The attention output is held to the attention tolerance; the appended K row
to the rounding rule of ``_util.assert_rounded_match``; the appended V row
and every other byte of the pools are bit-exact.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, assert_rounded_match, bits, f64, pair_scale, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402

EPS, THETA = wl.RMS_EPS, wl.ROPE_THETA
KEYS = ("q_new", "k_new", "v_new", "q_gain", "k_gain", "page_table", "seq_lens", "k_pages", "v_pages")


def run_step(w, **kw):
    d = {k: to_dev(w[k]) for k in KEYS}
    out = qa.qa_decode_step(d["q_new"], d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"],
                            d["seq_lens"], d["k_pages"], d["v_pages"], rms_eps=EPS, rope_theta=THETA, **kw)
    torch.cuda.synchronize()
    return out, d


def check_step(w, what):
    out, d = run_step(w, debug_checks=True)
    r = oracle.decode_append(w["q_new"], w["k_new"], w["v_new"], w["q_gain"], w["k_gain"], w["page_table"],
                             w["seq_lens"], w["k_pages"], w["v_pages"], eps=EPS, theta=THETA)
    ref = oracle.decode(r["q"], r["k_pages"], r["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, what)
    kp, vp = bits(d["k_pages"]), bits(d["v_pages"])
    pos = w["seq_lens"] - 1
    pages = w["page_table"][np.arange(len(pos)), pos // 16]
    slots = pos % 16
    assert_rounded_match(kp[pages, slots], r["k_rot"], pair_scale(w["k_new"], w["k_gain"]), f"{what}: k slot")
    np.testing.assert_array_equal(vp[pages, slots], w["v_new"])
    kp[pages, slots] = w["k_pages"][pages, slots]
    vp[pages, slots] = w["v_pages"][pages, slots]
    np.testing.assert_array_equal(kp, w["k_pages"])
    np.testing.assert_array_equal(vp, w["v_pages"])
    return out, d, r


@pytest.mark.parametrize("lengths", [
    (1, 15, 16, 17, 127, 128, 129),
    (2000,),
    (16,) * 40,
    (3000, 1, 2500, 33),
])
def test_small_lengths(lengths):
    n_pages = sum(-(-L // 16) for L in lengths) + 7
    w = wl.decode_append_workload(200 + len(lengths), lengths, num_pages=n_pages, max_pages=max(1, -(-max(lengths) // 16)))
    check_step(w, f"lengths {lengths}")


def test_only_the_new_token_returns_its_value():
    # seq_len 1: the new token is the only key, p = 1, out = v exactly
    w = wl.decode_append_workload(210, (1, 1, 1), num_pages=6, max_pages=1)
    out, _, _ = check_step(w, "single new token")
    np.testing.assert_array_equal(bits(out), np.repeat(w["v_new"], 2, axis=1))


def test_many_requests_share_ctas():
    rng = np.random.default_rng(211)
    lengths = rng.integers(1, 70, size=600)
    w = wl.decode_append_workload(211, lengths, num_pages=int(sum(-(-l // 16) for l in lengths)) + 3, max_pages=5)
    check_step(w, "600 short requests")


def test_mha_group_one():
    w = wl.decode_append_workload(212, (300, 45, 1), num_pages=40, max_pages=20)
    w["q_new"] = np.ascontiguousarray(w["q_new"][:, :8])
    check_step(w, "MHA 8/8")


def test_workload_decode_0p6b():
    check_step(wl.with_append(wl.decode_0p6b(), 2), "decode step 0.6B")


def test_matches_the_two_call_sequence():
    w = wl.with_append(wl.decode_0p6b(), 2)
    out_f, d_f = run_step(w)
    d = {k: to_dev(w[k]) for k in KEYS}
    q_rot = qa.qa_decode_append(d["q_new"], d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"],
                                d["seq_lens"], d["k_pages"], d["v_pages"], rms_eps=EPS, rope_theta=THETA)
    out_2 = qa.qa_decode_attn(q_rot, d["k_pages"], d["v_pages"], d["page_table"], d["seq_lens"])
    torch.cuda.synchronize()
    # same arithmetic up to fp32 evaluation order: near-identical outputs and pools
    assert_close(f64(out_f), f64(out_2), "fused vs two calls")
    assert (bits(d_f["k_pages"]) != bits(d["k_pages"])).sum() <= 64
    np.testing.assert_array_equal(bits(d_f["v_pages"]), bits(d["v_pages"]))


def test_empty_request_is_reported():
    w = wl.decode_append_workload(213, (20, 30), num_pages=8, max_pages=4)
    w["seq_lens"] = np.array([0, 30], np.int32)
    with pytest.raises(qa.QAError) as e:
        run_step(w, debug_checks=True)
    assert e.value.status == -6 and "bad length" in str(e.value)


def test_graph_replay():
    w = wl.decode_append_workload(214, (33, 250, 1000), num_pages=96, max_pages=64)
    d = {k: to_dev(w[k]) for k in KEYS}
    out = torch.empty_like(d["q_new"])
    ws = torch.zeros(qa.qa_decode_workspace_size(3, 1000, num_pages=96, max_pages_per_seq=64), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()

    def step():
        qa.qa_decode_step(d["q_new"], d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"],
                          d["seq_lens"], d["k_pages"], d["v_pages"], out, workspace=ws, rms_eps=EPS,
                          rope_theta=THETA, stream=s)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    r = oracle.decode_append(w["q_new"], w["k_new"], w["v_new"], w["q_gain"], w["k_gain"], w["page_table"],
                             w["seq_lens"], w["k_pages"], w["v_pages"], eps=EPS, theta=THETA)
    ref = oracle.decode(r["q"], r["k_pages"], r["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "graph replay")
    assert qa.qa_device_status() == 0


def test_new_token_with_two_pages_per_cta():
    # two pages per CTA: the request's last page (which the fused step
    # patches) sits in a short segment of a CTA that also merges
    w = wl.decode_append_workload(215, (2000, 2000, 1999), num_pages=400, max_pages=125)
    check_step(w, "two pages per CTA")
