"""GPU parity of qa_decode_append (per-head QK-norm, NEOX RoPE and the page
write of the new token) against the fp64 oracle, through the C ABI; and of
the decode step it feeds (append, then qa_decode_attn).

The append's bf16 outputs are checked with the rounding rule of
``_util.assert_rounded_match``.
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


def _dev_inputs(w):
    d = {k: to_dev(w[k]) for k in ("q_new", "k_new", "v_new", "q_gain", "k_gain", "page_table", "seq_lens",
                                   "k_pages", "v_pages")}
    return d


def run_append(w, **kw):
    d = _dev_inputs(w)
    q_out = qa.qa_decode_append(d["q_new"], d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"],
                                d["seq_lens"], d["k_pages"], d["v_pages"], rms_eps=EPS, rope_theta=THETA, **kw)
    torch.cuda.synchronize()
    return q_out, d


def oracle_append(w):
    return oracle.decode_append(w["q_new"], w["k_new"], w["v_new"], w["q_gain"], w["k_gain"], w["page_table"],
                                w["seq_lens"], w["k_pages"], w["v_pages"], eps=EPS, theta=THETA)


def check_append(w, what):
    q_out, d = run_append(w, debug_checks=True)
    r = oracle_append(w)
    assert_rounded_match(bits(q_out), r["q_rot"], pair_scale(w["q_new"], w["q_gain"]), f"{what}: q")
    kp, vp = bits(d["k_pages"]), bits(d["v_pages"])
    pos = w["seq_lens"] - 1
    pages = w["page_table"][np.arange(len(pos)), pos // 16]
    slots = pos % 16
    assert_rounded_match(kp[pages, slots], r["k_rot"], pair_scale(w["k_new"], w["k_gain"]), f"{what}: k slot")
    np.testing.assert_array_equal(vp[pages, slots], w["v_new"])
    # nothing else in the pools changed
    kp[pages, slots] = w["k_pages"][pages, slots]
    vp[pages, slots] = w["v_pages"][pages, slots]
    np.testing.assert_array_equal(kp, w["k_pages"])
    np.testing.assert_array_equal(vp, w["v_pages"])
    return q_out, d, r


@pytest.mark.parametrize("x_scale", [1.0, 1e-3, 40.0])
def test_small_batch(x_scale):
    # positions 0, 16, 39, 202: first slot, a page's first slot, mid-page
    w = wl.decode_append_workload(41, (1, 17, 40, 203), num_pages=32, max_pages=16, x_scale=x_scale)
    check_append(w, f"small batch x{x_scale}")


def test_page_boundaries():
    w = wl.decode_append_workload(42, (15, 16, 32, 33, 48, 255, 256, 257), num_pages=64, max_pages=20)
    check_append(w, "page boundaries")


def test_large_positions_share_a_page():
    # one small pool; every page-table entry of a request names the same page,
    # so positions up to 65535 need no large pool
    lengths = np.array([1, 1000, 16384, 40001, 65535, 65536], np.int32)
    B, maxp = len(lengths), 4096
    table = np.repeat(np.arange(B, dtype=np.int32)[:, None], maxp, axis=1)
    pool = wl.normal_bf16(wl.rng_for(44), (B, 16, wl.HKV, wl.D_DEC))
    w = dict(page_table=table, seq_lens=lengths, k_pages=pool, v_pages=pool.copy())
    w.update(wl.append_inputs(wl.rng_for(45), B))
    check_append(w, "large positions")


def test_mha_group_one():
    w = wl.decode_append_workload(46, (5, 70, 300), num_pages=40, max_pages=20)
    # 8 query heads over 8 KV heads: keep the first half of the query heads
    w["q_new"] = np.ascontiguousarray(w["q_new"][:, :8])
    check_append(w, "MHA 8/8")


def test_in_place_query():
    w = wl.decode_append_workload(47, (9, 100), num_pages=16, max_pages=8)
    d = _dev_inputs(w)
    q = d["q_new"].clone()
    out = qa.qa_decode_append(q, d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"], d["seq_lens"],
                              d["k_pages"], d["v_pages"], q_out=q, rms_eps=EPS, rope_theta=THETA)
    torch.cuda.synchronize()
    assert out.data_ptr() == q.data_ptr()
    r = oracle_append(w)
    assert_rounded_match(bits(q), r["q_rot"], pair_scale(w["q_new"], w["q_gain"]), "in place")


def test_bad_page_and_length_are_reported():
    w = wl.decode_append_workload(48, (20, 30), num_pages=8, max_pages=4)
    w["page_table"] = w["page_table"].copy()
    w["page_table"][1, 1] = 99
    with pytest.raises(qa.QAError) as e:
        run_append(w, debug_checks=True)
    assert e.value.status == -6 and "bad page" in str(e.value)
    w = wl.decode_append_workload(48, (20, 30), num_pages=8, max_pages=4)
    w["seq_lens"] = np.array([0, 65], np.int32)
    with pytest.raises(qa.QAError) as e:
        run_append(w, debug_checks=True)
    assert e.value.status == -6 and "bad length" in str(e.value)


def test_decode_step_workload_0p6b():
    """Append then decode on the batched-decode workload (B = 32, L ~ U[200,
    2000]): the decode output against the oracle's append + decode."""
    w = wl.with_append(wl.decode_0p6b(), 2)
    q_out, d, r = check_append(w, "decode 0.6B append")
    out = qa.qa_decode_attn(q_out, d["k_pages"], d["v_pages"], d["page_table"], d["seq_lens"], debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.decode(r["q"], r["k_pages"], r["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "decode step 0.6B")


def test_decode_step_graph_replay():
    """The two launches of a decode step captured in one CUDA graph and
    replayed: same results as eager calls (the append's early launch of the
    decode is graph-safe)."""
    w = wl.decode_append_workload(49, (33, 250, 1000), num_pages=96, max_pages=64)
    d = _dev_inputs(w)
    q_out = torch.empty_like(d["q_new"])
    out = torch.empty_like(d["q_new"])
    ws = torch.zeros(qa.qa_decode_workspace_size(3, 1000, num_pages=96, max_pages_per_seq=64), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()

    def step():
        qa.qa_decode_append(d["q_new"], d["k_new"], d["v_new"], d["q_gain"], d["k_gain"], d["page_table"],
                            d["seq_lens"], d["k_pages"], d["v_pages"], q_out=q_out, rms_eps=EPS, rope_theta=THETA,
                            stream=s)
        qa.qa_decode_attn(q_out, d["k_pages"], d["v_pages"], d["page_table"], d["seq_lens"], out, workspace=ws,
                          stream=s)

    with torch.cuda.stream(s):
        step()  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    r = oracle_append(w)
    ref = oracle.decode(r["q"], r["k_pages"], r["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "graph replay")
    assert qa.qa_device_status() == 0
