"""GPU parity of qa_prefill_attn (causal attention + KV page write) against
the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def run_prefill(w, **kw):
    d = {k: to_dev(w[k]) for k in ("q", "k", "v", "cu_seqlens", "page_table", "k_pages", "v_pages")}
    out = qa.qa_prefill_attn(d["q"], d["k"], d["v"], d["cu_seqlens"], d["page_table"], d["k_pages"], d["v_pages"], **kw)
    torch.cuda.synchronize()
    return out, d


def check(w, what):
    out, d = run_prefill(w, debug_checks=True)
    ref = oracle.prefill(w["q"], w["k"], w["v"], w["cu_seqlens"])
    assert_close(f64(out), ref, what)
    ekp, evp = oracle.page_write(w["k"], w["v"], w["cu_seqlens"], w["page_table"], w["k_pages"], w["v_pages"])
    np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
    np.testing.assert_array_equal(bits(d["v_pages"]), evp)
    return out, d


@pytest.mark.parametrize("lengths", [(1, 15, 16, 17), (127, 128, 129), (64,), (1,), (300, 2, 0, 45)])
def test_small_lengths(lengths):
    maxp = max(1, -(-max(lengths) // 16))
    w = wl.prefill_workload(200 + sum(lengths), lengths, num_pages=sum(-(-l // 16) for l in lengths) + 5, max_pages=maxp)
    check(w, f"lengths {lengths}")


def test_tiny_workload_and_cross_pin():
    t = wl.tiny()
    out, d = check(t, "tiny prefill")
    # decode of the last prefill query over the freshly written pages equals
    # the last prefill row
    dq = d["q"][63:64].contiguous()
    dout = qa.qa_decode_attn(dq, d["k_pages"], d["v_pages"], d["page_table"], to_dev(t["seq_lens"]), debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.prefill(t["q"], t["k"], t["v"], t["cu_seqlens"], rows=np.arange(63 * 16, 64 * 16))
    assert_close(f64(dout)[0], ref, "decode of prefill row 63")
    assert_close(f64(dout)[0], f64(out)[63], "decode vs prefill row 63 (GPU)")


def test_workload_prefill_bucket_full():
    w = wl.prefill_bucket()
    check(w, "prefill bucket workload")


def test_untouched_slots_keep_sentinels():
    w = wl.prefill_workload(9, (20, 3), num_pages=10, max_pages=2)
    _, d = run_prefill(w)
    kp = bits(d["k_pages"])
    used = set()
    for r, L in enumerate((20, 3)):
        for i in range(L):
            used.add((int(w["page_table"][r, i // 16]), i % 16))
    for p in range(10):
        for s in range(16):
            if (p, s) not in used:
                assert (kp[p, s] == wl.BF16_NAN).all()


def test_bad_page_id_is_reported_not_faulted():
    w = wl.prefill_workload(10, (40,), num_pages=4, max_pages=3)
    w["page_table"] = w["page_table"].copy()
    w["page_table"][0, 2] = -7
    with pytest.raises(qa.QAError) as e:
        run_prefill(w, debug_checks=True)
    assert e.value.status == -6


def test_overlong_request_is_reported_and_clipped():
    # request 0 has 40 rows but its page-table row holds 2 pages (32 rows)
    w = wl.prefill_workload(11, (40, 5), num_pages=8, max_pages=3)
    w["page_table"] = np.ascontiguousarray(w["page_table"][:, :2])
    d = {k: to_dev(w[k]) for k in ("q", "k", "v", "cu_seqlens", "page_table", "k_pages", "v_pages")}
    with pytest.raises(qa.QAError) as e:
        qa.qa_prefill_attn(d["q"], d["k"], d["v"], d["cu_seqlens"], d["page_table"], d["k_pages"], d["v_pages"],
                           debug_checks=True)
    assert e.value.status == -6 and "bad length" in str(e.value)
    # rows [0, 32) of request 0 and all of request 1 reach the pools, nothing else
    keep = np.r_[0:32, 40:45]
    ekp, evp = oracle.page_write(w["k"][keep], w["v"][keep], np.array([0, 32, 37], np.int32), w["page_table"],
                                 w["k_pages"], w["v_pages"])
    np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
    np.testing.assert_array_equal(bits(d["v_pages"]), evp)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (4, 2), (2, 1)])
def test_other_head_counts(hq, hkv):
    # plain MHA (one query head per KV head: that job writes both the K and
    # the V rows) and GQA 2:1 with fewer heads than the Thinker's
    lengths = (130, 7, 256)
    w = wl.prefill_workload(230 + hq, lengths, num_pages=30, max_pages=16, hq=hq, hkv=hkv)
    check(w, f"prefill {hq}/{hkv} heads")
