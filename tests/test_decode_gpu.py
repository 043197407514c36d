"""GPU parity of qa_decode_attn against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def run_decode(w, **kw):
    q = to_dev(w["q"])
    kp, vp = to_dev(w["k_pages"]), to_dev(w["v_pages"])
    pt, sl = to_dev(w["page_table"]), to_dev(w["seq_lens"])
    out = qa.qa_decode_attn(q, kp, vp, pt, sl, **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("lengths", [
    (1, 15, 16, 17, 127, 128, 129),
    (0, 5, 0, 33),
    (2000,),
    (16,) * 40,
])
def test_small_lengths(lengths):
    maxp = max(1, -(-max(lengths) // 16))
    w = wl.decode_workload(100 + len(lengths), lengths, num_pages=sum(-(-l // 16) for l in lengths) + 9, max_pages=maxp)
    out = run_decode(w, debug_checks=True)
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, f"lengths {lengths}")
    for b, L in enumerate(lengths):
        if L == 0:
            assert (bits(out[b]) == 0).all()


def test_many_requests_share_ctas():
    rng = np.random.default_rng(9)
    lengths = rng.integers(1, 70, size=600)
    w = wl.decode_workload(77, lengths, num_pages=int(sum(-(-l // 16) for l in lengths)) + 3, max_pages=5)
    out = run_decode(w, debug_checks=True)
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "600 short requests")


def test_mha_group_one():
    w = wl.decode_workload(31, (300, 45, 1), num_pages=40, max_pages=20, hq=8, hkv=8)
    out = run_decode(w, debug_checks=True)
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "MHA 8/8")


def test_single_key_returns_value_bit_exact():
    w = wl.decode_workload(5, (1, 1, 1, 1), num_pages=8, max_pages=2)
    out = run_decode(w)
    for b in range(4):
        v0 = w["v_pages"][w["page_table"][b, 0], 0]  # [Hkv, D]
        np.testing.assert_array_equal(bits(out[b]), np.repeat(v0, 2, axis=0))


def test_permuted_page_table_gives_identical_output():
    w = wl.decode_workload(6, (300, 17, 999), num_pages=128, max_pages=63)
    out_a = run_decode(w)
    ck, cv = np.full_like(w["k_pages"], wl.BF16_NAN), np.full_like(w["v_pages"], wl.BF16_NAN)
    table = np.full_like(w["page_table"], -1)
    nxt = 0
    for b, L in enumerate(w["seq_lens"]):
        for p in range(-(-int(L) // 16)):
            ck[nxt], cv[nxt] = w["k_pages"][w["page_table"][b, p]], w["v_pages"][w["page_table"][b, p]]
            table[b, p] = nxt
            nxt += 1
    w2 = dict(w, k_pages=ck, v_pages=cv, page_table=table)
    out_b = run_decode(w2)
    np.testing.assert_array_equal(bits(out_a), bits(out_b))


def test_workload_batched_decode_0p6b_full():
    w = wl.decode_0p6b()
    out = run_decode(w, debug_checks=True)
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "decode 0.6B workload")


def test_workload_long_context_1p7b_full():
    # the long-context decode workload, every (request, head) row checked
    # against the oracle over the whole output tensor
    w = wl.decode_1p7b()
    out = run_decode(w, debug_checks=True)
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "decode 1.7B workload (all rows)")


def test_tiny_workload_decode():
    t = wl.tiny()
    ekp, evp = oracle.page_write(t["k"], t["v"], t["cu_seqlens"], t["page_table"], t["k_pages"], t["v_pages"])
    w = dict(q=t["decode_q"], k_pages=ekp, v_pages=evp, page_table=t["page_table"], seq_lens=t["seq_lens"])
    out = run_decode(w, debug_checks=True)
    ref = oracle.decode(t["decode_q"], ekp, evp, t["page_table"], t["seq_lens"])
    assert_close(f64(out), ref, "tiny decode")


def test_bad_page_id_is_reported_not_faulted():
    w = wl.decode_workload(8, (40, 20), num_pages=8, max_pages=3)
    w["page_table"] = w["page_table"].copy()
    w["page_table"][0, 1] = 1 << 20  # outside the pool: must be skipped and reported
    with pytest.raises(qa.QAError) as e:
        run_decode(w, debug_checks=True)
    assert e.value.status == -6 and "bad page" in str(e.value)
    assert qa.qa_device_status() == 0  # cleared


def test_workspace_too_small_is_rejected():
    w = wl.decode_workload(8, (40,), num_pages=8, max_pages=3)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(qa.QAError) as e:
        run_decode(w, workspace=ws)
    assert e.value.status == -1 and "workspace" in str(e.value)


@pytest.mark.parametrize("lengths", [
    (2000, 2000),                # 250 pages over 152 CTAs: two pages each, some idle
    (31,) * 100 + (500,),        # many 2-page requests and one long one
    (1,) * 40 + (3000,) * 3,     # idle CTAs, single-page requests and long ones
])
def test_uneven_page_distributions(lengths):
    # few pages per CTA, idle CTAs, many split requests: every page must
    # reach exactly one partial and every partial the merge
    n_pages = sum(-(-L // 16) for L in lengths)
    w = wl.decode_workload(700 + len(lengths), lengths, num_pages=n_pages + 11, max_pages=max(-(-L // 16) for L in lengths))
    for call in range(3):  # the counters must be left at zero between calls
        out = run_decode(w, debug_checks=True)
        ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
        assert_close(f64(out), ref, f"lengths {lengths[:3]}... call {call}")


def test_host_mapped_query_table_lengths_and_output():
    # q, page table, lengths and out in page-locked host memory, passed to the
    # C ABI as they are (the device reaches them directly); the pools stay in
    # HBM.  Two calls in a row, each against the oracle.
    import ctypes

    w = wl.decode_workload(81, (1, 17, 300, 0, 129, 2000), num_pages=200, max_pages=125)
    kp, vp = to_dev(w["k_pages"]), to_dev(w["v_pages"])
    hq = torch.from_numpy(w["q"].view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    hpt = torch.from_numpy(w["page_table"].copy()).pin_memory()
    hsl = torch.from_numpy(w["seq_lens"].copy()).pin_memory()
    hout = torch.full(w["q"].shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    B = len(w["seq_lens"])
    ws = torch.zeros(qa.qa_decode_workspace_size(B, 2000, num_pages=200, max_pages_per_seq=125), dtype=torch.uint8,
                     device="cuda")
    p = qa._params(n_q_heads=16, n_kv_heads=8, head_dim=128, num_pages=200, max_pages_per_seq=125, workspace=ws,
                   debug_checks=True)
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    for call in range(2):
        hout.fill_(float("nan"))
        st = qa._lib.qa_decode_attn(ctypes.c_void_p(hq.data_ptr()), ctypes.c_void_p(kp.data_ptr()),
                                    ctypes.c_void_p(vp.data_ptr()), ctypes.c_void_p(hpt.data_ptr()),
                                    ctypes.c_void_p(hsl.data_ptr()), B, ctypes.c_void_p(hout.data_ptr()),
                                    ctypes.byref(p))
        assert st == 0, qa.qa_last_error()
        torch.cuda.synchronize()
        got = wl.bf16_to_f64(hout.view(torch.int16).numpy().view(np.uint16))
        assert_close(got, ref, f"host-mapped decode, call {call + 1}")
        assert (wl.bf16_to_f64(hout[3].view(torch.int16).numpy().view(np.uint16)) == 0).all()  # seq_len 0


def test_largest_batch():
    # 4096 requests, the most one call takes (the page prefix sums live in
    # shared memory), lengths 1..40; one more is rejected before any launch
    rng = np.random.default_rng(90)
    lengths = rng.integers(1, 41, size=4096).astype(np.int32)
    n_pages = int(sum(-(-int(L) // 16) for L in lengths))
    w = wl.decode_workload(91, lengths, num_pages=n_pages + 3, max_pages=3)
    out = run_decode(w, debug_checks=True)
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "4096 requests")
    big = wl.decode_workload(92, np.ones(4097, np.int32), num_pages=4097, max_pages=1)
    with pytest.raises(qa.QAError) as e:
        run_decode(big)
    assert e.value.status == -1 and "batch 4097" in str(e.value)
