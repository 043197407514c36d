"""GPU parity of qa_prefill_chunk_attn (chunked prefill after n_past cached
positions, with the positioned KV page write) against the fp64 oracle,
through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402

KEYS = ("q", "k", "v", "cu_seqlens", "n_past", "page_table", "k_pages", "v_pages")


def run_chunk(w, **kw):
    d = {k: to_dev(w[k]) for k in KEYS}
    out = qa.qa_prefill_chunk_attn(d["q"], d["k"], d["v"], d["cu_seqlens"], d["n_past"], d["page_table"],
                                   d["k_pages"], d["v_pages"], **kw)
    torch.cuda.synchronize()
    return out, d


def check(w, what):
    out, d = run_chunk(w, debug_checks=True)
    ref = oracle.prefill_chunk(w["q"], w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"], w["k_pages"],
                               w["v_pages"])
    assert_close(f64(out), ref, what)
    ekp, evp = oracle.page_write_at(w["k"], w["v"], w["cu_seqlens"], w["n_past"], w["page_table"], w["k_pages"],
                                    w["v_pages"])
    np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
    np.testing.assert_array_equal(bits(d["v_pages"]), evp)
    return out, d


def _workload(seed, past, new):
    need = [-(-(p + n) // 16) for p, n in zip(past, new)]
    return wl.chunk_workload(seed, past, new, num_pages=sum(need) + 5, max_pages=max(need))


@pytest.mark.parametrize("past,new", [
    ((0, 0), (7, 130)),                      # no cached positions: the prefill
    ((16, 32, 128), (1, 16, 5)),             # page-aligned history
    ((5, 17, 127, 129), (3, 40, 1, 128)),    # boundary page shared by cached and new rows
    ((300, 1000), (129, 300)),               # several cached tiles, several new tiles
    ((250, 0, 77), (0, 20, 1)),              # a request with no new rows
])
def test_small_chunks(past, new):
    check(_workload(600 + sum(past) + sum(new), past, new), f"past {past} new {new}")


def test_many_requests_mixed_costs():
    # more than 32 requests (the job order reads the lengths 32 at a time),
    # costs from 1 to 6 key tiles, empty requests and empty histories mixed
    rng = np.random.default_rng(615)
    past = tuple(int(x) for x in rng.choice([0, 3, 16, 130, 257, 400], size=45))
    new = tuple(int(x) for x in rng.choice([0, 1, 17, 128, 129, 200], size=45))
    check(_workload(615, past, new), "45 requests")


def test_split_prompt_equals_one_shot_on_the_gpu():
    # the first 200 rows by qa_prefill_attn, the remaining 157 by the chunked call
    L, split = 357, 200
    p = wl.prefill_workload(610, (L,), num_pages=30, max_pages=23)
    d = {k: to_dev(p[k]) for k in ("q", "k", "v", "page_table", "k_pages", "v_pages")}
    head = to_dev(np.array([0, split], np.int32))
    tail = to_dev(np.array([0, L - split], np.int32))
    out_head = qa.qa_prefill_attn(d["q"][:split].contiguous(), d["k"][:split].contiguous(), d["v"][:split].contiguous(),
                                  head, d["page_table"], d["k_pages"], d["v_pages"], debug_checks=True)
    out_tail = qa.qa_prefill_chunk_attn(d["q"][split:].contiguous(), d["k"][split:].contiguous(),
                                        d["v"][split:].contiguous(), tail, to_dev(np.array([split], np.int32)),
                                        d["page_table"], d["k_pages"], d["v_pages"], debug_checks=True)
    torch.cuda.synchronize()
    one_shot = oracle.prefill(p["q"], p["k"], p["v"], p["cu_seqlens"])
    assert_close(f64(out_head), one_shot[:split], "head")
    assert_close(f64(out_tail), one_shot[split:], "tail")
    ekp, evp = oracle.page_write(p["k"], p["v"], p["cu_seqlens"], p["page_table"], p["k_pages"], p["v_pages"])
    np.testing.assert_array_equal(bits(d["k_pages"]), ekp)
    np.testing.assert_array_equal(bits(d["v_pages"]), evp)


def test_workload_reprefill_bucket():
    w = wl.chunk_reprefill()
    check(w, "re-prefill bucket")


def test_bad_history_length_is_reported():
    w = _workload(620, (20, 30), (5, 5))
    w["n_past"] = np.array([20, w["max_pages"] * 16 + 1], np.int32)
    with pytest.raises(qa.QAError) as e:
        run_chunk(w, debug_checks=True)
    assert e.value.status == -6 and "bad length" in str(e.value)



@pytest.mark.parametrize("cached_page", [0, 9])
def test_bad_cached_page_id_is_reported_not_faulted(cached_page):
    # a cached page id outside the pool: reported, that page not loaded, and
    # the request that does not use it still right.  Page 0 sits in the first
    # cached key tile, page 9 in the second (each tile's page boxes are
    # requested from separate lanes).
    w = _workload(630 + cached_page, (200, 40), (20, 7))
    w["page_table"] = w["page_table"].copy()
    w["page_table"][0, cached_page] = w["num_pages"] + 3
    with pytest.raises(qa.QAError) as e:
        run_chunk(w, debug_checks=True)
    assert e.value.status == -6 and "bad page" in str(e.value)
    assert qa.qa_device_status() == 0  # cleared
    out, _ = run_chunk(w)
    qa.qa_device_status()  # clear this call's report too
    r0, r1 = int(w["cu_seqlens"][1]), int(w["cu_seqlens"][2])
    ref = oracle.prefill_chunk(w["q"][r0:r1], w["k"][r0:r1], w["v"][r0:r1], np.array([0, r1 - r0], np.int32),
                               w["n_past"][1:2], w["page_table"][1:2], w["k_pages"], w["v_pages"])
    assert_close(f64(out)[r0:r1], ref, "the request without the bad page")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (4, 2)])
def test_other_head_counts(hq, hkv):
    past, new = (130, 0, 16), (40, 129, 1)
    need = [-(-(p + n) // 16) for p, n in zip(past, new)]
    w = wl.chunk_workload(640 + hq, past, new, num_pages=sum(need) + 5, max_pages=max(need), hq=hq, hkv=hkv)
    check(w, f"chunked prefill {hq}/{hkv} heads")
