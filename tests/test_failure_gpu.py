"""Failure handling on the GPU without a fault: a bounded wait that nothing
completes gives up, reports QA_DEVICE_TIMEOUT through the device status word,
and the context keeps running the attention kernels."""
import time

import pytest

import oracle
import workloads as wl
from _util import assert_close, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def test_expired_wait_is_reported_and_the_context_stays_usable():
    assert qa.qa_device_status() == 0
    t0 = time.perf_counter()
    qa.qa_check_bounded_wait(20000)  # the wait gives up after 20 ms
    bits = qa.qa_device_status()  # synchronises, reads and clears
    elapsed = time.perf_counter() - t0
    assert bits == 0x8, f"status bits {bits:#x}"
    assert 0.019 < elapsed < 5.0
    assert qa.qa_device_status() == 0  # cleared
    # the same context still runs a decode, checked against the oracle
    w = wl.decode_workload(9, (40, 17), num_pages=8, max_pages=3)
    d = {k: to_dev(w[k]) for k in ("q", "k_pages", "v_pages", "page_table", "seq_lens")}
    out = qa.qa_decode_attn(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["seq_lens"], debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "decode after an expired wait")
