"""GPU parity of qa_window_attn against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def run_window(w, cu, **kw):
    q, k, v = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"])
    out = qa.qa_window_attn(q, k, v, to_dev(cu), **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("counts", [(1,), (103,), (104,), (105,), (13, 117, 250), (600, 7)])
def test_small_windows(counts):
    w = wl.window_workload(300 + sum(counts), counts)
    cu = oracle.window_plan(counts)
    np.testing.assert_array_equal(qa.qa_window_plan(counts), cu)
    out = run_window(w, cu, debug_checks=True)
    ref = oracle.window(w["q"], w["k"], w["v"], cu)
    assert_close(f64(out), ref, f"counts {counts}")


@pytest.mark.parametrize("d", [64, 128])
def test_window_sizes_around_the_store_boxes(d):
    # the output leaves in whole row boxes plus the rows of a partial box:
    # window sizes around multiples of 8, 16 and 32 rows and around the
    # 128-row tile, every row checked; the output starts NaN-filled, so a row
    # left unwritten (or overwritten by a neighbouring window's box) fails
    sizes = [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 95, 96, 97, 103, 104, 105, 127, 128, 129]
    T = sum(sizes)
    w = wl.window_workload(350 + d, (T,), h=3, d=d)
    cu = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    q, k, v = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"])
    out = torch.full_like(q, float("nan"))
    qa.qa_window_attn(q, k, v, to_dev(cu), out, debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.window(w["q"], w["k"], w["v"], cu)
    assert_close(f64(out), ref, f"D={d}, window sizes {sizes}")


def test_head_dim_128_and_long_windows():
    counts = (300, 129)
    w = wl.window_workload(41, counts, h=4, d=128)
    cu = oracle.window_plan(counts, 200)
    out = run_window(w, cu, debug_checks=True)
    ref = oracle.window(w["q"], w["k"], w["v"], cu)
    assert_close(f64(out), ref, "D=128, windows of 200")


def test_window_split_equals_separate_calls():
    counts = (250,)
    w = wl.window_workload(42, counts)
    cu = oracle.window_plan(counts)
    whole = bits(run_window(w, cu))
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        part = dict(q=w["q"][a:b], k=w["k"][a:b], v=w["v"][a:b])
        one = bits(run_window(part, np.array([0, b - a], np.int32)))
        np.testing.assert_array_equal(whole[a:b], one)


def test_workload_aut_window_full():
    # the AuT windowed-attention workload, every row of every window checked
    # against the oracle over the whole output tensor
    w = wl.window_aut()
    cu = qa.qa_window_plan(w["token_counts"])
    np.testing.assert_array_equal(cu, oracle.window_plan(w["token_counts"]))
    q, k, v = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"])
    out = torch.full_like(q, float("nan"))  # a row left unwritten fails
    qa.qa_window_attn(q, k, v, to_dev(cu), out, debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.window(w["q"], w["k"], w["v"], cu)
    got = f64(out)
    assert_close(got, ref, f"AuT window workload ({got.shape[0]} tokens x {got.shape[1]} heads, all rows)")
    # the worst window as a diagnostic on failure of a later change
    err = np.abs(got - ref).max(axis=(1, 2))
    worst = int(np.argmax(err))
    assert err[worst] <= 1e-2, f"token {worst}"


def test_many_jobs_with_empty_windows():
    # more (window, head) jobs than the grid's sub-CTAs, so each one claims
    # several; empty windows (repeated offsets) scattered among them are
    # skipped and leave the jobs around them intact
    rng = np.random.default_rng(7)
    sizes = [int(s) if rng.random() > 0.2 else 0 for s in rng.integers(1, 129, size=180)]
    sizes[0] = 0
    sizes[-1] = 0
    cu = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    w = wl.window_workload(77, (int(cu[-1]),), h=6)
    q, k, v = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"])
    out = torch.full_like(q, float("nan"))
    qa.qa_window_attn(q, k, v, to_dev(cu), out, debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.window(w["q"], w["k"], w["v"], cu)
    assert_close(f64(out), ref, f"{len(sizes)} windows, {sizes.count(0)} empty")


def test_repeated_calls_bit_identical():
    # which sub-CTA computes a job changes from call to call (jobs are
    # claimed dynamically); the result of a job does not
    w = wl.window_aut()
    cu = to_dev(qa.qa_window_plan(w["token_counts"]))
    q, k, v = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"])
    first = bits(qa.qa_window_attn(q, k, v, cu))
    for _ in range(3):
        np.testing.assert_array_equal(bits(qa.qa_window_attn(q, k, v, cu)), first)


def test_job_counter_workspace_same_bits_and_left_zero():
    # with a workspace the jobs are claimed from a counter in it; the result
    # is the same bit for bit, and every call leaves the counter zero for the
    # next one (several calls in a row, two workloads, head_dim 64 and 128,
    # windows longer than one tile)
    ws = torch.zeros(qa.qa_window_workspace_size(), dtype=torch.uint8, device="cuda")
    aut = wl.window_aut()
    cases = [(aut, qa.qa_window_plan(aut["token_counts"]))]
    w = wl.window_workload(43, (300, 129, 5), h=4, d=128)
    cases.append((w, oracle.window_plan((300, 129, 5), 200)))
    w = wl.window_workload(44, (700, 40), h=14, d=64)
    cases.append((w, oracle.window_plan((700, 40), 150)))
    for w, cu in cases:
        q, k, v, dcu = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"]), to_dev(cu)
        fixed = bits(qa.qa_window_attn(q, k, v, dcu))
        for _ in range(3):
            got = qa.qa_window_attn(q, k, v, dcu, workspace=ws, debug_checks=True)
            np.testing.assert_array_equal(bits(got), fixed)
            assert int(ws.sum()) == 0, "job counter not reset"
        if w is not aut:
            assert_close(f64(got), oracle.window(w["q"], w["k"], w["v"], cu), "workspace")


def test_job_counter_survives_malformed_windows():
    # windows whose bounds are out of range are skipped and reported; the
    # claims run on past them, so the counter still ends at zero and the
    # next call on the same workspace is whole
    ws = torch.zeros(qa.qa_window_workspace_size(), dtype=torch.uint8, device="cuda")
    w = wl.window_workload(45, (600,), h=14)
    q, k, v = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"])
    assert qa.qa_device_status() == 0
    bad = to_dev(np.array([0, 104, 9999, 600], np.int32))  # [104, 9999) and [9999, 600) are invalid
    out = torch.full_like(q, float("nan"))
    qa.qa_window_attn(q, k, v, bad, out, workspace=ws)
    bits_ = qa.qa_device_status()
    assert bits_ & 0x4, f"status {bits_:#x}"  # bad segments
    assert int(ws.sum()) == 0, "job counter not reset after skipped windows"
    ref0 = oracle.window(w["q"][:104], w["k"][:104], w["v"][:104], np.array([0, 104], np.int32))
    assert_close(f64(out[:104]), ref0, "the valid window beside the malformed ones")
    assert torch.isnan(out[104:]).all(), "rows of skipped windows were written"
    cu = oracle.window_plan((600,))
    fixed = bits(qa.qa_window_attn(q, k, v, to_dev(cu)))
    np.testing.assert_array_equal(bits(qa.qa_window_attn(q, k, v, to_dev(cu), workspace=ws)), fixed)
    assert int(ws.sum()) == 0


@pytest.mark.parametrize("d", [64, 128])
def test_late_keys_far_above_the_first_block(d):
    # A few keys of every window score tens of log2 units above the rest
    # for many rows (keys 30 and 100 are planted as multiples of rows 7 and
    # 5's queries, x2 and x4: exact in bf16): the row maximum sits late in
    # the window, far from the first keys, and most probabilities of those
    # rows underflow against it.
    counts = (104 * 6 + 40,)
    w = wl.window_workload(46 + d, counts, h=4, d=d)
    cu = oracle.window_plan(counts)
    k = w["k"].copy()
    qf = (w["q"].astype(np.uint32) << 16).view(np.float32)
    for s0, s1 in zip(cu[:-1], cu[1:]):
        for key, row, mult in ((30, 7, 2.0), (100, 5, 4.0)):
            if s0 + key < s1:
                k[s0 + key] = ((qf[s0 + row] * mult).view(np.uint32) >> 16).astype(np.uint16)
    w["k"] = k
    out = run_window(w, cu, debug_checks=True)
    ref = oracle.window(w["q"], w["k"], w["v"], cu)
    assert_close(f64(out), ref, f"D={d}, planted late keys")


def test_job_counter_under_graph_replay():
    # the counter is reset by the kernel itself, so a captured call replays
    # with the same result every time (a CUDA graph of three calls, replayed
    # three times on its own stream)
    w = wl.window_aut()
    cu = to_dev(qa.qa_window_plan(w["token_counts"]))
    q, k, v = to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"])
    ws = torch.zeros(qa.qa_window_workspace_size(), dtype=torch.uint8, device="cuda")
    fixed = bits(qa.qa_window_attn(q, k, v, cu))
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    qa.qa_window_attn(q, k, v, cu, out, workspace=ws, stream=s)  # loads the kernel before the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            qa.qa_window_attn(q, k, v, cu, out, workspace=ws, stream=s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(out), fixed)
        assert int(ws.sum()) == 0
