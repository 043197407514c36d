"""qa_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory -- a plugin whose host application owns every device
allocation, a real-time path that may not wait on or fail in an allocator,
plain C code with no allocator of its own.  Its split-K scratch is a fixed
4 MiB array built into the library instead of a caller workspace.

Called through the C ABI with ctypes, on two calls in a row through the
shared array, and checked against the fp64 oracle and against qa_decode_attn
(the entry point that takes a caller workspace), within the tolerances of
the other parity tests.  Also: the largest batch the array holds runs and the
next one is rejected, for both head groupings.  Kept in a file that pytest
collects last, so that a failure here does not stop the rest of the suite."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, f64, to_dev

pytestmark = pytest.mark.gpu

import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402

SCRATCH_BYTES = 4 << 20  # the built-in array's size, as include/qa.h states it


def _c_noalloc():
    lib = ctypes.CDLL(qa.lib_path)
    fn = lib.qa_decode_attn_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [P, P, P, P, P, ctypes.c_int, P, ctypes.POINTER(qa.qa_attn_params)]
    fn.restype = ctypes.c_int
    return fn


def _inputs(w):
    return {k: to_dev(w[k]) for k in ("q", "k_pages", "v_pages", "page_table", "seq_lens")}


def _call_noalloc(fn, d, out, stream, batch=None):
    B, Hq, D = d["q"].shape
    P, PS, Hkv, _ = d["k_pages"].shape
    p = qa.qa_attn_default_params()
    p.n_q_heads, p.n_kv_heads, p.head_dim, p.page_size = Hq, Hkv, D, PS
    p.num_pages, p.max_pages_per_seq = P, d["page_table"].shape[1]
    p.stream = ctypes.c_void_p(stream.cuda_stream)
    return fn(ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k_pages"].data_ptr()),
              ctypes.c_void_p(d["v_pages"].data_ptr()), ctypes.c_void_p(d["page_table"].data_ptr()),
              ctypes.c_void_p(d["seq_lens"].data_ptr()), B if batch is None else batch,
              ctypes.c_void_p(out.data_ptr()), ctypes.byref(p))


def _oracle(w):
    return oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])


def _check_against_both(fn, w, what):
    """Two calls in a row through the shared array; each compared with the
    oracle and with qa_decode_attn on the same inputs."""
    d = _inputs(w)
    stream = torch.cuda.current_stream()
    ref = _oracle(w)
    for call in range(2):
        got = torch.full_like(d["q"], float("nan"))
        assert _call_noalloc(fn, d, got, stream) == 0, qa.qa_last_error()
        with_ws = qa.qa_decode_attn(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["seq_lens"])
        torch.cuda.synchronize()
        assert_close(f64(got), ref, f"{what}, call {call + 1} against the oracle")
        assert_close(f64(got), f64(with_ws), f"{what}, call {call + 1} against qa_decode_attn")


def _largest_batch(n_q_heads, n_kv_heads):
    """Largest batch whose decode scratch fits the built-in array on this device."""
    lo, hi = 1, 4096
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if qa.qa_decode_workspace_size(mid, 16, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_noalloc_matches_the_oracle_and_the_workspace_decode_on_two_calls_in_a_row():
    fn = _c_noalloc()
    _check_against_both(fn, wl.decode_0p6b(), "batched decode 0.6B")
    w = wl.decode_workload(55, (1, 17, 300, 0, 129, 2000), num_pages=200, max_pages=125)
    _check_against_both(fn, w, "ragged lengths")
    assert qa.qa_device_status() == 0


@pytest.mark.parametrize("hq,hkv", [(16, 8), (8, 8)])
def test_noalloc_largest_batch_runs_and_the_next_is_rejected(hq, hkv):
    fn = _c_noalloc()
    B = _largest_batch(hq, hkv)
    assert B >= 32
    rng = np.random.default_rng(57 + hq)
    lengths = rng.integers(1, 70, size=B + 1).astype(np.int32)
    n_pages = int(sum(-(-int(L) // 16) for L in lengths))
    w = wl.decode_workload(58 + hq, lengths, num_pages=n_pages + 5, max_pages=5, hq=hq, hkv=hkv)
    # the first B requests: the largest batch the array holds
    wb = dict(w, q=w["q"][:B], page_table=w["page_table"][:B], seq_lens=w["seq_lens"][:B])
    _check_against_both(fn, wb, f"{hq}/{hkv} heads, largest batch {B}")
    # one more request does not fit: rejected before any launch
    d = _inputs(w)
    out = torch.full_like(d["q"], float("nan"))
    assert _call_noalloc(fn, d, out, torch.cuda.current_stream()) == -1
    assert "scratch" in qa.qa_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
