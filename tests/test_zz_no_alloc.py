"""qa_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (its split-K scratch is an array built into the
library).  Called through the C ABI with ctypes and checked against
qa_decode_attn, the entry point that takes a caller workspace, on two calls
in a row.  Kept in a file that runs last so a failure here does not hide the
rest of the suite."""
import ctypes

import numpy as np
import pytest

import workloads as wl
from _util import errors, f64, to_dev, MAX_ABS, REL_L2

pytestmark = pytest.mark.gpu

import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def _c_noalloc():
    lib = ctypes.CDLL(qa.lib_path)
    fn = lib.qa_decode_attn_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [P, P, P, P, P, ctypes.c_int, P, ctypes.POINTER(qa.qa_attn_params)]
    fn.restype = ctypes.c_int
    return lib, fn


def _inputs(w):
    return {k: to_dev(w[k]) for k in ("q", "k_pages", "v_pages", "page_table", "seq_lens")}


def _call_noalloc(fn, d, out, stream):
    B, Hq, D = d["q"].shape
    P, PS, Hkv, _ = d["k_pages"].shape
    p = qa.qa_attn_default_params()
    p.n_q_heads, p.n_kv_heads, p.head_dim, p.page_size = Hq, Hkv, D, PS
    p.num_pages, p.max_pages_per_seq = P, d["page_table"].shape[1]
    p.stream = ctypes.c_void_p(stream.cuda_stream)
    return fn(ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k_pages"].data_ptr()),
              ctypes.c_void_p(d["v_pages"].data_ptr()), ctypes.c_void_p(d["page_table"].data_ptr()),
              ctypes.c_void_p(d["seq_lens"].data_ptr()), B, ctypes.c_void_p(out.data_ptr()), ctypes.byref(p))


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    _, fn = _c_noalloc()
    stream = torch.cuda.current_stream()
    cases = [wl.decode_0p6b(), wl.decode_workload(55, (1, 17, 300, 0, 129, 2000), num_pages=200, max_pages=125)]
    for w in cases:  # two calls in a row through the shared scratch array
        d = _inputs(w)
        got = torch.empty_like(d["q"])
        assert _call_noalloc(fn, d, got, stream) == 0, qa.qa_last_error()
        ref = qa.qa_decode_attn(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["seq_lens"])
        torch.cuda.synchronize()
        a, b = f64(got), f64(ref)
        assert np.isfinite(a).all()
        max_abs, rel = errors(a, b)
        assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert qa.qa_device_status() == 0


def test_noalloc_rejects_a_batch_beyond_the_scratch_array():
    _, fn = _c_noalloc()
    lengths = np.full(1000, 3, np.int32)
    w = wl.decode_workload(56, lengths, num_pages=1000, max_pages=1)
    d = _inputs(w)
    out = torch.empty_like(d["q"])
    st = _call_noalloc(fn, d, out, torch.cuda.current_stream())
    assert st == -1
    assert "scratch" in qa.qa_last_error()
