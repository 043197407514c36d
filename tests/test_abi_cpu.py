"""C-ABI checks that need no GPU: the library builds, loads and exports
exactly the qa_* entry points declared in include/qa.h; the header compiles
as strict C99; host-side validation returns status codes without touching a
device; the host window planner matches the oracle's bit for bit."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qa.h")


@pytest.fixture(scope="session")
def libqa():
    import __graft_entry__

    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qa_[a-z_]+)\s*\(", src)))


def test_exports_exactly_the_declared_symbols(libqa):
    import __graft_entry__

    _build = __graft_entry__._builder()
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True, check=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    declared = declared_functions()
    assert declared, "no declarations parsed from qa.h"
    assert exported == declared
    for name in declared:
        assert hasattr(libqa, name)


def test_header_is_strict_c99(libqa, tmp_path):
    import __graft_entry__

    _build = __graft_entry__._builder()

    c = tmp_path / "abi_c.c"
    c.write_text(r'''
#include "qa.h"
#include <stddef.h>
#include <stdio.h>
#include <string.h>
int main(void) {
    qa_attn_params p = qa_attn_default_params();
    int32_t counts[2] = {117, 5};
    int32_t cu[8];
    if (p.abi_version != QA_ABI_VERSION || p.n_q_heads != 16 || p.n_kv_heads != 8) return 1;
    if (qa_decode_attn(NULL, NULL, NULL, NULL, NULL, 1, NULL, &p) != QA_STATUS_INVALID_PARAMS) return 2;
    if (strlen(qa_last_error()) == 0) return 3;
    if (qa_window_attn(NULL, NULL, NULL, NULL, 1, 0, NULL, NULL) != QA_STATUS_INVALID_PARAMS) return 4;
    p.abi_version = QA_ABI_VERSION + 1;
    if (qa_prefill_attn(NULL, NULL, NULL, NULL, 1, 0, NULL, NULL, NULL, NULL, &p) != QA_STATUS_INVALID_PARAMS) return 5;
    if (qa_decode_append(NULL, NULL, NULL, NULL, NULL, 1e-6f, 1e6f, NULL, NULL, 1, NULL, NULL, NULL, &p) !=
        QA_STATUS_INVALID_PARAMS) return 9;
    if (qa_window_plan(counts, 2, 0, cu, 8) != 3 || cu[1] != 104 || cu[2] != 117 || cu[3] != 122) return 6;
    {
        qa_graph *g = NULL;
        if (qa_decode_graph_create(0, NULL, NULL, NULL, NULL, NULL, 1, NULL, &p, &g) != QA_STATUS_INVALID_PARAMS) return 7;
        if (qa_graph_launch(NULL, NULL) != QA_STATUS_INVALID_PARAMS) return 8;
        qa_graph_destroy(g);
    }
    printf("%s\n", qa_version());
    printf("sizeof %u stable_metadata %u\n", (unsigned)sizeof(qa_attn_params),
           (unsigned)offsetof(qa_attn_params, stable_metadata));
    return 0;
}
''')
    exe = tmp_path / "abi_c"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(c), "-o", str(exe), _build.LIB, f"-Wl,-rpath,{os.path.dirname(_build.LIB)}"], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    import paged_kv_gqa_attention_gb300 as qa

    assert "abi 2" in res.stdout
    # the ctypes mirror of qa_attn_params has the C layout
    size, off = (int(x) for x in res.stdout.split()[-3::2])
    assert ctypes.sizeof(qa.qa_attn_params) == size
    assert qa.qa_attn_params.stable_metadata.offset == off


def _params(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    return qa.qa_attn_default_params()


def test_invalid_arguments_return_status_without_device(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    lib = qa._lib
    p = qa.qa_attn_default_params()
    fake = ctypes.c_void_p(0x1000)
    # NULL params
    assert lib.qa_decode_attn(fake, fake, fake, fake, fake, 1, fake, None) == -1
    assert "params is NULL" in qa.qa_last_error()
    # wrong abi version
    p.abi_version = 99
    assert lib.qa_window_attn(fake, fake, fake, fake, 1, 1, fake, ctypes.byref(p)) == -1
    assert "abi_version" in qa.qa_last_error()
    p = qa.qa_attn_default_params()
    p.num_pages, p.max_pages_per_seq = 4, 4
    # unsupported head_dim / heads / page size / batch
    for field, bad in (("head_dim", 96), ("n_kv_heads", 9), ("n_q_heads", 24), ("page_size", 32)):
        q = qa.qa_attn_default_params()
        q.num_pages, q.max_pages_per_seq = 4, 4
        setattr(q, field, bad)
        assert lib.qa_decode_attn(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(q)) == -1, field
    assert lib.qa_decode_attn(fake, fake, fake, fake, fake, 0, fake, ctypes.byref(p)) == -1
    assert "batch" in qa.qa_last_error()
    assert lib.qa_decode_attn(None, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "NULL" in qa.qa_last_error()
    # misaligned pointer
    odd = ctypes.c_void_p(0x1002)
    assert lib.qa_decode_attn(odd, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "aligned" in qa.qa_last_error()
    # prefill: negative total, window: n_kv != n_q, bad scale
    assert lib.qa_prefill_attn(fake, fake, fake, fake, 1, -1, fake, fake, fake, fake, ctypes.byref(p)) == -1
    w = qa.qa_attn_default_params()
    w.n_q_heads, w.n_kv_heads, w.head_dim = 14, 7, 64
    assert lib.qa_window_attn(fake, fake, fake, fake, 1, 1, fake, ctypes.byref(w)) == -1
    w.n_kv_heads, w.scale = 14, float("nan")
    assert lib.qa_window_attn(fake, fake, fake, fake, 1, 1, fake, ctypes.byref(w)) == -1
    assert "scale" in qa.qa_last_error()
    # window: an optional workspace must hold the job counter and be 4-byte aligned
    assert qa.qa_window_workspace_size() >= 8
    w.scale = 0.0
    w.workspace, w.workspace_bytes = fake, qa.qa_window_workspace_size() - 1
    assert lib.qa_window_attn(fake, fake, fake, fake, 1, 1, fake, ctypes.byref(w)) == -1
    assert "workspace" in qa.qa_last_error()
    w.workspace, w.workspace_bytes = odd, qa.qa_window_workspace_size()
    assert lib.qa_window_attn(fake, fake, fake, fake, 1, 1, fake, ctypes.byref(w)) == -1
    assert "workspace" in qa.qa_last_error()
    # decode append: eps and theta must be positive, pointers non-NULL, gains 8-byte aligned
    app = lib.qa_decode_append
    assert app(fake, fake, fake, fake, fake, 0.0, 1e6, fake, fake, 1, fake, fake, fake, ctypes.byref(p)) == -1
    assert "rms_eps" in qa.qa_last_error()
    assert app(fake, fake, fake, fake, fake, 1e-6, float("inf"), fake, fake, 1, fake, fake, fake, ctypes.byref(p)) == -1
    assert "rope_theta" in qa.qa_last_error()
    assert app(fake, fake, fake, None, fake, 1e-6, 1e6, fake, fake, 1, fake, fake, fake, ctypes.byref(p)) == -1
    assert "NULL" in qa.qa_last_error()
    assert app(fake, fake, fake, ctypes.c_void_p(0x1004), fake, 1e-6, 1e6, fake, fake, 1, fake, fake, fake,
               ctypes.byref(p)) == -1
    assert "aligned" in qa.qa_last_error()
    assert app(fake, fake, fake, fake, fake, 1e-6, 1e6, fake, fake, 0, fake, fake, fake, ctypes.byref(p)) == -1
    assert "batch" in qa.qa_last_error()
    big = qa.qa_attn_default_params()
    big.num_pages, big.max_pages_per_seq = 4, 20000  # positions up to 320000 > 2^18
    assert app(fake, fake, fake, fake, fake, 1e-6, 1e6, fake, fake, 1, fake, fake, fake, ctypes.byref(big)) == -1
    assert "positions" in qa.qa_last_error()
    # fused decode step: the append's checks, then the decode's
    stp = lib.qa_decode_step
    assert stp(fake, fake, fake, fake, fake, -1.0, 1e6, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "rms_eps" in qa.qa_last_error()
    assert stp(fake, fake, fake, ctypes.c_void_p(0x1008), fake, 1e-6, 1e6, fake, fake, fake, fake, 1, fake,
               ctypes.byref(p)) == -1
    assert "aligned" in qa.qa_last_error()
    # then the decode's own checks: no workspace (or, on a machine without a GPU, no device)
    assert stp(fake, fake, fake, fake, fake, 1e-6, 1e6, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) in (-1, -3)
    assert "workspace" in qa.qa_last_error() or "device" in qa.qa_last_error()


def test_graph_api_rejects_bad_arguments_without_device(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    lib = qa._lib
    p = qa.qa_attn_default_params()
    arr = (ctypes.c_void_p * 1)(0x1000)
    h = ctypes.c_void_p(0x1234)
    fake = ctypes.c_void_p(0x1000)
    assert lib.qa_decode_graph_create(0, arr, arr, arr, fake, fake, 1, arr, ctypes.byref(p), ctypes.byref(h)) == -1
    assert "n_layers" in qa.qa_last_error() and h.value is None
    p.debug_checks = 1
    assert lib.qa_prefill_graph_create(1, arr, arr, arr, fake, 1, 1, fake, arr, arr, arr, ctypes.byref(p),
                                       ctypes.byref(h)) == -1
    assert "debug_checks" in qa.qa_last_error()
    assert lib.qa_graph_launch(None, None) == -1
    lib.qa_graph_destroy(None)  # ignored


def test_window_plan_matches_oracle(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    rng = np.random.default_rng(7)
    for _ in range(50):
        counts = rng.integers(0, 1000, size=rng.integers(1, 12))
        np.testing.assert_array_equal(qa.qa_window_plan(counts), oracle.window_plan(counts))
        w = int(rng.integers(1, 200))
        np.testing.assert_array_equal(qa.qa_window_plan(counts, w), oracle.window_plan(counts, w))
    assert qa.qa_window_plan([117]).tolist() == [0, 104, 117]
    with pytest.raises(qa.QAError):
        qa.qa_window_plan([5, -1])


def test_window_plan_capacity_error(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    counts = np.array([300], np.int32)
    cu = np.zeros(2, np.int32)
    n = qa._lib.qa_window_plan(counts.ctypes.data_as(ctypes.c_void_p), 1, 0, cu.ctypes.data_as(ctypes.c_void_p), 2)
    assert n == -1 and "capacity" in qa.qa_last_error()


def test_stable_metadata_levels_are_checked(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    p = qa.qa_attn_default_params()
    fake = ctypes.c_void_p(0x1000)
    p.stable_metadata = 3
    assert qa._lib.qa_decode_attn(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "stable_metadata" in qa.qa_last_error()
    p.abi_version = 1  # ABI 1 callers have no such field: the value is ignored
    assert "stable_metadata" not in (qa._lib.qa_decode_attn(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(p)),
                                     qa.qa_last_error())[1]


def test_noalloc_decode_applies_the_decode_checks(libqa):
    # the no-alloc entry point takes the same argument checks as qa_decode_attn
    # (all of them run on the host, before any device is touched)
    import paged_kv_gqa_attention_gb300 as qa

    fn = qa._lib.qa_decode_attn_noalloc
    fake = ctypes.c_void_p(0x1000)
    p = qa.qa_attn_default_params()
    p.num_pages, p.max_pages_per_seq = 8, 2
    p.stable_metadata = 3
    assert fn(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "stable_metadata 3 outside [0, 2]" in qa.qa_last_error()
    p.stable_metadata = 0
    p.abi_version = qa.QA_ABI_VERSION + 1
    assert fn(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "abi_version" in qa.qa_last_error()
    p.abi_version = qa.QA_ABI_VERSION
    assert fn(fake, fake, fake, fake, fake, 0, fake, ctypes.byref(p)) == -1
    assert "batch 0" in qa.qa_last_error()
    assert fn(ctypes.c_void_p(0x1008), fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "aligned" in qa.qa_last_error()
    p.head_dim = 64
    assert fn(fake, fake, fake, fake, fake, 1, fake, ctypes.byref(p)) == -1
    assert "head_dim" in qa.qa_last_error()


def test_python_abi_version_matches_the_header(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    src = open(HEADER).read()
    m = re.search(r"#define\s+QA_ABI_VERSION\s+(\d+)", src)
    assert m and qa.QA_ABI_VERSION == int(m.group(1)) == qa.qa_attn_default_params().abi_version


def test_bounded_wait_check_rejects_bad_limits_without_device(libqa):
    import paged_kv_gqa_attention_gb300 as qa

    for limit in (0, 1000001):
        assert qa._lib.qa_check_bounded_wait(limit, None) == -1
        assert "limit_us" in qa.qa_last_error()
