"""Reference oracle for paged GQA attention -- TEST INFRASTRUCTURE ONLY.

Plain fp64 CPU statement of what the attention hot path computes, used to
check the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import it; the library itself never
does, and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain loops, bf16 widened exactly to
double, no intermediate rounding).  This module compiles it with gcc, wraps it
with ctypes, and adds the two pieces of host logic the pages define in integer
arithmetic:

* ``after_cnn_len`` -- the token count of one conv-stem chunk, the three
  stride-2 convolutions applied in turn (qwenasr.cpp ARCHITECTURE.md,
  "Conv2d subsampling stem");
* ``window_plan`` -- cutting each request's encoder tokens into consecutive
  windows of ``window_aftercnn = conv_out(chunk_mel) * window_chunks`` tokens
  (13 * 8 = 104 by default), the last one partial (same page, "Windowed audio
  tower"; GGUF keys n_window 50 and n_window_infer 800 in "GGUF layout").

The encoder layer around the window attention (``layer_norm``, ``linear``,
``encoder_layer``: the pre-norm AuT layer of "Windowed audio tower", bf16 at
every operator boundary) is in the same C file.

Parity status: every function here is pinned: the attention functions by
``tests/test_oracle_pins.py`` (brute force, torch float64 SDPA, mpmath,
closed forms, invariants, printed values under ``tests/golden/``), QK-norm,
RoPE and the decode append by ``tests/test_oracle_rope_pins.py`` (torch
float64 ``rms_norm``, closed-form rotations, rotation invariants, a numpy
scatter of the append), the encoder layer by
``tests/test_oracle_encoder_pins.py`` (torch float64 ``layer_norm`` and
``gelu``, numpy products, closed forms, a numpy statement of the layer with an
explicit block-diagonal mask, window locality, planted mistakes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# GGUF metadata of the audio tower (qwenasr.cpp ARCHITECTURE.md, "GGUF layout").
N_WINDOW = 50  # chunk_mel = n_window * 2 = 100 mel frames
N_WINDOW_INFER = 800  # window_chunks = n_window_infer / chunk_mel = 8


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` from ``oracle.c`` with gcc (plain C, -O2)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fvisibility=hidden",
                   "-D_POSIX_C_SOURCE=200809L", "-o", tmp, _SRC, "-lm", "-lpthread"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def bind_library(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P, I, Dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.oracle_attend_row.argtypes = [P, P, P, I, I, Dbl, P, P]
    lib.oracle_attend_row.restype = None
    lib.oracle_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, Dbl, P, I, P, I]
    lib.oracle_decode.restype = I
    lib.oracle_prefill.argtypes = [P, P, P, P, I, I, I, I, I, Dbl, P, I, P, I]
    lib.oracle_prefill.restype = I
    lib.oracle_page_write.argtypes = [P, P, P, I, P, I, I, I, I, I, P, P]
    lib.oracle_page_write.restype = I
    lib.oracle_window.argtypes = [P, P, P, P, I, I, I, I, Dbl, P, I, P, I]
    lib.oracle_window.restype = I
    lib.oracle_prefill_chunk.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, P, I, I, I, Dbl, P, I, P, I]
    lib.oracle_prefill_chunk.restype = I
    lib.oracle_page_write_at.argtypes = [P, P, P, P, I, P, I, I, I, I, I, P, P]
    lib.oracle_page_write_at.restype = I
    lib.oracle_qk_norm_rope.argtypes = [P, I, I, I, P, P, Dbl, Dbl, P]
    lib.oracle_qk_norm_rope.restype = I
    lib.oracle_decode_append.argtypes = [P, P, P, P, P, Dbl, Dbl, P, P, I, I, I, I, I, I, I, P, P, P, P, P]
    lib.oracle_decode_append.restype = I
    lib.oracle_layer_norm.argtypes = [P, I, I, P, P, Dbl, P, I]
    lib.oracle_layer_norm.restype = I
    lib.oracle_linear.argtypes = [P, I, I, P, I, P, I, P, P, I]
    lib.oracle_linear.restype = I
    lib.oracle_encoder_layer.argtypes = [P, P, I, I, I, I, I] + [P] * 12 + [Dbl, I, P, I]
    lib.oracle_encoder_layer.restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = bind_library(_LIB)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 data must be passed as its uint16 bit pattern, got {a.dtype}")
    return a


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def attend_row(q, K, V, scale):
    """softmax(scale * q.K^T) V for one row; returns (out, p) in float64."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    n, D = K.shape
    out = np.zeros(D, np.float64)
    p = np.zeros(max(n, 1), np.float64)
    _load().oracle_attend_row(_ptr(q), _ptr(K), _ptr(V), n, D, float(scale), _ptr(out), _ptr(p))
    return out, p[:n]


def decode(q, k_pages, v_pages, page_table, seq_lens, *, scale=None, rows=None, n_threads=0):
    """Paged GQA decode.  q [B,Hq,D], pools [P,page_size,Hkv,D] (bf16 bits as
    uint16), page_table [B,max_pages] int32, seq_lens [B] int32.  Returns
    float64 [B,Hq,D], or [len(rows),D] for rows = flat b*Hq+h indices."""
    q, k_pages, v_pages = _u16(q), _u16(k_pages), _u16(v_pages)
    page_table, seq_lens = _i32(page_table), _i32(seq_lens)
    B, Hq, D = q.shape
    P, PS, Hkv, D2 = k_pages.shape
    assert D2 == D and v_pages.shape == k_pages.shape and page_table.shape[0] == B
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    rows_a = None if rows is None else _i32(rows)
    n = B * Hq if rows_a is None else len(rows_a)
    out = np.zeros((n, D), np.float64)
    rc = _load().oracle_decode(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                               _ptr(seq_lens), B, Hq, Hkv, D, PS, page_table.shape[1], P,
                               float(scale), _ptr(rows_a), n, _ptr(out), _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out.reshape(B, Hq, D) if rows_a is None else out


def prefill(q, k, v, cu_seqlens, *, scale=None, rows=None, n_threads=0):
    """Packed causal GQA prefill.  q [T,Hq,D], k/v [T,Hkv,D], cu_seqlens [B+1].
    Returns float64 [T,Hq,D], or [len(rows),D] for rows = flat t*Hq+h."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu = _i32(cu_seqlens)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    rows_a = None if rows is None else _i32(rows)
    n = T * Hq if rows_a is None else len(rows_a)
    out = np.zeros((n, D), np.float64)
    rc = _load().oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, T, Hq, Hkv,
                                D, float(scale), _ptr(rows_a), n, _ptr(out), _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_prefill rejected its arguments")
    return out.reshape(T, Hq, D) if rows_a is None else out


def page_write(k, v, cu_seqlens, page_table, k_pages, v_pages):
    """Bit copy of packed K/V rows into their pages; returns new pool arrays."""
    k, v = _u16(k), _u16(v)
    kp, vp = _u16(k_pages).copy(), _u16(v_pages).copy()
    cu, pt = _i32(cu_seqlens), _i32(page_table)
    P, PS, Hkv, D = kp.shape
    rc = _load().oracle_page_write(_ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, _ptr(pt),
                                   pt.shape[1], PS, P, Hkv, D, _ptr(kp), _ptr(vp))
    if rc != 0:
        raise ValueError("oracle_page_write rejected its arguments")
    return kp, vp


def prefill_chunk(q, k, v, cu_seqlens, n_past, page_table, k_pages, v_pages, *, scale=None, rows=None,
                  n_threads=0):
    """Chunked causal GQA prefill: request r has n_past[r] cached positions in
    the pools [P,page_size,Hkv,D]; its packed new rows attend over those and
    over new rows j <= i.  Returns float64 [T,Hq,D], or [len(rows),D] for
    rows = flat t*Hq+h."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    kp, vp = _u16(k_pages), _u16(v_pages)
    cu, npast, pt = _i32(cu_seqlens), _i32(n_past), _i32(page_table)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    P, PS, Hkv2, D2 = kp.shape
    assert Hkv2 == Hkv and D2 == D and npast.shape == (len(cu) - 1,)
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    rows_a = None if rows is None else _i32(rows)
    n = T * Hq if rows_a is None else len(rows_a)
    out = np.zeros((n, D), np.float64)
    rc = _load().oracle_prefill_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), _ptr(npast), len(cu) - 1, T, Hq, Hkv, D,
                                      _ptr(kp), _ptr(vp), _ptr(pt), pt.shape[1], PS, P, float(scale), _ptr(rows_a), n,
                                      _ptr(out), _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_prefill_chunk rejected its arguments")
    return out.reshape(T, Hq, D) if rows_a is None else out


def page_write_at(k, v, cu_seqlens, n_past, page_table, k_pages, v_pages):
    """Bit copy of the new rows to positions n_past[r] + i of their pages;
    returns new pool arrays."""
    k, v = _u16(k), _u16(v)
    kp, vp = _u16(k_pages).copy(), _u16(v_pages).copy()
    cu, npast, pt = _i32(cu_seqlens), _i32(n_past), _i32(page_table)
    P, PS, Hkv, D = kp.shape
    rc = _load().oracle_page_write_at(_ptr(k), _ptr(v), _ptr(cu), _ptr(npast), len(cu) - 1, _ptr(pt), pt.shape[1],
                                      PS, P, Hkv, D, _ptr(kp), _ptr(vp))
    if rc != 0:
        raise ValueError("oracle_page_write_at rejected its arguments")
    return kp, vp


def window(q, k, v, cu_windows, *, scale=None, rows=None, n_threads=0):
    """Packed bidirectional window attention.  q/k/v [T,H,D], cu_windows [W+1].
    Returns float64 [T,H,D], or [len(rows),D] for rows = flat t*H+h."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu = _i32(cu_windows)
    T, H, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    rows_a = None if rows is None else _i32(rows)
    n = T * H if rows_a is None else len(rows_a)
    out = np.zeros((n, D), np.float64)
    rc = _load().oracle_window(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, T, H, D,
                               float(scale), _ptr(rows_a), n, _ptr(out), _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_window rejected its arguments")
    return out.reshape(T, H, D) if rows_a is None else out


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def qk_norm_rope(x, pos, gain, *, eps, theta):
    """Per-head RMSNorm (gain [D] float32) then NEOX RoPE at pos[t] for every
    head of row t.  x [T,H,D] bf16 bits.  Returns float64 [T,H,D]."""
    x, pos, gain = _u16(x), _i32(pos), _f32(gain)
    T, H, D = x.shape
    assert pos.shape == (T,) and gain.shape == (D,)
    out = np.zeros((T, H, D), np.float64)
    rc = _load().oracle_qk_norm_rope(_ptr(x), T, H, D, _ptr(pos), _ptr(gain), float(eps), float(theta), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_qk_norm_rope rejected its arguments")
    return out


def decode_append(q, k, v, q_gain, k_gain, page_table, seq_lens, k_pages, v_pages, *, eps, theta):
    """Decode KV append: QK-norm + NEOX RoPE of the new token (position
    seq_lens[b] - 1), its K/V written into the pools.  Returns a dict with
    q_rot/k_rot (float64, before rounding), q (bf16 bits, rounded) and the new
    k_pages/v_pages arrays."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    q_gain, k_gain = _f32(q_gain), _f32(k_gain)
    page_table, seq_lens = _i32(page_table), _i32(seq_lens)
    kp, vp = _u16(k_pages).copy(), _u16(v_pages).copy()
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    P, PS, Hkv2, D2 = kp.shape
    assert Hkv2 == Hkv and D2 == D and v.shape == k.shape and page_table.shape[0] == B
    q_rot = np.zeros((B, Hq, D), np.float64)
    k_rot = np.zeros((B, Hkv, D), np.float64)
    q_bf16 = np.zeros((B, Hq, D), np.uint16)
    rc = _load().oracle_decode_append(_ptr(q), _ptr(k), _ptr(v), _ptr(q_gain), _ptr(k_gain), float(eps),
                                      float(theta), _ptr(page_table), _ptr(seq_lens), B, Hq, Hkv, D, PS,
                                      page_table.shape[1], P, _ptr(q_rot), _ptr(k_rot), _ptr(q_bf16), _ptr(kp),
                                      _ptr(vp))
    if rc != 0:
        raise ValueError("oracle_decode_append rejected its arguments")
    return dict(q_rot=q_rot, k_rot=k_rot, q=q_bf16, k_pages=kp, v_pages=vp)


def after_cnn_len(mel_len: int) -> int:
    """Tokens out of one conv-stem chunk of mel_len frames: three convolutions
    of kernel 3, stride 2, padding 1, applied in turn."""
    n = mel_len
    for _ in range(3):
        n = (n - 1) // 2 + 1
    return n


def window_tokens(n_window: int = N_WINDOW, n_window_infer: int = N_WINDOW_INFER) -> int:
    """window_aftercnn = conv_out(chunk_mel) * window_chunks."""
    chunk_mel = n_window * 2
    window_chunks = n_window_infer // chunk_mel
    return after_cnn_len(chunk_mel) * window_chunks


def window_plan(token_counts, window: int | None = None) -> np.ndarray:
    """cu_windows for packed requests: each request's tokens are cut into
    consecutive windows of ``window`` tokens from its own start, the last one
    partial; a request shorter than a window is one window; a request with no
    token contributes no window."""
    w = window_tokens() if window is None else int(window)
    cu = [0]
    for n in token_counts:
        n = int(n)
        start = 0
        while start < n:
            take = min(w, n - start)
            cu.append(cu[-1] + take)
            start += take
    return np.asarray(cu, dtype=np.int32)


def layer_norm(x, gamma, beta, *, eps, n_threads=0):
    """LayerNorm over the last axis of x [T, d] with gain and bias [d] (all
    bf16 bits).  Returns float64 [T, d]."""
    x, gamma, beta = _u16(x), _u16(gamma), _u16(beta)
    T, d = x.shape
    assert gamma.shape == (d,) and beta.shape == (d,)
    y = np.zeros((T, d), np.float64)
    rc = _load().oracle_layer_norm(_ptr(x), T, d, _ptr(gamma), _ptr(beta), float(eps), _ptr(y), _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_layer_norm rejected its arguments")
    return y


def linear(x, w, bias=None, *, gelu=False, residual=None, n_threads=0):
    """act(x W^T + bias) + residual: x [T, K], w [N, K] (PyTorch Linear
    layout), bias [N], residual [T, N], all bf16 bits; act = exact gelu when
    gelu.  Returns float64 [T, N]."""
    x, w = _u16(x), _u16(w)
    T, K = x.shape
    N, K2 = w.shape
    assert K2 == K
    bias = None if bias is None else _u16(bias)
    residual = None if residual is None else _u16(residual)
    assert bias is None or bias.shape == (N,)
    assert residual is None or residual.shape == (T, N)
    y = np.zeros((T, N), np.float64)
    rc = _load().oracle_linear(_ptr(x), T, K, _ptr(w), N, _ptr(bias), 1 if gelu else 0, _ptr(residual), _ptr(y),
                               _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_linear rejected its arguments")
    return y


ENCODER_WEIGHTS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_fc1", "b_fc1", "w_fc2",
                   "b_fc2")


def encoder_layer(x, cu_windows, weights, *, n_heads, eps, blocks=2, n_threads=0):
    """One AuT encoder layer (pre-norm; bf16 at every operator boundary) over
    packed tokens x [T, d] (bf16 bits) cut into windows cu_windows.
    weights: dict of bf16 arrays named as in ENCODER_WEIGHTS (w_qkv [3d, d],
    w_o [d, d], w_fc1 [ffn, d], w_fc2 [d, ffn]).  blocks=1 stops after the
    attention block.  Returns float64 [T, d] (the last operator unrounded)."""
    x = _u16(x)
    T, d = x.shape
    cu = _i32(cu_windows)
    ws = [_u16(weights[k]) for k in ENCODER_WEIGHTS]
    d_ffn = ws[ENCODER_WEIGHTS.index("w_fc1")].shape[0]
    assert ws[2].shape == (3 * d, d) and ws[4].shape == (d, d) and ws[8].shape == (d_ffn, d)
    assert ws[10].shape == (d, d_ffn)
    y = np.zeros((T, d), np.float64)
    rc = _load().oracle_encoder_layer(_ptr(x), _ptr(cu), len(cu) - 1, T, d, int(n_heads), d_ffn,
                                      *[_ptr(a) for a in ws], float(eps), int(blocks), _ptr(y), _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_encoder_layer rejected its arguments")
    return y
