"""Python binding of libqa, the GB300 paged GQA attention library.

Thin argument marshalling over the C ABI declared in ``include/qa.h``: each
function takes torch CUDA tensors, checks dtype / device / contiguity, and
passes raw pointers, sizes and the current CUDA stream to the ``qa_*`` entry
point of the same name.  Every step of the computation runs in the library's
CUDA kernels; there is no other implementation behind these names, and
importing this package fails loudly when ``libqa.so`` has not been built.

    qa_decode_attn    paged GQA decode (split-K flash decode + combine)
    qa_prefill_attn   ragged causal prefill with the KV page write
    qa_window_attn    windowed bidirectional encoder attention
    qa_window_plan    cu_windows from per-request encoder token counts (host)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "QA_ABI_VERSION", "QAError", "lib_path", "qa_version", "qa_last_error", "qa_attn_default_params",
    "qa_decode_workspace_size", "qa_decode_attn", "qa_prefill_attn", "qa_window_attn", "qa_window_plan",
    "qa_window_workspace_size",
    "qa_device_status", "DEVICE_STATUS_BITS", "qa_decode_attn_noalloc", "qa_check_bounded_wait",
    "qa_encoder_workspace_size", "qa_encoder_layer", "qa_linear", "qa_layer_norm", "ENCODER_WEIGHT_NAMES",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libqa.so")

DEVICE_STATUS_BITS = {0x1: "bad page id", 0x2: "bad length", 0x4: "bad segments", 0x8: "timeout"}


class QAError(RuntimeError):
    """A qa_* call returned a non-zero status."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed with status {status}: {message}")
        self.status = status


class qa_attn_params(ctypes.Structure):
    _fields_ = [
        ("abi_version", ctypes.c_int),
        ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("max_pages_per_seq", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("stream", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("debug_checks", ctypes.c_int),
        ("stable_metadata", ctypes.c_int),
    ]


ENCODER_WEIGHT_NAMES = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_fc1", "b_fc1",
                        "w_fc2", "b_fc2")


class qa_encoder_weights(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in ENCODER_WEIGHT_NAMES]


def _load():
    if not os.path.exists(lib_path):
        raise ImportError(
            f"libqa.so is not built ({lib_path}); run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(lib_path)
    P, I, PP = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(qa_attn_params)
    lib.qa_attn_default_params.restype = qa_attn_params
    lib.qa_attn_default_params.argtypes = []
    lib.qa_decode_workspace_size.restype = ctypes.c_size_t
    lib.qa_decode_workspace_size.argtypes = [I, I, PP]
    lib.qa_window_workspace_size.restype = ctypes.c_size_t
    lib.qa_window_workspace_size.argtypes = []
    lib.qa_decode_attn.restype = I
    lib.qa_decode_attn.argtypes = [P, P, P, P, P, I, P, PP]
    lib.qa_decode_attn_noalloc.restype = I
    lib.qa_decode_attn_noalloc.argtypes = [P, P, P, P, P, I, P, PP]
    lib.qa_prefill_attn.restype = I
    lib.qa_prefill_attn.argtypes = [P, P, P, P, I, I, P, P, P, P, PP]
    lib.qa_decode_append.restype = I
    lib.qa_decode_append.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, P, P, I, P, P, P, PP]
    lib.qa_decode_step.restype = I
    lib.qa_decode_step.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, P, P, P, P, I, P, PP]
    PA = ctypes.POINTER(ctypes.c_void_p)
    lib.qa_decode_graph_create.restype = I
    lib.qa_decode_graph_create.argtypes = [I, PA, PA, PA, P, P, I, PA, PP, ctypes.POINTER(ctypes.c_void_p)]
    lib.qa_prefill_graph_create.restype = I
    lib.qa_prefill_graph_create.argtypes = [I, PA, PA, PA, P, I, I, P, PA, PA, PA, PP, ctypes.POINTER(ctypes.c_void_p)]
    lib.qa_graph_launch.restype = I
    lib.qa_graph_launch.argtypes = [P, P]
    lib.qa_graph_destroy.restype = None
    lib.qa_graph_destroy.argtypes = [P]
    lib.qa_prefill_chunk_attn.restype = I
    lib.qa_prefill_chunk_attn.argtypes = [P, P, P, P, P, I, I, P, P, P, P, PP]
    lib.qa_window_attn.restype = I
    lib.qa_window_attn.argtypes = [P, P, P, P, I, I, P, PP]
    lib.qa_window_plan.restype = I
    lib.qa_window_plan.argtypes = [P, I, I, P, I]
    lib.qa_encoder_workspace_size.restype = ctypes.c_size_t
    lib.qa_encoder_workspace_size.argtypes = [I, I, I]
    lib.qa_encoder_layer.restype = I
    lib.qa_encoder_layer.argtypes = [P, P, I, I, I, I, I, ctypes.POINTER(qa_encoder_weights), ctypes.c_float, P, PP]
    lib.qa_linear.restype = I
    lib.qa_linear.argtypes = [P, I, I, P, I, P, I, P, P, PP]
    lib.qa_layer_norm.restype = I
    lib.qa_layer_norm.argtypes = [P, I, I, P, P, ctypes.c_float, P, PP]
    lib.qa_device_status.restype = I
    lib.qa_device_status.argtypes = [P]
    lib.qa_check_bounded_wait.restype = I
    lib.qa_check_bounded_wait.argtypes = [ctypes.c_uint, P]
    lib.qa_last_error.restype = ctypes.c_char_p
    lib.qa_last_error.argtypes = []
    lib.qa_version.restype = ctypes.c_char_p
    lib.qa_version.argtypes = []
    return lib


_lib = _load()

# The library's ABI version (include/qa.h QA_ABI_VERSION), read from the
# library's own defaults so the two cannot disagree.
QA_ABI_VERSION = int(_lib.qa_attn_default_params().abi_version)


def qa_version() -> str:
    return _lib.qa_version().decode()


def qa_last_error() -> str:
    return _lib.qa_last_error().decode()


def _check(fn: str, status: int):
    if status != 0:
        raise QAError(fn, status, qa_last_error())


def _torch():
    import torch

    return torch


def _stream_ptr(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name, dtype=None, ndim=None, allow_host=False):
    """Device address of a tensor.  allow_host: a page-locked CPU tensor is
    accepted too (the decode's q, page table, lengths and output may live in
    host memory the device addresses directly; see qa.h)."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or (allow_host and t.is_pinned())):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or page-locked host memory" if allow_host else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def qa_attn_default_params() -> qa_attn_params:
    return _lib.qa_attn_default_params()


def _params(*, n_q_heads, n_kv_heads, head_dim, page_size=16, num_pages=0, max_pages_per_seq=0, scale=0.0,
            stream=None, workspace=None, debug_checks=False, stable_metadata=False):
    p = _lib.qa_attn_default_params()
    p.n_q_heads, p.n_kv_heads, p.head_dim = n_q_heads, n_kv_heads, head_dim
    p.page_size, p.num_pages, p.max_pages_per_seq = page_size, num_pages, max_pages_per_seq
    p.scale = float(scale)
    p.stream = _stream_ptr(stream)
    if workspace is not None:
        p.workspace = _dev(workspace, "workspace")
        p.workspace_bytes = workspace.numel() * workspace.element_size()
    p.debug_checks = 1 if debug_checks else 0
    p.stable_metadata = int(stable_metadata)  # False/True/2 -> 0/1/2
    return p


def qa_decode_workspace_size(batch: int, max_seq_len: int, *, n_q_heads=16, n_kv_heads=8, head_dim=128,
                             page_size=16, num_pages=1, max_pages_per_seq=1) -> int:
    """Bytes of decode workspace for `batch` requests on the current device."""
    p = _lib.qa_attn_default_params()
    p.n_q_heads, p.n_kv_heads, p.head_dim = n_q_heads, n_kv_heads, head_dim
    p.page_size, p.num_pages, p.max_pages_per_seq = page_size, num_pages, max_pages_per_seq
    n = _lib.qa_decode_workspace_size(int(batch), int(max_seq_len), ctypes.byref(p))
    if n == 0:
        raise QAError("qa_decode_workspace_size", -1, qa_last_error())
    return int(n)


def qa_decode_attn(q, k_pages, v_pages, page_table, seq_lens, out=None, *, workspace=None, scale=0.0,
                   stream=None, debug_checks=False, stable_metadata=False):
    """Paged GQA decode.  q bf16 [B,Hq,D]; pools bf16 [P,16,Hkv,D];
    page_table int32 [B,max_pages]; seq_lens int32 [B].  Returns out bf16
    [B,Hq,D].  q, page_table, seq_lens and out may be page-locked CPU
    tensors (the kernel reads and writes them over the host link; pass
    `out` then).  `workspace` is a zero-filled device byte tensor of at least
    qa_decode_workspace_size(B, ...) bytes (allocated here if omitted); the
    call leaves its arrival counters at zero, so it can be reused across
    calls without clearing.
    stable_metadata=True (1): the caller promises that page_table and
    seq_lens are not written by the kernel just before this call on the
    stream; 2: the same of the pools as well (see
    qa_attn_params::stable_metadata in qa.h)."""
    torch = _torch()
    B, Hq, D = q.shape
    P, PS, Hkv, D2 = k_pages.shape
    if D2 != D or tuple(v_pages.shape) != tuple(k_pages.shape) or page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = qa_decode_workspace_size(B, 0, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS,
                                          num_pages=P, max_pages_per_seq=page_table.shape[1])
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], scale=scale, stream=stream, workspace=workspace,
                debug_checks=debug_checks, stable_metadata=stable_metadata)
    st = _lib.qa_decode_attn(_dev(q, "q", torch.bfloat16, 3, True), _dev(k_pages, "k_pages", torch.bfloat16, 4),
                             _dev(v_pages, "v_pages", torch.bfloat16, 4),
                             _dev(page_table, "page_table", torch.int32, 2, True),
                             _dev(seq_lens, "seq_lens", torch.int32, 1, True), B,
                             _dev(out, "out", torch.bfloat16, 3, True), ctypes.byref(p))
    _check("qa_decode_attn", st)
    return out


def qa_decode_attn_noalloc(q, k_pages, v_pages, page_table, seq_lens, out=None, *, scale=0.0, stream=None,
                           debug_checks=False, stable_metadata=False):
    """qa_decode_attn without a workspace, for callers that cannot allocate
    device memory: the split-K scratch is a fixed 4 MiB array inside the
    library, shared by every call on the device (calls that overlap on the
    GPU race on it; calls ordered on one stream are fine).  Batches whose
    scratch would not fit are rejected.  With out=None the output tensor is allocated here by torch; pass `out` to keep
    the call allocation-free."""
    torch = _torch()
    B, Hq, D = q.shape
    P, PS, Hkv, D2 = k_pages.shape
    if D2 != D or tuple(v_pages.shape) != tuple(k_pages.shape) or page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    if out is None:
        out = torch.empty_like(q)
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], scale=scale, stream=stream, debug_checks=debug_checks,
                stable_metadata=stable_metadata)
    st = _lib.qa_decode_attn_noalloc(_dev(q, "q", torch.bfloat16, 3), _dev(k_pages, "k_pages", torch.bfloat16, 4),
                                     _dev(v_pages, "v_pages", torch.bfloat16, 4),
                                     _dev(page_table, "page_table", torch.int32, 2),
                                     _dev(seq_lens, "seq_lens", torch.int32, 1), B,
                                     _dev(out, "out", torch.bfloat16, 3), ctypes.byref(p))
    _check("qa_decode_attn_noalloc", st)
    return out


def qa_prefill_attn(q, k, v, cu_seqlens, page_table, k_pages, v_pages, out=None, *, scale=0.0, stream=None,
                    debug_checks=False, stable_metadata=False):
    """Ragged causal prefill with the KV page write.  q bf16 [T,Hq,D]; k/v
    bf16 [T,Hkv,D]; cu_seqlens int32 [B+1]; page_table int32 [B,max_pages];
    pools bf16 [P,16,Hkv,D] (written in place).  Returns out bf16 [T,Hq,D]."""
    torch = _torch()
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.shape[0] - 1
    P, PS = k_pages.shape[0], k_pages.shape[1]
    if out is None:
        out = torch.empty_like(q)
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], scale=scale, stream=stream, debug_checks=debug_checks,
                stable_metadata=stable_metadata)
    st = _lib.qa_prefill_attn(_dev(q, "q", torch.bfloat16, 3), _dev(k, "k", torch.bfloat16, 3),
                              _dev(v, "v", torch.bfloat16, 3), _dev(cu_seqlens, "cu_seqlens", torch.int32, 1), B, T,
                              _dev(page_table, "page_table", torch.int32, 2), _dev(k_pages, "k_pages", torch.bfloat16, 4),
                              _dev(v_pages, "v_pages", torch.bfloat16, 4), _dev(out, "out", torch.bfloat16, 3),
                              ctypes.byref(p))
    _check("qa_prefill_attn", st)
    return out


def qa_prefill_chunk_attn(q, k, v, cu_seqlens, n_past, page_table, k_pages, v_pages, out=None, *, scale=0.0,
                          stream=None, debug_checks=False, stable_metadata=False):
    """Chunked prefill: request r holds n_past[r] (int32 [B], device) cached
    positions in its pages; its packed new rows attend over those and over
    new rows j <= i, and are written to positions n_past[r] + i.  Shapes as
    for qa_prefill_attn.  Returns out bf16 [T,Hq,D]."""
    torch = _torch()
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.shape[0] - 1
    P, PS = k_pages.shape[0], k_pages.shape[1]
    if tuple(n_past.shape) != (B,):
        raise ValueError("n_past must be [batch]")
    if out is None:
        out = torch.empty_like(q)
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], scale=scale, stream=stream, debug_checks=debug_checks,
                stable_metadata=stable_metadata)
    st = _lib.qa_prefill_chunk_attn(_dev(q, "q", torch.bfloat16, 3), _dev(k, "k", torch.bfloat16, 3),
                                    _dev(v, "v", torch.bfloat16, 3), _dev(cu_seqlens, "cu_seqlens", torch.int32, 1),
                                    _dev(n_past, "n_past", torch.int32, 1), B, T,
                                    _dev(page_table, "page_table", torch.int32, 2),
                                    _dev(k_pages, "k_pages", torch.bfloat16, 4), _dev(v_pages, "v_pages", torch.bfloat16, 4),
                                    _dev(out, "out", torch.bfloat16, 3), ctypes.byref(p))
    _check("qa_prefill_chunk_attn", st)
    return out


def qa_decode_append(q, k, v, q_gain, k_gain, page_table, seq_lens, k_pages, v_pages, q_out=None, *,
                     rms_eps=1e-6, rope_theta=1e6, stream=None, debug_checks=False):
    """Decode KV append: per-head RMSNorm (gains float32 [D]) and NEOX RoPE
    of the new token at position seq_lens[b] - 1, its K/V written into the
    pools.  q bf16 [B,Hq,D]; k/v bf16 [B,Hkv,D]; page_table int32
    [B,max_pages]; seq_lens int32 [B]; pools bf16 [P,16,Hkv,D] (written in
    place).  Returns q_out bf16 [B,Hq,D], the rotated query (q_out=q is
    allowed: in place)."""
    torch = _torch()
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    P, PS = k_pages.shape[0], k_pages.shape[1]
    if tuple(k.shape) != (B, Hkv, D) or tuple(v.shape) != (B, Hkv, D) or page_table.shape[0] != B:
        raise ValueError("inconsistent append shapes")
    if tuple(q_gain.shape) != (D,) or tuple(k_gain.shape) != (D,):
        raise ValueError("gains must be [head_dim]")
    if q_out is None:
        q_out = torch.empty_like(q)
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], stream=stream, debug_checks=debug_checks)
    st = _lib.qa_decode_append(_dev(q, "q", torch.bfloat16, 3), _dev(k, "k", torch.bfloat16, 3),
                               _dev(v, "v", torch.bfloat16, 3), _dev(q_gain, "q_gain", torch.float32, 1),
                               _dev(k_gain, "k_gain", torch.float32, 1), float(rms_eps), float(rope_theta),
                               _dev(page_table, "page_table", torch.int32, 2), _dev(seq_lens, "seq_lens", torch.int32, 1),
                               B, _dev(k_pages, "k_pages", torch.bfloat16, 4), _dev(v_pages, "v_pages", torch.bfloat16, 4),
                               _dev(q_out, "q_out", torch.bfloat16, 3), ctypes.byref(p))
    _check("qa_decode_append", st)
    return q_out


def qa_decode_step(q, k, v, q_gain, k_gain, page_table, seq_lens, k_pages, v_pages, out=None, *, workspace=None,
                   rms_eps=1e-6, rope_theta=1e6, scale=0.0, stream=None, debug_checks=False, stable_metadata=False):
    """The fused decode step: qa_decode_append (QK-norm + NEOX RoPE of the
    new token at seq_lens[b] - 1, its K/V written into the pools) and
    qa_decode_attn on the rotated query, in one launch.  q pre-norm bf16
    [B,Hq,D]; k/v bf16 [B,Hkv,D]; gains float32 [D]; workspace as for
    qa_decode_attn.  Returns out bf16 [B,Hq,D]."""
    torch = _torch()
    B, Hq, D = q.shape
    P, PS, Hkv, D2 = k_pages.shape
    if (D2 != D or tuple(v_pages.shape) != tuple(k_pages.shape) or page_table.dim() != 2 or page_table.shape[0] != B
            or tuple(k.shape) != (B, Hkv, D) or tuple(v.shape) != (B, Hkv, D)):
        raise ValueError("inconsistent decode-step shapes")
    if tuple(q_gain.shape) != (D,) or tuple(k_gain.shape) != (D,):
        raise ValueError("gains must be [head_dim]")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = qa_decode_workspace_size(B, 0, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS,
                                          num_pages=P, max_pages_per_seq=page_table.shape[1])
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], scale=scale, stream=stream, workspace=workspace,
                debug_checks=debug_checks, stable_metadata=stable_metadata)
    st = _lib.qa_decode_step(_dev(q, "q", torch.bfloat16, 3), _dev(k, "k", torch.bfloat16, 3),
                             _dev(v, "v", torch.bfloat16, 3), _dev(q_gain, "q_gain", torch.float32, 1),
                             _dev(k_gain, "k_gain", torch.float32, 1), float(rms_eps), float(rope_theta),
                             _dev(k_pages, "k_pages", torch.bfloat16, 4), _dev(v_pages, "v_pages", torch.bfloat16, 4),
                             _dev(page_table, "page_table", torch.int32, 2), _dev(seq_lens, "seq_lens", torch.int32, 1),
                             B, _dev(out, "out", torch.bfloat16, 3), ctypes.byref(p))
    _check("qa_decode_step", st)
    return out


class QAGraph:
    """A captured step (qa_decode_graph_create / qa_prefill_graph_create).
    Holds the tensors it was captured with, so their storage stays alive;
    launch() replays it, reading the tensors' current contents."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep

    def launch(self, stream=None):
        _check("qa_graph_launch", _lib.qa_graph_launch(self._h, _stream_ptr(stream)))

    def close(self):
        if self._h:
            _lib.qa_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _ptr_array(ts, name, dtype, ndim, allow_host=False):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _dev(t, f"{name}[{i}]", dtype, ndim, allow_host).value
    return arr


def qa_decode_graph_create(qs, k_pages, v_pages, page_table, seq_lens, outs, *, workspace, scale=0.0,
                           stable_metadata=False):
    """Captures one decode step: layer i runs qa_decode_attn(qs[i],
    k_pages[i], v_pages[i], page_table, seq_lens, outs[i]) with the shared
    workspace.  stable_metadata as for qa_decode_attn (no layer writes the
    page table or the lengths).  Returns a QAGraph."""
    torch = _torch()
    n = len(qs)
    if not (len(k_pages) == len(v_pages) == len(outs) == n):
        raise ValueError("per-layer lists must have the same length")
    B, Hq, D = qs[0].shape
    P, PS, Hkv, _ = k_pages[0].shape
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], scale=scale, workspace=workspace,
                stable_metadata=stable_metadata)
    h = ctypes.c_void_p()
    st = _lib.qa_decode_graph_create(n, _ptr_array(qs, "q", torch.bfloat16, 3, True),
                                     _ptr_array(k_pages, "k_pages", torch.bfloat16, 4),
                                     _ptr_array(v_pages, "v_pages", torch.bfloat16, 4),
                                     _dev(page_table, "page_table", torch.int32, 2, True),
                                     _dev(seq_lens, "seq_lens", torch.int32, 1, True), B,
                                     _ptr_array(outs, "out", torch.bfloat16, 3, True), ctypes.byref(p),
                                     ctypes.byref(h))
    _check("qa_decode_graph_create", st)
    return QAGraph(h, (qs, k_pages, v_pages, page_table, seq_lens, outs, workspace))


def qa_prefill_graph_create(qs, ks, vs, cu_seqlens, page_table, k_pages, v_pages, outs, *, scale=0.0,
                            stable_metadata=False):
    """Captures one prefill step of a packed bucket: layer i runs
    qa_prefill_attn(qs[i], ks[i], vs[i], cu_seqlens, page_table, k_pages[i],
    v_pages[i], outs[i]).  Returns a QAGraph."""
    torch = _torch()
    n = len(qs)
    if not (len(ks) == len(vs) == len(k_pages) == len(v_pages) == len(outs) == n):
        raise ValueError("per-layer lists must have the same length")
    T, Hq, D = qs[0].shape
    Hkv = ks[0].shape[1]
    B = cu_seqlens.shape[0] - 1
    P, PS = k_pages[0].shape[0], k_pages[0].shape[1]
    p = _params(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=PS, num_pages=P,
                max_pages_per_seq=page_table.shape[1], scale=scale, stable_metadata=stable_metadata)
    h = ctypes.c_void_p()
    st = _lib.qa_prefill_graph_create(n, _ptr_array(qs, "q", torch.bfloat16, 3), _ptr_array(ks, "k", torch.bfloat16, 3),
                                      _ptr_array(vs, "v", torch.bfloat16, 3),
                                      _dev(cu_seqlens, "cu_seqlens", torch.int32, 1), B, T,
                                      _dev(page_table, "page_table", torch.int32, 2),
                                      _ptr_array(k_pages, "k_pages", torch.bfloat16, 4),
                                      _ptr_array(v_pages, "v_pages", torch.bfloat16, 4),
                                      _ptr_array(outs, "out", torch.bfloat16, 3), ctypes.byref(p), ctypes.byref(h))
    _check("qa_prefill_graph_create", st)
    return QAGraph(h, (qs, ks, vs, cu_seqlens, page_table, k_pages, v_pages, outs))


def qa_window_workspace_size() -> int:
    """Bytes of the optional qa_window_attn workspace (its job counter)."""
    return int(_lib.qa_window_workspace_size())


def qa_window_attn(q, k, v, cu_windows, out=None, *, scale=0.0, workspace=None, stream=None, debug_checks=False):
    """Windowed bidirectional attention.  q/k/v bf16 [T,H,D]; cu_windows
    int32 [W+1].  workspace: optional zero-filled device tensor of at least
    qa_window_workspace_size() bytes (jobs then claimed from a counter in
    it).  Returns out bf16 [T,H,D]."""
    torch = _torch()
    T, H, D = q.shape
    W = cu_windows.shape[0] - 1
    if out is None:
        out = torch.empty_like(q)
    p = _params(n_q_heads=H, n_kv_heads=k.shape[1], head_dim=D, scale=scale, stream=stream, workspace=workspace,
                debug_checks=debug_checks)
    st = _lib.qa_window_attn(_dev(q, "q", torch.bfloat16, 3), _dev(k, "k", torch.bfloat16, 3),
                             _dev(v, "v", torch.bfloat16, 3), _dev(cu_windows, "cu_windows", torch.int32, 1), W, T,
                             _dev(out, "out", torch.bfloat16, 3), ctypes.byref(p))
    _check("qa_window_attn", st)
    return out


def qa_encoder_workspace_size(total_tokens: int, d_model: int, d_ffn: int) -> int:
    """Bytes of workspace qa_encoder_layer needs for total_tokens tokens."""
    n = _lib.qa_encoder_workspace_size(int(total_tokens), int(d_model), int(d_ffn))
    if n == 0 and total_tokens > 0:
        raise QAError("qa_encoder_workspace_size", -1, qa_last_error())
    return int(n)


def qa_encoder_layer(x, cu_windows, weights, out=None, *, n_heads, ln_eps=1e-5, workspace=None, stream=None,
                     debug_checks=False):
    """One AuT encoder layer.  x bf16 [T, d]; cu_windows int32 [W+1];
    weights: dict of bf16 device tensors named as ENCODER_WEIGHT_NAMES
    (w_qkv [3d, d], w_o [d, d], w_fc1 [ffn, d], w_fc2 [d, ffn], vectors for
    the rest).  Returns out bf16 [T, d]."""
    torch = _torch()
    T, d = x.shape
    d_ffn = weights["w_fc1"].shape[0]
    if out is None:
        out = torch.empty_like(x)
    if workspace is None:
        workspace = torch.empty(max(1, qa_encoder_workspace_size(T, d, d_ffn)), dtype=torch.uint8, device=x.device)
    wt = qa_encoder_weights()
    for name in ENCODER_WEIGHT_NAMES:
        t = weights[name]
        setattr(wt, name, _dev(t, name, torch.bfloat16, t.dim()).value)
    p = _params(n_q_heads=n_heads, n_kv_heads=n_heads, head_dim=d // n_heads, stream=stream, workspace=workspace,
                debug_checks=debug_checks)
    st = _lib.qa_encoder_layer(_dev(x, "x", torch.bfloat16, 2), _dev(cu_windows, "cu_windows", torch.int32, 1),
                               cu_windows.shape[0] - 1, T, d, int(n_heads), d_ffn, ctypes.byref(wt), float(ln_eps),
                               _dev(out, "out", torch.bfloat16, 2), ctypes.byref(p))
    _check("qa_encoder_layer", st)
    return out


def qa_linear(x, w, bias=None, out=None, *, gelu=False, residual=None, stream=None, debug_checks=False):
    """out = act(x W^T + bias) + residual on the tensor cores.  x bf16 [m, k],
    w bf16 [n, k], bias [n], residual [m, n]; act = exact gelu when gelu."""
    torch = _torch()
    m, k = x.shape
    n = w.shape[0]
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=x.device)
    p = _params(n_q_heads=1, n_kv_heads=1, head_dim=128, stream=stream, debug_checks=debug_checks)
    st = _lib.qa_linear(_dev(x, "x", torch.bfloat16, 2), m, k, _dev(w, "w", torch.bfloat16, 2), n,
                        None if bias is None else _dev(bias, "bias", torch.bfloat16, 1), 1 if gelu else 0,
                        None if residual is None else _dev(residual, "residual", torch.bfloat16, 2),
                        _dev(out, "out", torch.bfloat16, 2), ctypes.byref(p))
    _check("qa_linear", st)
    return out


def qa_layer_norm(x, gain, bias, out=None, *, eps=1e-5, stream=None, debug_checks=False):
    """LayerNorm over the rows of x bf16 [t, d] with gain and bias bf16 [d]."""
    torch = _torch()
    t, d = x.shape
    if out is None:
        out = torch.empty_like(x)
    p = _params(n_q_heads=1, n_kv_heads=1, head_dim=128, stream=stream, debug_checks=debug_checks)
    st = _lib.qa_layer_norm(_dev(x, "x", torch.bfloat16, 2), t, d, _dev(gain, "gain", torch.bfloat16, 1),
                            _dev(bias, "bias", torch.bfloat16, 1), float(eps), _dev(out, "out", torch.bfloat16, 2),
                            ctypes.byref(p))
    _check("qa_layer_norm", st)
    return out


def qa_window_plan(token_counts, window_tokens: int = 0) -> np.ndarray:
    """cu_windows (int32 numpy) for per-request encoder token counts; windows
    of window_tokens (0 = 104) from each request's start, last one partial."""
    counts = np.ascontiguousarray(np.asarray(token_counts, dtype=np.int32))
    w = int(window_tokens) if window_tokens > 0 else 104
    cap = int(sum(-(-int(c) // w) for c in counts if c > 0)) + 1
    cu = np.zeros(max(cap, 1), dtype=np.int32)
    n = _lib.qa_window_plan(counts.ctypes.data_as(ctypes.c_void_p), len(counts), int(window_tokens),
                            cu.ctypes.data_as(ctypes.c_void_p), len(cu))
    if n < 0:
        raise QAError("qa_window_plan", -1, qa_last_error())
    return cu[: n + 1]


def qa_check_bounded_wait(limit_us=20000, stream=None) -> None:
    """Launches one CTA whose bounded wait (the one the kernels use) gives up
    after limit_us microseconds on a barrier that nothing completes, setting
    QA_DEVICE_TIMEOUT (read it with qa_device_status); the kernel then ends."""
    _check("qa_check_bounded_wait", _lib.qa_check_bounded_wait(int(limit_us), _stream_ptr(stream)))


def qa_device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status bits."""
    n = _lib.qa_device_status(_stream_ptr(stream))
    if n < 0:
        raise QAError("qa_device_status", -1, qa_last_error())
    return n
