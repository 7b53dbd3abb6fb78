"""GB300-native speculative-sampling verification (sm_103a CUDA + C ABI).

The compute lives in ``libspecverify.so`` (built in-tree from ``csrc/`` by
:func:`build`); this module only marshals arguments to its C ABI
(``include/spec_verify.h``).  PyTorch supplies device memory and streams.
There is no CPU fallback: every call fails loudly when the library is
missing or no CUDA device is present.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
LIB_PATH = os.path.join(_HERE, "libspecverify.so")
_SOURCES = [os.path.join(_HERE, "csrc", f) for f in ("spec_verify.cu", "spec_strip.cu", "spec_row.cu",
                                                      "spec_commit.cu", "spec_law.cu",
                                                      "spec_cascade.cu")]
_DEPS = _SOURCES + [os.path.join(_HERE, "csrc", f)
                    for f in ("sv_common.cuh", "sv_core.cuh", "sv_strip.h", "sv_row.h",
                              "sv_verify.h")] + [
    os.path.join(_ROOT, "include", "spec_verify.h")]

SPEC_F32, SPEC_BF16 = 0, 1
ROW_BAD_TOKEN, ROW_BAD_LOGIT, ROW_NO_FINITE, ROW_Q_ZERO, ROW_BAD_GAMMA, ROW_BAD_UNIFORM = (
    1, 2, 4, 8, 16, 32)
ROW_ERROR_MASK = ROW_BAD_TOKEN | ROW_BAD_LOGIT | ROW_NO_FINITE | ROW_BAD_GAMMA | ROW_BAD_UNIFORM

EXPORTS = ("spec_verify", "spec_sample", "spec_verify_workspace_size", "spec_status_string",
           "spec_read_diagnostics", "spec_verify_noalloc", "spec_commit", "spec_law",
           "spec_cascade_verify", "spec_cascade_workspace_size", "spec_law_ws",
           "spec_law_workspace_size", "spec_sample_ws", "spec_sample_workspace_size")


class SpecParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("gamma_max", ctypes.c_int32), ("V", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("temperature", ctypes.c_float), ("top_p", ctypes.c_float),
        ("top_k", ctypes.c_int32), ("flags", ctypes.c_int32),
        ("target_pos_stride", ctypes.c_int64), ("target_row_stride", ctypes.c_int64),
        ("draft_pos_stride", ctypes.c_int64), ("draft_row_stride", ctypes.c_int64),
        ("gamma_per_row", ctypes.c_void_p), ("cluster_size", ctypes.c_int32),
        ("list_capacity", ctypes.c_int32),
    ]


class SpecDebug(ctypes.Structure):
    _fields_ = [("p_draft", ctypes.c_void_p), ("q_draft", ctypes.c_void_p),
                ("residual_mass", ctypes.c_void_p), ("row_status", ctypes.c_void_p)]


class SpecAimd(ctypes.Structure):
    _fields_ = [("gamma_min", ctypes.c_int32), ("gamma_max", ctypes.c_int32),
                ("increase", ctypes.c_int32), ("decrease", ctypes.c_float)]


class SpecError(RuntimeError):
    pass


_NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
               "-Xcompiler", "-fPIC", "-I", os.path.join(_ROOT, "include"),
               "-I", os.path.join(_HERE, "csrc")]


def nvcc_cmd(out: str = LIB_PATH, extra=()) -> list:
    """One nvcc command that compiles and links every source (serially)."""
    return ["nvcc", *_NVCC_FLAGS, *extra, "-shared", *_SOURCES, "-o", out]


def _compile(out: str, extra=()):
    """Compile the sources in parallel (one nvcc per translation unit), then link."""
    tag = f".tmp{os.getpid()}"
    objs = [out + f".{i}{tag}.o" for i in range(len(_SOURCES))]
    procs = [subprocess.Popen(["nvcc", *_NVCC_FLAGS, *extra, "-c", src, "-o", obj])
             for src, obj in zip(_SOURCES, objs)]
    codes = [p.wait() for p in procs]
    try:
        if any(codes):
            raise subprocess.CalledProcessError(max(codes), "nvcc -c")
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                        *objs, "-o", out], check=True)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)


def build(force: bool = False, out: str = None, extra=()) -> str:
    """Compile libspecverify.so in-tree for sm_103a (skipped when up to date)."""
    out = out or LIB_PATH
    stale = (not os.path.exists(out)) or any(
        os.path.getmtime(p) > os.path.getmtime(out) for p in _DEPS)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        _compile(tmp, extra)
        os.replace(tmp, out)
    return out


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise SpecError(f"{LIB_PATH} is missing: call build() first")
            L = ctypes.CDLL(LIB_PATH)
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            L.spec_verify.argtypes = [vp, vp, vp, vp, ctypes.POINTER(SpecParams), vp, vp,
                                      ctypes.POINTER(SpecDebug), vp, sz, vp]
            L.spec_verify.restype = ctypes.c_int
            L.spec_verify_noalloc.argtypes = [vp, vp, vp, vp, ctypes.POINTER(SpecParams), vp, vp,
                                              ctypes.POINTER(SpecDebug), vp]
            L.spec_verify_noalloc.restype = ctypes.c_int
            L.spec_sample.argtypes = [vp, vp, ctypes.POINTER(SpecParams), vp, vp, vp]
            L.spec_sample.restype = ctypes.c_int
            L.spec_verify_workspace_size.argtypes = [ctypes.POINTER(SpecParams)]
            L.spec_verify_workspace_size.restype = sz
            L.spec_status_string.argtypes = [ctypes.c_int]
            L.spec_status_string.restype = ctypes.c_char_p
            L.spec_read_diagnostics.argtypes = [vp, vp, ctypes.c_int, vp]
            L.spec_read_diagnostics.restype = ctypes.c_int
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            L.spec_commit.argtypes = [i32, i32, vp, vp, vp, vp, vp, i64, i32, vp, vp, vp,
                                      ctypes.POINTER(SpecAimd), vp]
            L.spec_commit.restype = ctypes.c_int
            L.spec_law.argtypes = [vp, vp, vp, ctypes.POINTER(SpecParams), vp, vp, vp, vp, vp]
            L.spec_law.restype = ctypes.c_int
            L.spec_sample_ws.argtypes = [vp, vp, ctypes.POINTER(SpecParams), vp, vp, vp, sz, vp]
            L.spec_sample_ws.restype = ctypes.c_int
            L.spec_sample_workspace_size.argtypes = [ctypes.POINTER(SpecParams)]
            L.spec_sample_workspace_size.restype = sz
            L.spec_law_ws.argtypes = [vp, vp, vp, ctypes.POINTER(SpecParams), vp, vp, vp, vp,
                                      vp, sz, vp]
            L.spec_law_ws.restype = ctypes.c_int
            L.spec_law_workspace_size.argtypes = [ctypes.POINTER(SpecParams)]
            L.spec_law_workspace_size.restype = sz
            L.spec_cascade_workspace_size.argtypes = [ctypes.POINTER(SpecParams), i32]
            L.spec_cascade_workspace_size.restype = sz
            L.spec_cascade_verify.argtypes = [ctypes.POINTER(vp), i32, vp, vp,
                                              ctypes.POINTER(SpecParams), vp, vp, vp, vp, vp,
                                              sz, vp]
            L.spec_cascade_verify.restype = ctypes.c_int
            _lib = L
    return _lib


def _check(code: int):
    if code != 0:
        raise SpecError(lib().spec_status_string(code).decode())


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise SpecError("no CUDA device: this library has no CPU path")
    return torch


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


SPEC_FLAG_CLUSTER_KERNEL = 1


def make_params(target, draft, temperature, top_k=0, top_p=1.0, gamma_per_row=None,
                cluster_size=0, list_capacity=0, flags=0) -> SpecParams:
    B, G1, _ = target.shape
    V = int(target.shape[2])
    if target.stride(2) != 1 or (draft is not None and draft.numel() and draft.stride(2) != 1):
        raise ValueError("the vocabulary axis must be contiguous")
    return SpecParams(
        B=B, gamma_max=G1 - 1, V=V, dtype=_dtype_code(target), temperature=float(temperature),
        top_p=float(top_p), top_k=int(top_k), flags=int(flags),
        target_pos_stride=target.stride(1), target_row_stride=target.stride(0),
        draft_pos_stride=draft.stride(1) if draft is not None and draft.dim() == 3 else V,
        draft_row_stride=draft.stride(0) if draft is not None and draft.dim() == 3 else 0,
        gamma_per_row=gamma_per_row.data_ptr() if gamma_per_row is not None else None,
        cluster_size=int(cluster_size), list_capacity=int(list_capacity))


_ws_lock = threading.Lock()
_ws_cache = {}


def auto_workspace(params: SpecParams, device, stream=None):
    """A workspace of the size the call needs, cached per device and stream
    (calls on one stream run in order, so they may share it)."""
    torch = _torch()
    need = int(lib().spec_verify_workspace_size(ctypes.byref(params)))
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (torch.device(device).index, s.cuda_stream)
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < need:
            buf = torch.zeros(max(need, 4096), dtype=torch.uint8, device=device)
            _ws_cache[key] = buf
    return buf


def spec_verify(target, draft, draft_tokens, uniforms, temperature, top_k=0, top_p=1.0,
                gamma_per_row=None, debug=False, workspace="auto", cluster_size=0,
                list_capacity=0, out=None, stream=None, kernel="auto"):
    """Verify a batch on the GPU.

    target [B, G+1, V] and draft [B, G, V] (float32 or bfloat16, CUDA, any
    row / position strides, contiguous vocabulary axis); draft_tokens [B, G]
    int32; uniforms [B, G+1, 2] float32; gamma_per_row [B] int32 or None.
    workspace: "auto" (a cached buffer of the size the call needs, which
    enables the strip-parallel kernel for greedy and top-k problems), a
    uint8 CUDA tensor, or None (no workspace: the cluster-per-row kernel).
    Vocabularies of at most 1024 with greedy or unfiltered sampling run on
    the warp-per-row kernel whatever the workspace.  kernel="cluster" forces
    the cluster-per-row kernel (same results; for comparisons).
    Returns (accepted_len, next_token) int32 tensors, plus a dict of debug
    outputs (p_draft, q_draft, residual_mass, row_status) when debug=True.
    """
    torch = _torch()
    B, G1, V = target.shape
    G = G1 - 1
    dev = target.device
    for name, t in (("draft_tokens", draft_tokens), ("uniforms", uniforms)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if draft_tokens is not None and draft_tokens.dtype != torch.int32:
        raise TypeError("draft_tokens must be int32")
    if uniforms is not None and uniforms.dtype != torch.float32:
        raise TypeError("uniforms must be float32")
    if kernel not in ("auto", "cluster"):
        raise ValueError("kernel must be 'auto' or 'cluster'")
    P = make_params(target, draft, temperature, top_k, top_p, gamma_per_row, cluster_size,
                    list_capacity, SPEC_FLAG_CLUSTER_KERNEL if kernel == "cluster" else 0)
    if out is None:
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        nxt = torch.empty(B, dtype=torch.int32, device=dev)
    else:
        acc, nxt = out
    dbg = None
    dbg_t = None
    if debug:
        dbg_t = {"p_draft": torch.empty((B, G), dtype=torch.float32, device=dev),
                 "q_draft": torch.empty((B, G), dtype=torch.float32, device=dev),
                 "residual_mass": torch.empty(B, dtype=torch.float32, device=dev),
                 "row_status": torch.empty(B, dtype=torch.int32, device=dev)}
        dbg = SpecDebug(*(dbg_t[k].data_ptr() if dbg_t[k].numel() else None
                          for k in ("p_draft", "q_draft", "residual_mass", "row_status")))
    ws_ptr, ws_bytes = (None, 0)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', a tensor or None")
        workspace = auto_workspace(P, dev, stream) if B > 0 else None
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().spec_verify(
        target.data_ptr(), draft.data_ptr() if draft is not None and draft.numel() else None,
        draft_tokens.data_ptr() if draft_tokens is not None and draft_tokens.numel() else None,
        uniforms.data_ptr() if uniforms is not None else None, ctypes.byref(P),
        acc.data_ptr(), nxt.data_ptr(), ctypes.byref(dbg) if dbg is not None else None,
        ws_ptr, ws_bytes, _stream_ptr(stream)))
    if debug:
        return acc, nxt, dbg_t
    return acc, nxt


def spec_verify_noalloc(target, draft, draft_tokens, uniforms, temperature, top_k=0, top_p=1.0,
                        gamma_per_row=None, debug=False, cluster_size=0, list_capacity=0,
                        out=None, stream=None):
    """spec_verify with the library's fixed device block as its workspace
    (no caller workspace, no allocation by the library).  Same arguments and
    results as spec_verify; problems too large for the block raise SpecError
    (SPEC_ERR_WORKSPACE).  Calls must not overlap in time."""
    torch = _torch()
    B, G1, V = target.shape
    G = G1 - 1
    dev = target.device
    for name, t in (("draft_tokens", draft_tokens), ("uniforms", uniforms)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    P = make_params(target, draft, temperature, top_k, top_p, gamma_per_row, cluster_size,
                    list_capacity)
    if out is None:
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        nxt = torch.empty(B, dtype=torch.int32, device=dev)
    else:
        acc, nxt = out
    dbg = dbg_t = None
    if debug:
        dbg_t = {"p_draft": torch.empty((B, G), dtype=torch.float32, device=dev),
                 "q_draft": torch.empty((B, G), dtype=torch.float32, device=dev),
                 "residual_mass": torch.empty(B, dtype=torch.float32, device=dev),
                 "row_status": torch.empty(B, dtype=torch.int32, device=dev)}
        dbg = SpecDebug(*(dbg_t[k].data_ptr() if dbg_t[k].numel() else None
                          for k in ("p_draft", "q_draft", "residual_mass", "row_status")))
    _check(lib().spec_verify_noalloc(
        target.data_ptr(), draft.data_ptr() if draft is not None and draft.numel() else None,
        draft_tokens.data_ptr() if draft_tokens is not None and draft_tokens.numel() else None,
        uniforms.data_ptr() if uniforms is not None else None, ctypes.byref(P),
        acc.data_ptr(), nxt.data_ptr(), ctypes.byref(dbg) if dbg is not None else None,
        _stream_ptr(stream)))
    if debug:
        return acc, nxt, dbg_t
    return acc, nxt


def spec_sample(logits, u, temperature, top_k=0, top_p=1.0, cluster_size=0, list_capacity=0,
                stream=None, with_status=False, workspace="auto"):
    """One draw per row of logits [n, V] (CUDA, float32/bfloat16) with
    uniforms u [n] float32: the filtered tempered law's inverse CDF.
    workspace: "auto" (a cached buffer of the size the call can use: the
    strip-parallel or CTA-per-row kernels), a uint8 CUDA tensor, or None
    (the warp-per-row or cluster kernels)."""
    torch = _torch()
    n, V = logits.shape
    if logits.stride(1) != 1:
        raise ValueError("the vocabulary axis must be contiguous")
    P = SpecParams(B=n, gamma_max=0, V=V, dtype=_dtype_code(logits),
                   temperature=float(temperature), top_p=float(top_p), top_k=int(top_k),
                   flags=0, target_pos_stride=V, target_row_stride=logits.stride(0),
                   draft_pos_stride=V, draft_row_stride=0, gamma_per_row=None,
                   cluster_size=int(cluster_size), list_capacity=int(list_capacity))
    tok = torch.empty(n, dtype=torch.int32, device=logits.device)
    st = torch.empty(n, dtype=torch.int32, device=logits.device)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', a tensor or None")
        workspace = auto_workspace(P, logits.device, stream) if n > 0 else None
    ws_ptr, ws_bytes = (None, 0)
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().spec_sample_ws(logits.data_ptr(), u.data_ptr() if u is not None else None,
                                ctypes.byref(P), tok.data_ptr(), st.data_ptr(), ws_ptr, ws_bytes,
                                _stream_ptr(stream)))
    return (tok, st) if with_status else tok


def workspace_bytes(params: SpecParams = None) -> int:
    """Workspace bytes a call with these parameters can use (the diagnostics
    block alone when params is None or the strip kernel does not apply)."""
    return int(lib().spec_verify_workspace_size(ctypes.byref(params) if params is not None
                                                else None))


def read_diagnostics(workspace, n=4, stream=None):
    import numpy as np
    out = np.zeros(n, np.uint32)
    _check(lib().spec_read_diagnostics(workspace.data_ptr(), out.ctypes.data, n,
                                       _stream_ptr(stream)))
    return out


def spec_commit(accepted_len, next_token, draft_tokens, seq, seq_len, gamma_per_row=None,
                aimd=None, stream=None):
    """The step after spec_verify (see spec_commit in include/spec_verify.h):
    appends each row's accepted drafts and next token to seq [B, capacity]
    (int32 CUDA, updated in place, row stride seq.stride(0)), updates seq_len
    [B] in place, and returns (kv_len, gamma_next) int32 tensors; gamma_next
    is None unless aimd = (gamma_min, gamma_max, increase, decrease)."""
    torch = _torch()
    B = int(accepted_len.shape[0])
    for name, t in (("accepted_len", accepted_len), ("next_token", next_token),
                    ("draft_tokens", draft_tokens), ("seq", seq), ("seq_len", seq_len)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    if seq.dim() != 2 or seq.stride(1) != 1:
        raise ValueError("seq must be [B, capacity] with contiguous rows")
    if not draft_tokens.is_contiguous():
        raise ValueError("draft_tokens must be contiguous")
    G = int(draft_tokens.shape[1]) if draft_tokens.dim() == 2 else 0
    kv = torch.empty(B, dtype=torch.int32, device=seq.device)
    gn = torch.empty(B, dtype=torch.int32, device=seq.device) if aimd is not None else None
    A = SpecAimd(int(aimd[0]), int(aimd[1]), int(aimd[2]), float(aimd[3])) if aimd else None
    ptr = lambda t: t.data_ptr() if t is not None and t.numel() else None
    _check(lib().spec_commit(B, G, ptr(accepted_len), ptr(next_token), ptr(draft_tokens),
                             ptr(gamma_per_row), ptr(seq), seq.stride(0), int(seq.shape[1]),
                             ptr(seq_len), ptr(kv), ptr(gn),
                             ctypes.byref(A) if A is not None else None, _stream_ptr(stream)))
    return kv, gn


def spec_law(target, draft, tokens, temperature, top_k=0, top_p=1.0, stream=None,
             workspace="auto", cluster_size=0, list_capacity=0):
    """The emitted-token law of the speculative sampler at each row's token
    (see spec_law and spec_law_ws in include/spec_verify.h): target and draft
    [n, V] logits (float32 / bfloat16 CUDA, contiguous rows), tokens [n]
    int32, the laws tempered and filtered (top-k then top-p) as in
    spec_verify.  workspace: "auto" (a fresh buffer of the size the call can
    use: filtered laws then run on the strip-parallel kernel), a uint8 CUDA
    tensor, or None (the one-CTA-per-row kernels).  Returns (p_spec, beta,
    p_x, q_x) float32 tensors [n]."""
    torch = _torch()
    n, V = target.shape
    if target.stride(1) != 1 or draft.stride(1) != 1 or draft.shape != target.shape:
        raise ValueError("target and draft must be [n, V] with contiguous rows")
    if tokens.dtype != torch.int32:
        raise TypeError("tokens must be int32")
    P = SpecParams(B=n, gamma_max=0, V=V, dtype=_dtype_code(target),
                   temperature=float(temperature), top_p=float(top_p), top_k=int(top_k),
                   flags=0, target_pos_stride=V, target_row_stride=target.stride(0),
                   draft_pos_stride=V, draft_row_stride=draft.stride(0), gamma_per_row=None,
                   cluster_size=int(cluster_size), list_capacity=int(list_capacity))
    out = [torch.empty(n, dtype=torch.float32, device=target.device) for _ in range(4)]
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', a tensor or None")
        need = int(lib().spec_law_workspace_size(ctypes.byref(P)))
        workspace = torch.empty(need, dtype=torch.uint8, device=target.device) if need else None
    ws_ptr, ws_bytes = (None, 0)
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().spec_law_ws(target.data_ptr(), draft.data_ptr(), tokens.data_ptr(),
                             ctypes.byref(P), *(o.data_ptr() for o in out), ws_ptr, ws_bytes,
                             _stream_ptr(stream)))
    return tuple(out)


def law_workspace_bytes(params: SpecParams) -> int:
    return int(lib().spec_law_workspace_size(ctypes.byref(params)))


def cascade_params(levels, temperature, top_k=0, top_p=1.0, gamma_per_row=None,
                   flags=0) -> SpecParams:
    """spec_params of a cascade: the target strides from levels[0] (shared by
    every level but the smallest), the draft strides from levels[-1]."""
    torch = _torch()
    tgt, small = levels[0], levels[-1]
    B, G1, V = tgt.shape
    for lv in levels[:-1]:
        if lv.shape != tgt.shape or lv.stride() != tgt.stride() or lv.dtype != tgt.dtype:
            raise ValueError("every level but the smallest must match the target's "
                             "shape, strides and dtype")
    if small is not None and (small.shape != (B, G1 - 1, V) or small.dtype != tgt.dtype):
        raise ValueError("the smallest level must be [B, gamma_max, V] in the target's dtype")
    if gamma_per_row is not None and gamma_per_row.dtype != torch.int32:
        raise TypeError("gamma_per_row must be int32")
    return make_params(tgt, small, temperature, top_k, top_p, gamma_per_row, flags=flags)


def cascade_workspace_bytes(params: SpecParams, n_levels: int) -> int:
    return int(lib().spec_cascade_workspace_size(ctypes.byref(params), int(n_levels)))


def spec_cascade_verify(levels, draft_tokens, uniforms, temperature, top_k=0, top_p=1.0,
                        gamma_per_row=None, workspace="auto", stream=None, kernel="auto"):
    """Verify a multi-stage draft cascade on the GPU (see spec_cascade_verify
    in include/spec_verify.h).  levels: [target, level 1, ..., smallest]
    CUDA logits, every level but the smallest [B, G+1, V] with the target's
    strides, the smallest [B, G, V]; draft_tokens [B, G] int32 (drawn from
    the smallest level); uniforms [L, B, G+1, 2] float32 (stage k uses
    uniforms[k]); gamma_per_row [B] int32 or None.  workspace: "auto" (a
    fresh buffer of the size the call can use), a uint8 CUDA tensor.
    Returns (out_tokens [B, G+1], out_len [B], stage_accepted [L, B],
    row_status [B]) int32 tensors."""
    torch = _torch()
    L = len(levels) - 1
    if L < 1:
        raise ValueError("a cascade needs the target and at least one draft level")
    tgt = levels[0]
    B, G1, V = tgt.shape
    dev = tgt.device
    for name, t in (("draft_tokens", draft_tokens), ("uniforms", uniforms)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if draft_tokens.dtype != torch.int32:
        raise TypeError("draft_tokens must be int32")
    if uniforms is not None and (uniforms.dtype != torch.float32 or
                                 tuple(uniforms.shape) != (L, B, G1, 2)):
        raise ValueError("uniforms must be float32 [L, B, gamma_max+1, 2]")
    if kernel not in ("auto", "cluster"):
        raise ValueError("kernel must be 'auto' or 'cluster'")
    P = cascade_params(levels, temperature, top_k, top_p, gamma_per_row,
                       SPEC_FLAG_CLUSTER_KERNEL if kernel == "cluster" else 0)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto' or a tensor")
        workspace = torch.empty(max(cascade_workspace_bytes(P, L + 1), 256), dtype=torch.uint8,
                                device=dev)
    out_tok = torch.empty((B, G1), dtype=torch.int32, device=dev)
    out_len = torch.empty(B, dtype=torch.int32, device=dev)
    stage_acc = torch.empty((L, B), dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    ptrs = (ctypes.c_void_p * (L + 1))(*[lv.data_ptr() if lv is not None and lv.numel() else None
                                         for lv in levels])
    _check(lib().spec_cascade_verify(
        ptrs, L + 1, draft_tokens.data_ptr() if draft_tokens.numel() else None,
        uniforms.data_ptr() if uniforms is not None else None, ctypes.byref(P),
        out_tok.data_ptr(), out_len.data_ptr(), stage_acc.data_ptr(), status.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out_tok, out_len, stage_acc, status
