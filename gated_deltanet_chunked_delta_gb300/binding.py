"""ctypes binding of libgdr (``include/gdr.h``).

Argument marshalling only: every step of the forward and backward runs in the
library's CUDA kernels.  PyTorch provides device memory and the stream.  There
is no fallback: if ``libgdr.so`` is missing or cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

GDR_BF16, GDR_F32 = 0, 1
GDR_PATH_AUTO, GDR_PATH_SIMT, GDR_PATH_TC = 0, 1, 2
ERRORS = {1: "GDR_ERR_ARG", 2: "GDR_ERR_SHAPE", 3: "GDR_ERR_DTYPE", 4: "GDR_ERR_ALIGN",
          5: "GDR_ERR_WORKSPACE", 6: "GDR_ERR_CUDA", 7: "GDR_ERR_TIMEOUT", 8: "GDR_ERR_DEVICE"}
EXPORTS = ("gdr_num_chunks", "gdr_get_plan", "gdr_fwd_workspace_size", "gdr_bwd_workspace_size", "gdr_fwd",
           "gdr_bwd", "gdr_check_status", "gdr_last_error", "gdr_version")


class GdrError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class gdr_buf(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int)]


class gdr_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hq", ctypes.c_int), ("Hv", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int), ("n_seqs", ctypes.c_int),
                ("cu_seqlens", ctypes.c_void_p), ("cu_seqlens_host", ctypes.c_void_p)]


class gdr_opts(ctypes.Structure):
    _fields_ = [("cp_segments", ctypes.c_int), ("path", ctypes.c_int), ("debug_checks", ctypes.c_int),
                ("timeout_spins", ctypes.c_longlong), ("events", ctypes.POINTER(ctypes.c_void_p)),
                ("names", ctypes.POINTER(ctypes.c_char_p)), ("max_events", ctypes.c_int),
                ("n_launched", ctypes.POINTER(ctypes.c_int)), ("cp_warmup", ctypes.c_int)]


class gdr_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("n_chunks", ctypes.c_longlong), ("n_segments", ctypes.c_int),
                ("seg_len", ctypes.c_int), ("cp_warmup", ctypes.c_int)]


class KernelTimer:
    """Caller-owned CUDA events that a call records around each of its kernel
    launches (``gdr_opts.events``).  ``elapsed()`` gives (name, ms) per launch
    after the stream has been synchronised."""

    def __init__(self, max_launches: int = 64):
        self.max = max_launches
        self.torch_events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_launches)]
        for e in self.torch_events:  # creates the underlying cudaEvent_t
            e.record()
        torch.cuda.synchronize()
        self.handles = (ctypes.c_void_p * (2 * max_launches))(*[e.cuda_event for e in self.torch_events])
        self.names = (ctypes.c_char_p * max_launches)()
        self.count = ctypes.c_int(0)

    def attach(self, opts):
        opts.events = ctypes.cast(self.handles, ctypes.POINTER(ctypes.c_void_p))
        opts.names = ctypes.cast(self.names, ctypes.POINTER(ctypes.c_char_p))
        opts.max_events = 2 * self.max
        opts.n_launched = ctypes.pointer(self.count)
        return opts

    def elapsed(self):
        n = min(self.count.value, self.max)
        return [(self.names[i].decode() if self.names[i] else f"k{i}",
                 self.torch_events[2 * i].elapsed_time(self.torch_events[2 * i + 1])) for i in range(n)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libgdr.so (raises if it is missing and ``build_if_missing`` is False)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libgdr.so is not built ({path}); run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    P, vp, sz = ctypes.POINTER, ctypes.c_void_p, ctypes.c_size_t
    lib.gdr_num_chunks.argtypes = [P(gdr_shape)]
    lib.gdr_num_chunks.restype = ctypes.c_longlong
    lib.gdr_get_plan.argtypes = [P(gdr_shape), ctypes.c_int, P(gdr_opts), P(gdr_plan)]
    lib.gdr_get_plan.restype = ctypes.c_int
    for f in (lib.gdr_fwd_workspace_size, lib.gdr_bwd_workspace_size):
        f.argtypes = [P(gdr_shape), P(gdr_opts)]
        f.restype = sz
    lib.gdr_fwd.argtypes = [P(gdr_shape), gdr_buf, gdr_buf, gdr_buf, vp, vp, ctypes.c_float, vp, gdr_buf, vp,
                            vp, vp, vp, sz, P(gdr_opts), vp]
    lib.gdr_fwd.restype = ctypes.c_int
    lib.gdr_bwd.argtypes = [P(gdr_shape), gdr_buf, gdr_buf, gdr_buf, vp, vp, vp, gdr_buf, vp, ctypes.c_float, vp,
                            gdr_buf, gdr_buf, gdr_buf, vp, vp, vp, vp, sz, P(gdr_opts), vp]
    lib.gdr_bwd.restype = ctypes.c_int
    lib.gdr_check_status.argtypes = [vp]
    lib.gdr_check_status.restype = ctypes.c_int
    lib.gdr_last_error.restype = ctypes.c_char_p
    lib.gdr_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDR_BF16
    if t.dtype == torch.float32:
        return GDR_F32
    raise GdrError(3, f"unsupported dtype {t.dtype}")


def _buf(t: Optional[torch.Tensor]) -> gdr_buf:
    if t is None:
        return gdr_buf(None, 0)
    return gdr_buf(t.data_ptr(), _dt(t))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check_dev(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise GdrError(1, "every tensor must live on the GPU")
            if not t.is_contiguous():
                raise GdrError(1, "every tensor must be contiguous")


class Problem:
    """Sizes of one call, with the host copy of cu_seqlens kept alive."""

    def __init__(self, q, v, cu_seqlens=None, cu_seqlens_host=None):
        B, T, Hq, K = q.shape
        Hv, V = v.shape[2], v.shape[3]
        self.B, self.T, self.Hq, self.Hv, self.K, self.V = B, T, Hq, Hv, K, V
        self.cu_dev = cu_seqlens
        if cu_seqlens is not None:
            if cu_seqlens.dtype != torch.int32:
                raise GdrError(3, "cu_seqlens must be int32")
            host = cu_seqlens_host if cu_seqlens_host is not None else cu_seqlens.cpu()
            self.cu_host = host.to(torch.int32).contiguous()
            self.n_seqs = self.cu_host.numel() - 1
        else:
            self.cu_host = None
            self.n_seqs = 0
        self.shape = gdr_shape(B, T, Hq, Hv, K, V, self.n_seqs,
                               None if cu_seqlens is None else cu_seqlens.data_ptr(),
                               None if self.cu_host is None else self.cu_host.data_ptr())

    @property
    def N(self):
        return self.n_seqs if self.n_seqs else self.B

    def num_chunks(self) -> int:
        n = load().gdr_num_chunks(ctypes.byref(self.shape))
        if n < 0:
            raise GdrError(2, load().gdr_last_error().decode())
        return int(n)


def make_opts(cp_segments=0, path=GDR_PATH_AUTO, debug_checks=0, timeout_spins=0, timer=None,
              cp_warmup=0) -> gdr_opts:
    o = gdr_opts(int(cp_segments), int(path), int(debug_checks), int(timeout_spins), None, None, 0, None,
                 int(cp_warmup))
    return timer.attach(o) if timer is not None else o


def get_plan(prob: Problem, in_dtype: int = GDR_BF16, opts: Optional[gdr_opts] = None) -> dict:
    """The plan a call with these sizes, input dtype and options would take
    (host-side query: path, chunks, context-parallel segments, warm-up)."""
    out = gdr_plan()
    rc = load().gdr_get_plan(ctypes.byref(prob.shape), int(in_dtype), ctypes.byref(opts or make_opts()),
                             ctypes.byref(out))
    if rc:
        raise GdrError(rc, load().gdr_last_error().decode())
    return {"path": out.path, "n_chunks": out.n_chunks, "n_segments": out.n_segments, "seg_len": out.seg_len,
            "cp_warmup": out.cp_warmup}


def fwd_workspace_size(prob: Problem, opts: gdr_opts) -> int:
    n = load().gdr_fwd_workspace_size(ctypes.byref(prob.shape), ctypes.byref(opts))
    if n == 0:
        raise GdrError(2, load().gdr_last_error().decode())
    return int(n)


def bwd_workspace_size(prob: Problem, opts: gdr_opts) -> int:
    n = load().gdr_bwd_workspace_size(ctypes.byref(prob.shape), ctypes.byref(opts))
    if n == 0:
        raise GdrError(2, load().gdr_last_error().decode())
    return int(n)


def tc_available(K: int = 128, V: int = 128) -> bool:
    """Whether the loaded library carries the tensor-core path for these head sizes."""
    shp = gdr_shape(1, 64, 1, 1, K, V, 0, None, None)
    opts = make_opts(path=GDR_PATH_TC)
    return load().gdr_fwd_workspace_size(ctypes.byref(shp), ctypes.byref(opts)) > 0


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def gdr_fwd(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None, cu_seqlens_host=None, *, o_dtype=None,
            output_final_state=True, want_A=True, want_h=False, cp_segments=0, path=GDR_PATH_AUTO,
            debug_checks=0, timeout_spins=0, workspace=None, out=None, stream=None, timer=None, cp_warmup=0):
    """Forward.  Returns dict(o, final_state, A, h) (entries None when not requested).

    ``out`` may hold preallocated output tensors under the same keys."""
    _check_dev(q, k, v, g, beta, h0, cu_seqlens)
    lib = load()
    prob = Problem(q, v, cu_seqlens, cu_seqlens_host)
    if scale is None:
        scale = prob.K ** -0.5
    opts = make_opts(cp_segments, path, debug_checks, timeout_spins, timer=timer, cp_warmup=cp_warmup)
    out = dict(out or {})
    dev = q.device
    if out.get("o") is None:
        out["o"] = torch.empty(prob.B, prob.T, prob.Hv, prob.V, device=dev, dtype=o_dtype or q.dtype)
    if output_final_state and out.get("final_state") is None:
        out["final_state"] = torch.empty(prob.N, prob.Hv, prob.K, prob.V, device=dev, dtype=torch.float32)
    if want_A and out.get("A") is None:
        out["A"] = torch.empty(prob.B, prob.T, prob.Hv, 64, device=dev, dtype=torch.float32)
    if want_h and out.get("h") is None:
        out["h"] = torch.empty(prob.num_chunks(), prob.Hv, prob.K, prob.V, device=dev, dtype=torch.float32)
    for key in ("final_state", "A", "h"):
        out.setdefault(key, None)
    _check_dev(*out.values())
    if workspace is None:
        workspace = alloc_workspace(fwd_workspace_size(prob, opts), dev)
    rc = lib.gdr_fwd(ctypes.byref(prob.shape), _buf(q), _buf(k), _buf(v), _ptr(g), _ptr(beta), float(scale),
                     _ptr(h0), _buf(out["o"]), _ptr(out["final_state"]), _ptr(out["A"]), _ptr(out["h"]),
                     workspace.data_ptr(), workspace.numel(), ctypes.byref(opts), _stream(stream))
    if rc:
        raise GdrError(rc, lib.gdr_last_error().decode())
    return out


def gdr_bwd(q, k, v, g, beta, A, do, dht=None, scale=None, h0=None, cu_seqlens=None, cu_seqlens_host=None, *,
            want_dh0=True, cp_segments=0, path=GDR_PATH_AUTO, debug_checks=0, timeout_spins=0, workspace=None,
            out=None, stream=None, timer=None, cp_warmup=0):
    """Backward.  Returns dict(dq, dk, dv, dbeta, dg, dh0)."""
    _check_dev(q, k, v, g, beta, A, do, dht, h0, cu_seqlens)
    lib = load()
    prob = Problem(q, v, cu_seqlens, cu_seqlens_host)
    if scale is None:
        scale = prob.K ** -0.5
    opts = make_opts(cp_segments, path, debug_checks, timeout_spins, timer=timer, cp_warmup=cp_warmup)
    out = dict(out or {})
    dev = q.device
    for key, like in (("dq", q), ("dk", k), ("dv", v)):
        if out.get(key) is None:
            out[key] = torch.empty_like(like)
    for key in ("dbeta", "dg"):
        if out.get(key) is None:
            out[key] = torch.empty_like(g, dtype=torch.float32)
    if want_dh0 and out.get("dh0") is None:
        out["dh0"] = torch.empty(prob.N, prob.Hv, prob.K, prob.V, device=dev, dtype=torch.float32)
    out.setdefault("dh0", None)
    _check_dev(*out.values())
    if workspace is None:
        workspace = alloc_workspace(bwd_workspace_size(prob, opts), dev)
    rc = lib.gdr_bwd(ctypes.byref(prob.shape), _buf(q), _buf(k), _buf(v), _ptr(g), _ptr(beta), _ptr(A), _buf(do),
                     _ptr(dht), float(scale), _ptr(h0), _buf(out["dq"]), _buf(out["dk"]), _buf(out["dv"]),
                     _ptr(out["dbeta"]), _ptr(out["dg"]), _ptr(out["dh0"]), workspace.data_ptr(),
                     workspace.numel(), ctypes.byref(opts), _stream(stream))
    if rc:
        raise GdrError(rc, lib.gdr_last_error().decode())
    return out


def check_status(stream=None) -> None:
    lib = load()
    rc = lib.gdr_check_status(_stream(stream))
    if rc:
        raise GdrError(rc, lib.gdr_last_error().decode())


def version() -> str:
    return load().gdr_version().decode()
