"""fp64 CPU oracle for the Gated DeltaNet chunked-prefill hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path (the
CUDA library and its binding) never touches it, and it shares no code with
that path.

Functions (FlashQLA pages, page 1 "usage and requirements": the low-level
forward returns ``(g, A, o, h, final_state)`` and the backward returns
``(dq, dk, dv, db, dg, dh0)``):

* ``fwd``         -- the gated delta rule token by token (``gdr_oracle.c``);
* ``A_matrix``    -- ``A = (I + L)^-1`` of every chunk by its definition;
* ``bwd``         -- reverse mode of the token recurrence;
* ``chunked_fwd`` -- an independent chunked/WY form with the exact segment
  (context-parallel) split (``gdr_chunked.c``), used only to pin the chunk
  algebra, ``A`` and ``h``.

Inputs are numpy arrays or CPU torch tensors of any float dtype; they are
upcast exactly to fp64.  Shapes follow the FlashQLA signature:
q, k ``[B,T,Hq,K]``; v ``[B,T,Hv,V]``; g, beta ``[B,T,Hv]``; h0 ``[N,Hv,K,V]``.
With ``cu_seqlens`` (varlen), ``B`` must be 1 and ``N = len(cu_seqlens) - 1``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = ("gdr_oracle.c", "gdr_chunked.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain C, fp64, pthreads)."""
    srcs = [os.path.join(_HERE, s) for s in _SRCS]
    if not force and os.path.exists(_LIB_PATH):
        newest = max(os.path.getmtime(s) for s in srcs)
        if os.path.getmtime(_LIB_PATH) >= newest:
            return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-o", tmp, *srcs, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(mutation: int, out_dir: str) -> str:
    """Build the oracle with a planted mistake (``-DGDR_ORACLE_MUTATION=n``), for
    the oracle's own self-test that its pins catch it."""
    srcs = [os.path.join(_HERE, s) for s in _SRCS]
    path = os.path.join(out_dir, f"liboracle_mut{mutation}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    f"-DGDR_ORACLE_MUTATION={int(mutation)}", "-o", path, *srcs, "-lm"], check=True)
    return path


def use_library(path):
    """Point this module at another build of the oracle (``None``: the default one)."""
    global _lib
    _lib = None
    if path is not None:
        _lib = _configure(ctypes.CDLL(path))


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _configure(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    i, d = ctypes.c_int, ctypes.c_double
    lib.gdr_oracle_fwd.argtypes = [i, ip, i, i, i, i, i, dp, dp, dp, dp, dp, d, dp, dp, dp, dp, i, i]
    lib.gdr_oracle_A.argtypes = [i, ip, i, i, i, i, dp, dp, dp, dp, i]
    lib.gdr_oracle_bwd.argtypes = [i, ip, i, i, i, i, dp, dp, dp, dp, dp, d, dp, dp, dp,
                                   dp, dp, dp, dp, dp, dp, i, i]
    lib.gdr_chunked_fwd.argtypes = [i, ip, i, i, i, i, i, i, dp, dp, dp, dp, dp, d, dp, dp,
                                    dp, dp, dp, i]
    for f in (lib.gdr_oracle_fwd, lib.gdr_oracle_A, lib.gdr_oracle_bwd, lib.gdr_chunked_fwd):
        f.restype = ctypes.c_int
    return lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _seqs(B, T, cu_seqlens):
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int32) * T
    else:
        if B != 1:
            raise ValueError("varlen inputs need B == 1")
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int32))
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must start at 0, be non-decreasing and end at T")
    return cu


def n_chunks(cu, C=64):
    lens = np.diff(np.asarray(cu))
    return int(np.sum((lens + C - 1) // C))


def _dims(q, v):
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    return B, T, Hq, Hv, K, V


def fwd(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64, want_h=False,
        nthreads=None, vblock=None):
    """Token-by-token forward.  Returns dict(o, final_state[, h])."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, Hq, Hv, K, V = _dims(q, v)
    cu = _seqs(B, T, cu_seqlens)
    N = len(cu) - 1
    o = np.zeros((B, T, Hv, V))
    fs = np.zeros((N, Hv, K, V))
    nt = n_chunks(cu, chunk)
    hc = np.zeros((nt, Hv, K, V)) if want_h else None
    rc = _load().gdr_oracle_fwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), Hq, Hv, K, V,
                                chunk, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                float(scale), _ptr(h0), _ptr(o), _ptr(fs), _ptr(hc),
                                _threads(nthreads), int(vblock or V))
    if rc:
        raise ValueError("oracle fwd: bad arguments")
    out = {"o": o, "final_state": fs}
    if want_h:
        out["h"] = hc.reshape(B, nt // B, Hv, K, V) if cu_seqlens is None else hc[None]
    return out


def A_matrix(k, g, beta, cu_seqlens=None, chunk=64, Hv=None, nthreads=None):
    """A = (I + strict_tril(diag(b)(KK^T o D)))^-1 per chunk, laid out [B,T,Hv,chunk]."""
    k, g, beta = map(_f64, (k, g, beta))
    B, T, Hq, K = k.shape
    Hv = g.shape[2]
    cu = _seqs(B, T, cu_seqlens)
    A = np.zeros((B, T, Hv, chunk))
    rc = _load().gdr_oracle_A(len(cu) - 1, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), Hq, Hv,
                              K, chunk, _ptr(k), _ptr(g), _ptr(beta), _ptr(A), _threads(nthreads))
    if rc:
        raise ValueError("oracle A: bad arguments")
    return A


def bwd(q, k, v, g, beta, scale, do, dht=None, h0=None, cu_seqlens=None, nthreads=None,
        checkpoint=64):
    """Reverse mode of the token recurrence.  Returns dict(dq, dk, dv, dbeta, dg, dh0).

    ``checkpoint`` is the token interval of the saved fp64 states (a memory
    knob; the result does not depend on it)."""
    q, k, v, g, beta, do, dht, h0 = map(_f64, (q, k, v, g, beta, do, dht, h0))
    B, T, Hq, Hv, K, V = _dims(q, v)
    cu = _seqs(B, T, cu_seqlens)
    N = len(cu) - 1
    dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    dbeta = np.zeros_like(beta); dg = np.zeros_like(g); dh0 = np.zeros((N, Hv, K, V))
    rc = _load().gdr_oracle_bwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), Hq, Hv, K, V,
                                _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                _ptr(h0), _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(dbeta), _ptr(dg), _ptr(dh0), _threads(nthreads),
                                int(checkpoint))
    if rc:
        raise ValueError("oracle bwd: bad arguments")
    return {"dq": dq, "dk": dk, "dv": dv, "dbeta": dbeta, "dg": dg, "dh0": dh0}


def chunked_fwd(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64, seg_chunks=0,
                nthreads=None):
    """Independent chunked/WY form with segments of ``seg_chunks`` chunks (0 = one segment)."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, Hq, Hv, K, V = _dims(q, v)
    cu = _seqs(B, T, cu_seqlens)
    N = len(cu) - 1
    nt = n_chunks(cu, chunk)
    o = np.zeros((B, T, Hv, V)); fs = np.zeros((N, Hv, K, V))
    hc = np.zeros((nt, Hv, K, V)); A = np.zeros((B, T, Hv, chunk))
    rc = _load().gdr_chunked_fwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), Hq, Hv, K, V,
                                 chunk, int(seg_chunks), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), float(scale), _ptr(h0), _ptr(o), _ptr(fs), _ptr(hc),
                                 _ptr(A), _threads(nthreads))
    if rc:
        raise ValueError("oracle chunked fwd: bad arguments")
    hc = hc.reshape(B, nt // B, Hv, K, V) if cu_seqlens is None else hc[None]
    return {"o": o, "final_state": fs, "h": hc, "A": A}
