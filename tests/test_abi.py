"""The C ABI on the CPU: the library loads, exports every entry point that
include/gdr.h declares, and rejects bad arguments with the documented codes
before launching anything."""
import ctypes
import os
import re

import pytest

import gated_deltanet_chunked_delta_gb300 as gdr
from gated_deltanet_chunked_delta_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_chunked_delta_gb300 import build
    build.build()
    return gdr.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "gdr.h")).read()
    return sorted(set(re.findall(r"GDR_API\s+[\w\s\*]+?\b(gdr_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) >= set(B.EXPORTS)


def test_version(lib):
    assert "sm_103a" in gdr.version()


def shape(B_=1, T=128, Hq=2, Hv=4, K=128, V=128, n_seqs=0, cu=None, cu_host=None):
    return B.gdr_shape(B_, T, Hq, Hv, K, V, n_seqs, cu, cu_host)


def sizes(lib, shp, opts=None):
    opts = opts or B.make_opts()
    return lib.gdr_fwd_workspace_size(ctypes.byref(shp), ctypes.byref(opts))


def test_workspace_size_and_chunks(lib):
    assert sizes(lib, shape()) > 0
    assert lib.gdr_num_chunks(ctypes.byref(shape(B_=3, T=130))) == 9
    assert lib.gdr_bwd_workspace_size(ctypes.byref(shape()), ctypes.byref(B.make_opts())) > sizes(lib, shape())


@pytest.mark.parametrize("bad", [dict(K=96), dict(V=32), dict(K=256), dict(V=320), dict(Hq=3, Hv=4), dict(T=0), dict(B_=0),
                                 dict(B_=2, n_seqs=2)])
def test_bad_shapes_rejected(lib, bad):
    assert sizes(lib, shape(**bad)) == 0
    assert lib.gdr_num_chunks(ctypes.byref(shape(**bad))) == -1
    assert lib.gdr_last_error()


def test_varlen_host_table_checked(lib):
    arr = (ctypes.c_int32 * 4)(0, 10, 5, 20)  # decreasing
    shp = shape(T=20, n_seqs=3, cu=ctypes.addressof(arr), cu_host=ctypes.addressof(arr))
    assert sizes(lib, shp) == 0
    good = (ctypes.c_int32 * 4)(0, 10, 10, 20)
    shp = shape(T=20, n_seqs=3, cu=ctypes.addressof(good), cu_host=ctypes.addressof(good))
    assert sizes(lib, shp) > 0
    assert lib.gdr_num_chunks(ctypes.byref(shp)) == 2


def _fwd(lib, shp, q=(0x10000, 0), k=(0x20000, 0), v=(0x30000, 0), g=0x40000, beta=0x50000, o=(0x60000, 0),
         ws=0x100000, ws_bytes=1 << 40, opts=None):
    opts = opts or B.make_opts()
    return lib.gdr_fwd(ctypes.byref(shp), B.gdr_buf(*q), B.gdr_buf(*k), B.gdr_buf(*v), g, beta, 0.1, None,
                       B.gdr_buf(*o), None, None, None, ws, ws_bytes, ctypes.byref(opts), None)


def test_fwd_argument_errors_launch_nothing(lib):
    shp = shape()
    assert _fwd(lib, shp, q=(0, 0)) == 1                       # null q
    assert _fwd(lib, shp, g=0) == 1                            # null g
    assert _fwd(lib, shp, q=(0x10008, 0)) == 4                 # misaligned
    assert _fwd(lib, shp, k=(0x20000, 1)) == 3                 # mixed dtypes
    assert _fwd(lib, shp, o=(0x60000, 7)) == 3                 # unknown dtype
    assert _fwd(lib, shp, ws=0) == 5                           # no workspace
    assert _fwd(lib, shp, ws_bytes=16) == 5                    # too small
    assert _fwd(lib, shp, ws=0x100010) == 4                    # workspace alignment
    assert _fwd(lib, shape(K=80)) == 2                         # shape
    assert _fwd(lib, shp, q=(0x10000, 1), k=(0x20000, 1), v=(0x30000, 1),
                opts=B.make_opts(path=2)) == 3                 # tensor-core path needs bf16
    assert _fwd(lib, shp, opts=B.make_opts(cp_segments=-1)) == 1


def test_bwd_argument_errors(lib):
    shp = shape()
    opts = B.make_opts()
    z = B.gdr_buf(0, 0)
    b = lambda a: B.gdr_buf(a, 0)  # noqa: E731
    rc = lib.gdr_bwd(ctypes.byref(shp), b(0x1000), b(0x2000), b(0x3000), 0x4000, 0x5000, None, b(0x6000), None,
                     0.1, None, b(0x7000), b(0x8000), b(0x9000), 0xa000, 0xb000, None, 0x100000, 1 << 40,
                     ctypes.byref(opts), None)
    assert rc == 1  # A is required
    rc = lib.gdr_bwd(ctypes.byref(shp), b(0x1000), b(0x2000), b(0x3000), 0x4000, 0x5000, 0xc000, z, None,
                     0.1, None, b(0x7000), b(0x8000), b(0x9000), 0xa000, 0xb000, None, 0x100000, 1 << 40,
                     ctypes.byref(opts), None)
    assert rc == 1  # do is required


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 64, 1, 64)
    with pytest.raises(gdr.GdrError):
        gdr.gdr_fwd(q, q, q, torch.zeros(1, 64, 1), torch.zeros(1, 64, 1))


def test_high_level_call_refuses_cpu_tensors(lib):
    # no CPU fallback behind the differentiable call either
    import torch
    q = torch.zeros(1, 64, 1, 64, requires_grad=True)
    with pytest.raises(gdr.GdrError):
        gdr.chunk_gated_delta_rule(q, q, q, torch.zeros(1, 64, 1), torch.zeros(1, 64, 1), output_final_state=True)


def test_plain_c_client_compiles_links_and_runs(lib, tmp_path):
    """include/gdr.h compiles as C11 and libgdr links with C linkage: a plain-C
    program calls the host-side entry points (no device needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(B.library_path())
    exe = str(tmp_path / "abi_smoke")
    src = os.path.join(ROOT, "tests", "c_abi", "abi_smoke.c")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), src,
                    "-o", exe, "-L", libdir, "-lgdr", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
