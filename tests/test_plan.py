"""The host-side plan on the CPU (gdr_get_plan): which path a call takes and how
the intra-card context-parallel split cuts the sequences.  With no device
visible the library plans for 152 SMs, the GB300's count.  The plan never
changes a result (the split is exact); these tests pin its bookkeeping and
the choices the measured workloads rely on."""
import math

import pytest
import torch

import gated_deltanet_chunked_delta_gb300 as gdr
from gated_deltanet_chunked_delta_gb300 import binding as B


@pytest.fixture(scope="module", autouse=True)
def lib():
    from gated_deltanet_chunked_delta_gb300 import build
    build.build()
    return gdr.load()


def problem(B_=1, T=8192, Hq=4, Hv=8, K=128, V=128, lengths=None):
    if lengths is not None:
        B_, T = 1, sum(lengths)
    q = torch.empty(B_, T, Hq, K, device="meta")
    v = torch.empty(B_, T, Hv, V, device="meta")
    if lengths is None:
        return gdr.Problem(q, v)
    cu = torch.tensor([0] + [sum(lengths[:i + 1]) for i in range(len(lengths))], dtype=torch.int32)
    # the host-side query reads only the host copy; any non-null device pointer will do
    return gdr.Problem(q, v, cu_seqlens=cu, cu_seqlens_host=cu)


def plan(prob, dtype=B.GDR_BF16, **opts):
    return gdr.get_plan(prob, dtype, gdr.make_opts(**opts))


def segments_of(lengths, seg_len):
    return sum(max(1, math.ceil(math.ceil(n / 64) / seg_len)) for n in lengths)


def test_bench_workload_splits_to_fill_the_sms_once():
    # B=1, T=8192, Hv=8: 8 scans alone would use 8 of 152 SMs
    p = plan(problem())
    assert p["path"] == B.GDR_PATH_TC and p["n_chunks"] == 128
    assert p["n_segments"] == math.ceil(128 / p["seg_len"])
    # one scan CTA per (segment, v-head): a single wave that fills at least 90 % of the SMs
    assert 0.9 * 152 <= p["n_segments"] * 8 <= 152
    assert p["seg_len"] >= 4
    assert p["cp_warmup"] == 0  # segments shorter than four 8-chunk windows


def test_many_heads_need_no_split():
    # B=2, T=16384, Hv=64: 128 scans, a split would only add waves
    p = plan(problem(B_=2, T=16384, Hq=32, Hv=64))
    assert p["n_segments"] == 2 and p["seg_len"] == 256 and p["n_chunks"] == 512


def test_long_sequence_takes_warm_up_starts():
    p = plan(problem(T=262144, Hq=8, Hv=16))
    assert p["n_chunks"] == 4096 and p["n_segments"] > 1
    assert p["n_segments"] == math.ceil(4096 / p["seg_len"])
    assert p["seg_len"] >= 32 and p["cp_warmup"] == 8
    assert plan(problem(T=262144, Hq=8, Hv=16), cp_warmup=-1)["cp_warmup"] == 0
    assert plan(problem(T=262144, Hq=8, Hv=16), cp_warmup=3)["cp_warmup"] == 3


def _model(n_scans, maxc, nseg, warm_req=0, share=0.3, sms=152):
    # the planner's estimate in chunk steps, written out: the scan's waves times
    # the segment (with its warm-up chunks), the summary's waves for the share
    # of heads that run it (all of them without warm-up starts), the combine
    L = math.ceil(maxc / nseg)
    wc = 0 if nseg == 1 or warm_req < 0 else (warm_req if warm_req > 0 else (8 if L >= 32 else 0))
    f = share if wc > 0 else 1.0
    t = math.ceil(n_scans * nseg / sms) * (L + wc)
    if nseg > 1:
        t += math.ceil(2 * f * n_scans * nseg / sms) * L * 0.8 + 0.7 * nseg
    return t, L


def _best(n_scans, maxc, warm_req=0):
    best = None
    for nseg in range(1, 65):
        t, L = _model(n_scans, maxc, nseg, warm_req)
        if nseg > 1 and L < 4:
            break
        if best is None or t < best[0] - 1e-9:
            best = (t, L)
    return best[1]


@pytest.mark.parametrize("T,Hv,warm", [(262144, 16, 0), (262144, 16, -1), (32768, 16, 0), (8192, 8, 0),
                                       (16384 * 2, 64, 0), (65536, 4, 0)])
def test_split_follows_the_cost_model(T, Hv, warm):
    # with warm-up starts only the heads whose gates barely decay run the
    # summary, so the long forward takes more, shorter segments than the exact
    # split alone would (28 of 147 chunks against 19 of 216)
    p = plan(problem(T=T, Hq=max(1, Hv // 2), Hv=Hv), cp_warmup=warm)
    assert p["seg_len"] == _best(Hv, math.ceil(T / 64), warm)
    if (T, Hv) == (262144, 16):
        assert p["n_segments"] == (28 if warm == 0 else 19)


@pytest.mark.parametrize("n", [1, 2, 5, 19, 128, 500])
def test_forced_segment_count(n):
    p = plan(problem(), cp_segments=n)
    if n == 1:
        assert p["n_segments"] == 1 and p["seg_len"] == 128
    else:
        assert p["seg_len"] == max(1, math.ceil(128 / n))
        assert p["n_segments"] == math.ceil(128 / p["seg_len"])


def test_varlen_segments_cover_every_sequence():
    lengths = (1000, 0, 70000, 64, 1)
    p = plan(problem(Hq=2, Hv=4, lengths=lengths))
    assert p["n_chunks"] == sum(math.ceil(n / 64) for n in lengths)
    assert p["n_segments"] == segments_of(lengths, p["seg_len"])
    assert p["n_segments"] > len(lengths)  # 4 heads: the long sequence is split
    forced = plan(problem(Hq=2, Hv=4, lengths=lengths), cp_segments=1)
    assert forced["n_segments"] == len(lengths)


def test_path_follows_dtype_and_head_size():
    assert plan(problem(), B.GDR_F32)["path"] == B.GDR_PATH_SIMT
    assert plan(problem(K=64, V=64))["path"] == B.GDR_PATH_SIMT
    assert plan(problem(), path=B.GDR_PATH_SIMT)["path"] == B.GDR_PATH_SIMT
    # the CUDA-core split: two 32-column CTAs per SM, segments of at least 4 chunks
    p = plan(problem(), B.GDR_F32)
    assert p["seg_len"] >= 4 and p["n_segments"] == math.ceil(128 / p["seg_len"])
    assert p["cp_warmup"] == 0
    with pytest.raises(gdr.GdrError) as e:
        plan(problem(), B.GDR_F32, path=B.GDR_PATH_TC)
    assert e.value.code == 3


def test_bad_arguments():
    with pytest.raises(gdr.GdrError) as e:
        gdr.get_plan(problem(), 7)
    assert e.value.code == 3
    bad = B.gdr_shape(1, 64, 3, 4, 128, 128, 0, None, None)
    out = B.gdr_plan()
    assert gdr.load().gdr_get_plan(bad, 0, None, out) == 2


@pytest.mark.parametrize("K,V", [(128, 256), (192, 192), (64, 256), (192, 64)])
def test_wide_head_sizes_take_the_cuda_core_path(K, V):
    """Head sizes beyond 128 are accepted and planned on the CUDA-core path,
    bf16 inputs included (the tensor-core path takes K = V = 128 only)."""
    assert plan(problem(K=K, V=V))["path"] == B.GDR_PATH_SIMT
    assert plan(problem(K=K, V=V), B.GDR_F32)["path"] == B.GDR_PATH_SIMT
