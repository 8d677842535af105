"""Helpers shared by the GPU parity tests: run the C ABI through the binding
and the fp64 oracle on the same seeded inputs, and measure the error as
max|x - ref| / rms(ref) per tensor."""
import numpy as np
import torch

import oracle
from gated_deltanet_chunked_delta_gb300 import inputs

TOL = {"f32": 2e-3, "bf16": 2e-2}


# Unit roundoff of a stored bf16 value (8 significant bits, round to nearest).
BF16_U = 2.0 ** -8


# Every comparison made through err() during a test session, for the report
# that tests/conftest.py writes when GDR_PARITY_REPORT names a file:
# (test id, tensor, dtype, elements, err, raw_err).
RECORDS = []
CURRENT = {"test": "?"}


def err(x, ref, key=None):
    """max|x - ref| / rms(ref).  For a tensor stored in bf16 the stored value
    cannot be nearer to the fp64 result than its own rounding, so the error
    counted is what exceeds that rounding: max(|x - ref| - u |x|, 0).  The
    plain figure (raw_err) is recorded beside it."""
    slack = 0.0
    dt = "f64"
    if torch.is_tensor(x):
        dt = str(x.dtype).replace("torch.", "")
        if x.dtype == torch.bfloat16:
            slack = BF16_U * 1.01
        x = x.detach().float().cpu().double().numpy()
    else:
        x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if not x.size:
        return 0.0
    ad = np.abs(x - ref)
    d = np.maximum(ad - slack * np.abs(x), 0.0)
    rms = float(np.sqrt(np.mean(ref * ref)))
    e = float(np.max(d)) / rms if rms else float(np.max(d))
    raw = float(np.max(ad)) / rms if rms else float(np.max(ad))
    RECORDS.append((CURRENT["test"], key or f"#{len(RECORDS)}", dt, int(x.size), e, raw))
    return e


def raw_err(x, ref):
    """The plain max|x - ref| / rms(ref), rounding of the stored value included."""
    x = x.detach().float().cpu().double().numpy() if torch.is_tensor(x) else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) or 1.0
    return float(np.max(np.abs(x - ref))) / rms if x.size else 0.0


def write_report(path):
    """A markdown summary of every recorded comparison, both figures per tensor:
    the workload-sized checks row by row, then the largest figures of each
    test function over its parameters."""
    full = [r for r in RECORDS if "workload" in r[0]]
    lines = ["## Workload-sized checks", "",
             "| test | tensor | dtype | elements | err (beyond bf16 storage rounding) | raw max-abs / rms |",
             "|---|---|---|---|---|---|"]
    for t, k, dt, n, e, raw in full:
        lines.append(f"| {t} | {k} | {dt} | {n} | {e:.2e} | {raw:.2e} |")
    groups = {}
    for t, k, dt, n, e, raw in RECORDS:
        if "workload" in t:
            continue
        key = (t.split("[", 1)[0], k.split(" ")[0] if not k.startswith("#") else "?", dt)
        c, me, mr = groups.get(key, (0, 0.0, 0.0))
        groups[key] = (c + 1, max(me, e), max(mr, raw))
    lines += ["", "## Small-size checks: largest figures per test function and tensor", "",
              "| test function | tensor | dtype | comparisons | max err | max raw |", "|---|---|---|---|---|---|"]
    for (t, k, dt), (c, me, mr) in sorted(groups.items()):
        lines.append(f"| {t} | {k} | {dt} | {c} | {me:.2e} | {mr:.2e} |")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def _nans(shape, dtype, like):
    return torch.full(shape, float("nan"), dtype=dtype, device=like.device)


def _n_seqs(d):
    return d["cu_seqlens"].numel() - 1 if d["cu_seqlens"] is not None else d["v"].shape[0]


def gpu_fwd(gdr, d, **kw):
    """The forward into NaN-filled outputs, so that an element the kernels never
    write shows up as a parity failure."""
    if "out" not in kw:
        B, T, Hv, V = d["v"].shape
        K = d["q"].shape[-1]
        kw["out"] = {"o": _nans((B, T, Hv, V), kw.get("o_dtype") or d["q"].dtype, d["v"]),
                     "final_state": _nans((_n_seqs(d), Hv, K, V), torch.float32, d["v"]),
                     "A": _nans((B, T, Hv, 64), torch.float32, d["v"])}
        if kw.get("want_h"):
            if d["cu_seqlens"] is not None:
                lens = (d["cu_seqlens"][1:] - d["cu_seqlens"][:-1]).cpu()
                nt = int(((lens + 63) // 64).sum())
            else:
                nt = B * ((T + 63) // 64)
            kw["out"]["h"] = _nans((nt, Hv, K, V), torch.float32, d["v"])
    return gdr.gdr_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                       cu_seqlens=d["cu_seqlens"], **kw)


def gpu_bwd(gdr, d, A, **kw):
    """The backward into NaN-filled outputs (see gpu_fwd)."""
    if "out" not in kw:
        Hv, V = d["v"].shape[2:]
        K = d["q"].shape[-1]
        kw["out"] = {"dq": torch.full_like(d["q"], float("nan")), "dk": torch.full_like(d["k"], float("nan")),
                     "dv": torch.full_like(d["v"], float("nan")),
                     "dbeta": _nans(d["g"].shape, torch.float32, d["g"]),
                     "dg": _nans(d["g"].shape, torch.float32, d["g"]),
                     "dh0": _nans((_n_seqs(d), Hv, K, V), torch.float32, d["g"])}
    return gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], A, d["do"], dht=d.get("dht"),
                       scale=d["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"], **kw)


def oracle_fwd(x, want_h=False):
    return oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                      cu_seqlens=x["cu_seqlens"], want_h=want_h)


def oracle_bwd(x):
    return oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["do"], dht=x.get("dht"),
                      h0=x["h0"], cu_seqlens=x["cu_seqlens"])


def oracle_A(x):
    return oracle.A_matrix(x["k"], x["g"], x["beta"], cu_seqlens=x["cu_seqlens"])


def select_heads(x, hq):
    """Inputs restricted to qk-head hq and the v-heads of its group."""
    spec = x["spec"]
    G = spec.Hv // spec.Hq
    hv = slice(hq * G, (hq + 1) * G)
    y = dict(x)
    y["q"] = x["q"][:, :, hq:hq + 1].contiguous()
    y["k"] = x["k"][:, :, hq:hq + 1].contiguous()
    for key in ("v", "g", "beta", "do"):
        if key in x and x[key] is not None:
            y[key] = x[key][:, :, hv].contiguous()
    for key in ("h0", "dht"):
        if key in x and x[key] is not None:
            y[key] = x[key][:, hv].contiguous()
    return y, hv
