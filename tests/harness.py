"""Shared test harness: move a workload to the GPU, run the library, fetch
results, and compare with the fp64 oracle under the stated tolerances."""

from __future__ import annotations

import json
import os

import numpy as np

import oracle
import workloads as W

# Tolerances (max|gpu - ref| / max|ref| over the whole tensor):
#   o:  1e-2 for bf16 inputs, 1e-4 for fp32 inputs;
#   S1: 1e-4;
#   U:  1e-4 (U feeds S1 linearly, so it is held to the commit's bound).
TOL_O = {W.BF16: 1e-2, W.F32: 1e-4}
TOL_S1 = 1e-4
TOL_U = 1e-4


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.isfinite(ref)
    if not m.any():
        return 0.0
    den = np.abs(ref[m]).max()
    num = np.abs(gpu[m] - ref[m]).max()
    return float(num / max(den, 1e-30))


def ensure_state(w: W.Workload) -> W.Workload:
    """Workloads that carry warm-up draws get S0 from the oracle's recurrence."""
    if w.S0 is None:
        wu = w.warmup
        w.S0 = oracle.warmup_state(wu["k"], wu["v"], wu["log_alpha"], wu["beta"], w.Hv,
                                   w.dk, w.dv)
    return w


def to_device(w: W.Workload, device="cuda"):
    import torch
    dt = torch.bfloat16 if w.dtype == W.BF16 else torch.float32

    def t(x, dtype=None):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=dtype)

    return dict(q=t(w.q, dt), k=t(w.k, dt), v=t(w.v, dt), log_alpha=t(w.log_alpha),
                beta=t(w.beta), parent=t(w.parent), S0=t(w.S0), path=t(w.path),
                path_len=t(w.path_len))


def run_gpu(w: W.Workload, inplace: bool = False, with_parent: bool = True):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    x = to_device(w)
    st_v = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    st_c = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                     dev_status=st_v)
    S1 = gt.commit(x["path"], x["path_len"], U, x["k"], x["log_alpha"], x["S0"],
                   S1=x["S0"] if inplace else None,
                   parent=x["parent"] if with_parent else None, dev_status=st_c)
    torch.cuda.synchronize()
    return dict(o=o.float().cpu().numpy(), U=U.cpu().numpy(), S1=S1.cpu().numpy(),
                status_verify=st_v.cpu().numpy(), status_commit=st_c.cpu().numpy())


def run_oracle(w: W.Workload, units=None):
    o, U = oracle.verify_workload(w, mode="memo", units=units)
    S1 = oracle.commit_workload(w, units=units)
    return dict(o=o, U=U, S1=S1)


def unit_mask(w: W.Workload, units):
    """Boolean masks selecting the listed (b, h) units in o/U/S1 layouts."""
    sel = np.zeros((w.B, w.Hv), dtype=bool)
    for u in units:
        sel[u // w.Hv, u % w.Hv] = True
    return sel


def compare(w: W.Workload, gpu, ref, units=None):
    if units is not None:
        sel = unit_mask(w, units)
        o_g, o_r = gpu["o"].transpose(0, 2, 1, 3)[sel], ref["o"].transpose(0, 2, 1, 3)[sel]
        U_g, U_r = gpu["U"][sel], ref["U"][sel]
        S_g, S_r = gpu["S1"][sel], ref["S1"][sel]
    else:
        o_g, o_r, U_g, U_r, S_g, S_r = (gpu["o"], ref["o"], gpu["U"], ref["U"], gpu["S1"],
                                        ref["S1"])
    return dict(o=rel_err(o_g, o_r), U=rel_err(U_g, U_r), S1=rel_err(S_g, S_r))


def report(w: W.Workload, errs, tag: str = "") -> None:
    """Append the errors to $GDN_PARITY_REPORT (JSON lines) when set."""
    path = os.environ.get("GDN_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(workload=w.name, tag=tag, dtype=w.dtype,
                                    kernel=os.environ.get("GDN_TREE_KERNEL", "auto"),
                                    **errs)) + "\n")


def assert_parity(w: W.Workload, errs):
    report(w, errs)
    assert errs["o"] <= TOL_O[w.dtype], f"{w.name}: o rel err {errs['o']:.3e}"
    assert errs["U"] <= TOL_U, f"{w.name}: U rel err {errs['U']:.3e}"
    assert errs["S1"] <= TOL_S1, f"{w.name}: S1 rel err {errs['S1']:.3e}"
