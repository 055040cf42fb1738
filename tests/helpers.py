"""Shared helpers for the GPU tests: device transfer, error measures, oracle subsets."""
import numpy as np
import torch

import oracle
from gated_deltanet_cpr_gb300 import synth

f64 = synth.as_f64


def to_dev(x, dev="cuda"):
    return {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def rel_err(a, ref):
    """max |a - ref| / max |ref| (normwise, per tensor)."""
    a = a.detach().double().cpu().numpy() if isinstance(a, torch.Tensor) else np.asarray(a)
    ref = np.asarray(ref)
    den = np.abs(ref).max()
    return float(np.abs(a - ref).max() / (den if den > 0 else 1.0))


def oracle_full(x, chunk=0):
    return oracle.fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                      x["cu_seqlens"].numpy(), state_in=f64(x["state_in"]), chunk=chunk)


def oracle_pairs(x, pairs, chunk=0):
    """Oracle on selected (sequence, value head) pairs, each run as its own 1-head problem.
    Returns {(s, h): (o [L, d], state [d, d], bnd [nchunks, d, d] or None)}."""
    cu = x["cu_seqlens"].tolist()
    hqk, hv = x["k"].shape[1], x["v"].shape[1]
    grp = hv // hqk
    out = {}
    for s, h in pairs:
        a, b = cu[s], cu[s + 1]
        hq = h // grp
        sin = None if x["state_in"] is None else f64(x["state_in"][s:s + 1, h:h + 1])
        o, st, bnd = oracle.fwd(f64(x["q"][a:b, hq:hq + 1]), f64(x["k"][a:b, hq:hq + 1]),
                                f64(x["v"][a:b, h:h + 1]), f64(x["g"][a:b, h:h + 1]),
                                f64(x["beta"][a:b, h:h + 1]), [0, b - a], state_in=sin,
                                chunk=chunk)
        out[(s, h)] = (o[:, 0], st[0, 0], None if bnd is None else bnd[:, 0])
    return out
