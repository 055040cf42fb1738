"""Calls through the C ABI covering every kernel, for comparing the bounds-checked build with
the ordinary one (tests/test_gpu_checked.py).  run_cases returns CPU copies of every output
and the device error code of every call."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gated_deltanet_cpr_gb300 import api, synth  # noqa: E402


def _prefill(x, C, dev, out=torch.float32, cache=None):
    t = {n: (v.to(dev) if isinstance(v, torch.Tensor) else v) for n, v in x.items()}
    shape = api.make_shape(len(x["cu_seqlens"]) - 1, int(x["cu_seqlens"][-1]), x["k"].shape[1], x["v"].shape[1],
                           x["k"].shape[2], C, x["q"].dtype, out)
    ws = api.alloc_workspace(api.workspace_bytes(shape, api.MODE_PREFILL, x["cu_seqlens"]), dev)
    o, st = api.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                        state_in=t["state_in"], out_dtype=out, cache=cache, cu_seqlens_host=x["cu_seqlens"], ws=ws)
    return o, st, api.device_error(ws)


def run_cases(dev="cuda"):
    res, errs = {}, {}
    # prefill, tensor-core boundary path (bf16, d = 128, C = 64) and fp32 SIMT path (d = 64, C = 32)
    for name, (lengths, hqk, hv, d, C, dt) in {
            "tc": ([300, 64, 0, 130, 7], 2, 4, 128, 64, synth.BF16),
            "simt": ([100, 32, 3, 65], 2, 4, 64, 32, synth.F32)}.items():
        x = synth.make_inputs(lengths, hqk, hv, d, dtype=dt, seed=61, decay="slow", state_in=True, dout=True,
                              out_dtype=synth.F32)
        o, st, e = _prefill(x, C, dev)
        res[f"{name}_o"], res[f"{name}_state"], errs[f"{name}_prefill"] = o.cpu(), st.cpu(), e
        # trainer forward + backward
        t = {n: (v.to(dev) if isinstance(v, torch.Tensor) else v) for n, v in x.items()}
        o2, st2, saved = api.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                                 state_in=t["state_in"], out_dtype=torch.float32, cu_seqlens_host=x["cu_seqlens"])
        shape = api.make_shape(len(lengths), sum(lengths), hqk, hv, d, C, x["q"].dtype, torch.float32)
        ws = api.alloc_workspace(api.workspace_bytes(shape, api.MODE_BWD, x["cu_seqlens"]), dev)
        gr = api.bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], saved, t["dout"], chunk=C,
                     state_in=t["state_in"], cu_seqlens_host=x["cu_seqlens"], ws=ws)
        errs[f"{name}_bwd"] = api.device_error(ws)
        for k, v in gr.items():
            res[f"{name}_{k}"] = v.cpu()
        # decode through two resynchronisations, then a continued prefill, from a cache
        cache = api.Cache(2, hqk, hv, d, C, dtype=x["q"].dtype, device=dev)
        y = synth.make_inputs([2 * C - 3, C + 5], hqk, hv, d, dtype=dt, seed=62)
        _, _, e = _prefill(y, C, dev, cache=cache)
        errs[f"{name}_cache_prefill"] = e
        slots = torch.tensor([1, 0], dtype=torch.int32, device=dev)
        z = synth.make_inputs([2 * (C + 2)], hqk, hv, d, dtype=dt, seed=63)
        zt = {n: z[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
        shp = api.make_shape(2, 2, hqk, hv, d, C, x["q"].dtype, torch.float32)
        wsd = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_DECODE), dev)
        outs = []
        for i in range(C + 2):
            sl = slice(2 * i, 2 * i + 2)
            outs.append(api.decode_step(zt["q"][sl], zt["k"][sl], zt["v"][sl], zt["g"][sl], zt["beta"][sl],
                                        slots, cache, out_dtype=torch.float32, ws=wsd).cpu())
            errs[f"{name}_decode_{i}"] = api.device_error(wsd)
        res[f"{name}_decode_o"] = torch.stack(outs)
        c = synth.make_inputs([37, 70], hqk, hv, d, dtype=dt, seed=64)
        ct = {n: c[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
        shc = api.make_shape(2, 107, hqk, hv, d, C, x["q"].dtype, torch.float32)
        wsc = api.alloc_workspace(api.workspace_bytes(shc, api.MODE_CONTINUE, c["cu_seqlens"]), dev)
        oc, sc = api.prefill_continue(ct["q"], ct["k"], ct["v"], ct["g"], ct["beta"], c["cu_seqlens"].to(dev),
                                      slots, cache, cu_seqlens_host=c["cu_seqlens"], out_dtype=torch.float32,
                                      want_state=True, ws=wsc)
        errs[f"{name}_continue"] = api.device_error(wsc)
        res[f"{name}_continue_o"], res[f"{name}_continue_state"] = oc.cpu(), sc.cpu()
        for n in api.Cache.TENSORS:
            res[f"{name}_cache_{n}"] = getattr(cache, n).cpu()
    torch.cuda.synchronize()
    return res, errs


if __name__ == "__main__":
    out = sys.argv[1]
    r, e = run_cases()
    torch.save({"res": r, "errs": e, "lib": api.LIB_PATH}, out)
