"""Thin Python binding of the C ABI in include/gdn_cpr.h.

Argument marshalling only: torch tensors supply device memory and the current stream,
their data pointers go through ctypes, and every step of the operator runs in the CUDA
kernels of libgdn_cpr.so.  There is no fallback: if the library is missing or a call
fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# GDN_CPR_CHECKED=1 selects the bounds-checked debug build (build.build(checked=True))
LIB_PATH = os.path.join(HERE, "libgdn_cpr_checked.so" if os.environ.get("GDN_CPR_CHECKED") == "1"
                        else "libgdn_cpr.so")

GDN_F32, GDN_BF16 = 0, 1
MODE_PREFILL, MODE_DECODE, MODE_FWD, MODE_BWD, MODE_CONTINUE = 0, 1, 2, 3, 4
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
          4: "workspace missing, misaligned or too small", 5: "device-side error recorded"}
DEVERR = {0: "none", 1: "cu_seqlens mismatch", 2: "slot out of range", 3: "negative position",
          4: "bounded wait timed out", 5: "index range outside a buffer (bounds-checked build)",
          6: "host positions disagree with the cache (step skipped)"}

# every function the header declares (checked by the CPU test suite)
EXPORTS = ("gdn_cpr_version", "gdn_cpr_status_string", "gdn_cpr_workspace_size",
           "gdn_cpr_prefill", "gdn_cpr_decode_step", "gdn_cpr_fwd", "gdn_cpr_bwd",
           "gdn_cpr_get_device_error", "gdn_cpr_set_profile", "gdn_cpr_decode_step_noalloc",
           "gdn_cpr_policy_digest", "gdn_cpr_prefill_continue", "gdn_cpr_running_state",
           "gdn_cpr_noalloc_device_error", "gdn_cpr_test_wait_timeout", "gdn_cpr_decode_step_pos")
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class GdnError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("h_qk", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("chunk", ctypes.c_int32), ("in_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int)]


class CacheStruct(ctypes.Structure):
    _fields_ = [("s_run", ctypes.c_void_p), ("c_run", ctypes.c_void_p), ("s_bnd", ctypes.c_void_p),
                ("tail_k", ctypes.c_void_p), ("tail_v", ctypes.c_void_p),
                ("tail_g", ctypes.c_void_p), ("tail_beta", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("slots", ctypes.c_int32)]


class ProfileStruct(ctypes.Structure):
    _fields_ = [("events", ctypes.c_void_p * 16), ("n_events", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("kernels", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def load():
    """Load libgdn_cpr.so (built by __graft_entry__.build() / build.py).  Raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(LIB_PATH)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.gdn_cpr_version.restype = I
            lib.gdn_cpr_status_string.restype = ctypes.c_char_p
            lib.gdn_cpr_status_string.argtypes = [I]
            lib.gdn_cpr_workspace_size.argtypes = [P, I, P, ctypes.POINTER(S)]
            lib.gdn_cpr_prefill.argtypes = [P] * 14 + [S, P]
            lib.gdn_cpr_decode_step.argtypes = [P] * 10 + [S, P]
            lib.gdn_cpr_decode_step_pos.argtypes = [P] * 11 + [S, P]
            lib.gdn_cpr_decode_step_pos.restype = I
            lib.gdn_cpr_fwd.argtypes = [P] * 13 + [S, P]
            lib.gdn_cpr_bwd.argtypes = [P] * 19 + [S, P]
            lib.gdn_cpr_get_device_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
            lib.gdn_cpr_decode_step_noalloc.argtypes = [P] * 10
            lib.gdn_cpr_decode_step_noalloc.restype = I
            lib.gdn_cpr_set_profile.argtypes = [P]
            lib.gdn_cpr_set_profile.restype = None
            lib.gdn_cpr_policy_digest.argtypes = [P, P, P, S]
            lib.gdn_cpr_policy_digest.restype = I
            lib.gdn_cpr_prefill_continue.argtypes = [P] * 14 + [S, P]
            lib.gdn_cpr_prefill_continue.restype = I
            lib.gdn_cpr_running_state.argtypes = [P, P, P, ctypes.c_int32, P, P]
            lib.gdn_cpr_running_state.restype = I
            lib.gdn_cpr_noalloc_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
            lib.gdn_cpr_noalloc_device_error.restype = I
            lib.gdn_cpr_test_wait_timeout.argtypes = [ctypes.c_int32]
            lib.gdn_cpr_test_wait_timeout.restype = None
            for fn in ("gdn_cpr_workspace_size", "gdn_cpr_prefill", "gdn_cpr_decode_step",
                       "gdn_cpr_fwd", "gdn_cpr_bwd", "gdn_cpr_get_device_error"):
                getattr(lib, fn).restype = I
            _lib = lib
    return _lib


def _dt(x: torch.dtype) -> int:
    if x == torch.float32:
        return GDN_F32
    if x == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"unsupported dtype {x}")


def _tdt(code: int) -> torch.dtype:
    return torch.float32 if code == GDN_F32 else torch.bfloat16


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.numel() and not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(fn, rc):
    if rc != 0:
        raise GdnError(fn, rc)


def make_shape(num_seqs, total_tokens, h_qk, h_v, d, chunk, in_dtype, out_dtype) -> Shape:
    return Shape(int(num_seqs), int(total_tokens), int(h_qk), int(h_v), int(d), int(d),
                 int(chunk), _dt(in_dtype), _dt(out_dtype))


def policy_digest(d, chunk, in_dtype=torch.bfloat16, out_dtype=None, h_qk=1, h_v=1,
                  num_seqs=1, total_tokens=0):
    """gdn_cpr_policy_digest: (hex SHA-256 of the numerical policy, its canonical text)."""
    lib = load()
    shape = make_shape(num_seqs, total_tokens, h_qk, h_v, d, chunk, in_dtype,
                       in_dtype if out_dtype is None else out_dtype)
    dig = (ctypes.c_ubyte * 32)()
    buf = ctypes.create_string_buffer(4096)
    _check("gdn_cpr_policy_digest",
           lib.gdn_cpr_policy_digest(ctypes.byref(shape), dig, buf, ctypes.sizeof(buf)))
    return bytes(dig).hex(), buf.value.decode()


def _host_cu(cu_seqlens, cu_seqlens_host):
    if cu_seqlens_host is None:
        cu_seqlens_host = cu_seqlens.cpu()
    if not isinstance(cu_seqlens_host, torch.Tensor):
        cu_seqlens_host = torch.tensor(list(cu_seqlens_host), dtype=torch.int32)
    return cu_seqlens_host.to(torch.int32).contiguous()


def workspace_bytes(shape: Shape, mode: int, cu_host=None) -> int:
    lib = load()
    n = ctypes.c_size_t(0)
    cu = None if cu_host is None else _p(cu_host)
    _check("gdn_cpr_workspace_size", lib.gdn_cpr_workspace_size(ctypes.byref(shape), mode, cu,
                                                                 ctypes.byref(n)))
    return int(n.value)


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


class Cache:
    """Decode cache (see gdn_cpr_cache): running state (held as c_run * s_run, see
    running_state), boundary state, chunk tail, position.
    Also the full checkpoint of every decoding sequence: copying these tensors out and back
    resumes decoding bit-exactly."""

    def __init__(self, slots, h_qk, h_v, d, chunk, dtype=torch.bfloat16, device="cuda"):
        self.slots, self.h_qk, self.h_v, self.d, self.chunk, self.dtype = slots, h_qk, h_v, d, chunk, dtype
        self.s_run = torch.zeros((slots, h_v, d, d), dtype=torch.float32, device=device)
        self.c_run = torch.ones((slots, h_v), dtype=torch.float32, device=device)
        self.s_bnd = torch.zeros((slots, h_v, d, d), dtype=torch.float32, device=device)
        self.tail_k = torch.zeros((slots, chunk, h_qk, d), dtype=dtype, device=device)
        self.tail_v = torch.zeros((slots, chunk, h_v, d), dtype=dtype, device=device)
        self.tail_g = torch.zeros((slots, chunk, h_v), dtype=torch.float32, device=device)
        self.tail_beta = torch.zeros((slots, chunk, h_v), dtype=torch.float32, device=device)
        self.pos = torch.zeros((slots,), dtype=torch.int32, device=device)

    TENSORS = ("s_run", "c_run", "s_bnd", "tail_k", "tail_v", "tail_g", "tail_beta", "pos")

    def running_state(self, slots=None):
        """gdn_cpr_running_state: the explicit running state c_run * s_run of the given
        slots (a sequence or device tensor of indices; all slots if None), fp32
        [n, H_v, d, d], formed by the library as the kernels form state_out."""
        lib = load()
        dev = self.s_run.device
        if slots is None:
            sel, n = None, self.slots
        else:
            sel = torch.as_tensor(slots, device=dev).to(torch.int32).reshape(-1).contiguous()
            n = sel.numel()
        out = torch.empty((n, self.h_v, self.d, self.d), dtype=torch.float32, device=dev)
        shape = make_shape(n, n, self.h_qk, self.h_v, self.d, self.chunk, self.dtype, torch.float32)
        cs = self.struct()
        _check("gdn_cpr_running_state",
               lib.gdn_cpr_running_state(ctypes.byref(shape), ctypes.byref(cs), _p(sel), n, _p(out),
                                         _stream(dev)))
        if slots is not None and not isinstance(slots, torch.Tensor) and \
                not isinstance(slots, (list, tuple)):
            return out[0]  # a single slot index
        return out

    def struct(self) -> CacheStruct:
        return CacheStruct(*(_p(getattr(self, n)) for n in self.TENSORS), self.slots)

    def state_dict(self):
        return {n: getattr(self, n).detach().cpu().clone() for n in self.TENSORS}

    def load_state_dict(self, sd):
        for n in self.TENSORS:
            getattr(self, n).copy_(sd[n])


def prefill(q, k, v, g, beta, cu_seqlens, chunk=64, state_in=None, out_dtype=None,
            cache: Cache | None = None, slot_of_seq=None, cu_seqlens_host=None,
            want_state=True, ws=None, o=None, state_out=None):
    """gdn_cpr_prefill.  Returns (o, state_out)."""
    lib = load()
    cu_host = _host_cu(cu_seqlens, cu_seqlens_host)
    N = cu_host.numel() - 1
    T, hqk, d = k.shape
    hv = v.shape[1]
    od = out_dtype or q.dtype
    shape = make_shape(N, T, hqk, hv, d, chunk, q.dtype, od)
    if o is None:
        o = torch.empty((T, hv, d), dtype=od, device=q.device)
    if state_out is None and want_state:
        state_out = torch.empty((N, hv, d, d), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(shape, MODE_PREFILL, cu_host), q.device)
    cs = cache.struct() if cache is not None else None
    rc = lib.gdn_cpr_prefill(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta),
                             _p(state_in), _p(cu_seqlens), _p(cu_host), _p(o), _p(state_out),
                             ctypes.byref(cs) if cs is not None else None, _p(slot_of_seq),
                             _p(ws), ws.numel(), _stream(q.device))
    _check("gdn_cpr_prefill", rc)
    return o, state_out


def prefill_continue(q, k, v, g, beta, cu_seqlens, slots, cache: Cache, pos_host=None,
                     cu_seqlens_host=None, out_dtype=None, want_state=False, ws=None, o=None,
                     state_out=None):
    """gdn_cpr_prefill_continue: append the packed tokens of sequence i to cache slot
    slots[i] at its current position.  pos_host defaults to a host copy of cache.pos[slots]
    (a device read).  Returns (o, state_out)."""
    lib = load()
    cu_host = _host_cu(cu_seqlens, cu_seqlens_host)
    N = cu_host.numel() - 1
    T, hqk, d = k.shape
    hv = v.shape[1]
    od = out_dtype or q.dtype
    shape = make_shape(N, T, hqk, hv, d, cache.chunk, q.dtype, od)
    if pos_host is None:
        pos_host = cache.pos.index_select(0, slots.long()).cpu()
    if not isinstance(pos_host, torch.Tensor):
        pos_host = torch.tensor(list(pos_host), dtype=torch.int32)
    pos_host = pos_host.to(torch.int32).contiguous()
    if o is None:
        o = torch.empty((T, hv, d), dtype=od, device=q.device)
    if state_out is None and want_state:
        state_out = torch.empty((N, hv, d, d), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(shape, MODE_CONTINUE, cu_host), q.device)
    cs = cache.struct()
    rc = lib.gdn_cpr_prefill_continue(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta),
                                      _p(cu_seqlens), _p(cu_host), _p(slots), _p(pos_host),
                                      ctypes.byref(cs), _p(o), _p(state_out), _p(ws), ws.numel(),
                                      _stream(q.device))
    _check("gdn_cpr_prefill_continue", rc)
    return o, state_out


def fwd(q, k, v, g, beta, cu_seqlens, chunk=64, state_in=None, out_dtype=None,
        cu_seqlens_host=None, ws=None, o=None, state_out=None, saved_bnd=None):
    """gdn_cpr_fwd.  Returns (o, state_out, saved_bnd)."""
    lib = load()
    cu_host = _host_cu(cu_seqlens, cu_seqlens_host)
    N = cu_host.numel() - 1
    T, hqk, d = k.shape
    hv = v.shape[1]
    od = out_dtype or q.dtype
    shape = make_shape(N, T, hqk, hv, d, chunk, q.dtype, od)
    n_chunks = int(sum((int(cu_host[i + 1]) - int(cu_host[i]) + chunk - 1) // chunk for i in range(N)))
    if o is None:
        o = torch.empty((T, hv, d), dtype=od, device=q.device)
    if state_out is None:
        state_out = torch.empty((N, hv, d, d), dtype=torch.float32, device=q.device)
    if saved_bnd is None:
        saved_bnd = torch.empty((max(n_chunks, 1), hv, d, d), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(shape, MODE_FWD, cu_host), q.device)
    rc = lib.gdn_cpr_fwd(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta),
                         _p(state_in), _p(cu_seqlens), _p(cu_host), _p(o), _p(state_out),
                         _p(saved_bnd), _p(ws), ws.numel(), _stream(q.device))
    _check("gdn_cpr_fwd", rc)
    return o, state_out, saved_bnd[:n_chunks]


def decode_step(q, k, v, g, beta, slot, cache: Cache, out_dtype=None, ws=None, o=None, pos_host=None):
    """gdn_cpr_decode_step: one token per slot.  q,k [N,Hqk,d], v [N,Hv,d], g,beta [N,Hv],
    slot [N] int32 (device).  With pos_host (the host's copy of cache.pos[slot], a sequence
    or CPU tensor), gdn_cpr_decode_step_pos: the resync kernels are skipped when no token
    completes a chunk.  Returns o [N,Hv,d]."""
    lib = load()
    N, hqk, d = k.shape
    hv = v.shape[1]
    od = out_dtype or q.dtype
    shape = make_shape(N, N, hqk, hv, d, cache.chunk, q.dtype, od)
    if o is None:
        o = torch.empty((N, hv, d), dtype=od, device=q.device)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(shape, MODE_DECODE), q.device)
    cs = cache.struct()
    if pos_host is not None:
        ph = torch.as_tensor(pos_host, dtype=torch.int32).cpu().contiguous()
        rc = lib.gdn_cpr_decode_step_pos(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta),
                                         _p(slot), _p(ph), ctypes.byref(cs), _p(o), _p(ws), ws.numel(),
                                         _stream(q.device))
        _check("gdn_cpr_decode_step_pos", rc)
        return o
    rc = lib.gdn_cpr_decode_step(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta),
                                 _p(slot), ctypes.byref(cs), _p(o), _p(ws), ws.numel(),
                                 _stream(q.device))
    _check("gdn_cpr_decode_step", rc)
    return o


def decode_step_noalloc(q, k, v, g, beta, slot, cache: Cache, out_dtype=None, o=None):
    """gdn_cpr_decode_step_noalloc: the decode step with its workspace in the library's
    built-in device array, for callers that cannot allocate device memory.  The library
    allocates nothing; only the output `o`, if not given, is allocated here by torch."""
    lib = load()
    N, hqk, d = k.shape
    hv = v.shape[1]
    od = out_dtype or q.dtype
    shape = make_shape(N, N, hqk, hv, d, cache.chunk, q.dtype, od)
    if o is None:
        o = torch.empty((N, hv, d), dtype=od, device=q.device)
    cs = cache.struct()
    rc = lib.gdn_cpr_decode_step_noalloc(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g),
                                         _p(beta), _p(slot), ctypes.byref(cs), _p(o),
                                         _stream(q.device))
    _check("gdn_cpr_decode_step_noalloc", rc)
    return o


def bwd(q, k, v, g, beta, cu_seqlens, saved_bnd, dout, chunk=64, state_in=None,
        dstate_out=None, cu_seqlens_host=None, ws=None, want_dstate_in=True, out=None):
    """gdn_cpr_bwd.  Returns dict dq, dk, dv, dg, dbeta, dstate_in (fp32); `out`, if given, is
    such a dict of preallocated tensors to write into."""
    lib = load()
    cu_host = _host_cu(cu_seqlens, cu_seqlens_host)
    N = cu_host.numel() - 1
    T, hqk, d = k.shape
    hv = v.shape[1]
    shape = make_shape(N, T, hqk, hv, d, chunk, q.dtype, dout.dtype)
    dev = q.device
    if out is None:
        out = dict(dq=torch.empty((T, hqk, d), dtype=torch.float32, device=dev),
                   dk=torch.empty((T, hqk, d), dtype=torch.float32, device=dev),
                   dv=torch.empty((T, hv, d), dtype=torch.float32, device=dev),
                   dg=torch.empty((T, hv), dtype=torch.float32, device=dev),
                   dbeta=torch.empty((T, hv), dtype=torch.float32, device=dev),
                   dstate_in=torch.empty((N, hv, d, d), dtype=torch.float32, device=dev)
                   if want_dstate_in else None)
    if ws is None:
        ws = alloc_workspace(workspace_bytes(shape, MODE_BWD, cu_host), dev)
    rc = lib.gdn_cpr_bwd(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta),
                         _p(state_in), _p(cu_seqlens), _p(cu_host), _p(saved_bnd), _p(dout),
                         _p(dstate_out), _p(out["dq"]), _p(out["dk"]), _p(out["dv"]),
                         _p(out["dg"]), _p(out["dbeta"]), _p(out["dstate_in"]), _p(ws),
                         ws.numel(), _stream(dev))
    _check("gdn_cpr_bwd", rc)
    return out


def noalloc_device_error(device=None) -> int:
    """gdn_cpr_noalloc_device_error: synchronise the current stream and return the device
    error code of the last no-alloc decode step on the current device."""
    lib = load()
    dev = torch.device("cuda") if device is None else torch.device(device)
    code = ctypes.c_int32(0)
    rc = lib.gdn_cpr_noalloc_device_error(_stream(dev), ctypes.byref(code))
    if rc not in (0, 5):
        raise GdnError("gdn_cpr_noalloc_device_error", rc)
    return int(code.value)


def test_wait_timeout(calls: int) -> None:
    """gdn_cpr_test_wait_timeout (test hook): the next `calls` tensor-core prefills from
    this thread make one boundary-chain CTA's bounded wait run out."""
    load().gdn_cpr_test_wait_timeout(int(calls))


def device_error(ws: torch.Tensor) -> int:
    """Synchronise the current stream and return the device error code of `ws`."""
    lib = load()
    code = ctypes.c_int32(0)
    rc = lib.gdn_cpr_get_device_error(_p(ws), _stream(ws.device), ctypes.byref(code))
    if rc not in (0, 5):
        raise GdnError("gdn_cpr_get_device_error", rc)
    return int(code.value)


class Profiler:
    """Per-thread profiling hook (gdn_cpr_set_profile): the library records CUDA events at
    its stage boundaries on the launching stream and counts the kernels it launches.

    with Profiler(n_events=6) as p:
        api.prefill(...)
    p.stage_ms()  ->  [ms of stage 1, ms of stage 2, ...] of the last call (after a sync)
    p.kernels     ->  kernels launched by all calls made while active
    """

    def __init__(self, n_events: int = 8):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(n_events)]
        for e in self.events:  # creates the underlying cudaEvent_t
            e.record()
        self.struct = ProfileStruct()
        for i, e in enumerate(self.events):
            self.struct.events[i] = e.cuda_event
        self.struct.n_events = n_events
        self.struct.kernels = 0

    def __enter__(self):
        load().gdn_cpr_set_profile(ctypes.cast(ctypes.pointer(self.struct), ctypes.c_void_p))
        return self

    def __exit__(self, *exc):
        load().gdn_cpr_set_profile(None)
        return False

    @property
    def kernels(self) -> int:
        return int(self.struct.kernels)

    def stage_ms(self):
        n = int(self.struct.stages)
        return [self.events[i].elapsed_time(self.events[i + 1]) for i in range(n - 1)]
