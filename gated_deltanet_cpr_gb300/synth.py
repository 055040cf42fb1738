"""Seeded synthetic inputs for the CPR Gated DeltaNet operator.

This module only draws random numbers; it contains none of the operator's arithmetic.
It is shared by the tests, the benchmark and the smoke check, and it is the only code
the CPU oracle and the CUDA path have in common.

Distributions (the workloads the IsoExec pages time are Qwen3.5-35B-A3B layers on
DAPO-Math-17k; neither weights nor data are available, so these seeded tensors stand in):
  q, k   ~ N(0, 1), L2-normalised per (token, head) over d_k in fp32, then cast
  v      ~ N(0, 1), cast to the input dtype
  beta   = sigmoid(N(0, 1))                       fp32
  g      = -softplus(N(0, 1))                     fp32  ("default" decay)
         = -0.02 * sigmoid(N(0, 1))               fp32  ("slow" decay: state carries memory)
  dO     ~ N(0, 1) in the output dtype (backward only)
Sequence lengths come from their own generator (seed + 1) so that the token tensors of a
batch do not depend on how its lengths were drawn.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

F32, BF16 = "f32", "bf16"
_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


@dataclass
class Workload:
    name: str
    lengths: list
    h_qk: int
    h_v: int
    d: int
    chunk: int
    dtype: str
    decode_steps: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))


def lengths_uniform(n: int, lo: int, hi: int, seed: int) -> list:
    gen = torch.Generator().manual_seed(seed + 1)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def lengths_loguniform(n: int, lo: int, hi: int, seed: int) -> list:
    gen = torch.Generator().manual_seed(seed + 1)
    u = torch.rand(n, generator=gen, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def workloads(seed: int = 0) -> dict:
    """The five named workloads (tiny, prefill, decode, trainer, long-context)."""
    return {
        "tiny": Workload("tiny B=1 H=2 T=256 d=32 C=16 fp32", [256], 2, 2, 32, 16, F32),
        "prefill": Workload("prefill B=4 T=4096 Hqk=16 Hv=32 d=128 C=64 bf16", [4096] * 4, 16, 32,
                            128, 64, BF16),
        "decode": Workload("decode 256 seqs x 2048 prefill + 128 steps Hqk=16 Hv=32 d=128 C=64 bf16",
                           [2048] * 256, 16, 32, 128, 64, BF16, decode_steps=128),
        "trainer": Workload("trainer fwd+bwd 8 seqs U[512,8192] Hqk=16 Hv=32 d=128 C=64 bf16",
                            lengths_uniform(8, 512, 8192, seed), 16, 32, 128, 64, BF16),
        "longctx": Workload("long context 64 seqs logU[128,32768] Hqk=16 Hv=32 d=128 C=64 bf16",
                            lengths_loguniform(64, 128, 32768, seed), 16, 32, 128, 64, BF16),
    }


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(lengths, h_qk: int, h_v: int, d_k: int, d_v: int | None = None,
                dtype: str = BF16, seed: int = 0, decay: str = "default",
                state_in: bool = False, dout: bool = False, out_dtype: str | None = None,
                device=None):
    """Draw one packed batch.  Returns a dict of tensors on `device` (default: the CPU):
    q, k [T,Hqk,dk] and v [T,Hv,dv] in `dtype`; g, beta [T,Hv] fp32; cu_seqlens [N+1] int32
    (always on the CPU); state_in [N,Hv,dv,dk] fp32 (N(0,1)/sqrt(dk)) or None; dout [T,Hv,dv]
    or None.  A device generator draws the same distributions but not the same values as
    the CPU one (used where the CPU would take too long to draw a large workload)."""
    d_v = d_k if d_v is None else d_v
    T = int(sum(lengths))
    dev = torch.device("cpu") if device is None else torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    td = _TORCH_DTYPE[dtype]

    def randn(shape):
        return torch.randn(shape, generator=gen, dtype=torch.float32, device=dev)

    def unit_rows(shape):
        x = randn(shape)
        return (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)).to(td)

    q = unit_rows((T, h_qk, d_k))
    k = unit_rows((T, h_qk, d_k))
    v = randn((T, h_v, d_v)).to(td)
    beta = torch.sigmoid(randn((T, h_v)))
    z = randn((T, h_v))
    if decay == "default":
        g = -torch.nn.functional.softplus(z)
    elif decay == "slow":
        g = -0.02 * torch.sigmoid(z)
    elif decay == "none":
        g = torch.zeros_like(z)
    else:
        raise ValueError(decay)
    out = dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(),
               cu_seqlens=cu_seqlens_of(lengths), state_in=None, dout=None)
    n = len(lengths)
    if state_in:
        out["state_in"] = randn((n, h_v, d_v, d_k)) / math.sqrt(d_k)
    if dout:
        od = _TORCH_DTYPE[out_dtype or dtype]
        out["dout"] = randn((T, h_v, d_v)).to(od)
    return out


def as_f64(x):
    """The exact values a kernel sees, widened to float64 numpy (None passes through)."""
    if x is None:
        return None
    return x.detach().to("cpu").to(torch.float64).numpy()
