"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the
oracle.  This module draws random numbers and picks row samples; it holds
none of attention's arithmetic.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws Q, K, V and then
(when asked) dO, in that order, each ``torch.randn`` in fp32 of shape
[B, H, N, d] (iid N(0, 1)); for bf16 workloads each tensor is then rounded to
bf16 (round-to-nearest-even).  The same host tensors feed the GPU and, after
an exact widening to float64, the oracle.

The named workloads are the shapes the pages measure on (GPT-2 medium and
Llama-3.1-8B attention shapes, a long-context sweep and a training step),
filled with synthetic data: no dataset or trained weights are involved.
"""
import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "bf16" or "f32"
    scale: float
    causal: tuple       # causal settings the workload is run with
    passes: str         # "fwd" or "fwd+bwd"
    seed: int


def _w(name, B, H, N, d, dtype, causal, passes, seed):
    return Workload(name, B, H, N, d, dtype, 1.0 / math.sqrt(d), causal,
                    passes, seed)


# Seeds are 1000 + workload index (+ N for the long-context sweep).
WORKLOADS = {
    "single_head_f32": _w("single_head_f32", 1, 1, 256, 64, "f32", (False,),
                          "fwd", 1000),
    "gpt2_medium_fwd": _w("gpt2_medium_fwd", 8, 16, 1024, 64, "bf16",
                          (False, True), "fwd", 1001),
    "llama3_8b_fwd": _w("llama3_8b_fwd", 4, 32, 4096, 128, "bf16",
                        (False, True), "fwd", 1002),
    "long_ctx_8k": _w("long_ctx_8k", 1, 32, 8192, 128, "bf16", (True,), "fwd",
                      1003 + 8192),
    "long_ctx_16k": _w("long_ctx_16k", 1, 32, 16384, 128, "bf16", (True,),
                       "fwd", 1003 + 16384),
    "long_ctx_32k": _w("long_ctx_32k", 1, 32, 32768, 128, "bf16", (True,),
                       "fwd", 1003 + 32768),
    "train_fwd_bwd": _w("train_fwd_bwd", 8, 16, 2048, 128, "bf16", (True,),
                        "fwd+bwd", 1004),
    # head dimension 256 (the d^2/M wall): a 4096-token forward, and the
    # training step's shape at d = 256
    "d256_fwd": _w("d256_fwd", 2, 16, 4096, 256, "bf16", (False, True), "fwd",
                   1005),
    "d256_train": _w("d256_train", 4, 16, 2048, 256, "bf16", (True,),
                     "fwd+bwd", 1006),
}


def seeded_inputs(B, H, N, d, seed, dtype="bf16", with_dO=False):
    """Returns a dict of CPU tensors Q, K, V (and dO) of shape [B, H, N, d] in
    ``dtype`` ("bf16" or "f32"), drawn as the module docstring describes."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    names = ["Q", "K", "V"] + (["dO"] if with_dO else [])
    out = {}
    for n in names:
        t = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        out[n] = t.to(torch.bfloat16) if dtype == "bf16" else t
    return out


def seeded_inputs_cuda(B, H, N, d, seed, with_dO=False):
    """For tensors too large to draw on the host in reasonable time: Q, K, V
    (and dO) as bf16 CUDA tensors drawn by torch's seeded CUDA generator
    (``torch.randn`` in bf16, same order).  The oracle is given exact copies
    of the heads it checks."""
    g = torch.Generator(device="cuda")
    g.manual_seed(int(seed))
    names = ["Q", "K", "V"] + (["dO"] if with_dO else [])
    return {n: torch.randn((B, H, N, d), generator=g, device="cuda",
                           dtype=torch.bfloat16) for n in names}


def workload_inputs(w: Workload, with_dO=None):
    if with_dO is None:
        with_dO = w.passes == "fwd+bwd"
    return seeded_inputs(w.B, w.H, w.N, w.d, w.seed, w.dtype, with_dO)


E4M3_MAX = 448.0  # largest finite OCP FP8 E4M3 value


def e4m3_inputs(B, H, N, d, seed):
    """Q, K, V as E4M3 with per-tensor factors, for the 8-bit forward: the
    fp32 draws of ``seeded_inputs`` (same seed, same order), each divided by
    its factor amax/448 (rounded to an fp32 value, which both sides then use
    exactly) and rounded to E4M3 by torch (round to nearest even).
    Returns ({"Q": q8, "K": k8, "V": v8} as torch.float8_e4m3fn CPU tensors,
    {"Q": qd, "K": kd, "V": vd} the factors)."""
    x = seeded_inputs(B, H, N, d, seed, dtype="f32")
    out, fac = {}, {}
    for n in ("Q", "K", "V"):
        amax = float(x[n].abs().max())
        f = float(torch.tensor(amax / E4M3_MAX if amax > 0 else 1.0,
                               dtype=torch.float32))
        out[n] = (x[n] / f).to(torch.float8_e4m3fn)
        fac[n] = f
    return out, fac


def e4m3_to_f64(t, factor):
    """The values an E4M3 tensor stands for: exact widening times its factor
    (one rounding of the product in float64)."""
    return t.detach().to("cpu").to(torch.float32).to(torch.float64).numpy() * factor


def to_f64(t):
    """Exact widening of a bf16/fp32 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def sample_rows(B, H, N, per_head=512, seed=0, tile=128):
    """A seeded sample of flat row indices (b*H + h)*N + r, ``per_head`` rows
    per head (fewer when N is smaller): rows 0 and N-1, the rows on both sides
    of every ``tile`` boundary, and uniform random rows for the rest."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    fixed = {0, N - 1}
    for b in range(tile, N, tile):
        fixed.add(b - 1)
        fixed.add(b)
    fixed = sorted(r for r in fixed if 0 <= r < N)
    rows = []
    for bh in range(B * H):
        if N <= per_head:
            chosen = list(range(N))
        else:
            keep = fixed[:per_head]
            if len(fixed) > per_head:
                pick = torch.randperm(len(fixed), generator=g)[:per_head]
                keep = sorted(fixed[i] for i in pick.tolist())
            extra = per_head - len(keep)
            pool = torch.randint(0, N, (extra * 2 + 8,), generator=g).tolist()
            seen = set(keep)
            for r in pool:
                if extra == 0:
                    break
                if r not in seen:
                    seen.add(r)
                    keep.append(r)
                    extra -= 1
            chosen = sorted(keep)
        rows.extend(bh * N + r for r in chosen)
    return torch.tensor(rows, dtype=torch.int64)
