"""Seeded synthetic inputs for the local MoE forward.

This module only draws random numbers and shapes them into the workloads'
structure (forced ties, poisoned rows, a per-expert logit bias).  It holds none
of the method's arithmetic and imports nothing else from this package, so the
CUDA path and the CPU oracle can both be fed from it.

Recipe (all workloads): a ``torch.Generator`` on the target device seeded with
the workload's seed draws, in this order, x ``[T,H]``, logits ``[T,E]``, then
gate, up and down one expert at a time (``e = 0..E-1``).  Each draw is FP32
``randn`` times its standard deviation, rounded to the storage dtype
(round-to-nearest-even, as torch casts).  Standard deviations: x and logits 1,
gate/up ``1/sqrt(H)``, down ``1/sqrt(I)``.  Structural choices (which rows are
poisoned, in which column) come from a CPU generator seeded with the same seed,
so they do not depend on the device.
"""
from __future__ import annotations

import dataclasses
import math

import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    E: int
    top_k: int
    H: int
    I: int
    dtype: str
    renormalize: bool
    seed: int
    forced_ties: bool = False      # the tiny workload's eight tied rows
    skew: float = 0.0              # per-expert logit bias skew * log(1/(e+1))
    poison_frac: float = 0.0       # fraction of rows holding NaN / +inf / all -inf

    @property
    def N(self) -> int:
        return self.T * self.top_k

    @property
    def flops(self) -> int:
        return 6 * self.T * self.top_k * self.H * self.I


# The five workloads: a tiny FP32 case, Mixtral-like shapes, the fine-grained
# headline case, a skewed-routing case with poisoned rows and a decode case.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=64, E=4, top_k=2, H=64, I=128, dtype="f32",
                          renormalize=True, seed=0, forced_ties=True),
    "mixtral_bf16": Workload("mixtral_bf16", T=4096, E=8, top_k=2, H=4096, I=14336,
                             dtype="bf16", renormalize=True, seed=1),
    "finegrained_bf16": Workload("finegrained_bf16", T=16384, E=64, top_k=6, H=2048, I=1408,
                                 dtype="bf16", renormalize=False, seed=2),
    "skewed_bf16": Workload("skewed_bf16", T=8192, E=128, top_k=8, H=2048, I=768,
                            dtype="bf16", renormalize=True, seed=3, skew=2.0, poison_frac=0.01),
    "decode_bf16": Workload("decode_bf16", T=32, E=256, top_k=8, H=7168, I=2048,
                            dtype="bf16", renormalize=True, seed=4),
}


def _randn(gen: torch.Generator, shape, std: float, dtype: str, device) -> torch.Tensor:
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v.to(TORCH_DTYPES[dtype])


def _force_ties(logits: torch.Tensor) -> None:
    """Overwrite rows 0..7 of a [T,4] logits tensor with exact ties."""
    rows = [
        [0.5, 0.5, 0.5, 0.5],        # all equal
        [0.0, 2.0, 2.0, -1.0],       # experts 1 and 2 equal and largest
        [3.0, 1.0, -2.0, 1.0],       # 2nd and 3rd largest equal (tie across the k=2 boundary)
        [2.0, 2.0, -1.0, 2.0],       # three equal at the top
        [-0.0, -1.0, 0.0, -2.0],     # -0.0 and +0.0 as the top two
        [0.1, 0.5, 0.5, 1.0],        # tie at the boundary, the largest has the highest id
        [0.0, 0.0, 0.0, 0.0],        # all equal at zero
        [1.0, 0.2, 0.3, 1.0],        # experts 3 and 0 tied for first
    ]
    assert logits.shape[1] == 4
    t = torch.tensor(rows, dtype=torch.float32).to(logits.dtype)
    logits[:8] = t.to(logits.device)


def _poison(logits: torch.Tensor, frac: float, seed: int) -> dict:
    """Make round(frac*T) rows hold NaN, +inf or only -inf (cycling), plus one
    control row with some (not all) -inf entries.  Returns the chosen rows."""
    T, E = logits.shape
    g = torch.Generator(device="cpu").manual_seed(seed)
    order = torch.randperm(T, generator=g)
    n = int(round(frac * T))
    cols = torch.randint(0, E, (n,), generator=g)
    rows = order[:n].tolist()
    kinds = []
    for i, r in enumerate(rows):
        kind = i % 3
        if kind == 0:
            logits[r, int(cols[i])] = float("nan")
        elif kind == 1:
            logits[r, int(cols[i])] = float("inf")
        else:
            logits[r, :] = float("-inf")
        kinds.append(("nan", "+inf", "all-inf")[kind])
    control = int(order[n]) if n < T else None
    if control is not None:
        logits[control, : max(1, E // 2)] = float("-inf")
    return {"rows": rows, "kinds": kinds, "control": control}


def make_routing_logits(T: int, E: int, dtype: str, seed: int, device="cpu",
                        skew: float = 0.0) -> torch.Tensor:
    """Router logits alone: FP32 ``randn`` from a generator seeded with ``seed``,
    plus the optional per-expert bias, rounded to ``dtype``."""
    gen = torch.Generator(device=device).manual_seed(seed)
    v = torch.randn((T, E), generator=gen, device=device, dtype=torch.float32)
    if skew:
        bias = skew * torch.log(1.0 / torch.arange(1, E + 1, device=device, dtype=torch.float32))
        v += bias
    return v.to(TORCH_DTYPES[dtype])


def make_inputs(w: Workload, device="cuda", weights: bool = True, logits_dtype: str | None = None):
    """Draw one workload.  Returns a dict with x, logits, gate, up, down (device
    tensors) and ``meta`` (poisoned rows etc.)."""
    gen = torch.Generator(device=device).manual_seed(w.seed)
    ldt = logits_dtype or w.dtype
    x = _randn(gen, (w.T, w.H), 1.0, w.dtype, device)
    lf = torch.randn((w.T, w.E), generator=gen, device=device, dtype=torch.float32)
    if w.skew:
        lf += w.skew * torch.log(1.0 / torch.arange(1, w.E + 1, device=device, dtype=torch.float32))
    logits = lf.to(TORCH_DTYPES[ldt])
    del lf
    meta = {}
    if w.forced_ties:
        _force_ties(logits)
    if w.poison_frac:
        meta["poison"] = _poison(logits, w.poison_frac, w.seed)
    out = {"x": x, "logits": logits, "meta": meta}
    if weights:
        tdt = TORCH_DTYPES[w.dtype]
        gate = torch.empty((w.E, w.I, w.H), dtype=tdt, device=device)
        up = torch.empty((w.E, w.I, w.H), dtype=tdt, device=device)
        down = torch.empty((w.E, w.H, w.I), dtype=tdt, device=device)
        sg = 1.0 / math.sqrt(w.H)
        sd = 1.0 / math.sqrt(w.I)
        for e in range(w.E):
            gate[e] = _randn(gen, (w.I, w.H), sg, w.dtype, device)
        for e in range(w.E):
            up[e] = _randn(gen, (w.I, w.H), sg, w.dtype, device)
        for e in range(w.E):
            down[e] = _randn(gen, (w.H, w.I), sd, w.dtype, device)
        out.update(gate=gate, up=up, down=down)
    return out


def with_dtype(w: Workload, dtype: str) -> Workload:
    """The same workload stored in another dtype (same seed and draws)."""
    if dtype == w.dtype:
        return w
    return dataclasses.replace(w, name=f"{w.name.rsplit('_', 1)[0]}_{dtype}", dtype=dtype)


def small_workload(T, E, top_k, H, I, dtype="bf16", renormalize=True, seed=0, **kw) -> Workload:
    """An ad-hoc workload for parity cases (several tiles plus ragged tails)."""
    return Workload(f"T{T}_E{E}_k{top_k}_H{H}_I{I}_{dtype}", T=T, E=E, top_k=top_k, H=H, I=I,
                    dtype=dtype, renormalize=renormalize, seed=seed, **kw)


def to_stored_numpy(t: torch.Tensor):
    """Host numpy view of a tensor's stored bits (BF16/F16 as uint16, F32 as float32)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view("uint16")
    raise TypeError(t.dtype)
