"""Seeded synthetic inputs for the fused linear log-prob LM head.

This module only draws random numbers; it holds none of the method's
arithmetic, and both the CUDA path's tests/bench and the oracle consume what it
produces.  Every array is created on the CPU from a ``torch.Generator`` with a
fixed seed, normals drawn in fp32 and rounded to bf16 (round-to-nearest-even,
torch's conversion), so the same bytes can be copied to the GPU and handed to
the oracle.

Workloads (shapes from the Liger-Kernel native fused scaled linear
cross-entropy commit, "Performance methodology" and "Model-shape campaign",
and the SkyRL fused LM-head page, "H100 benchmark"):

* ``tiny``: M=256, H=256, V=4096; X ~ N(0,1), W ~ N(0, 0.02); 10% ignored
  targets; s = 1; entropy on; upstream grads 1/M on valid rows.
* ``m4096_h4096_v131072`` (the headline shape): X ~ N(0,1), W ~ N(0, 1/sqrt(H))
  (standard deviation); 5% ignored; s = 1; entropy on; N(0,1) grads.
* ``m8192_h8192_v131072``: same recipe, no ignored rows, s = 1/0.7
  (temperature 0.7), entropy off, N(0,1) grad on logprob only.
* ``ragged_m20001_h4096_v128257``: 1% of X rows (seeded choice) scaled by 50;
  5% ignored; entropy on; N(0,1) grads on both outputs.
* ``large_m32768_h5120_v152064``: targets drawn Zipf(1.1) over the vocabulary
  (P(k) proportional to (k+1)^-1.1, inverse CDF, no permutation), no ignored
  rows, entropy on, N(0,1) grads on both outputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

IGNORE_INDEX = -100


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    H: int
    V: int
    x_std: float = 1.0
    w_std: float | None = None  # None -> 1/sqrt(H)
    ignore_frac: float = 0.0
    scale: float = 1.0
    compute_entropy: bool = True
    grads: str = "normal"  # "normal" | "normal_lp" | "inv_m"
    hot_row_frac: float = 0.0
    hot_row_mult: float = 1.0
    targets: str = "uniform"  # "uniform" | "zipf"
    zipf_a: float = 1.1
    seed: int = 1000
    notes: dict = field(default_factory=dict)

    @property
    def flops_fwd(self) -> float:
        return 2.0 * self.M * self.H * self.V

    @property
    def flops_fwd_bwd(self) -> float:
        return 8.0 * self.M * self.H * self.V


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 256, 256, 4096, w_std=0.02, ignore_frac=0.10, grads="inv_m", seed=1001),
        Workload("m4096_h4096_v131072", 4096, 4096, 131072, ignore_frac=0.05, seed=1002),
        Workload("m8192_h8192_v131072", 8192, 8192, 131072, scale=1.0 / 0.7,
                 compute_entropy=False, grads="normal_lp", seed=1003),
        Workload("ragged_m20001_h4096_v128257", 20001, 4096, 128257, ignore_frac=0.05,
                 hot_row_frac=0.01, hot_row_mult=50.0, seed=1004),
        Workload("large_m32768_h5120_v152064", 32768, 5120, 152064, targets="zipf", seed=1005),
        # the headline recipe with a quarter of the vocabulary: every operand is
        # still larger than L2 but the device footprint stays near 1 GB, the
        # size used for full ncu captures of the kernels
        Workload("quarter_vocab_m4096_h4096_v32768", 4096, 4096, 32768, ignore_frac=0.05,
                 seed=1006),
        # the model-shape campaign of the native commit (M = 8192 tokens, random
        # inputs): small H makes the per-logit epilogue relatively heavier
        Workload("m8192_h2048_v151936", 8192, 2048, 151936, seed=1007),
        Workload("m8192_h5120_v202048", 8192, 5120, 202048, seed=1008),
        Workload("m8192_h7168_v129280", 8192, 7168, 129280, seed=1009),
    ]
}

HEADLINE = "m4096_h4096_v131072"
# the other synthetic workloads timed beside the headline (tiny, temperature 0.7, ragged, large)
REPORTED_WORKLOADS = ("tiny", "m8192_h8192_v131072", "ragged_m20001_h4096_v128257",
                      "large_m32768_h5120_v152064")


def custom(name: str, M: int, H: int, V: int, **kw) -> Workload:
    """A workload of another size with the same recipe knobs."""
    return Workload(name, M, H, V, **kw)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def make_inputs(w: Workload, seed: int | None = None, with_grads: bool = True) -> dict:
    """Draw X, W, targets and upstream grads on the CPU.

    Returns a dict of CPU tensors: X, W (bf16, contiguous), y (int64), g_lp and
    g_ent (fp32 or None), plus scale, ignore_index and compute_entropy.
    """
    seed = w.seed if seed is None else seed
    g = _gen(seed)
    M, H, V = w.M, w.H, w.V
    w_std = (1.0 / math.sqrt(H)) if w.w_std is None else w.w_std
    X = torch.randn(M, H, generator=g, dtype=torch.float32) * w.x_std
    if w.hot_row_frac > 0 and M > 0:
        n_hot = max(1, int(round(w.hot_row_frac * M)))
        hot = torch.randperm(M, generator=g)[:n_hot]
        X[hot] *= w.hot_row_mult
    X = X.to(torch.bfloat16).contiguous()
    W = (torch.randn(V, H, generator=g, dtype=torch.float32) * w_std).to(torch.bfloat16).contiguous()
    if w.targets == "zipf":
        ranks = torch.arange(1, V + 1, dtype=torch.float64)
        pmf = ranks.pow(-w.zipf_a)
        cdf = torch.cumsum(pmf, 0)
        cdf = cdf / cdf[-1]
        u = torch.rand(M, generator=g, dtype=torch.float64)
        y = torch.searchsorted(cdf, u).clamp_(max=V - 1).to(torch.int64)
    else:
        y = torch.randint(0, V, (M,), generator=g, dtype=torch.int64)
    if w.ignore_frac > 0 and M > 0:
        drop = torch.rand(M, generator=g) < w.ignore_frac
        y[drop] = IGNORE_INDEX
    out = dict(X=X, W=W, y=y.contiguous(), scale=float(w.scale), ignore_index=IGNORE_INDEX,
               compute_entropy=bool(w.compute_entropy), g_lp=None, g_ent=None)
    if with_grads:
        valid = (y != IGNORE_INDEX)
        if w.grads == "inv_m":
            g_lp = valid.to(torch.float32) / max(M, 1)
            g_ent = g_lp.clone() if w.compute_entropy else None
        else:
            g_lp = torch.randn(M, generator=g, dtype=torch.float32)
            g_ent = (torch.randn(M, generator=g, dtype=torch.float32)
                     if (w.compute_entropy and w.grads == "normal") else None)
        out["g_lp"] = g_lp.contiguous()
        out["g_ent"] = None if g_ent is None else g_ent.contiguous()
    return out


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a CPU bf16 tensor, as a numpy array."""
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def sample_rows(M: int, n: int, seed: int = 7) -> torch.Tensor:
    """A seeded sample of row indices that always includes the first and last
    row and the rows around 128-row tile boundaries near the end."""
    g = _gen(seed)
    base = torch.randperm(M, generator=g)[: max(0, min(n, M))]
    extra = [0, M - 1]
    if M > 129:
        t = (M - 1) // 128 * 128
        extra += [t - 1, t]
    idx = torch.unique(torch.cat([base, torch.tensor([e for e in extra if 0 <= e < M],
                                                     dtype=torch.int64)]))
    return idx
