"""Seeded synthetic workloads: logits shaped like decode batches, plus per-row sampling parameters.

This module only draws inputs. It holds none of the sampler's arithmetic, so the CUDA path and
the float64 oracle can both be fed from it without sharing any of the method.

Every workload is a pure function of (name, seed, device, overrides). Random numbers come from a
``torch.Generator`` on the requested device; the CPU stream is what the parity tests use, the CUDA
stream is what the benchmark uses for multi-hundred-MB inputs.
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = ["Workload", "make", "NAMES", "describe"]


@dataclasses.dataclass
class Workload:
    name: str
    logits: torch.Tensor          # [B, V] float32 or bfloat16
    temperature: torch.Tensor     # [B] float32
    top_k: torch.Tensor           # [B] int32
    top_p: torch.Tensor           # [B] float32
    min_p: torch.Tensor           # [B] float32
    seed: torch.Tensor            # [B] int64 (read as uint64 by the library)
    step: int = 0

    @property
    def B(self) -> int:
        return int(self.logits.shape[0])

    @property
    def V(self) -> int:
        return int(self.logits.shape[1])

    def to(self, device) -> "Workload":
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
             for k, v in dataclasses.asdict(self).items()}
        return Workload(**f)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _distinct_positions(B, V, n, g, device):
    """n distinct random column indices per row ([B, n] int64)."""
    keys = torch.rand((B, V), generator=g, device=device)
    return torch.topk(keys, n, dim=1).indices


def _peaked_rows(B, V, g, device):
    """Four head logits 8, 3, 2, 1 at random distinct positions over an N(0, 1) tail."""
    z = torch.randn((B, V), generator=g, device=device)
    pos = _distinct_positions(B, V, 4, g, device)
    head = torch.tensor([8.0, 3.0, 2.0, 1.0], device=device).expand(B, 4)
    z.scatter_(1, pos, head)
    return z


def _flat_rows(B, V, g, device):
    """Logits evenly spaced from 1 down to 0 plus N(0, 0.01^2) noise."""
    base = torch.linspace(1.0, 0.0, V, device=device).expand(B, V)
    return base + 0.01 * torch.randn((B, V), generator=g, device=device)


def _seeds(B, device, base=1000):
    return (torch.arange(B, device=device, dtype=torch.int64) + base)


def cfg_small(device="cpu", seed=0, B=8, V=32000, dtype=torch.float32):
    """B=8, V=32,000 fp32 logits ~ N(0, 2^2); T cycles {0, 0.5, 1, 2}; top_p ~ U[0.05, 1]."""
    g = _gen(device, seed)
    z = 2.0 * torch.randn((B, V), generator=g, device=device)
    T = torch.tensor([0.0, 0.5, 1.0, 2.0], device=device).repeat(B // 4 + 1)[:B]
    p = 0.05 + 0.95 * torch.rand(B, generator=g, device=device)
    return Workload("small_b8_v32000_f32", z.to(dtype), T.float(), torch.zeros(B, dtype=torch.int32, device=device),
                    p.float(), torch.zeros(B, device=device), _seeds(B, device))


def cfg_mixed(device="cpu", seed=0, B=64, V=128256, dtype=torch.float32):
    """B=64, V=128,256: even rows peaked, odd rows flat; T ~ U[0.5, 1.5], top_p ~ U[0.5, 0.99];
    top_k = 50 on odd rows; min_p = 0.05 on every fourth row."""
    g = _gen(device, seed)
    peaked = _peaked_rows(B, V, g, device)
    flat = _flat_rows(B, V, g, device)
    odd = (torch.arange(B, device=device) % 2 == 1).unsqueeze(1)
    z = torch.where(odd, flat, peaked)
    T = 0.5 + torch.rand(B, generator=g, device=device)
    p = 0.5 + 0.49 * torch.rand(B, generator=g, device=device)
    r = torch.arange(B, device=device)
    k = torch.where(r % 2 == 1, 50, 0).to(torch.int32)
    m = torch.where(r % 4 == 0, 0.05, 0.0).float()
    return Workload("mixed_b64_v128256_f32", z.to(dtype), T.float(), k, p.float(), m, _seeds(B, device))


def cfg_ties_masked(device="cpu", seed=0, B=256, V=151936, dtype=torch.bfloat16, mask_frac=0.3):
    """B=256, V=151,936 bf16: a third integer logits {0..4} (heavy ties), a third N(0, 3^2), a third
    peaked; 30% of each row set to -inf (a grammar mask); top_p in {0.5, 0.9, 1}, T in {0, 0.7, 1}."""
    g = _gen(device, seed)
    ints = torch.randint(0, 5, (B, V), generator=g, device=device).float()
    normal = 3.0 * torch.randn((B, V), generator=g, device=device)
    peaked = _peaked_rows(B, V, g, device)
    r = torch.arange(B, device=device).unsqueeze(1)
    z = torch.where(r % 3 == 0, ints, torch.where(r % 3 == 1, normal, peaked))
    n_mask = int(round(mask_frac * V))
    if n_mask > 0:
        pos = _distinct_positions(B, V, n_mask, g, device)
        z.scatter_(1, pos, float("-inf"))
    choice = torch.randint(0, 3, (B,), generator=g, device=device)
    p = torch.tensor([0.5, 0.9, 1.0], device=device)[choice]
    choice_t = torch.randint(0, 3, (B,), generator=g, device=device)
    T = torch.tensor([0.0, 0.7, 1.0], device=device)[choice_t]
    return Workload("ties_masked_b256_v151936_bf16", z.to(dtype), T.float(),
                    torch.zeros(B, dtype=torch.int32, device=device), p.float(),
                    torch.zeros(B, device=device), _seeds(B, device))


def cfg_decode(device="cpu", seed=0, B=1024, V=128256, dtype=torch.float32, step=0):
    """Decode batch: B=1024, V=128,256 fp32 logits ~ N(0, 2.5^2) with a 20-token head offset by +6;
    every row T=0.7, top_k=50, top_p=0.9, min_p=0.05, distinct per-row seeds."""
    g = _gen(device, seed)
    z = 2.5 * torch.randn((B, V), generator=g, device=device)
    n_head = min(20, V)
    pos = _distinct_positions(B, V, n_head, g, device)
    z.scatter_add_(1, pos, torch.full((B, n_head), 6.0, device=device))
    full = lambda v, dt=torch.float32: torch.full((B,), v, dtype=dt, device=device)
    return Workload(f"decode_b{B}_v{V}_{'f32' if dtype == torch.float32 else 'bf16'}", z.to(dtype),
                    full(0.7), full(50, torch.int32), full(0.9), full(0.05), _seeds(B, device), step)


def cfg_sweep(device="cpu", seed=0, B=64, V=32000, dtype=torch.float32):
    """Sweep point: logits ~ N(0, 2^2); top_p ~ U[0.1, 1]; T ~ U[0.3, 2]; no top-k, no min-p."""
    g = _gen(device, seed)
    z = 2.0 * torch.randn((B, V), generator=g, device=device)
    p = 0.1 + 0.9 * torch.rand(B, generator=g, device=device)
    T = 0.3 + 1.7 * torch.rand(B, generator=g, device=device)
    tag = "f32" if dtype == torch.float32 else "bf16"
    return Workload(f"sweep_b{B}_v{V}_{tag}", z.to(dtype), T.float(),
                    torch.zeros(B, dtype=torch.int32, device=device), p.float(),
                    torch.zeros(B, device=device), _seeds(B, device))


_MAKERS = {
    "small": cfg_small,
    "mixed": cfg_mixed,
    "ties_masked": cfg_ties_masked,
    "decode": cfg_decode,
    "sweep": cfg_sweep,
}
NAMES = tuple(_MAKERS)

SWEEP_B = (1, 8, 64, 256, 1024, 4096)
SWEEP_V = (32000, 128256, 256000)


def make(name: str, device="cpu", seed: int = 0, **overrides) -> Workload:
    """Build a named workload; keyword overrides (B, V, dtype, ...) resize it for tests."""
    return _MAKERS[name](device=device, seed=seed, **overrides)


def describe(name: str) -> str:
    return (_MAKERS[name].__doc__ or "").strip()


def bytes_per_row(V: int, dtype: torch.dtype) -> int:
    """One read of the row plus the per-row parameters and the token written back."""
    elem = 4 if dtype == torch.float32 else 2
    return V * elem + 4 + 4 + 4 + 4 + 8 + 4


def tiny_grid(seed: int, n_batches: int = 300, rows: int = 4, max_v: int = 39):
    """Small-vocabulary batches (V in 1..max_v) for brute-force checks: temperatures {0, .5, 1, 2},
    top_p in [0.05, 1], a third of the batches on the five-value integer logit set so ties are
    common, plus random top_k / min_p on half the rows."""
    g = torch.Generator().manual_seed(int(seed))
    out = []
    temps = torch.tensor([0.0, 0.5, 1.0, 2.0])
    for bi in range(n_batches):
        V = int(torch.randint(1, max_v + 1, (1,), generator=g))
        if bi % 3 == 0:
            z = torch.randint(0, 5, (rows, V), generator=g).float()
        else:
            z = 2.0 * torch.randn((rows, V), generator=g)
        if bi % 7 == 3 and V > 1:
            mask = torch.rand((rows, V), generator=g) < 0.3
            z = z.masked_fill(mask, float("-inf"))
        T = temps[torch.randint(0, 4, (rows,), generator=g)]
        p = 0.05 + 0.95 * torch.rand(rows, generator=g)
        use = torch.rand(rows, generator=g) < 0.5
        k = torch.where(use, torch.randint(0, max(V, 1) + 2, (rows,), generator=g), 0).to(torch.int32)
        m = torch.where(torch.rand(rows, generator=g) < 0.3, 0.3 * torch.rand(rows, generator=g),
                        torch.zeros(rows))
        seeds = torch.randint(0, 2**62, (rows,), generator=g)
        out.append(Workload(f"tiny{bi}", z, T.float(), k, p.float(), m.float(), seeds, step=bi))
    return out



@dataclasses.dataclass
class PenaltyInputs:
    history: torch.Tensor     # [B, H] int32 token ids (-1 pads; a few ids >= V)
    hist_len: torch.Tensor    # [B] int32
    repetition: torch.Tensor  # [B] float32
    frequency: torch.Tensor   # [B] float32
    presence: torch.Tensor    # [B] float32


def penalty_inputs(B: int, V: int, H: int, device="cpu", seed: int = 0, bad_rows: int = 0) -> PenaltyInputs:
    """Token histories shaped like a decode batch's generated text: 70% of the entries come from a
    per-row pool of 32 ids (so tokens repeat), the rest uniformly from the vocabulary; 5% of the
    entries are -1 padding and 1% are ids >= V.  Lengths are uniform in [H/2, H].  Penalty values:
    repetition in [1, 1.5], frequency and presence in [0, 1].  The last `bad_rows` rows get an
    invalid penalty value (repetition 0 or -1, or a NaN/inf frequency or presence)."""
    g = _gen(device, seed + 7919)
    pool = torch.randint(0, V, (B, 32), generator=g, device=device)
    pick = torch.randint(0, 32, (B, H), generator=g, device=device)
    from_pool = torch.gather(pool, 1, pick)
    uniform = torch.randint(0, V, (B, H), generator=g, device=device)
    r = torch.rand((B, H), generator=g, device=device)
    hist = torch.where(r < 0.7, from_pool, uniform)
    hist = torch.where(r > 0.95, torch.full_like(hist, -1), hist)
    hist = torch.where((r > 0.94) & (r <= 0.95), hist + V, hist)
    lens = torch.randint(H // 2, H + 1, (B,), generator=g, device=device)
    rep = 1.0 + 0.5 * torch.rand(B, generator=g, device=device)
    freq = torch.rand(B, generator=g, device=device)
    pres = torch.rand(B, generator=g, device=device)
    bad = [(0.0, 0.0, 0.0), (-1.0, 0.0, 0.0), (1.2, float("nan"), 0.0), (1.2, 0.0, float("inf"))]
    for i in range(min(bad_rows, B)):
        rep[B - 1 - i], freq[B - 1 - i], pres[B - 1 - i] = bad[i % len(bad)]
    return PenaltyInputs(hist.to(torch.int32), lens.to(torch.int32), rep.float(), freq.float(), pres.float())
