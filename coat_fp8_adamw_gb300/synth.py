"""Seeded synthetic inputs for the fused FP8 AdamW + DRE step.

This module only draws random numbers: it holds none of the optimizer's or
the quantizer's arithmetic.  Both the CUDA path's tests/benchmark and the CPU
oracle's tests take their inputs from here.

The parameter sets stand in for the models the COAT paper-review page
(xllm-io) trains (section 5: OLMo-1B pretraining, Llama-2-7B memory and
throughput table; figure 1(c): Llama-2-13B).  No weights or datasets are
used: every tensor is drawn from the distributions listed per workload.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np

try:  # torch is only needed for the on-device generators
    import torch
except ImportError:  # pragma: no cover
    torch = None

#: AdamW hyper-parameters used by every workload
HYPER = dict(beta1=0.9, beta2=0.95, lr=1e-4, eps=1e-8, weight_decay=0.1)


@dataclasses.dataclass(frozen=True)
class Tensor:
    name: str
    numel: int
    is_norm: bool = False


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tensors: Tuple[Tensor, ...]
    G: int
    seed: int
    grad: str  # "tiny", "rowscale" or "lognormal"

    @property
    def n(self) -> int:
        return sum(t.numel for t in self.tensors)

    def offsets(self) -> List[int]:
        out, o = [], 0
        for t in self.tensors:
            out.append(o)
            o += t.numel
        return out


def _llama_like(name: str, layers: int, d: int, mlp: int, vocab: int, tied: bool,
                G: int, seed: int) -> Workload:
    ts: List[Tensor] = []
    for i in range(layers):
        for p in ("q", "k", "v", "o"):
            ts.append(Tensor(f"l{i}.{p}", d * d))
        for p in ("gate", "up", "down"):
            ts.append(Tensor(f"l{i}.{p}", d * mlp))
        ts.append(Tensor(f"l{i}.norm_attn", d, True))
        ts.append(Tensor(f"l{i}.norm_mlp", d, True))
    ts.append(Tensor("embed", vocab * d))
    if not tied:
        ts.append(Tensor("head", vocab * d))
    ts.append(Tensor("final_norm", d, True))
    return Workload(name, tuple(ts), G, seed, "lognormal")


def workload(name: str, G: Optional[int] = None) -> Workload:
    """The parameter sets.

    * ``tiny``     one tensor of 4096 params; g ~ N(0, 1e-3^2) with 1% x100
                   outliers; group 30 all-zero gradient, group 31 one non-zero.
    * ``mat4096``  one 4096x4096 matrix; row r has g ~ N(0, s_r^2),
                   s_r log-uniform in [1e-5, 1e-2].
    * ``mat16384`` one 16384x16384 matrix (3.8 GB of state: every access goes to
                   HBM, yet small enough for a full profiler capture); gradients
                   like the model-shaped sets (log-normal scale, 0.1% x1000).
    * ``olmo1b``   OLMo-1B-shaped: 16 layers, d=2048, MLP 8192, tied vocab 50304.
    * ``llama7b``  Llama-2-7B-shaped: 32 layers, d=4096, MLP 11008, vocab 32000.
    * ``llama13b`` Llama-2-13B-shaped: 40 layers, d=5120, MLP 13824, vocab 32000.
    """
    if name == "tiny":
        return Workload("tiny", (Tensor("w", 4096),), G or 128, 0, "tiny")
    if name == "mat4096":
        return Workload("mat4096", (Tensor("w", 4096 * 4096),), G or 128, 1, "rowscale")
    if name == "mat16384":
        return Workload("mat16384", (Tensor("w", 16384 * 16384),), G or 128, 5, "lognormal")
    if name == "olmo1b":
        return _llama_like("olmo1b", 16, 2048, 8192, 50304, True, G or 128, 2)
    if name == "llama7b":
        return _llama_like("llama7b", 32, 4096, 11008, 32000, False, G or 128, 3)
    if name == "llama13b":
        return _llama_like("llama13b", 40, 5120, 13824, 32000, False, G or 128, 4)
    raise KeyError(name)


WORKLOADS = ("tiny", "mat4096", "mat16384", "olmo1b", "llama7b", "llama13b")


# ---------------------------------------------------------------------------
# host (numpy) generators: small sizes, used directly by the oracle tests
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def init_weights_np(wl: Workload) -> np.ndarray:
    """fp32 master weights: N(0, 0.02^2); norm vectors are 1."""
    rng = np.random.default_rng([wl.seed, 0])
    w = (rng.standard_normal(wl.n) * 0.02).astype(np.float32)
    for off, t in zip(wl.offsets(), wl.tensors):
        if t.is_norm:
            w[off:off + t.numel] = 1.0
    return w


def _tensor_sigmas(wl: Workload) -> np.ndarray:
    rng = np.random.default_rng([wl.seed, 1])
    z = rng.standard_normal(len(wl.tensors))
    return 1e-3 * np.exp(1.5 * z)


def _row_sigmas(wl: Workload) -> np.ndarray:
    rng = np.random.default_rng([wl.seed, 2])
    return 10.0 ** rng.uniform(-5.0, -2.0, size=4096)


def grad_np(wl: Workload, step: int) -> np.ndarray:
    """bf16 gradient bits for ``step`` (host generator; small workloads)."""
    rng = np.random.default_rng([wl.seed, 100 + step])
    n = wl.n
    if wl.grad == "tiny":
        g = rng.standard_normal(n) * 1e-3
        out = rng.random(n) < 0.01
        g[out] *= 100.0
        G = wl.G
        g[30 * G:31 * G] = 0.0               # an all-zero group
        g[31 * G:32 * G] = 0.0               # a group with a single non-zero
        g[31 * G + 5] = 2.5e-3 * (1 + step % 3)
    elif wl.grad == "rowscale":
        s = np.repeat(_row_sigmas(wl), 4096)
        g = rng.standard_normal(n) * s
    else:
        g = np.empty(n)
        for off, t, sig in zip(wl.offsets(), wl.tensors, _tensor_sigmas(wl)):
            g[off:off + t.numel] = rng.standard_normal(t.numel) * sig
        out = rng.random(n) < 1e-3
        g[out] *= 1000.0
    return f32_to_bf16_bits(g.astype(np.float32))


def zero_state_np(n: int, G: int):
    """Initial optimizer state: all-zero codes, meta (S, k) = (0, 1) for both moments."""
    ng = (n + G - 1) // G
    meta = np.zeros((ng, 4), dtype=np.float32)
    meta[:, 1] = 1.0
    meta[:, 3] = 1.0
    return np.zeros(n, np.uint8), np.zeros(n, np.uint8), meta


def random_state_np(n: int, G: int, seed: int):
    """A synthetic non-zero optimizer state: random finite codes and random (S, k).

    m codes cover every finite E4M3 code of either sign; v codes are the
    finite non-negative codes.  log2 S_m ~ U[-90, -20], k_m ~ U[1, 8];
    log2 S_v ~ U[-110, -30], k_v ~ U[0.6, 4].
    """
    rng = np.random.default_rng([seed, 7])
    r = rng.integers(0, 254, size=n)
    mq = np.where(r < 127, r, r + 1).astype(np.uint8)       # skips 0x7F; 0xFF never drawn
    vq = rng.integers(0, 127, size=n).astype(np.uint8)
    ng = (n + G - 1) // G
    meta = np.empty((ng, 4), dtype=np.float32)
    meta[:, 0] = np.exp2(rng.uniform(-90.0, -20.0, ng))
    meta[:, 1] = rng.uniform(1.0, 8.0, ng)
    meta[:, 2] = np.exp2(rng.uniform(-110.0, -30.0, ng))
    meta[:, 3] = rng.uniform(0.6, 4.0, ng)
    return mq, vq, meta


# ---------------------------------------------------------------------------
# device (torch) generators: full-size parameter sets, drawn on the GPU
# ---------------------------------------------------------------------------

def _gen(device, seed: int):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def init_weights_torch(wl: Workload, device) -> "torch.Tensor":
    w = torch.empty(wl.n, dtype=torch.float32, device=device)
    w.normal_(0.0, 0.02, generator=_gen(device, wl.seed * 1000 + 1))
    for off, t in zip(wl.offsets(), wl.tensors):
        if t.is_norm:
            w[off:off + t.numel] = 1.0
    return w


def grad_torch(wl: Workload, step: int, device, out=None) -> "torch.Tensor":
    """bf16 gradient for ``step`` drawn on ``device`` (full-size workloads)."""
    n = wl.n
    gen = _gen(device, wl.seed * 1000003 + 17 * step + 5)
    if out is None:
        out = torch.empty(n, dtype=torch.bfloat16, device=device)
    chunk = 1 << 28
    if wl.grad == "rowscale":
        s = torch.from_numpy(_row_sigmas(wl).astype(np.float32)).to(device)
        for a in range(0, n, chunk):
            b = min(n, a + chunk)
            x = torch.randn(b - a, generator=gen, device=device, dtype=torch.float32)
            x.mul_(s.repeat_interleave(4096)[a:b])
            out[a:b] = x.to(torch.bfloat16)
        return out
    sig = _tensor_sigmas(wl) if wl.grad == "lognormal" else None
    offs = wl.offsets()
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        x = torch.randn(b - a, generator=gen, device=device, dtype=torch.float32)
        if sig is None:
            x.mul_(1e-3)
        else:
            scale = torch.empty(b - a, dtype=torch.float32, device=device)
            for off, t, s in zip(offs, wl.tensors, sig):
                lo, hi = max(a, off), min(b, off + t.numel)
                if lo < hi:
                    scale[lo - a:hi - a] = float(s)
            x.mul_(scale)
        u = torch.rand(b - a, generator=gen, device=device)
        x = torch.where(u < 1e-3, x * 1000.0, x)
        out[a:b] = x.to(torch.bfloat16)
    return out


def random_state_torch(n: int, G: int, seed: int, device):
    """Device version of :func:`random_state_np` (same distributions, torch RNG).

    Codes are drawn in chunks so that no full-size int32 temporary exists.
    """
    gen = _gen(device, seed * 7919 + 3)
    ng = (n + G - 1) // G
    mq = torch.empty(n, dtype=torch.uint8, device=device)
    vq = torch.empty(n, dtype=torch.uint8, device=device)
    chunk = 1 << 28
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        r = torch.randint(0, 254, (b - a,), generator=gen, device=device, dtype=torch.int32)
        mq[a:b] = torch.where(r < 127, r, r + 1).to(torch.uint8)
        r = torch.randint(0, 127, (b - a,), generator=gen, device=device, dtype=torch.int32)
        vq[a:b] = r.to(torch.uint8)
    meta = torch.empty(ng, 4, dtype=torch.float32, device=device)
    meta[:, 0] = torch.exp2(torch.empty(ng, device=device).uniform_(-90.0, -20.0, generator=gen))
    meta[:, 1] = torch.empty(ng, device=device).uniform_(1.0, 8.0, generator=gen)
    meta[:, 2] = torch.exp2(torch.empty(ng, device=device).uniform_(-110.0, -30.0, generator=gen))
    meta[:, 3] = torch.empty(ng, device=device).uniform_(0.6, 4.0, generator=gen)
    return mq, vq, meta


def adamw_like_moments_np(n: int, G: int, seed: int):
    """fp32 first and second moments coupled like real AdamW moments.

    Per group a gradient scale s is drawn log-uniform in [1e-6, 1e-2]; per
    element s_e = s exp(0.5 z); then m ~ 0.23 s_e N(0, 1) (the spread of an
    EMA with beta1 = 0.9 of i.i.d. gradients) and v ~ s_e^2 (0.5 + U[0, 1]).
    """
    rng = np.random.default_rng([seed, 31])
    ng = (n + G - 1) // G
    s = np.repeat(10.0 ** rng.uniform(-6, -2, ng), G)[:n]
    se = s * np.exp(0.5 * rng.standard_normal(n))
    m = (0.23 * se * rng.standard_normal(n)).astype(np.float32)
    v = (se * se * (0.5 + rng.random(n))).astype(np.float32)
    return m, v


def adamw_like_moments_torch(n: int, G: int, seed: int, device):
    """Device version of :func:`adamw_like_moments_np` (same distributions, torch RNG)."""
    import torch
    gen = _gen(device, seed * 7919 + 3)
    ng = (n + G - 1) // G
    s = torch.pow(10.0, torch.rand(ng, generator=gen, device=device) * 4.0 - 6.0)
    se = s.repeat_interleave(G)[:n] * torch.exp(0.5 * torch.randn(n, generator=gen, device=device))
    m = 0.23 * se * torch.randn(n, generator=gen, device=device)
    v = se * se * (0.5 + torch.rand(n, generator=gen, device=device))
    return m.float(), v.float()


def fp8_operand_codes_np(rows: int, cols: int, seed: int) -> np.ndarray:
    """E4M3 codes of a per-tensor-quantized linear-layer operand, uint8 [rows, cols]:
    a random sign and a magnitude code drawn around 0x58 (the value 16) with a
    spread of 10 codes (about 1.25 binades), clipped to the finite codes 0..0x7E,
    so that the largest values come near 448 as after an absmax scaling."""
    rng = np.random.default_rng([seed, 17])
    mag = np.clip(np.rint(rng.normal(88.0, 10.0, (rows, cols))), 0, 126).astype(np.uint8)
    sign = (rng.random((rows, cols)) < 0.5).astype(np.uint8) << 7
    return mag | sign


def sample_groups(num_groups: int, count: int, seed: int) -> np.ndarray:
    """Sorted sample of group indices: the first, the last and ``count`` random ones."""
    rng = np.random.default_rng([seed, 99])
    pick = rng.choice(num_groups, size=min(count, num_groups), replace=False)
    return np.unique(np.concatenate([pick, [0, num_groups - 1]])).astype(np.int64)


def human(n: float) -> str:
    for unit in ("", "K", "M", "G", "T"):
        if abs(n) < 1000:
            return f"{n:.3g}{unit}"
        n /= 1000.0
    return f"{n:.3g}P"

