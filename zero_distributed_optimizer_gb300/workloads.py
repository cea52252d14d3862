"""Synthetic workloads for the ZeRO-1 step: param size lists, weight-decay
masks, AdamW hyper-parameters and seeded generators of the step's inputs.

This module holds none of the step's arithmetic.  It only says what the
buffers look like and fills them with seeded random numbers; both the CUDA
path and the CPU oracle are fed from it.

Shapes follow the workloads described for the Megatron-LM distributed
optimizer ("04 · 分布式优化器", §3 ownership demo) and the model families the
tutorial pages discuss:

* ``toy_1000``: the page's ownership demo, one 1000-element buffer, DP 4,
  shard 250, five params of 130/260/90/310/210 elements.
* ``gpt2_small``: GPT-2 small (12 layers, hidden 768, vocab 50257, context
  1024, fused qkv, tied head), 124,439,808 elements, DP 8, 40 Mi buckets.
* ``llama_1p3b``: Llama-style 1.3B (24 layers, hidden 2048, SwiGLU 5632,
  RMSNorm, vocab 32000, untied), 1,364,297,728 elements, DP 8, 64 Mi buckets.
* ``sweep_256m``: 4096 params with log-uniform sizes on a 256 Mi buffer,
  DP in {1,2,4,8,16}, buckets in {1,4,16,64} Mi.
* ``moe_many_small``: 16 layers x 64 experts (two 512x1408 matrices each),
  router 2048x64 and two norms per layer (2096 tensors), fp32 grads, DP 8,
  scaling factor 1/32.

"Mi" is 2**20 elements.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field, replace

MI = 1 << 20


@dataclass(frozen=True)
class Workload:
    name: str
    sizes: tuple
    wd_mask: tuple          # 1: the param decays, 0: no weight decay
    D: int
    bucket_elems: int       # 0: one bucket
    pad_unit: int
    grad_dtype: str         # "bf16", "fp16" or "fp32"
    grad_dist: str          # "uniform1", "normal1e-3", "normal1e-3_outliers"
    m_init: str             # "zero" or "normal1e-4"
    v_init: str             # "zero" or "absnormal1e-6"
    steps: int
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    grad_scale: float = 1.0
    param_names: tuple = field(default=(), compare=False)

    @property
    def numel(self) -> int:
        """Unpadded element count N."""
        return int(sum(self.sizes))

    @property
    def grad_bytes(self) -> int:
        return 4 if self.grad_dtype == "fp32" else 2

    def adam_kwargs(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, grad_scale=self.grad_scale)

    def algorithmic_bytes_per_element(self) -> int:
        """Bytes one element moves: D grads read, master/m/v read+written,
        D 16-bit params written."""
        return self.D * self.grad_bytes + 24 + 2 * self.D

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def toy_1000() -> Workload:
    sizes = (130, 260, 90, 310, 210)
    return Workload("toy_1000", sizes, (1,) * 5, D=4, bucket_elems=0, pad_unit=1,
                    grad_dtype="bf16", grad_dist="uniform1", m_init="zero", v_init="zero",
                    steps=3, grad_scale=1.0 / 4, param_names=tuple(f"p{i}" for i in range(5)))


def gpt2_small() -> Workload:
    V, C, H, F, L = 50257, 1024, 768, 3072, 12
    names, sizes, wd = [], [], []

    def add(name, n, decays):
        names.append(name)
        sizes.append(n)
        wd.append(1 if decays else 0)

    add("wte", V * H, True)
    add("wpe", C * H, True)
    for i in range(L):
        add(f"h{i}.ln_1.weight", H, False)
        add(f"h{i}.ln_1.bias", H, False)
        add(f"h{i}.attn.c_attn.weight", H * 3 * H, True)
        add(f"h{i}.attn.c_attn.bias", 3 * H, False)
        add(f"h{i}.attn.c_proj.weight", H * H, True)
        add(f"h{i}.attn.c_proj.bias", H, False)
        add(f"h{i}.ln_2.weight", H, False)
        add(f"h{i}.ln_2.bias", H, False)
        add(f"h{i}.mlp.c_fc.weight", H * F, True)
        add(f"h{i}.mlp.c_fc.bias", F, False)
        add(f"h{i}.mlp.c_proj.weight", F * H, True)
        add(f"h{i}.mlp.c_proj.bias", H, False)
    add("ln_f.weight", H, False)
    add("ln_f.bias", H, False)
    return Workload("gpt2_small", tuple(sizes), tuple(wd), D=8, bucket_elems=40 * MI,
                    pad_unit=64, grad_dtype="bf16", grad_dist="normal1e-3", m_init="normal1e-4",
                    v_init="absnormal1e-6", steps=10, grad_scale=1.0 / 8,
                    param_names=tuple(names))


def llama_1p3b() -> Workload:
    V, H, F, L = 32000, 2048, 5632, 24
    names, sizes = [], []

    def add(name, n):
        names.append(name)
        sizes.append(n)

    add("embed_tokens", V * H)
    for i in range(L):
        add(f"l{i}.input_norm", H)
        for proj in ("q", "k", "v", "o"):
            add(f"l{i}.attn.{proj}_proj", H * H)
        add(f"l{i}.post_norm", H)
        for proj in ("gate", "up", "down"):
            add(f"l{i}.mlp.{proj}_proj", H * F)
    add("norm", H)
    add("lm_head", V * H)
    return Workload("llama_1p3b", tuple(sizes), (1,) * len(sizes), D=8, bucket_elems=64 * MI,
                    pad_unit=64, grad_dtype="bf16", grad_dist="normal1e-3_outliers",
                    m_init="zero", v_init="zero", steps=5, grad_scale=1.0 / 8,
                    param_names=tuple(names))


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return z ^ (z >> 31)


def sweep_sizes(count: int = 4096, total: int = 256 * MI, lo: int = 64, hi: int = 4 * MI,
                seed: int = 4096) -> tuple:
    """Log-uniform sizes on [lo, hi], scaled to sum to `total`, rounded and
    clamped to [lo, hi]; the residual goes to the largest param."""
    raw = []
    for i in range(count):
        u = (_splitmix64(seed * 1_000_003 + i) >> 11) / float(1 << 53)
        raw.append(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    scale = total / sum(raw)
    sizes = [min(hi, max(lo, int(round(r * scale)))) for r in raw]
    big = max(range(count), key=lambda i: sizes[i])
    sizes[big] += total - sum(sizes)
    if sizes[big] < lo:
        raise ValueError("residual made the largest param too small")
    return tuple(sizes)


def sweep_256m(D: int = 8, bucket_mi: int = 64) -> Workload:
    sizes = sweep_sizes()
    return Workload(f"sweep_256m_D{D}_b{bucket_mi}M", sizes, (1,) * len(sizes), D=D,
                    bucket_elems=bucket_mi * MI, pad_unit=64, grad_dtype="bf16",
                    grad_dist="normal1e-3", m_init="zero", v_init="zero", steps=3,
                    grad_scale=1.0 / D)


SWEEP_D = (1, 2, 4, 8, 16)
SWEEP_BUCKET_MI = (1, 4, 16, 64)


def moe_many_small() -> Workload:
    L, E, H = 16, 64, 2048
    names, sizes, wd = [], [], []
    for i in range(L):
        names += [f"l{i}.router", f"l{i}.norm1", f"l{i}.norm2"]
        sizes += [H * 64, H, H]
        wd += [0, 0, 0]
        for e in range(E):
            names += [f"l{i}.e{e}.w_in", f"l{i}.e{e}.w_out"]
            sizes += [512 * 1408, 1408 * 512]
            wd += [1, 1]
    return Workload("moe_many_small", tuple(sizes), tuple(wd), D=8, bucket_elems=64 * MI,
                    pad_unit=64, grad_dtype="fp32", grad_dist="normal1e-3", m_init="zero",
                    v_init="zero", steps=5, grad_scale=1.0 / 32, param_names=tuple(names))


def all_configs() -> list:
    """The five workloads, with the sweep at its D=8, 64 Mi point."""
    return [toy_1000(), gpt2_small(), llama_1p3b(), sweep_256m(8, 64), moe_many_small()]


# ---------------------------------------------------------------------------
# Seeded inputs (torch; the same call gives the same numbers on one device).
# ---------------------------------------------------------------------------

def seed_of(*parts) -> int:
    """Stable 63-bit seed from a tuple of names and numbers."""
    h = zlib.crc32("/".join(str(p) for p in parts).encode())
    return (h * 0x9E3779B1 + len(parts)) & 0x7FFFFFFFFFFFFFFF


def _gen(torch, device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_grads(w: Workload, numel: int, t: int, device="cpu", ranks=None):
    """Fresh replica gradients for step t: a list of D tensors of `numel`
    (padded) elements, bf16 or fp32, seeded by (workload, step, rank).
    Padding positions are filled like the rest; the step never reads them."""
    import torch

    out = []
    for r in (range(w.D) if ranks is None else ranks):
        g = _gen(torch, device, seed_of(w.name, "grad", t, r))
        if w.grad_dist == "uniform1":
            x = torch.rand(numel, generator=g, device=device, dtype=torch.float32) * 2 - 1
        else:
            x = torch.randn(numel, generator=g, device=device, dtype=torch.float32) * 1e-3
            if w.grad_dist == "normal1e-3_outliers":
                hit = torch.rand(numel, generator=g, device=device, dtype=torch.float32) < 0.01
                x = torch.where(hit, x * 100, x)
        out.append(_to_grad_dtype(torch, x, w.grad_dtype))
        del x
    return out


def make_state(w: Workload, numel: int, device="cpu"):
    """Initial fp32 master/m/v (buffer-indexed, `numel` padded elements)."""
    import torch

    g = _gen(torch, device, seed_of(w.name, "state"))
    master = torch.randn(numel, generator=g, device=device, dtype=torch.float32) * 0.02
    if w.m_init == "normal1e-4":
        m = torch.randn(numel, generator=g, device=device, dtype=torch.float32) * 1e-4
    else:
        m = torch.zeros(numel, device=device, dtype=torch.float32)
    if w.v_init == "absnormal1e-6":
        v = (torch.randn(numel, generator=g, device=device, dtype=torch.float32) * 1e-6).abs()
    else:
        v = torch.zeros(numel, device=device, dtype=torch.float32)
    return master, m, v


def make_params(master, D: int):
    """D bf16 param replicas, each the bf16 rounding of the initial master."""
    import torch

    p = master.to(torch.bfloat16)
    return [p.clone() for _ in range(D)]


def _to_grad_dtype(torch, x, grad_dtype: str):
    """fp32 draws cast to the grads' type ("bf16", "fp16" or "fp32")."""
    return x.to({"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[grad_dtype])


def random_case(numel: int, D: int, steps: int, grad_dtype: str = "bf16", seed: int = 0):
    """Seeded inputs for a small parity case (CPU tensors): fp32 master/m/v,
    D distinct random bf16 replicas (so untouched padding is visible) and
    per-step grads mixing magnitudes: N(0, 1e-3), 1% near 1, 1% zeros and
    1% below eps (1e-10)."""
    import torch

    g = _gen(torch, "cpu", seed_of("random_case", numel, D, seed))
    master = torch.randn(numel, generator=g) * 0.02
    m = torch.randn(numel, generator=g) * 1e-4
    v = (torch.randn(numel, generator=g) * 1e-6).abs()
    params = [(torch.randn(numel, generator=g) * 0.02).to(torch.bfloat16) for _ in range(D)]
    grads = []
    for _ in range(steps):
        per_rank = []
        for _ in range(D):
            x = torch.randn(numel, generator=g) * 1e-3
            u = torch.rand(numel, generator=g)
            x = torch.where(u < 0.01, x * 1000, x)
            x = torch.where((u >= 0.01) & (u < 0.02), torch.zeros_like(x), x)
            x = torch.where((u >= 0.02) & (u < 0.03), x * 1e-7, x)
            per_rank.append(_to_grad_dtype(torch, x, grad_dtype))
        grads.append(per_rank)
    return master, m, v, params, grads
