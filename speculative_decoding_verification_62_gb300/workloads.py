"""Seeded synthetic inputs for the verify step.

This module only draws inputs.  It holds none of the verify step's arithmetic
(no softmax, ratio, residual or inverse CDF): draft tokens are drawn from q by
the Gumbel-max trick (argmax of logits/T plus Gumbel noise), which samples
softmax(logits/T) exactly without forming it.  Both the CUDA path's tests and
the oracle consume the same bytes produced here.  Every draw runs on the CPU
with torch's CPU generator, whatever device the batch is then moved to, so a
workload name and seed always name the same bytes (the bench's GPU arm, its
CPU baseline and the reference arm hash identical inputs).

The five standard workloads restate the configurations of the verify-step
benchmark: vocabulary sizes of Llama-3-style (128256) and Qwen2.5-style
(152064) models, fixed or load-adaptive draft lengths, and acceptance rates in
the 0.3-0.9 range the pages report.  The pages' public prompt sets (MTBench,
ShareGPT, CNN/DailyMail, InstructCoder, WMT) are not used; these logits stand
in for them.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field

import torch

# name -> (B, G, V, dtype, description)
CONFIGS = {
    "1": dict(B=1, G=4, V=32000, dtype="f32",
              desc="B=1, gamma=4, V=32000, fp32, T=1.0; t~N(0,2^2), d=t+N(0,1)"),
    "2": dict(B=8, G=3, V=128256, dtype="bf16",
              desc="B=8, gamma=3, V=128256, bf16, T=0.8; t~N(0,3^2)+8 on 1%, d=t+N(0,0.7^2)"),
    "3": dict(B=64, G=5, V=152064, dtype="bf16",
              desc="B=64, gamma=5, V=152064, bf16, T=1.0; t=N(0,2.5^2)-1.1*ln(rank), "
                   "d=t+N(0,1.2^2), per-request seeds"),
    "4": dict(B=256, G=7, V=128256, dtype="bf16",
              desc="B=256, gamma_b~U{1..7}, V=128256, bf16, T=1.0; t~N(0,3^2), "
                   "d=t+N(0,sigma_b^2), sigma_b~U[0.3,2.0]"),
    "5a": dict(B=512, G=1, V=128256, dtype="bf16",
               desc="B=512, gamma=1, V=128256, bf16, T in {0.5,1.0,1.5}; t~N(0,3^2), d=t+N(0,1)"),
    "5b": dict(B=512, G=3, V=128256, dtype="bf16",
               desc="B=512, gamma=3, V=128256, bf16, T in {0.5,1.0,1.5}; t~N(0,3^2), d=t+N(0,1)"),
}


@dataclass
class Workload:
    """One batch of verify-step inputs (all tensors on one device)."""
    name: str
    target: torch.Tensor        # [B][G+1][V] float32 or bfloat16
    draft: torch.Tensor         # [B][G][V]
    draft_tokens: torch.Tensor  # [B][G] int32
    gamma: torch.Tensor         # [B] int32
    uniforms: torch.Tensor      # [B][G+1] float32 in [0,1)
    temperature: torch.Tensor   # [B] float32
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.target.shape[0]

    @property
    def G(self):
        return self.target.shape[1] - 1

    @property
    def V(self):
        return self.target.shape[2]

    @property
    def elem_bytes(self):
        return self.target.element_size()

    def gamma_sum(self) -> int:
        return int(self.gamma.sum().item())

    def bytes_min(self, mode: str = "sample") -> int:
        """One read of every valid logit row plus the small inputs and outputs."""
        gsum = self.gamma_sum()
        rows = (2 * gsum + self.B) if mode == "sample" else (gsum + self.B)
        small = self.B * (4 * self.G + 4 + 8) + self.B * 4 * (self.G + 2)
        if mode == "sample":
            small += self.B * 4 * (self.G + 1)
        return rows * self.V * self.elem_bytes + small

    def bytes_needed(self, mode: str, num_accepted, lazy: bool, ctas: int = 1) -> int:
        """The logit rows a call must read given its outcomes, plus the small
        inputs and outputs.  Read position by position (lazy), a sampled
        request with k accepted drafts needs target and draft rows
        0..min(k, gamma_b - 1) and, when k == gamma_b, the bonus row; a greedy
        request needs target rows 0..k.  In sampling mode the request-claims
        schedules (`ctas` CTAs, one per SM) read a sampled request lazily only
        in a batch of at least two requests per CTA, and then not when its rows
        alone reach 80 % of a CTA's share of the batch (such a request is read
        whole: 2 gamma_b + 1 rows); a request with T == 0 takes the greedy
        steps, target rows 0..k.  Read eagerly, every row: bytes_min()."""
        if not lazy:
            return self.bytes_min(mode)
        k = torch.as_tensor(num_accepted).cpu().to(torch.int64)
        g = self.gamma.cpu().to(torch.int64)
        if mode != "sample":
            small = self.B * (4 * self.G + 4 + 8) + self.B * 4 * (self.G + 2)
            return int((k + 1).sum().item()) * self.V * self.elem_bytes + small
        sampled = self.temperature.cpu() != 0
        full = torch.where(sampled, 2 * g + 1, g + 1)
        total = int(full.sum().item())
        by_stage = 2 * torch.minimum(k + 1, g) + (k == g).to(torch.int64)
        lazy_req = sampled & (5 * full * ctas < 4 * total) & (self.B >= 2 * ctas)
        rows = int(torch.where(lazy_req, by_stage, torch.where(sampled, full, k + 1)).sum().item())
        small = self.B * (4 * self.G + 4 + 8) + self.B * 4 * (self.G + 2) + self.B * 4 * (self.G + 1)
        return rows * self.V * self.elem_bytes + small

    def to(self, device):
        return Workload(self.name, *(getattr(self, k).to(device) for k in
                                     ("target", "draft", "draft_tokens", "gamma",
                                      "uniforms", "temperature")), dict(self.meta))

    def sha256(self) -> str:
        """SHA-256 of the input bytes (target, draft, draft tokens, gamma,
        uniforms, temperature in that order, each row-major), so that a
        measurement names exactly what it ran on."""
        h = hashlib.sha256()
        for k in ("target", "draft", "draft_tokens", "gamma", "uniforms", "temperature"):
            t = getattr(self, k).detach().contiguous().cpu()
            h.update(t.view(torch.uint8).numpy().tobytes() if t.numel() else b"")
        return h.hexdigest()


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gumbel_max_tokens(draft: torch.Tensor, temperature: torch.Tensor, gen) -> torch.Tensor:
    """Draw x ~ softmax(draft/T) per row by argmax(draft/T + Gumbel noise).

    Rows are processed one position at a time to bound temporary memory.
    """
    B, G, V = draft.shape
    out = torch.empty((B, G), dtype=torch.int32, device=draft.device)
    inv_t = (1.0 / temperature.float()).view(B, 1)
    for i in range(G):
        u = torch.rand((B, V), generator=gen, device=draft.device, dtype=torch.float32)
        u.clamp_(min=torch.finfo(torch.float32).tiny)
        g = -torch.log(-torch.log(u))
        out[:, i] = torch.argmax(draft[:, i, :].float() * inv_t + g, dim=1).to(torch.int32)
    return out


def _round(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def make(name: str, device="cpu", seed: int | None = None) -> Workload:
    """Build one of the standard workloads ("1", "2", "3", "4", "5a", "5b").

    The inputs are drawn on the CPU and then moved to `device`."""
    w = _make_cpu(name, seed)
    return w if torch.device(device) == torch.device("cpu") else w.to(device)


def _make_cpu(name: str, seed: int | None) -> Workload:
    device = "cpu"
    cfg = CONFIGS[name]
    B, G, V, dt = cfg["B"], cfg["G"], cfg["V"], cfg["dtype"]
    base = 620 + int(name[0]) if seed is None else int(seed)
    gen = _gen(device, base)
    f32 = dict(device=device, dtype=torch.float32)

    if name == "1":
        t = torch.randn((B, G + 1, V), generator=gen, **f32) * 2.0
        d = t[:, :G] + torch.randn((B, G, V), generator=gen, **f32)
        temp = torch.full((B,), 1.0, **f32)
        gamma = torch.full((B,), G, dtype=torch.int32, device=device)
    elif name == "2":
        t = torch.randn((B, G + 1, V), generator=gen, **f32) * 3.0
        peak = torch.rand((B, G + 1, V), generator=gen, **f32) < 0.01
        t = t + 8.0 * peak.float()
        d = t[:, :G] + 0.7 * torch.randn((B, G, V), generator=gen, **f32)
        temp = torch.full((B,), 0.8, **f32)
        gamma = torch.full((B,), G, dtype=torch.int32, device=device)
    elif name == "3":
        t = torch.empty((B, G + 1, V), **f32)
        d = torch.empty((B, G, V), **f32)
        for b in range(B):  # per-request seeds
            gb = _gen(device, base * 100003 + b)
            for i in range(G + 1):
                rank = torch.randperm(V, generator=gb, device=device).float() + 1.0
                t[b, i] = 2.5 * torch.randn((V,), generator=gb, **f32) - 1.1 * torch.log(rank)
            d[b] = t[b, :G] + 1.2 * torch.randn((G, V), generator=gb, **f32)
        temp = torch.full((B,), 1.0, **f32)
        gamma = torch.full((B,), G, dtype=torch.int32, device=device)
    elif name == "4":
        gamma = torch.randint(1, G + 1, (B,), generator=gen, device=device).to(torch.int32)
        sigma = 0.3 + 1.7 * torch.rand((B,), generator=gen, **f32)
        t = torch.randn((B, G + 1, V), generator=gen, **f32) * 3.0
        d = t[:, :G] + sigma.view(B, 1, 1) * torch.randn((B, G, V), generator=gen, **f32)
        temp = torch.full((B,), 1.0, **f32)
    elif name in ("5a", "5b"):
        t = torch.randn((B, G + 1, V), generator=gen, **f32) * 3.0
        d = t[:, :G] + torch.randn((B, G, V), generator=gen, **f32)
        temp = torch.tensor([0.5, 1.0, 1.5], **f32).repeat(math.ceil(B / 3))[:B].contiguous()
        gamma = torch.full((B,), G, dtype=torch.int32, device=device)
    else:
        raise KeyError(name)

    target, draft = _round(t, dt), _round(d, dt)
    del t, d
    tok_gen = _gen(device, base * 7919 + 1)
    tokens = gumbel_max_tokens(draft, temp, tok_gen)
    if name == "3":
        u = torch.empty((B, G + 1), **f32)
        for b in range(B):
            u[b] = torch.rand((G + 1,), generator=_gen(device, base * 100019 + b), **f32)
    else:
        u = torch.rand((B, G + 1), generator=_gen(device, base * 7919 + 2), **f32)
    for b in range(B):  # positions past gamma_b carry no draft
        tokens[b, int(gamma[b]):] = 0
    return Workload(name, target.contiguous(), draft.contiguous(), tokens.contiguous(),
                    gamma.contiguous(), u.contiguous(), temp.contiguous(),
                    dict(desc=cfg["desc"], seed=base, dtype=dt))


def make_random(B: int, G: int, V: int, dtype: str = "bf16", device="cpu", seed: int = 0,
                gamma=None, temperature=None, sigma_t: float = 3.0,
                sigma_d: float = 1.0) -> Workload:
    """Small generic workload: t ~ N(0, sigma_t^2), d = t + N(0, sigma_d^2).

    gamma: None (all G), "ragged" (U{0..G}), or an explicit list.
    temperature: None (1.0), a float, or a list of per-request values.
    Drawn on the CPU, then moved to `device`.
    """
    w = _make_random_cpu(B, G, V, dtype, seed, gamma, temperature, sigma_t, sigma_d)
    return w if torch.device(device) == torch.device("cpu") else w.to(device)


def _make_random_cpu(B, G, V, dtype, seed, gamma, temperature, sigma_t, sigma_d) -> Workload:
    device = "cpu"
    gen = _gen(device, seed)
    f32 = dict(device=device, dtype=torch.float32)
    t = torch.randn((B, G + 1, V), generator=gen, **f32) * sigma_t
    d = t[:, :G] + sigma_d * torch.randn((B, G, V), generator=gen, **f32)
    if gamma is None:
        g = torch.full((B,), G, dtype=torch.int32, device=device)
    elif isinstance(gamma, str) and gamma == "ragged":
        g = torch.randint(0, G + 1, (B,), generator=gen, device=device).to(torch.int32)
    else:
        g = torch.as_tensor(gamma, dtype=torch.int32, device=device).reshape(B)
    if temperature is None:
        temp = torch.ones((B,), **f32)
    elif isinstance(temperature, (int, float)):
        temp = torch.full((B,), float(temperature), **f32)
    else:
        temp = torch.as_tensor(temperature, **f32).reshape(B)
    target, draft = _round(t, dtype), _round(d, dtype)
    tokens = gumbel_max_tokens(draft, temp, _gen(device, seed * 7919 + 1)) if G > 0 else \
        torch.zeros((B, 0), dtype=torch.int32, device=device)
    for b in range(B):
        tokens[b, int(g[b]):] = 0
    u = torch.rand((B, G + 1), generator=_gen(device, seed * 7919 + 2), **f32)
    return Workload(f"random-B{B}-G{G}-V{V}-{dtype}", target.contiguous(), draft.contiguous(),
                    tokens.contiguous(), g.contiguous(), u.contiguous(), temp.contiguous(),
                    dict(seed=seed, dtype=dtype))


def logits_numpy(x: torch.Tensor):
    """Host copy of logits in the oracle's input form: float32, or bf16 bit patterns."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view("uint16")
    return x.numpy()


def oracle_inputs(w: Workload, requests=None):
    """Numpy arrays (optionally for a subset of requests) for the oracle."""
    idx = slice(None) if requests is None else torch.as_tensor(requests, dtype=torch.long)

    def pick(x):
        return x[idx.to(x.device)] if not isinstance(idx, slice) else x

    return dict(target=logits_numpy(pick(w.target)), draft=logits_numpy(pick(w.draft)),
                draft_tokens=pick(w.draft_tokens).cpu().numpy(),
                gamma=pick(w.gamma).cpu().numpy(),
                uniforms=pick(w.uniforms).cpu().numpy(),
                temperature=pick(w.temperature).cpu().numpy())


@dataclass
class Packed:
    """A workload in the packed (varlen) layout: rows back to back, no padding."""
    target: torch.Tensor        # [total + B][V]
    draft: torch.Tensor         # [total][V]
    cu_draft: torch.Tensor      # [B + 1] int32 prefix of the draft lengths
    draft_tokens: torch.Tensor  # [total] int32
    uniforms: torch.Tensor      # [total + B] float32: acceptance draws, then the final draw
    temperature: torch.Tensor   # [B]
    G: int

    @property
    def B(self):
        return self.cu_draft.numel() - 1

    @property
    def total(self):
        return self.draft_tokens.numel()


def pack(w: Workload) -> Packed:
    """Re-lay a padded workload out packed (data movement only)."""
    g = [int(x) for x in w.gamma.cpu().tolist()]
    if any(x < 0 or x > w.G for x in g):
        raise ValueError("gamma outside [0, G]")
    cu = [0]
    for x in g:
        cu.append(cu[-1] + x)
    dev = w.target.device
    target = torch.cat([w.target[b, :g[b] + 1] for b in range(w.B)], dim=0)
    if cu[-1]:
        draft = torch.cat([w.draft[b, :g[b]] for b in range(w.B)], dim=0)
        tokens = torch.cat([w.draft_tokens[b, :g[b]] for b in range(w.B)])
    else:
        draft = torch.empty((0, w.V), dtype=w.target.dtype, device=dev)
        tokens = torch.empty((0,), dtype=torch.int32, device=dev)
    uniforms = torch.cat([torch.cat([w.uniforms[b, :g[b]], w.uniforms[b, w.G:]]) for b in range(w.B)])
    return Packed(target.contiguous(), draft.contiguous(),
                  torch.tensor(cu, dtype=torch.int32, device=dev), tokens.contiguous(),
                  uniforms.contiguous(), w.temperature, w.G)


def unpack_per_draft(values: torch.Tensor, cu_draft: torch.Tensor, G: int, fill=float("nan")):
    """[total] per-draft values -> [B][G] padded with `fill` (data movement only)."""
    cu = [int(x) for x in cu_draft.cpu().tolist()]
    B = len(cu) - 1
    out = torch.full((B, G), fill, dtype=values.dtype, device=values.device)
    for b in range(B):
        n = cu[b + 1] - cu[b]
        out[b, :n] = values[cu[b]:cu[b + 1]]
    return out
