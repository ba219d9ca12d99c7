"""Seeded synthetic inputs for the verify step.

This module only draws random inputs; it holds none of the verify step's
arithmetic.  The same CPU tensors feed both the CUDA library and the CPU
oracle, so the two always see identical bytes.

Recipe (torch CPU generator, one stream per input, drawn in this order):
  stream 0: target logits  t[B, K+1, V] = target_std * N(0,1)  (+ an optional
            Zipf(s) log-prior  -s * ln(j + 1)  on token id j)
  stream 1: draft logits   d[B, K, V]   = t[:, :K] + draft_noise * N(0,1),
            or an independent  target_std * N(0,1)  draw
  stream 2: draft tokens   x[b, i] ~ softmax(d[b, i] / T) after the dtype cast
            (the draft model's own sampling), or, for the greedy workload,
            argmax(t[b, i] + greedy_noise * N(0,1)) over the fp32 target
  stream 3: uniforms       u[B, K+1] ~ U[0, 1), fp32
Stream k of seed s is ``torch.Generator().manual_seed(16 * s + k)``.
Logits are cast to the workload dtype (fp32 or bf16) once and then frozen.

Reward scores for Speculative Rejection's cut (``make_scores``, stream 4):
prompt g gets a shift mu_g = 2 * N(0,1) and a spread sigma_g = exp(0.5 * N(0,1))
(reward distributions differ a lot between prompts), and its N partial scores
are mu_g + sigma_g * N(0,1) in fp32; kind "ties" draws integers in [-3, 3]
instead (many equal scores, signed zeros included).
"""
from dataclasses import dataclass, field
from typing import Optional

import torch

MODE_SAMPLE = 0
MODE_GREEDY = 1


@dataclass
class Inputs:
    name: str
    mode: int
    B: int
    K: int
    V: int
    temperature: float
    target: torch.Tensor                 # [B, K+1, V] float32 or bfloat16 (CPU)
    draft: Optional[torch.Tensor]        # [B, K, V] or None (greedy)
    tokens: torch.Tensor                 # [B, K] int32
    uniforms: Optional[torch.Tensor]     # [B, K+1] float32 or None (greedy)
    recipe: dict = field(default_factory=dict)

    @property
    def dtype_name(self) -> str:
        return "bf16" if self.target.dtype == torch.bfloat16 else "f32"

    def algorithmic_bytes(self) -> int:
        """Bytes one verify call must move: every logit row read once, the
        tokens, the uniforms and the two outputs."""
        s = self.target.element_size()
        n = self.B * (self.K + 1) * self.V * s + self.B * self.K * 4
        n += self.B * 4 + self.B * (self.K + 1) * 4
        if self.mode == MODE_SAMPLE:
            n += self.B * self.K * self.V * s + self.B * (self.K + 1) * 4
        return n


def _gen(seed: int, k: int) -> torch.Generator:
    return torch.Generator().manual_seed(16 * seed + k)


def make_inputs(B, K, V, *, dtype=torch.float32, mode=MODE_SAMPLE, temperature=1.0,
                target_std=3.0, zipf_s=0.0, draft_noise=0.5, independent_draft=False,
                greedy_noise=1.0, seed=0, name=None) -> Inputs:
    """Draw one seeded batch following the recipe in the module docstring."""
    if K < 0 or B < 0 or V < 1:
        raise ValueError("need B >= 0, K >= 0, V >= 1")
    g_t, g_d, g_x, g_u = (_gen(seed, k) for k in range(4))
    t32 = torch.randn((B, K + 1, V), generator=g_t, dtype=torch.float32) * target_std
    if zipf_s:
        t32 += -zipf_s * torch.log(torch.arange(1, V + 1, dtype=torch.float32))
    target = t32.to(dtype).contiguous()
    draft = None
    uniforms = None
    if mode == MODE_SAMPLE:
        if independent_draft:
            d32 = torch.randn((B, K, V), generator=g_d, dtype=torch.float32) * target_std
        else:
            d32 = t32[:, :K] + draft_noise * torch.randn((B, K, V), generator=g_d,
                                                         dtype=torch.float32)
        draft = d32.to(dtype).contiguous()
        if K > 0 and B > 0:
            w = torch.softmax(draft.float().reshape(B * K, V) / temperature, dim=-1)
            tokens = torch.multinomial(w, 1, generator=g_x).reshape(B, K)
        else:
            tokens = torch.zeros((B, K), dtype=torch.int64)
        uniforms = torch.rand((B, K + 1), generator=g_u, dtype=torch.float32)
    else:
        noisy = t32[:, :K] + greedy_noise * torch.randn((B, K, V), generator=g_x,
                                                        dtype=torch.float32)
        tokens = noisy.argmax(dim=-1) if K > 0 else torch.zeros((B, 0), dtype=torch.int64)
    recipe = dict(target_std=target_std, zipf_s=zipf_s, draft_noise=draft_noise,
                  independent_draft=independent_draft, greedy_noise=greedy_noise,
                  seed=seed)
    return Inputs(name or f"B{B}_K{K}_V{V}", mode, B, K, V, float(temperature), target,
                  draft, tokens.to(torch.int32).contiguous(), uniforms, recipe)


# The five seeded workloads (B, K, V, dtype, logit statistics, temperature).
WORKLOADS = {
    "tiny_sample_f32_B4_K4_V1000": dict(
        B=4, K=4, V=1000, dtype=torch.float32, mode=MODE_SAMPLE, temperature=1.0,
        target_std=3.0, draft_noise=0.5),
    "greedy_bf16_B64_K8_V32000": dict(
        B=64, K=8, V=32000, dtype=torch.bfloat16, mode=MODE_GREEDY,
        target_std=4.0, greedy_noise=1.0),
    "sample_bf16_B64_K5_V128256_T1.0": dict(
        B=64, K=5, V=128256, dtype=torch.bfloat16, mode=MODE_SAMPLE, temperature=1.0,
        target_std=4.0, zipf_s=1.1, draft_noise=1.0),
    "sample_bf16_B64_K5_V128256_T0.7": dict(
        B=64, K=5, V=128256, dtype=torch.bfloat16, mode=MODE_SAMPLE, temperature=0.7,
        target_std=4.0, zipf_s=1.1, draft_noise=1.0),
    "best_of_n_bf16_B1024_K4_V32000": dict(
        B=1024, K=4, V=32000, dtype=torch.bfloat16, mode=MODE_SAMPLE, temperature=1.0,
        target_std=3.0, draft_noise=0.3),
    "long_draft_f32_B16_K16_V152064_T0.8": dict(
        B=16, K=16, V=152064, dtype=torch.float32, mode=MODE_SAMPLE, temperature=0.8,
        target_std=5.0, independent_draft=True),
}


def make_scd_inputs(B, K, V, *, dtype=torch.float32, temperature=1.0, target_std=3.0,
                    zipf_s=0.0, amateur_noise=1.0, independent_amateur=False, seed=0,
                    name=None) -> Inputs:
    """Inputs of speculative contrastive decoding's verify step: the expert's
    logits as make_inputs' target; the amateur's [B, K+1, V] logits (held in
    ``draft``) = the expert's + amateur_noise * N(0,1) (stream 5), or an
    independent target_std * N(0,1) draw; draft tokens drawn from
    softmax(amateur[:, :K] / T) after the dtype cast (stream 6); uniforms as
    make_inputs'."""
    base = make_inputs(B, K, V, dtype=dtype, temperature=temperature, target_std=target_std,
                       zipf_s=zipf_s, seed=seed, name=name)
    g_a, g_x = _gen(seed, 5), _gen(seed, 6)
    if independent_amateur:
        a32 = torch.randn((B, K + 1, V), generator=g_a, dtype=torch.float32) * target_std
    else:
        a32 = base.target.float() + amateur_noise * torch.randn((B, K + 1, V), generator=g_a,
                                                                dtype=torch.float32)
    amateur = a32.to(dtype).contiguous()
    if K > 0 and B > 0:
        w = torch.softmax(amateur[:, :K].float().reshape(B * K, V) / temperature, dim=-1)
        tokens = torch.multinomial(w, 1, generator=g_x).reshape(B, K)
    else:
        tokens = torch.zeros((B, K), dtype=torch.int64)
    recipe = dict(target_std=target_std, zipf_s=zipf_s, amateur_noise=amateur_noise,
                  independent_amateur=independent_amateur, seed=seed)
    return Inputs(name or f"scd_B{B}_K{K}_V{V}", MODE_SAMPLE, B, K, V, float(temperature),
                  base.target, amateur, tokens.to(torch.int32).contiguous(), base.uniforms, recipe)


# Speculative contrastive decoding on the sampling workload's shapes: the
# amateur is the expert plus N(0,1) noise, plausibility cut alpha = 0.1.
SCD_WORKLOADS = {
    "scd_bf16_B64_K5_V128256_T1.0_a0.1": dict(
        B=64, K=5, V=128256, dtype=torch.bfloat16, temperature=1.0, target_std=4.0,
        zipf_s=1.1, amateur_noise=1.0, alpha=0.1),
}


def make_scores(G: int, N: int, *, kind: str = "normal", seed: int = 0) -> torch.Tensor:
    """[G, N] float32 partial reward scores following the recipe above."""
    g = _gen(seed, 4)
    if kind == "normal":
        mu = 2.0 * torch.randn((G, 1), generator=g, dtype=torch.float64)
        sigma = torch.exp(0.5 * torch.randn((G, 1), generator=g, dtype=torch.float64))
        z = torch.randn((G, N), generator=g, dtype=torch.float64)
        return (mu + sigma * z).to(torch.float32).contiguous()
    if kind == "ties":
        v = torch.randint(-3, 4, (G, N), generator=g).to(torch.float32)
        neg0 = torch.rand((G, N), generator=g) < 0.5
        return torch.where((v == 0) & neg0, torch.full_like(v, -0.0), v).contiguous()
    raise ValueError(f"unknown score kind {kind!r}")


# Speculative Rejection's cut: G prompts of N = 1000 scored partial responses
# (the number of responses per prompt the review's Figure 2 uses), cut at
# alpha = 0.5.
REJECTION_WORKLOADS = {
    "rejection_cut_f32_G16384_N1000_a0.5": dict(G=16384, N=1000, alpha=0.5, kind="normal"),
}


def workload(name: str, seed: int = 0, B: Optional[int] = None) -> Inputs:
    """One of the named workloads; ``B`` overrides the batch (same statistics)."""
    kw = dict(WORKLOADS[name])
    if B is not None:
        kw["B"] = B
    return make_inputs(seed=seed, name=name, **kw)


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bfloat16 CPU tensor, as numpy."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def as_numpy_logits(t: Optional[torch.Tensor]):
    """fp32 logits as float32 numpy; bf16 logits as their uint16 bits."""
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.contiguous().numpy()
