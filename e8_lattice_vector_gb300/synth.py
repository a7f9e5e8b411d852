"""Seeded synthetic KV caches shaped like the method's model caches.

This module only draws random numbers: it holds none of the codec's
arithmetic and is shared, as plain input data, by the tests, the benchmark and
the smoke check.  The models and datasets the method was measured on
(Mistral-7B, Phi-3-mini, Llama-3.1-8B, Qwen2.5-14B on wikitext-2 / C4) are not
available here; these caches stand in for them with the same shapes (plus one
head_dim-64 cache shaped like Llama-3.2-1B's, for the head_dim-64 kernels).

Recipe, per layer l (generator seeded with seed * 1000 + l on the target
device):
  K: z ~ N(0, 1) [batch, heads, tokens, head_dim], times a per-(head, channel)
     scale exp(sigma * N(0, 1)); the first ceil(p * head_dim) channels of a
     seeded permutation per head are multiplied by `outlier_mult` (p =
     outlier_frac).  Then the model's own rotary embedding is applied
     (split-half, base theta, positions 0..T-1, fp32 like a HF forward pass), and
     the result is cast to fp16.
  V: N(0, 1), or Student-t with 5 degrees of freedom scaled to unit variance.
"""
import math
from dataclasses import dataclass, field

import torch

from .codec import CodecParams


@dataclass(frozen=True)
class CacheConfig:
    name: str
    layers: int
    batch: int
    kv_heads: int
    tokens: int
    head_dim: int
    sigma: float
    outlier_frac: float
    outlier_mult: float
    theta: float
    v_dist: str  # "normal" | "student_t5"
    seed: int
    modes: tuple = field(default_factory=tuple)  # CodecParams served on this cache

    @property
    def shape(self):
        return (self.layers, self.batch, self.kv_heads, self.tokens, self.head_dim)

    @property
    def rows(self):
        return self.layers * self.batch * self.kv_heads * self.tokens

    @property
    def fp16_bytes(self):
        """fp16 K + V bytes."""
        return 2 * self.rows * self.head_dim * 2


def _p(kb, vb, strict, delta, theta):
    return CodecParams(key_bits=kb, value_bits=vb, group_size=64, strict=strict, delta_chunk=delta,
                       rope_theta=theta)


CONFIGS = {
    "tiny": CacheConfig("tiny", 1, 1, 8, 512, 128, 0.5, 0.0, 1.0, 1e4, "normal", 0,
                        (_p(3, 2, False, 0, 1e4),)),
    "mistral7b": CacheConfig("mistral7b", 32, 1, 8, 4096, 128, 0.7, 0.02, 8.0, 1e4, "normal", 1,
                             (_p(2, 2, True, 0, 1e4), _p(2, 2, False, 0, 1e4))),
    "phi3mini": CacheConfig("phi3mini", 32, 2, 32, 2048, 96, 0.5, 0.0, 1.0, 1e4, "normal", 2,
                            (_p(3, 2, False, 256, 1e4),)),
    "llama31_8b": CacheConfig("llama31_8b", 32, 4, 8, 32768, 128, 0.7, 0.0, 1.0, 5e5, "student_t5", 3,
                              (_p(2, 2, False, 0, 5e5), _p(2, 2, True, 0, 5e5))),
    # head_dim 64 (the shape of Llama-3.2-1B's cache: 16 layers, 8 KV heads), for the kernels'
    # head_dim-64 path; not one of the pages' measured models
    "llama32_1b": CacheConfig("llama32_1b", 16, 1, 8, 32768, 64, 0.7, 0.0, 1.0, 5e5, "student_t5", 5,
                              (_p(2, 2, False, 0, 5e5), _p(2, 2, True, 0, 5e5))),
    "qwen25_14b": CacheConfig("qwen25_14b", 48, 1, 8, 131072, 128, 1.0, 0.01, 16.0, 1e6, "normal", 4,
                              (_p(3, 2, False, 256, 1e6), _p(3, 2, True, 256, 1e6),
                               _p(2, 2, False, 256, 1e6), _p(2, 2, True, 256, 1e6))),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _model_rope(k, theta, tokens):
    """The model's forward rotary embedding (what a prefill writes to the cache)."""
    D = k.shape[-1]
    inv_freq = 1.0 / (theta ** (torch.arange(0, D, 2, device=k.device, dtype=torch.float32) / D))
    t = torch.arange(tokens, device=k.device, dtype=torch.float32)
    ang = torch.outer(t, inv_freq)  # [T, D/2]
    cos = torch.cat([ang.cos(), ang.cos()], dim=-1)
    sin = torch.cat([ang.sin(), ang.sin()], dim=-1)
    rot = torch.cat([-k[..., D // 2:], k[..., : D // 2]], dim=-1)
    return k * cos + rot * sin


def layer_kv(cfg, layer, device="cuda", tokens=None, batch=None):
    """fp16 K, V of one layer: [batch, kv_heads, tokens, head_dim] (`batch` and
    `tokens` restrict the draw to a smaller sample of the same distribution)."""
    T = cfg.tokens if tokens is None else tokens
    B = cfg.batch if batch is None else batch
    H, D = cfg.kv_heads, cfg.head_dim
    g = _gen(device, cfg.seed * 1000 + layer)
    z = torch.randn((B, H, T, D), generator=g, device=device, dtype=torch.float32)
    scale = torch.exp(cfg.sigma * torch.randn((H, 1, D), generator=g, device=device))
    if cfg.outlier_frac > 0:
        n_out = math.ceil(cfg.outlier_frac * D)
        for h in range(H):
            perm = torch.randperm(D, generator=g, device=device)
            scale[h, 0, perm[:n_out]] *= cfg.outlier_mult
    k = z * scale
    if cfg.theta > 0:
        k = _model_rope(k, cfg.theta, T)
    if cfg.v_dist == "student_t5":
        z0 = torch.randn((B, H, T, D), generator=g, device=device)
        chi2 = torch.zeros_like(z0)
        for _ in range(5):
            chi2 += torch.randn((B, H, T, D), generator=g, device=device) ** 2
        v = z0 / torch.sqrt(chi2 / 5.0) * math.sqrt(3.0 / 5.0)
    else:
        v = torch.randn((B, H, T, D), generator=g, device=device)
    return k.to(torch.float16), v.to(torch.float16)


def make_cache(cfg, device="cuda", layers=None, tokens=None):
    """fp16 K, V [layers, batch, kv_heads, tokens, head_dim] (first `layers`
    layers when given, first `tokens` tokens' shape when given)."""
    nl = cfg.layers if layers is None else layers
    T = cfg.tokens if tokens is None else tokens
    shape = (nl, cfg.batch, cfg.kv_heads, T, cfg.head_dim)
    K = torch.empty(shape, dtype=torch.float16, device=device)
    V = torch.empty(shape, dtype=torch.float16, device=device)
    for l in range(nl):
        k, v = layer_kv(cfg, l, device, tokens=T)
        K[l].copy_(k)
        V[l].copy_(v)
        del k, v
    return K, V
