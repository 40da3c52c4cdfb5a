"""Seeded synthetic KV-cache workloads.

This module only draws inputs; it holds none of the codec's arithmetic, so
the library's tests, its benchmark and the fp64 oracle can all take their
inputs from it.

The pages measure the codec on real model caches (Llama-3-8B, SmolLM2-1.7B);
no weights or corpora are used here, so caches are drawn with the statistics
those caches are known for:

* keys: N(0,1), with 4 channels per (layer, head), chosen uniformly without
  replacement, scaled by 20 -- the per-channel key outliers that motivate
  keeping K at 8 bits ("PolyKV", 2.B.1);
* values: Student-t with 5 degrees of freedom, times 0.5 -- heavier tails
  than a Gaussian, which the Walsh-Hadamard rotation has to spread
  ("PolyKV", 2.B.2); drawn as Z / sqrt(W/5) with W a sum of 5 squared
  standard normals, the textbook construction of the t distribution;
* CacheCard bitwidths: i.i.d. per token from {2,4,8,16} with probabilities
  {0.25, 0.40, 0.25, 0.10} ("QKVShare", Methodology 1 names the set);
* LoRA value adapters ("LRAgent"): the shared low-rank cache X A ~ N(0,1)
  per entry, each agent's up-projection B ~ N(0, 0.02^2), so the adapter term
  is a small perturbation of the base values, as that page describes it.

Both are rounded to bf16 (round-to-nearest-even), laid out per layer as
[H][T][d], the Hugging Face past_key_values layout at batch 1.
"""
import numpy as np
import torch

# Shapes of the configurations the library is measured and tested on.
# (L layers, H KV heads, d head_dim, T tokens, N agents)
WORKLOADS = {
    "llama3-8b-1layer-512": dict(L=1, H=8, d=128, T=512, N=1),
    "smollm2-1.7b-1851": dict(L=24, H=32, d=64, T=1851, N=3),
    "llama3-8b-4k-15agents": dict(L=32, H=8, d=128, T=4096, N=15),
    "llama3-8b-32k-4agents": dict(L=32, H=8, d=128, T=32768, N=4),
    "llama31-8b-cachecard-8k": dict(L=32, H=8, d=128, T=8192, N=1),
}

CARD_BITS = (2, 4, 8, 16)
CARD_PROBS = (0.25, 0.40, 0.25, 0.10)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def kv_layer(H, T, d, gen, device="cpu"):
    """One layer's (K, V) as bf16 tensors of shape [H, T, d]."""
    k = torch.randn(H, T, d, generator=gen, device=device, dtype=torch.float32)
    # 4 distinct outlier channels per head: the first 4 of a random ordering.
    order = torch.rand(H, d, generator=gen, device=device).argsort(dim=1)[:, :4]
    scale = torch.ones(H, d, device=device)
    scale.scatter_(1, order, 20.0)
    k.mul_(scale[:, None, :])
    z = torch.randn(H, T, d, generator=gen, device=device, dtype=torch.float32)
    w = torch.zeros(H, T, d, device=device, dtype=torch.float32)
    for _ in range(5):
        e = torch.randn(H, T, d, generator=gen, device=device, dtype=torch.float32)
        w.addcmul_(e, e)
    v = z.mul_(0.5).div_(torch.sqrt(w.div_(5.0)))
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def kv_layers(L, H, T, d, seed=0, device="cpu"):
    """Lists of L bf16 key and value tensors, each [H, T, d] and contiguous."""
    g = _gen(seed, device)
    ks, vs = [], []
    for _ in range(L):
        k, v = kv_layer(H, T, d, g, device)
        ks.append(k)
        vs.append(v)
    return ks, vs


def card_bits(T, seed=0, device="cpu"):
    """Per-token bitwidths (uint8 tensor of length T)."""
    g = _gen(seed + 0x5EED, device)
    u = torch.rand(T, generator=g, device=device)
    edges = np.cumsum(CARD_PROBS)[:-1]
    out = torch.full((T,), CARD_BITS[-1], dtype=torch.uint8, device=device)
    for b, e in zip(reversed(CARD_BITS[:-1]), reversed(edges)):
        out[u < float(e)] = b
    return out


def lora_inputs(T, H, d, n_agents, rank, seed=0, device="cpu"):
    """Shared low-rank value cache (bf16 [T, rank]) and per-agent value
    up-projections (bf16 [n_agents, rank, H*d], rank-major rows)."""
    g = _gen(seed + 0x10AA, device)
    vlr = torch.randn(T, rank, generator=g, device=device)
    b = torch.randn(n_agents, rank, H * d, generator=g, device=device) * 0.02
    return vlr.to(torch.bfloat16), b.to(torch.bfloat16)


def bits16(t):
    """Raw uint16 bit pattern of a bf16 tensor, as a numpy array (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits16(a, device="cpu"):
    """bf16 tensor from a numpy uint16 bit-pattern array."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)
