"""Seeded synthetic inputs for the MoE routing layer.

This module builds inputs only: weights, token activations, router logits
shaped by a skewed expert popularity, expert-similarity and protection
matrices, and per-token load weights. It holds none of the layer's own
arithmetic (no softmax, top-k, reroute, capacity or FFN), so the CUDA path
and the CPU oracle can both draw from it without sharing any of the method.

Workloads (sizes follow the Qwen3-30B-A3B MoE layer: hidden 2048, 128
experts, top-8, SwiGLU intermediate 768):

* ``tiny``    T=16, H=64, N=8, k=2, I=128, everything fp32.
* ``decode``  T tokens (1..128), bf16 expert weights N(0, 0.02), fp32 router.
* ``prefill`` T=8192 with 70% "visual" tokens (load weight ~ Beta(2,5)) and
  30% "text" tokens (load weight 1).
* ``stack``   48 decode layers (generated on the device by the bench).

Seeds follow ``1000*config + 10*layer + stream`` so that every array of every
workload is reproducible on its own.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# Popularity skew of the experts: pi ~ Dirichlet(ALPHA * 1_N).  With the
# Gumbel-perturbed preference below, ALPHA = 0.29 gives a mean union of about
# 60 distinct top-8 experts over a batch of 32 tokens (about 82 at batch 128),
# the regime the SERE article reports for Qwen3-30B-A3B decode.
ALPHA_POPULARITY = 0.29

STREAM_WEIGHTS, STREAM_ROUTER, STREAM_TOKENS, STREAM_SIM, STREAM_PROTECT, STREAM_LOADW = range(6)

CONFIG_TINY, CONFIG_DECODE, CONFIG_SWEEP, CONFIG_PREFILL, CONFIG_STACK = 1, 2, 3, 4, 5


def seed_for(config: int, layer: int, stream: int) -> int:
    return 1000 * config + 10 * layer + stream


def rng_for(config: int, layer: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(seed_for(config, layer, stream))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest even) and return the raw uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Layer:
    """One MoE layer's inputs.  Array layouts are the ones the C-ABI expects.

    x       [T][H]   fp32 values; ``x_bf16`` holds the bf16 bits when dtype is bf16
    w_r     [N][H]   fp32 router weight
    w_gate  [N][I][H], w_up [N][I][H], w_down [N][H][I]: fp32 arrays (tiny) or
            uint16 bf16 bits (all other workloads)
    sim     [N][N]   fp32 expert similarity, symmetric, unit diagonal
    protect [N]      uint8 0/1 protection bit per source expert (or None)
    token_w [T]      fp32 per-token load weight (capacity mode) or None
    """
    T: int
    H: int
    N: int
    k: int
    I: int
    dtype: str                 # "f32" or "bf16"
    x: np.ndarray              # fp32 values (already rounded to bf16 when dtype is bf16)
    x_bf16: Optional[np.ndarray]
    w_r: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray
    sim: np.ndarray
    protect: Optional[np.ndarray]
    token_w: Optional[np.ndarray]
    k_primary: int = 2
    rho: float = 0.5
    gamma: float = 1.25
    R: int = 8
    is_visual: Optional[np.ndarray] = None


def _sym_uniform_sim(rng: np.random.Generator, N: int) -> np.ndarray:
    a = rng.random((N, N), dtype=np.float32)
    s = np.triu(a, 1)
    s = s + s.T
    np.fill_diagonal(s, 1.0)
    return s.astype(np.float32)


def clustered_sim(rng: np.random.Generator, N: int, cluster: int = 8) -> np.ndarray:
    """Block-structured similarity: a seeded permutation groups the experts into
    N/cluster clusters; same-cluster pairs ~ U[0.55, 0.95], others ~ U[0, 0.45],
    symmetric with a unit diagonal."""
    perm = rng.permutation(N)
    group = np.empty(N, dtype=np.int64)
    group[perm] = np.arange(N) // cluster
    same = group[:, None] == group[None, :]
    hi = rng.uniform(0.55, 0.95, size=(N, N))
    lo = rng.uniform(0.0, 0.45, size=(N, N))
    s = np.where(same, hi, lo)
    s = np.triu(s, 1)
    s = s + s.T
    np.fill_diagonal(s, 1.0)
    return s.astype(np.float32)


def protect_bits(rng: np.random.Generator, N: int, count: int) -> np.ndarray:
    p = np.zeros(N, dtype=np.uint8)
    p[rng.choice(N, size=count, replace=False)] = 1
    return p


def skewed_logits(rng: np.random.Generator, T: int, N: int, alpha: float = ALPHA_POPULARITY) -> np.ndarray:
    """Per-token expert preference drawn around a Dirichlet popularity.

    pi ~ Dirichlet(alpha * 1_N) is shared by the batch; token t's logits are
    log(pi) + g_t with g_t i.i.d. standard Gumbel, centred per token.  By the
    Gumbel-max property each token's top-k is then k experts drawn without
    replacement from pi, so a smaller alpha means a more skewed popularity and
    a smaller batch union.  The logits are continuous, so exact ties have
    probability zero."""
    pi = rng.dirichlet(alpha * np.ones(N))
    g = rng.gumbel(size=(T, N))
    l = np.log(pi)[None, :] + g
    l = l - l.mean(axis=1, keepdims=True)
    return l


def tokens_for_logits(rng: np.random.Generator, w_r: np.ndarray, logits: np.ndarray) -> np.ndarray:
    """Token activations whose router logits are (up to rounding) the given ones:
    x = pinv(W_r) l + a N(0,1) component in the null space of W_r."""
    W = w_r.astype(np.float64)
    pinv = np.linalg.pinv(W)                     # [H][N]
    x = logits @ pinv.T                          # [T][H], min-norm solution
    z = rng.standard_normal((logits.shape[0], W.shape[1]))
    z = z - (z @ W.T) @ pinv.T                   # project onto the null space of W
    return (x + z).astype(np.float32)


def _bf16_normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """N(0, std) rounded to bf16, as raw bits; generated expert by expert."""
    out = np.empty(shape, dtype=np.uint16)
    for e in range(shape[0]):
        out[e] = f32_to_bf16_bits(rng.standard_normal(shape[1:], dtype=np.float32) * np.float32(std))
    return out


def tiny(seed_layer: int = 0, capacity: bool = False) -> Layer:
    """The tiny fp32 layer: T=16, H=64, N=8, k=2, I=128."""
    T, H, N, k, I = 16, 64, 8, 2, 128
    c, l = CONFIG_TINY, seed_layer
    rw = rng_for(c, l, STREAM_WEIGHTS)
    w_gate = (rw.standard_normal((N, I, H)) / np.sqrt(H)).astype(np.float32)
    w_up = (rw.standard_normal((N, I, H)) / np.sqrt(H)).astype(np.float32)
    w_down = (rw.standard_normal((N, H, I)) / np.sqrt(I)).astype(np.float32)
    w_r = (rng_for(c, l, STREAM_ROUTER).standard_normal((N, H)) / np.sqrt(H)).astype(np.float32)
    x = rng_for(c, l, STREAM_TOKENS).standard_normal((T, H)).astype(np.float32)
    sim = _sym_uniform_sim(rng_for(c, l, STREAM_SIM), N)
    token_w = None
    vis = None
    if capacity:
        rl = rng_for(c, l, STREAM_LOADW)
        vis = np.zeros(T, dtype=bool)
        vis[rl.choice(T, size=11, replace=False)] = True
        token_w = np.ones(T, dtype=np.float32)
        token_w[vis] = rl.beta(2.0, 5.0, size=int(vis.sum())).astype(np.float32)
    return Layer(T=T, H=H, N=N, k=k, I=I, dtype="f32", x=x, x_bf16=None, w_r=w_r,
                 w_gate=w_gate, w_up=w_up, w_down=w_down, sim=sim, protect=None,
                 token_w=token_w, k_primary=1, rho=0.5, gamma=1.25, R=min(10, N), is_visual=vis)


def qwen_layer(T: int, config: int = CONFIG_DECODE, layer: int = 0, n_protect: int = 0,
               capacity: bool = False, visual_frac: float = 0.7,
               H: int = 2048, N: int = 128, k: int = 8, I: int = 768,
               with_weights: bool = True, token_stream_offset: int = 0) -> Layer:
    """A Qwen3-30B-A3B-shaped layer: bf16 experts ~ N(0, 0.02), fp32 router ~ N(0, 0.02).

    ``token_stream_offset`` selects an independent token batch over the same weights."""
    rw = rng_for(config, layer, STREAM_WEIGHTS)
    if with_weights:
        w_gate = _bf16_normal(rw, (N, I, H), 0.02)
        w_up = _bf16_normal(rw, (N, I, H), 0.02)
        w_down = _bf16_normal(rw, (N, H, I), 0.02)
    else:
        w_gate = w_up = w_down = None
    w_r = (rng_for(config, layer, STREAM_ROUTER).standard_normal((N, H)) * 0.02).astype(np.float32)
    rt = np.random.default_rng(seed_for(config, layer, STREAM_TOKENS) + 7919 * token_stream_offset)
    logits = skewed_logits(rt, T, N)
    x = tokens_for_logits(rt, w_r, logits)
    x_bits = f32_to_bf16_bits(x)
    x = bf16_bits_to_f32(x_bits)
    sim = clustered_sim(rng_for(config, layer, STREAM_SIM), N)
    protect = protect_bits(rng_for(config, layer, STREAM_PROTECT), N, n_protect) if n_protect else None
    token_w = None
    vis = None
    if capacity:
        rl = rng_for(config, layer, STREAM_LOADW)
        n_vis = int(round(visual_frac * T))
        vis = np.zeros(T, dtype=bool)
        vis[rl.choice(T, size=n_vis, replace=False)] = True
        token_w = np.ones(T, dtype=np.float32)
        token_w[vis] = rl.beta(2.0, 5.0, size=n_vis).astype(np.float32)
    return Layer(T=T, H=H, N=N, k=k, I=I, dtype="bf16", x=x, x_bf16=x_bits, w_r=w_r,
                 w_gate=w_gate, w_up=w_up, w_down=w_down, sim=sim, protect=protect,
                 token_w=token_w, k_primary=2, rho=0.5, gamma=1.25, R=min(10, N) if capacity else k,
                 is_visual=vis)


def decode(T: int = 32, layer: int = 0, n_protect: int = 0, **kw) -> Layer:
    """Single decode layer (batch T, default 32) with the 16x8 clustered similarity."""
    return qwen_layer(T, config=CONFIG_DECODE, layer=layer, n_protect=n_protect, **kw)


def sweep(T: int, layer: int = 0, **kw) -> Layer:
    """Decode batch-sweep layer with 16 protected experts."""
    return qwen_layer(T, config=CONFIG_SWEEP, layer=layer, n_protect=16, **kw)


def prefill(T: int = 8192, layer: int = 0, **kw) -> Layer:
    """Capacity-mode prefill layer: 70% visual (w ~ Beta(2,5)), 30% text (w = 1)."""
    return qwen_layer(T, config=CONFIG_PREFILL, layer=layer, capacity=True, **kw)


# ---------------------------------------------------------------------------
# 48-layer decode stack: x_{l+1} = x_l + y_l over layers with their own weights.
# ---------------------------------------------------------------------------
STACK_LAYERS, STACK_BATCH, STACK_PROTECT = 48, 64, 16


def stack_tokens(T: int = STACK_BATCH, H: int = 2048, token_stream_offset: int = 0):
    """x_0 [T][H] ~ N(0,1), rounded to bf16: (fp32 values, bf16 bits)."""
    rt = np.random.default_rng(seed_for(CONFIG_STACK, 0, STREAM_TOKENS) + 7919 * token_stream_offset)
    bits = f32_to_bf16_bits(rt.standard_normal((T, H), dtype=np.float32))
    return bf16_bits_to_f32(bits), bits


def stack_router(x0: np.ndarray, layer: int, N: int = 128) -> np.ndarray:
    """Router of stack layer `layer` [N][H] fp32: the minimum-norm W_r with
    x_0 W_r^T equal to that layer's Dirichlet-skewed logits, so every layer
    keeps its own expert popularity while the residual stream stays close to
    x_0 (the layers' outputs are small next to it)."""
    logits = skewed_logits(rng_for(CONFIG_STACK, layer, STREAM_ROUTER), x0.shape[0], N)
    w = np.linalg.pinv(x0.astype(np.float64)) @ logits      # [H][N]
    return np.ascontiguousarray(w.T).astype(np.float32)


def stack_sim(layer: int, N: int = 128) -> np.ndarray:
    return clustered_sim(rng_for(CONFIG_STACK, layer, STREAM_SIM), N)


def stack_protect(layer: int, N: int = 128) -> np.ndarray:
    return protect_bits(rng_for(CONFIG_STACK, layer, STREAM_PROTECT), N, STACK_PROTECT)


def stack_weight_seed(layer: int) -> int:
    """Seed of the torch generator that draws a stack layer's expert weights
    (N(0, 0.02), fp32 then bf16) on the device, in the order gate, up, down."""
    return seed_for(CONFIG_STACK, layer, STREAM_WEIGHTS)


STREAM_MODALITY = 6


def modality_bias(N: int = 128, config: int = CONFIG_PREFILL, layer: int = 0) -> np.ndarray:
    """Expert modality groups for the per-expert capacity: a seeded quarter of
    the experts visual (+1), a quarter text (-1), the rest shared (0).  It
    stands in for the grouping by activation frequency on a calibration set,
    which needs a trained model."""
    perm = rng_for(config, layer, STREAM_MODALITY).permutation(N)
    m = np.zeros(N, dtype=np.int8)
    m[perm[: N // 4]] = 1
    m[perm[N // 4: N // 2]] = -1
    return m
