"""Seeded synthetic inputs for the latent-routed top-k MoE layer.

This module is shared by the fp64 oracle (``oracle/``) and by the CUDA path
(``fine_grained_moe_02_b300``).  It holds the workload table and the random
draws only: nothing here computes any step of the layer.  Every tensor is
drawn from its own counter-addressed PCG64 stream (``SeedSequence(seed,
spawn_key=(tensor_id, chunk))``) so that the result does not depend on the
number of host threads, and float32 draws are rounded to bfloat16 with
round-to-nearest-even.  bfloat16 tensors are returned as ``uint16`` bit
patterns; the consumer widens them itself.

Workload shapes follow the pages' geometry (MAGI-2 Preview specification
table, "Routing" row: 12 latent heads of 256 dims, top-6; MAGI-1 page: 8x
spatial / 4x temporal VAE and 24-frame chunks; MAGI-2 page "Output specs":
10 s clips, 512x896 preview and 1088x1920 refiner).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

N_HEADS = 12
HEAD_DIM = 256
TOP_K = 6

_CHUNK = 1 << 22  # elements per independent RNG stream


@dataclass(frozen=True)
class MoeConfig:
    """One workload: layer dimensions plus how its inputs are drawn."""

    name: str
    T: int
    d: int
    E: int
    inter: int
    top_k: int = TOP_K
    n_heads: int = N_HEADS
    head_dim: int = HEAD_DIM
    router_init: str = "normal"      # "normal": N(0,1/fan_in); "uniform": U(+-1/sqrt(fan_in))
    bias: str = "none"               # "none" | "zipf"
    zipf_s: float = 1.2
    modality_split: tuple = ()       # ((n_tokens, x_scale), ...) in sequence order
    modality_experts: tuple = ()     # ((begin, end), ...) routed experts of each modality; () = no masking
    n_shared: int = 0                # shared experts, stored after the E routed experts
    head_local: bool = False         # head-local MoE: d = n_heads*head_dim split into heads, E experts per head
    seed: int = 0
    note: str = ""

    @property
    def L(self) -> int:
        return self.n_heads * self.head_dim

    def dims(self) -> dict:
        return dict(T=self.T, d=self.d, n_heads=self.n_heads, head_dim=self.head_dim,
                    E=self.E, inter=self.inter, top_k=self.top_k)


# The five workloads.  Token counts: 512x896 / 8 = 64x112 latent, 2x2 patches
# -> 32x56 = 1792 tokens per latent frame; a 24-frame chunk is 6 latent frames
# (4x temporal); a 10 s clip at 24 fps is 240 frames -> 60 latent frames;
# 1088x1920 / 8 / 2 = 68x120 tokens per refiner latent frame.
CONFIGS = {
    "tiny": MoeConfig("tiny", T=256, d=512, E=16, inter=128,
                      note="T=256, d=512, E=16, inter=128, top-6; x~N(0,1), weights N(0,1/fan_in), seed 0"),
    "frame": MoeConfig("frame", T=1792, d=2048, E=64, inter=1024, router_init="uniform",
                       note="one 512x896 preview latent frame (32x56 tokens), uniform router init"),
    "chunk": MoeConfig("chunk", T=10752 + 256 + 384, d=4096, E=128, inter=1024,
                       modality_split=((10752, 1.0), (256, 0.5), (384, 0.8)),
                       note="24-frame preview chunk: 10752 video + 256 text + 384 audio tokens, x scale 1.0/0.5/0.8"),
    "clip": MoeConfig("clip", T=107520, d=4096, E=128, inter=1024, bias="zipf",
                      note="full 10 s preview clip: 60 latent frames x 1792 tokens, Zipf(1.2) router bias"),
    "refiner": MoeConfig("refiner", T=48960, d=4096, E=256, inter=512, router_init="uniform",
                         note="refiner chunk: 6 latent frames x 68x120 tokens, E=256, inter=512, uniform routing"),
    # the chunk's video|text|audio stream with modality-specific routed experts
    # (video 0-95, text 96-111, audio 112-127) and one shared expert
    "chunk_mm": MoeConfig("chunk_mm", T=10752 + 256 + 384, d=4096, E=128, inter=1024,
                          modality_split=((10752, 1.0), (256, 0.5), (384, 0.8)),
                          modality_experts=((0, 96), (96, 112), (112, 128)), n_shared=1,
                          note="24-frame chunk with modality-specific experts (video 96, text 16, audio 16) "
                               "and one shared expert"),
    # head-local MultiHead MoE: 3072 = 12 x 256 split into heads, 256 experts
    # per head, top-6 per head (72 experts per token), head-local experts
    # 256 -> 512 -> 256; one 24-frame chunk of video tokens
    "headlocal": MoeConfig("headlocal", T=10752, d=3072, E=256, inter=512, head_local=True,
                           note="head-local MoE: 12 heads x 256 dims, 256 experts per head, top-6 per head, "
                                "expert inter 512, T=10752"),
    # not one of the pages' workloads: the head-local layer with a quarter of
    # the experts per head and a quarter of the tokens (the same ~252 rows per
    # expert; under 1 GB on the device), small enough for full profiler captures
    "headlocal_slice": MoeConfig("headlocal_slice", T=2688, d=3072, E=64, inter=512, head_local=True,
                                 note="profiling size: head-local MoE, 12 heads x 256 dims, 64 experts per head, "
                                      "top-6 per head, expert inter 512, T=2688"),
    # not one of the pages' workloads: a 4096-token slice at clip width with 32
    # experts, small enough (~1.5 GB on the device) for full profiler captures
    "slice": MoeConfig("slice", T=4096, d=4096, E=32, inter=1024,
                       note="profiling size: 4096 tokens, d=4096, E=32, inter=1024"),
    # not one of the pages' workloads: the first 16384 tokens' worth of the clip
    # workload (same width, experts and Zipf bias, about 4.6 GB on the device),
    # small enough for counter captures whose DRAM bytes scale to the clip
    "clip_slice": MoeConfig("clip_slice", T=16384, d=4096, E=128, inter=1024, bias="zipf",
                            note="profiling size: 16384 tokens at the clip workload's width, experts and bias"),
}
CONFIG_ORDER = ["tiny", "frame", "chunk", "clip", "refiner", "chunk_mm", "headlocal", "slice", "clip_slice",
                "headlocal_slice"]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32 (for harness use)."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill(out: np.ndarray, seed: int, tensor_id: int, kind: str, scale: float) -> None:
    """Fill a flat float32 array chunk by chunk, one PCG64 stream per chunk."""
    n = out.size
    starts = range(0, n, _CHUNK)

    def work(start: int) -> None:
        ss = np.random.SeedSequence(seed, spawn_key=(tensor_id, start // _CHUNK))
        g = np.random.Generator(np.random.PCG64(ss))
        view = out[start:start + _CHUNK]
        if kind == "normal":
            g.standard_normal(out=view, dtype=np.float32)
        elif kind == "uniform":
            view[:] = g.random(view.size, dtype=np.float32)
            view *= np.float32(2.0)
            view -= np.float32(1.0)
        else:
            raise ValueError(kind)
        if scale != 1.0:
            view *= np.float32(scale)

    if len(starts) == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))


def draw_bf16(shape, seed: int, tensor_id: int, kind: str = "normal", scale: float = 1.0) -> np.ndarray:
    """A bfloat16 tensor (uint16 bits) of i.i.d. draws times ``scale``."""
    n = int(np.prod(shape))
    f = np.empty(n, dtype=np.float32)
    _fill(f, seed, tensor_id, kind, scale)
    out = np.empty(n, dtype=np.uint16)

    def cvt(start: int) -> None:
        out[start:start + _CHUNK] = f32_to_bf16_bits(f[start:start + _CHUNK])

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(cvt, range(0, n, _CHUNK)))
    return out.reshape(shape)


# tensor ids: one independent stream family per tensor
_TID = dict(x=1, w_lat=2, w_head=3, w_gate=4, w_up=5, w_down=6, perm=7, surrogate=8)


def zipf_capped_shares(E: int, s: float, k: int) -> np.ndarray:
    """Zipf(s) shares over ranks 1..E, capped at 1/k and water-filled.

    With top-k routing over distinct experts no expert can hold more than a
    1/k share of the T*k assignments, so the raw Zipf head is clipped at 1/k
    and the clipped mass is spread over the rest in proportion to their
    shares, repeated until no share exceeds the cap.  Result sums to 1.
    """
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    cap = 1.0 / k
    capped = np.zeros(E, dtype=bool)
    for _ in range(E):
        over = (p > cap * (1 + 1e-12)) & ~capped
        if not over.any():
            break
        capped |= over
        p[capped] = cap
        free = ~capped
        rest = 1.0 - cap * capped.sum()
        p[free] *= rest / p[free].sum()
    return p


def router_bias(cfg: MoeConfig) -> np.ndarray | None:
    """The router bias b[E] (float32) or None.

    "zipf": the bias that makes the expert load follow the capped Zipf shares
    q (``zipf_capped_shares``), assigned to experts through a seeded
    permutation pi.  It is fitted on a Gaussian surrogate of the unbiased
    summed head scores, i.i.d. N(0, sigma^2) with sigma = sqrt(n_heads) (the
    score spread under this generator's weight scales: var(h) = 1,
    var(W_head) = 1/head_dim, summed over n_heads*head_dim terms).  Start at
    b = sigma * ln q and take 60 damped fixed-point steps
    b += 0.3 * sigma * (ln q - ln p_hat), p_hat the surrogate's top-k
    selection shares over 16384 draws.  The surrogate never sees the layer's
    inputs or weights; the fit is deterministic.
    """
    if cfg.bias == "none":
        return None
    if cfg.bias != "zipf":
        raise ValueError(cfg.bias)
    E, k = cfg.E, cfg.top_k
    q = zipf_capped_shares(E, cfg.zipf_s, k)
    sigma = math.sqrt(cfg.L / cfg.head_dim)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(cfg.seed, spawn_key=(_TID["surrogate"],))))
    Z = g.standard_normal((16384, E)).astype(np.float32) * np.float32(sigma)
    b = sigma * np.log(q)
    for _ in range(60):
        sel = np.argpartition(-(Z + b.astype(np.float32)), k - 1, axis=1)[:, :k]
        p_hat = np.bincount(sel.ravel(), minlength=E) / sel.size
        b = b + 0.3 * sigma * (np.log(q) - np.log(np.maximum(p_hat, 0.25 / sel.size)))
        b -= b.max()
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(cfg.seed, spawn_key=(_TID["perm"],))))
    perm = g.permutation(E)           # expert e takes Zipf rank perm[e]
    return b[perm].astype(np.float32)


def x_row_scales(cfg: MoeConfig) -> np.ndarray | None:
    if not cfg.modality_split:
        return None
    scales = np.concatenate([np.full(n, s, dtype=np.float32) for n, s in cfg.modality_split])
    assert scales.size == cfg.T
    return scales


def make_x(cfg: MoeConfig) -> np.ndarray:
    """Token activations x[T, d] (bf16 bits): N(0,1), per-modality scaled."""
    scales = x_row_scales(cfg)
    if scales is None:
        return draw_bf16((cfg.T, cfg.d), cfg.seed, _TID["x"])
    n = cfg.T * cfg.d
    f = np.empty(n, dtype=np.float32)
    _fill(f, cfg.seed, _TID["x"], "normal", 1.0)
    f = f.reshape(cfg.T, cfg.d)
    f *= scales[:, None]
    return f32_to_bf16_bits(f)


def _w(cfg: MoeConfig, name: str, shape, fan_in: int, router: bool) -> np.ndarray:
    if router and cfg.router_init == "uniform":
        return draw_bf16(shape, cfg.seed, _TID[name], "uniform", 1.0 / math.sqrt(fan_in))
    return draw_bf16(shape, cfg.seed, _TID[name], "normal", 1.0 / math.sqrt(fan_in))


def make_weights(cfg: MoeConfig) -> dict:
    """Router and expert weights, all bf16 bits, "[out, in]" row-major.

    w_lat [L, d], w_head [E, L], w_gate/w_up [E, inter, d], w_down [E, d, inter],
    bias [E] float32 or None.
    """
    if cfg.head_local:
        H, Dh = cfg.n_heads, cfg.head_dim
        assert cfg.d == H * Dh
        return dict(
            w_router=_w(cfg, "w_head", (H, cfg.E, Dh), Dh, True),
            w_gate=_w(cfg, "w_gate", (H, cfg.E, cfg.inter, Dh), Dh, False),
            w_up=_w(cfg, "w_up", (H, cfg.E, cfg.inter, Dh), Dh, False),
            w_down=_w(cfg, "w_down", (H, cfg.E, Dh, cfg.inter), cfg.inter, False),
            bias=None,
        )
    n_exp = cfg.E + cfg.n_shared   # shared experts follow the routed ones
    return dict(
        w_lat=_w(cfg, "w_lat", (cfg.L, cfg.d), cfg.d, True),
        w_head=_w(cfg, "w_head", (cfg.E, cfg.L), cfg.head_dim, True),
        w_gate=_w(cfg, "w_gate", (n_exp, cfg.inter, cfg.d), cfg.d, False),
        w_up=_w(cfg, "w_up", (n_exp, cfg.inter, cfg.d), cfg.d, False),
        w_down=_w(cfg, "w_down", (n_exp, cfg.d, cfg.inter), cfg.inter, False),
        bias=router_bias(cfg),
    )


def make_modality(cfg: MoeConfig) -> np.ndarray:
    """Modality id of each token (int32 [T]): its index in modality_split."""
    if not cfg.modality_split:
        return np.zeros(cfg.T, dtype=np.int32)
    return np.concatenate([np.full(n, m, dtype=np.int32) for m, (n, _) in enumerate(cfg.modality_split)])


def make_inputs(cfg: MoeConfig | str) -> dict:
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    out = make_weights(cfg)
    out["x"] = make_x(cfg)
    out["modality"] = make_modality(cfg)
    out["cfg"] = cfg
    return out


def custom_config(name: str = "custom", **kw) -> MoeConfig:
    """A config with explicit dims (for edge-case tests)."""
    return MoeConfig(name, **kw)


def sample_tokens(T: int, n: int, seed: int = 1234) -> np.ndarray:
    """A sorted, seeded sample of n distinct token indices in [0, T)."""
    n = min(n, T)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(99,))))
    return np.sort(g.choice(T, size=n, replace=False)).astype(np.int64)
