"""Seeded synthetic inputs for the Dory looped nGPT token forward.

This module describes workloads and draws their inputs: model shapes, random
unit-row weights, token ids, loop schedules and synthetic KV context rows. It
holds none of the forward's arithmetic, so both the CPU oracle and the CUDA
path can take their inputs from it without sharing any of the method.

Random numbers come from one counter-based generator defined here
(SplitMix64's finaliser over (stream key + counter), Box-Muller for normals),
so the same seed gives the same values on any machine and under any threading.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    a = np.array([(seed * 0x100000001B3 + stream * 0x51ED27 + 1) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(_mix(a))[0]


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n draws in (0, 1), float64, counters start..start+n of (seed, stream)."""
    c = np.arange(start, start + n, dtype=np.uint64)
    z = _mix(c * _GOLDEN + _stream_key(seed, stream))
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n standard normal draws (Box-Muller over consecutive uniform pairs).

    `start` must be even; draw 2i and 2i+1 share one uniform pair.
    """
    assert start % 2 == 0
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m, start)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = 2.0 * math.pi * u[1::2]
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); raw uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen raw bfloat16 bits to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(w: np.ndarray) -> np.ndarray:
    """Weights as float32 values, whatever their storage (uint16 bf16 bits or f32)."""
    return bf16_bits_to_f32(w) if w.dtype == np.uint16 else np.asarray(w, dtype=np.float32)


# ----------------------------------------------------------------------------------------
# Workload descriptions
# ----------------------------------------------------------------------------------------


@dataclasses.dataclass
class DoryConfig:
    """Shape, cache and scale recipe of one Dory model. Layer counts are physical sub-layers."""

    name: str
    hidden: int
    ffn: int
    vocab: int
    nh: int
    nk: int
    hd: int
    window: int
    pattern: str  # one char per physical layer: 'S' sliding attention, '*' full attention, '-' MLP
    n_in: int
    n_rec: int
    n_out: int
    loops: int = 4
    max_loops: int = 16
    full_window: int = 0  # 0: full layers read every earlier row
    max_context: int = 4096  # rows a full layer without full_window can hold
    kv_mode: str = "last_loop"  # or "per_loop"
    kv_quant: str = "f32"  # or "q8_2f"
    prompt_loops: int = 0
    max_batch: int = 1
    max_seqs: int = 1
    weight_dtype: str = "bf16"  # or "f32"
    rope_theta_sliding: float = 1.0e4
    rope_theta_full: float = 1.0e7
    # effective scales (already folded): s_q^2 per element, gate s_g^2, MLP s*sqrt(hidden)
    sq: float = 1.0
    attn_sg: float = 1.0
    mlp_suv: float = 1.0  # raw suv; the effective MLP scale is suv*sqrt(hidden)
    logit_scale: float = 1.0
    alpha: tuple = (0.05, 0.05)  # |alpha| drawn uniformly in [lo, hi] per element
    # per-element spread of the folded scale vectors (s_q^2, the gate's s_g^2, the MLP's
    # s_g and s_u, logit_scale): each element is its base value above times a uniform draw
    # in [1 - spread, 1 + spread]; 0 gives every element the base value
    scale_spread: float = 0.0

    @property
    def n_layers(self) -> int:
        return len(self.pattern)

    @property
    def attn_layers(self) -> int:
        return sum(1 for c in self.pattern if c != "-")

    def replace(self, **kw) -> "DoryConfig":
        return dataclasses.replace(self, **kw)


def pattern_of(in_kinds, rec_kinds, out_kinds) -> tuple[str, int, int, int]:
    """Pattern from (attention kind) per attention+MLP pair of each block."""
    blocks = ["".join(k + "-" for k in ks) for ks in (in_kinds, rec_kinds, out_kinds)]
    return "".join(blocks), len(blocks[0]), len(blocks[1]), len(blocks[2])


def tiny() -> DoryConfig:
    """Tiny fp32 Dory: hidden 256, 4 q heads over 1 kv head, hd 64, ffn 768, vocab 512,
    one input pair, two recurrent pairs, one output pair, loops 2, window 64, last_loop f32."""
    pat, a, b, c = pattern_of("S", "SS", "S")
    return DoryConfig(
        name="tiny-fp32", hidden=256, ffn=768, vocab=512, nh=4, nk=1, hd=64, window=64,
        pattern=pat, n_in=a, n_rec=b, n_out=c, loops=2, max_loops=16, kv_mode="last_loop",
        kv_quant="f32", weight_dtype="f32", sq=1.0, attn_sg=1.0, mlp_suv=1.0, logit_scale=1.0,
        alpha=(0.05, 0.05), max_context=512,
    )


def dory2b(rec_kinds: str = "SSSS", **kw) -> DoryConfig:
    """The 2B-shaped bf16 model: hidden 2048, 16 q over 4 kv heads, hd 128, ffn 5632,
    vocab 32000, 2/4/2 attention+MLP pairs, sliding window 512."""
    pat, a, b, c = pattern_of("SS", rec_kinds, "SS")
    base = dict(
        name="dory-2b", hidden=2048, ffn=5632, vocab=32000, nh=16, nk=4, hd=128, window=512,
        pattern=pat, n_in=a, n_rec=b, n_out=c, loops=4, max_loops=16, kv_mode="last_loop",
        kv_quant="f32", weight_dtype="bf16", sq=128.0, attn_sg=1.0, mlp_suv=1.0,
        logit_scale=1.0, alpha=(0.02, 0.1), max_context=16384 + 64, scale_spread=0.25,
    )
    base.update(kw)
    return DoryConfig(**base)


def small(rec_kinds: str = "S*", **kw) -> DoryConfig:
    """A reduced model with the 2B model's structure (GQA 4:1, several tiles per GEMM,
    sliding and full layers) that the oracle runs in seconds."""
    pat, a, b, c = pattern_of("S", rec_kinds, "S")
    base = dict(
        name="small", hidden=512, ffn=1024, vocab=1000, nh=8, nk=2, hd=64, window=48,
        pattern=pat, n_in=a, n_rec=b, n_out=c, loops=3, max_loops=16, kv_mode="last_loop",
        kv_quant="f32", weight_dtype="bf16", sq=64.0, attn_sg=6.0, mlp_suv=1.0,
        logit_scale=1.5, alpha=(0.02, 0.1), max_context=2048, scale_spread=0.5,
    )
    base.update(kw)
    return DoryConfig(**base)


# ----------------------------------------------------------------------------------------
# Draws
# ----------------------------------------------------------------------------------------

_POOL = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        import os

        _POOL = ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4))
    return _POOL


def unit_rows(seed: int, stream: int, rows: int, cols: int, dtype: str) -> np.ndarray:
    """[rows][cols] matrix, each row N(0,1) draws scaled to unit L2 norm, stored as
    float32 ("f32") or raw bfloat16 bits ("bf16", rounded from float32)."""
    out = np.empty((rows, cols), dtype=np.uint16 if dtype == "bf16" else np.float32)
    block = max(1, (1 << 20) // cols)

    def work(r0: int) -> None:
        r1 = min(rows, r0 + block)
        z = normal(seed, stream, (r1 - r0) * cols, start=r0 * cols).reshape(r1 - r0, cols)
        z /= np.sqrt(np.sum(z * z, axis=1, keepdims=True))
        z32 = z.astype(np.float32)
        out[r0:r1] = f32_to_bf16_bits(z32) if dtype == "bf16" else z32

    list(_pool().map(work, range(0, rows, block)))
    return out


def _uniform_range(seed: int, stream: int, n: int, lo: float, hi: float) -> np.ndarray:
    if lo == hi:
        return np.full(n, lo, dtype=np.float32)
    return (lo + (hi - lo) * uniform(seed, stream, n)).astype(np.float32)


def _scales(cfg: DoryConfig, seed: int, stream: int, n: int, base: float) -> np.ndarray:
    """n folded scale values: `base` times a uniform draw in [1 - spread, 1 + spread] each."""
    sp = cfg.scale_spread
    return (np.float64(base) * _uniform_range(seed, stream, n, 1.0 - sp, 1.0 + sp)).astype(np.float32)


def weights(cfg: DoryConfig, seed: int) -> dict:
    """Random-init weights of the given architecture, with the effective (folded) scales."""
    dt = cfg.weight_dtype
    q_size = cfg.nh * cfg.hd
    kv_row = cfg.nk * cfg.hd
    layers = []
    for li, kind in enumerate(cfg.pattern):
        s = 1000 + 32 * li
        alpha = _uniform_range(seed, s + 31, cfg.hidden, *cfg.alpha)
        if kind == "-":
            eff = cfg.mlp_suv * math.sqrt(cfg.hidden)
            layers.append(dict(
                kind="mlp",
                gate=unit_rows(seed, s + 0, cfg.ffn, cfg.hidden, dt),
                up=unit_rows(seed, s + 1, cfg.ffn, cfg.hidden, dt),
                down=unit_rows(seed, s + 2, cfg.hidden, cfg.ffn, dt),
                sg=_scales(cfg, seed, s + 5, cfg.ffn, eff),
                su=_scales(cfg, seed, s + 6, cfg.ffn, eff),
                alpha=alpha,
            ))
        else:
            layers.append(dict(
                kind="attn",
                sliding=(kind == "S"),
                q=unit_rows(seed, s + 0, q_size, cfg.hidden, dt),
                k=unit_rows(seed, s + 1, kv_row, cfg.hidden, dt),
                v=unit_rows(seed, s + 2, kv_row, cfg.hidden, dt),
                g=unit_rows(seed, s + 3, q_size, cfg.hidden, dt),
                o=unit_rows(seed, s + 4, cfg.hidden, q_size, dt),
                sq=_scales(cfg, seed, s + 5, q_size, cfg.sq),
                sg=_scales(cfg, seed, s + 6, q_size, cfg.attn_sg),
                alpha=alpha,
            ))
    return dict(
        embed=unit_rows(seed, 1, cfg.vocab, cfg.hidden, dt),
        head=unit_rows(seed, 2, cfg.vocab, cfg.hidden, dt),
        logit_scale=_scales(cfg, seed, 3, cfg.vocab, cfg.logit_scale),
        layers=layers,
    )


def token_ids(seed: int, stream: int, n: int, vocab: int) -> np.ndarray:
    """n uniform token ids in [0, vocab), int32."""
    return np.minimum((uniform(seed, 50_000 + stream, n) * vocab).astype(np.int64), vocab - 1).astype(np.int32)


def loop_schedule(seed: int, n: int, choices=(2, 4, 8)) -> np.ndarray:
    """One loop count per step, drawn uniformly from `choices`."""
    u = uniform(seed, 60_000, n)
    idx = np.minimum((u * len(choices)).astype(np.int64), len(choices) - 1)
    return np.asarray(choices, dtype=np.int32)[idx]


def kv_rows(seed: int, stream: int, n: int, nk: int, hd: int, start_row: int = 0) -> np.ndarray:
    """[n][nk][hd] float32 rows, each (row, kv head) vector N(0,1) scaled to unit norm."""
    z = normal(seed, 70_000 + stream, n * nk * hd, start=start_row * nk * hd).reshape(n, nk, hd)
    z /= np.sqrt(np.sum(z * z, axis=2, keepdims=True))
    return z.astype(np.float32)


def plain_rows(seed: int, stream: int, n: int, width: int) -> np.ndarray:
    """[n][width] float32 N(0,1) draws (no normalisation)."""
    return normal(seed, 80_000 + stream, n * width).reshape(n, width).astype(np.float32)
