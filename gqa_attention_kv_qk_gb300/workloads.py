"""Named decode workloads and their seeded synthetic inputs.

This module holds no arithmetic of the method: it names the workloads (shapes,
dtypes, rotary and masking parameters as plain data) and draws seeded random
tensors for them. Both the CUDA path's tests and benchmark and the oracle's
tests take their inputs from here, so the two sides see identical data; each
side then does its own arithmetic (quantising a vq8 cache included).

Draws are ~N(0, 1) in fp32 from torch's CPU generator, then cast to bf16
(round to nearest even) where the workload's dtype is bf16. Every tensor, and
every (sequence, kv head) slice of a cache, has its own generator seeded from
(workload seed, tensor tag, slice index), so slices can be drawn on their own
and the result never depends on the order of the draws.
"""
from __future__ import annotations

import copy

import numpy as np
import torch

TILE = 64  # cache capacities are rounded up to a multiple of this many slots

# The workloads. Method keys follow the oracle / library vocabulary;
# workload keys: batch, seq_len (int, or (lo, hi) inclusive for ragged lengths),
# steps, seed, layers (per-layer overrides; one cache per layer), page_size (a
# paged cache: pages of that many positions, assigned by block_table below), q_len
# (tokens per sequence in each step: a prefill chunk or draft tokens to verify).
CONFIGS: dict[str, dict] = {
    # Tiny Llama-3.2-1B-like step: fp32 everything, seed 0.
    "llama32_1b_tiny": dict(
        batch=1, n_q_heads=32, n_kv_heads=8, head_dim=64, seq_len=256, steps=1, seed=0,
        kv_dtype="f32", io_dtype="f32", out_dtype="f32",
        rope_style="interleaved", rope_theta=500000.0, rope_scaling="llama3", factor=32.0,
        low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192),
    # Llama-3.1-8B-like decode: 16 sequences at 8192 cached tokens, 64 steps.
    "llama31_8b_decode": dict(
        batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, seq_len=8192, steps=64, seed=1,
        kv_dtype="bf16", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=500000.0, rope_scaling="llama3", factor=8.0,
        low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192),
    # Qwen3-8B-like ragged decode: lengths uniform in [1024, 32768], QK RMSNorm.
    "qwen3_8b_ragged": dict(
        batch=32, n_q_heads=32, n_kv_heads=8, head_dim=128, seq_len=(1024, 32768), steps=1,
        seed=2, kv_dtype="bf16", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=1000000.0, rope_scaling="none",
        qk_norm=True, norm_eps=1e-6, norm_w_range=(0.5, 1.5)),
    # Gemma-2-9B-like decode: two layers per step (4096-token window, then global),
    # softcap 50, scale 1/sqrt(256).
    "gemma2_9b_swa": dict(
        batch=8, n_q_heads=16, n_kv_heads=8, head_dim=256, seq_len=16384, steps=1, seed=3,
        kv_dtype="bf16", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=10000.0, rope_scaling="none",
        softcap=50.0, scale=1.0 / 16.0, layers=[dict(window=4096), dict(window=0)]),
    # gpt-oss-like decode: vq8 cache, per-head sink logits, YaRN factor 32.
    "gptoss_vq8_sink": dict(
        batch=64, n_q_heads=64, n_kv_heads=8, head_dim=64, seq_len=4096, steps=1, seed=4,
        kv_dtype="vq8", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=150000.0, rope_scaling="yarn", factor=32.0,
        original_max_pos=4096, beta_fast=32.0, beta_slow=1.0, has_sink=True),
    # The Llama-3.1-8B-like decode over a q8 cache (int8 keys and values, one fp32
    # scale per token and kv head for each).
    "llama31_8b_q8": dict(
        batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, seq_len=8192, steps=64, seed=6,
        kv_dtype="q8", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=500000.0, rope_scaling="llama3", factor=8.0,
        low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192),
    # The Llama-3.1-8B-like decode over a paged bf16 cache: pages of 16 positions,
    # in seeded random order over a pool with spare pages.
    "llama31_8b_paged": dict(
        batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, seq_len=8192, steps=64, seed=7,
        kv_dtype="bf16", io_dtype="bf16", out_dtype="f32", page_size=16,
        rope_style="neox", rope_theta=500000.0, rope_scaling="llama3", factor=8.0,
        low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192),
    # The Llama-3.1-8B-like cache with 4 tokens per sequence and step (draft tokens
    # to verify), each attending the cache and the chunk's earlier tokens.
    "llama31_8b_verify": dict(
        batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, seq_len=8192, steps=16, seed=8, q_len=4,
        kv_dtype="bf16", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=500000.0, rope_scaling="llama3", factor=8.0,
        low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192),
    # The Llama-3.1-8B-like cache with a 512-token prefill chunk per sequence and step
    # (each token attends the cache and the chunk's earlier tokens).
    "llama31_8b_prefill": dict(
        batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, seq_len=8192, steps=1, seed=9, q_len=512,
        kv_dtype="bf16", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=500000.0, rope_scaling="llama3", factor=8.0,
        low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192),
    # Gemma-3-12B-like decode: QK RMSNorm whose weights are stored as deltas from
    # one (applied as 1 + w), scale 1/sqrt(256), no softcap; one layer of each
    # kind per step (the model runs five local layers per global one): a local
    # layer with a 1024-token window and base 10^4, a global one with base 10^6
    # and linear scaling 8.
    "gemma3_12b_local_global": dict(
        batch=8, n_q_heads=16, n_kv_heads=8, head_dim=256, seq_len=(1024, 16384), steps=1, seed=5,
        kv_dtype="bf16", io_dtype="bf16", out_dtype="f32",
        rope_style="neox", rope_theta=1000000.0, rope_scaling="linear", factor=8.0,
        qk_norm=True, norm_offset=True, norm_eps=1e-6, norm_w_range=(-0.5, 0.5), scale=1.0 / 16.0,
        layers=[dict(window=1024, rope_theta=10000.0, rope_scaling="none", factor=1.0), dict(window=0)]),
}

_TAGS = {"q": 1, "k_new": 2, "v_new": 3, "k_cache": 4, "v_cache": 5, "q_norm_w": 6,
         "k_norm_w": 7, "sink": 8, "seq_lens": 9, "block_table": 10}


def config(name: str, **overrides) -> dict:
    """A copy of a named workload with keys overridden (for smaller test cases)."""
    cfg = copy.deepcopy(CONFIGS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


def layer_configs(cfg: dict) -> list[dict]:
    """One config per layer (a workload without 'layers' has one layer)."""
    layers = cfg.get("layers") or [{}]
    out = []
    for i, over in enumerate(layers):
        c = copy.deepcopy(cfg)
        c.pop("layers", None)
        c.update(over)
        c["layer"] = i
        out.append(c)
    return out


def _gen(seed: int, tag: str, idx: int = 0, layer: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + _TAGS[tag] * 10_007 + layer * 101 + idx) % (2**62))
    return g


def _cast(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return x
    if dtype in ("bf16", "vq8"):
        return x.to(torch.bfloat16)
    raise ValueError(dtype)


def capacity(cfg: dict, extra: int = 0) -> int:
    """Slots per (sequence, kv head): the longest cached length + extra (tokens the
    steps append), rounded up to a multiple of 64 and of the page size of a paged
    workload."""
    sl = cfg["seq_len"]
    longest = sl[1] if isinstance(sl, (tuple, list)) else sl
    need = longest + max(extra, int(cfg.get("q_len", 1) or 1))
    unit = max(TILE, int(cfg.get("page_size", 0) or 0))
    return (need + unit - 1) // unit * unit


def block_table(cfg: dict, pages_per_seq: int, n_pages: int) -> torch.Tensor:
    """A paged workload's block table [B][pages_per_seq] int32: distinct pages of a
    pool of n_pages, in seeded random order (the pool's other pages stay unused)."""
    B = cfg["batch"]
    assert n_pages >= B * pages_per_seq
    perm = torch.randperm(n_pages, generator=_gen(cfg["seed"], "block_table", 0, cfg.get("layer", 0)))
    return perm[: B * pages_per_seq].reshape(B, pages_per_seq).to(torch.int32)


def seq_lens(cfg: dict) -> torch.Tensor:
    """Cached tokens per sequence before the first step (int32 [B])."""
    B = cfg["batch"]
    sl = cfg["seq_len"]
    if isinstance(sl, (tuple, list)):
        return torch.randint(int(sl[0]), int(sl[1]) + 1, (B,), generator=_gen(cfg["seed"], "seq_lens"),
                             dtype=torch.int64).to(torch.int32)
    return torch.full((B,), int(sl), dtype=torch.int32)


def step_inputs(cfg: dict, step: int = 0) -> dict:
    """q [B][Hq][D], k_new and v_new [B][Hkv][D] in the io dtype, fresh for each step;
    with cfg q_len = T > 1 a chunk of T tokens per sequence, [B][T][H][D]."""
    B, Hq, Hkv, D = cfg["batch"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    layer = cfg.get("layer", 0)
    io = cfg.get("io_dtype", "bf16")
    T = int(cfg.get("q_len", 1) or 1)
    tok = (T,) if T > 1 else ()
    out = {}
    for tag, shape in (("q", (B, *tok, Hq, D)), ("k_new", (B, *tok, Hkv, D)), ("v_new", (B, *tok, Hkv, D))):
        x = torch.randn(shape, generator=_gen(cfg["seed"], tag, step, layer), dtype=torch.float32)
        out[tag] = _cast(x, io)
    return out


def norm_weights(cfg: dict) -> dict:
    """QK RMSNorm weights [D] fp32, ~U(lo, hi); None when the workload has no norm."""
    if not cfg.get("qk_norm"):
        return {"q_norm_w": None, "k_norm_w": None}
    lo, hi = cfg.get("norm_w_range", (1.0, 1.0))
    D = cfg["head_dim"]
    layer = cfg.get("layer", 0)
    out = {}
    for tag in ("q_norm_w", "k_norm_w"):
        u = torch.rand((D,), generator=_gen(cfg["seed"], tag, 0, layer), dtype=torch.float32)
        out[tag] = (lo + (hi - lo) * u).to(torch.float32)
    return out


def sinks(cfg: dict):
    """Per-query-head sink logits [Hq] fp32 ~N(0, 1); None without sinks."""
    if not cfg.get("has_sink"):
        return None
    return torch.randn((cfg["n_q_heads"],), generator=_gen(cfg["seed"], "sink", 0, cfg.get("layer", 0)),
                       dtype=torch.float32)


def cache_slice(cfg: dict, b: int, g: int, n: int, which: str) -> torch.Tensor:
    """Rows [0, n) of cache slice (b, g): k in the key storage dtype (f32 / bf16);
    v in f32 / bf16, or as fp32 values for a vq8 cache (each side quantises them);
    a q8 cache has both k and v as fp32 values."""
    D, Hkv = cfg["head_dim"], cfg["n_kv_heads"]
    idx = b * Hkv + g
    x = torch.randn((n, D), generator=_gen(cfg["seed"], which, idx, cfg.get("layer", 0)),
                    dtype=torch.float32)
    kv = cfg.get("kv_dtype", "bf16")
    if kv in ("f32", "q8"):
        return x
    if which == "k_cache" or kv == "bf16":
        return x.to(torch.bfloat16)
    return x  # vq8 values, fp32


def cache(cfg: dict, cap: int, lens: torch.Tensor, fill_unused: str = "zero") -> dict:
    """Host caches [B][Hkv][cap][D] with rows [0, lens[b]) drawn; unused rows are
    zero or NaN (fill_unused='nan', to prove they are never read into a result).
    For vq8 'v_values' holds fp32 values, for q8 'k_values' too; each side
    quantises them itself."""
    B, Hkv, D = cfg["batch"], cfg["n_kv_heads"], cfg["head_dim"]
    kv = cfg.get("kv_dtype", "bf16")
    kdt = torch.float32 if kv in ("f32", "q8") else torch.bfloat16
    vdt = torch.float32 if kv in ("f32", "vq8", "q8") else torch.bfloat16
    fill = float("nan") if fill_unused == "nan" else 0.0
    k = torch.full((B, Hkv, cap, D), fill, dtype=kdt)
    v = torch.full((B, Hkv, cap, D), fill, dtype=vdt)
    for b in range(B):
        n = int(lens[b])
        for g in range(Hkv):
            k[b, g, :n] = cache_slice(cfg, b, g, n, "k_cache")
            v[b, g, :n] = cache_slice(cfg, b, g, n, "v_cache")
    kkey = "k_values" if kv == "q8" else "k_cache"
    vkey = "v_values" if kv in ("vq8", "q8") else "v_cache"
    return {kkey: k, vkey: v}


def host_case(cfg: dict, lens=None, cap=None, step: int = 0, fill_unused: str = "zero") -> dict:
    """One step's seeded inputs and cache on the host: cfg, lens [B] int32, cap,
    the cache tensors of cache(), the step inputs of step_inputs(), the norm
    weights and the sinks. cap defaults to the workload's longest length plus
    every token its steps append."""
    lens = seq_lens(cfg) if lens is None else torch.as_tensor(lens, dtype=torch.int32)
    cap = cap or capacity(cfg, extra=cfg.get("steps", 1) * int(cfg.get("q_len", 1) or 1))
    case = dict(cfg=cfg, lens=lens.clone(), cap=cap)
    case.update(cache(cfg, cap, lens, fill_unused=fill_unused))
    case.update(step_inputs(cfg, step))
    case.update(norm_weights(cfg))
    case["sink"] = sinks(cfg)
    return case


# ---------------------------------------------------------------- numpy views

def bits(t: torch.Tensor) -> np.ndarray:
    """A CPU tensor as the numpy array the oracle takes (bf16 -> uint16 bit patterns)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
