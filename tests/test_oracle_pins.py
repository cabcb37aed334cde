"""Pins of the CPU oracle against things other than itself.

Each pin is a value the pages print (tests/golden/pages_facts.json), a closed
form, an invariant of the mathematics, a library routine (torch's bf16 cast,
numpy float32 arithmetic) or the matrix-form brute force of tests/bruteforce.py
on tiny inputs. The negative controls at the end plant mistakes in the oracle's
inputs and check that the parity tolerance sees them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from gqa_attention_kv_qk_gb300 import workloads as W
from tests import bruteforce as BF
from tests.cases import host_case, oracle_arrays, run_oracle_step

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")))
TOL_MAX, TOL_MEAN = 2e-3, 2e-4  # the GPU parity bar; used by the negative controls


def rope_cfg(**kw):
    c = dict(n_q_heads=4, n_kv_heads=1, head_dim=64, rope_style="neox", rope_theta=10000.0,
             rope_scaling="none")
    c.update(kw)
    return c


def unscaled(oracle_mod, cfg):
    """The oracle's own plain table (pinned to the closed form in
    test_unscaled_table_is_the_closed_form), so divisor ratios are exact."""
    return oracle_mod.rope_inv_freq(dict(cfg, rope_scaling="none"))[0]


@pytest.mark.parametrize("D,base", [(64, 500000.0), (128, 500000.0), (256, 10000.0), (64, 150000.0)])
def test_unscaled_table_is_the_closed_form(oracle_mod, D, base):
    inv, ms = oracle_mod.rope_inv_freq(rope_cfg(head_dim=D, rope_theta=base))
    assert ms == 1.0 and inv[0] == 1.0
    assert np.allclose(inv, BF.plain_inv_freq(D, base), rtol=4e-16, atol=0)


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_matches_torch_cast(oracle_mod):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(4000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(4000, generator=g) * 20)
    # exact ties: a bf16 value plus half an ulp
    base = torch.randn(200, generator=g).to(torch.bfloat16).to(torch.float32)
    ties = (base.view(torch.int32) + 0x8000).view(torch.float32)
    special = torch.tensor([0.0, -0.0, 1e-40, -1e-40, 3.4e38, -3.4e38, 3.3895e38, 1.0, -1.0],
                           dtype=torch.float32)
    x = torch.cat([x, ties, special])
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.bf16_from_f64(x.to(torch.float64).numpy())
    assert np.array_equal(got, want)
    back = oracle_mod.bf16_to_f64(want)
    assert np.array_equal(back, x.to(torch.bfloat16).to(torch.float64).numpy())


# ------------------------------------------------------------------ RoPE frequencies

@pytest.mark.parametrize("model", GOLD["llama3_recovered"]["models"], ids=lambda m: m["name"])
def test_llama3_max_divisor_is_factor_and_rederives(oracle_mod, model):
    """FreeToken PR #722: factor = max(divisors) and re-deriving reproduces them."""
    fx = GOLD["llama3_recovered"]
    cfg = rope_cfg(head_dim=model["head_dim"], rope_theta=model["rope_theta"],
                   rope_scaling="llama3", factor=model["factor"],
                   low_freq_factor=fx["low_freq_factor"], high_freq_factor=fx["high_freq_factor"],
                   original_max_pos=fx["original_max_pos"])
    inv, ms = oracle_mod.rope_inv_freq(cfg)
    plain = unscaled(oracle_mod, cfg)
    div = plain / inv
    assert ms == 1.0
    assert div.max() == pytest.approx(model["factor"], rel=1e-14)
    recovered = dict(cfg, factor=float(div.max()))
    inv2, _ = oracle_mod.rope_inv_freq(recovered)
    assert np.allclose(plain / inv2, div, rtol=1e-13, atol=0)


@pytest.mark.parametrize("D,factor", [(64, 32.0), (128, 8.0)])
def test_llama3_regions_by_closed_form(oracle_mod, D, factor):
    """Regions solved for the pair index: wavelength 2 pi base^(2p/D) < 8192/4 keeps
    theta, > 8192/1 divides it by factor, in between the divisor rises monotonically."""
    base, orig = 500000.0, 8192
    cfg = rope_cfg(head_dim=D, rope_theta=base, rope_scaling="llama3", factor=factor,
                   low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=orig)
    inv, _ = oracle_mod.rope_inv_freq(cfg)
    div = unscaled(oracle_mod, cfg) / inv
    p = np.arange(D // 2)
    p_short = (D / 2) * math.log(orig / 4 / (2 * math.pi)) / math.log(base)
    p_long = (D / 2) * math.log(orig / 1 / (2 * math.pi)) / math.log(base)
    assert np.all(div[p < p_short] == 1.0)
    assert np.allclose(div[p > p_long], factor, rtol=1e-14)
    mid = div[(p >= p_short) & (p <= p_long)]
    assert mid.size > 0 and np.all(mid > 1.0) and np.all(mid < factor)
    assert np.all(np.diff(div) >= 0)
    # The decoder page's numeric check: the first 8 frequencies of the Llama-3.1-8B
    # configuration are the plain ones (those pairs are all short-wavelength).
    if D == 128:
        assert np.array_equal(inv[:8], unscaled(oracle_mod, cfg)[:8])
        assert np.allclose(inv[:8], np.power(base, -np.arange(8) * 2.0 / 128), rtol=4e-16)


def test_llama3_smooth_region_values(oracle_mod):
    """In the smooth region 1/divisor is linear in original/wavelength: it runs from
    1/factor at wavelength = original/low to 1 at wavelength = original/high."""
    D, base, factor, orig = 64, 500000.0, 32.0, 8192.0
    cfg = rope_cfg(head_dim=D, rope_theta=base, rope_scaling="llama3", factor=factor,
                   low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=int(orig))
    inv, _ = oracle_mod.rope_inv_freq(cfg)
    plain = unscaled(oracle_mod, cfg)
    r = orig * plain / (2 * math.pi)              # rotations in the original context
    sel = (r > 1.0) & (r < 4.0)
    # (1/div - 1/factor) / (1 - 1/factor) must equal (r - 1) / (4 - 1)
    t = (inv[sel] / plain[sel] - 1 / factor) / (1 - 1 / factor)
    assert np.allclose(t, (r[sel] - 1.0) / 3.0, rtol=0, atol=1e-13)
    assert sel.sum() == 3  # pairs 15, 16, 17 for this configuration


def test_unscaled_first_frequency_and_yarn_reductions(oracle_mod):
    inv, ms = oracle_mod.rope_inv_freq(rope_cfg(rope_theta=500000.0))
    assert inv[0] == 1.0 and ms == 1.0
    # YaRN with factor 1 is plain RoPE with multiplier 1
    y1, m1 = oracle_mod.rope_inv_freq(rope_cfg(rope_theta=150000.0, rope_scaling="yarn",
                                               factor=1.0, original_max_pos=4096))
    assert np.array_equal(y1, unscaled(oracle_mod, rope_cfg(rope_theta=150000.0))) and m1 == 1.0


def test_yarn_ramp_endpoints_and_mscale(oracle_mod):
    D, base, factor, orig = 64, 150000.0, 32.0, 4096
    inv, ms = oracle_mod.rope_inv_freq(rope_cfg(head_dim=D, rope_theta=base, rope_scaling="yarn",
                                                factor=factor, original_max_pos=orig,
                                                beta_fast=32.0, beta_slow=1.0))
    div = unscaled(oracle_mod, rope_cfg(head_dim=D, rope_theta=base)) / inv
    # pair whose wavelength fits n times into the original context: solve
    # orig / (2 pi base^(2p/D)) = n for p
    lo = D * math.log(orig / (2 * math.pi * 32.0)) / (2 * math.log(base))
    hi = D * math.log(orig / (2 * math.pi * 1.0)) / (2 * math.log(base))
    assert 8.0 < lo < 8.2 and 17.3 < hi < 17.5
    p = np.arange(D // 2)
    assert np.all(div[p <= math.floor(lo)] == 1.0)
    assert np.allclose(div[p >= math.ceil(hi)], factor, rtol=1e-14)
    assert np.all(np.diff(div) >= 0)
    assert ms == pytest.approx(1.0 + 0.1 * math.log(32.0), rel=1e-15)


def rotations_in_original_context(D, base, orig, p):
    """How many turns pair p (a real number here) makes over the original context:
    orig / wavelength = orig * base^(-2p/D) / (2 pi)."""
    return orig * np.power(base, -2.0 * np.asarray(p, dtype=np.float64) / D) / (2 * math.pi)


def yarn_ramp_violations(inv, plain, D, base, factor, orig, beta_fast, beta_slow):
    """Checks a YaRN frequency table against the reading of the gpt-oss YaRN ramp
    (llamay "Architectures": gpt-oss uses YaRN; the pages give no formula): the
    kept share u_p = (theta'_p / theta_p - 1/factor) / (1 - 1/factor) of every pair
    is 1 where the pair turns more than beta_fast times over the original context,
    0 where it turns fewer than beta_slow times, and in between lies on ONE straight
    line in the pair index whose ends, extended to u = 1 and u = 0, fall on the
    (real-valued) pair indices that turn exactly beta_fast and beta_slow times.
    Returns the list of violated conditions (empty when the table passes)."""
    bad = []
    u = (inv / plain - 1.0 / factor) / (1.0 - 1.0 / factor)
    p = np.arange(D // 2, dtype=np.float64)
    r = rotations_in_original_context(D, base, orig, p)
    keep, squash = r > beta_fast, r < beta_slow
    mid = ~keep & ~squash
    if not np.allclose(u[keep], 1.0, rtol=0, atol=1e-13):
        bad.append("pairs above beta_fast turns are changed")
    if not np.allclose(u[squash], 0.0, rtol=0, atol=1e-13):
        bad.append("pairs below beta_slow turns are not divided by the factor")
    pm, um = p[mid], u[mid]
    if pm.size < 3:
        bad.append("fewer than three pairs inside the ramp")
        return bad
    if np.any(um <= 0.0) or np.any(um >= 1.0):
        bad.append("a ramp pair is at an end value")
    if np.abs(np.diff(um, 2)).max() > 1e-12:
        bad.append("the ramp is not a straight line in the pair index")
    slope, icpt = np.polyfit(pm, um, 1)
    p_one, p_zero = (1.0 - icpt) / slope, -icpt / slope
    if abs(rotations_in_original_context(D, base, orig, p_one) / beta_fast - 1) > 1e-9:
        bad.append("the ramp does not leave 1 where a pair turns beta_fast times")
    if abs(rotations_in_original_context(D, base, orig, p_zero) / beta_slow - 1) > 1e-9:
        bad.append("the ramp does not reach 0 where a pair turns beta_slow times")
    return bad


YARN_RAMP_CASES = [(64, 150000.0, 32.0, 4096), (128, 150000.0, 32.0, 4096),
                   (64, 10000.0, 16.0, 4096), (128, 10000.0, 32.0, 4096), (128, 1e6, 4.0, 32768)]


@pytest.mark.parametrize("D,base,factor,orig", YARN_RAMP_CASES)
def test_yarn_ramp_interior(oracle_mod, D, base, factor, orig):
    """Every pair of the oracle's YaRN table, the interior of the ramp included,
    against the turn counts over the original context (no rounding of the ends)."""
    cfg = rope_cfg(head_dim=D, rope_theta=base, rope_scaling="yarn", factor=factor,
                   original_max_pos=orig, beta_fast=32.0, beta_slow=1.0)
    inv, _ = oracle_mod.rope_inv_freq(cfg)
    plain = BF.plain_inv_freq(D, base)
    assert yarn_ramp_violations(inv, plain, D, base, factor, orig, 32.0, 1.0) == []


@pytest.mark.parametrize("variant", ["rounded_ends", "linear_in_divisor", "linear_in_turns"])
@pytest.mark.parametrize("D,base,factor,orig", YARN_RAMP_CASES[:4])
def test_yarn_ramp_pin_rejects_other_ramps(D, base, factor, orig, variant):
    """Negative controls for the interior pin: the other common readings of the YaRN
    ramp (ends rounded down / up to whole pairs; a ramp on the divisor instead of
    the frequency; a ramp linear in the turn count) are tables the pin must refuse."""
    plain = BF.plain_inv_freq(D, base)
    p = np.arange(D // 2, dtype=np.float64)
    lo = D * math.log(orig / (2 * math.pi * 32.0)) / (2 * math.log(base))
    hi = D * math.log(orig / (2 * math.pi * 1.0)) / (2 * math.log(base))
    if variant == "rounded_ends":
        ramp = np.clip((p - math.floor(lo)) / (math.ceil(hi) - math.floor(lo)), 0, 1)
        inv = plain / factor * ramp + plain * (1 - ramp)
    elif variant == "linear_in_divisor":
        ramp = np.clip((p - lo) / (hi - lo), 0, 1)
        inv = plain / (1 + ramp * (factor - 1))
    else:
        r = rotations_in_original_context(D, base, orig, p)
        keep = np.clip((r - 1.0) / (32.0 - 1.0), 0, 1)
        inv = plain * keep + plain / factor * (1 - keep)
    assert yarn_ramp_violations(inv, plain, D, base, factor, orig, 32.0, 1.0) != []


# ------------------------------------------------------------------ RoPE rotation

@pytest.mark.parametrize("style", ["neox", "interleaved"])
@pytest.mark.parametrize("scaling", ["none", "llama3"])
def test_rotation_is_a_rotation(oracle_mod, style, scaling):
    cfg = rope_cfg(rope_style=style, rope_scaling=scaling, rope_theta=500000.0, factor=32.0,
                   low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192)
    rng = np.random.default_rng(1)
    x = rng.standard_normal(64)
    ia, ib = BF.pair_indices(64, style)
    for pos in (0, 1, 7, 4097, 32768):
        y = oracle_mod.rope_rotate(cfg, x, pos)
        # every pair keeps its length
        assert np.allclose(np.hypot(y[ia], y[ib]), np.hypot(x[ia], x[ib]), rtol=1e-12, atol=0)
        if pos == 0:
            assert np.array_equal(y, x)


@pytest.mark.parametrize("style", ["neox", "interleaved"])
def test_rotation_matches_complex_multiplication(oracle_mod, style):
    """Pair (a, b) as a + ib multiplied by exp(i pos theta_p)."""
    cfg = rope_cfg(rope_style=style, rope_theta=10000.0)
    rng = np.random.default_rng(2)
    x = rng.standard_normal(64)
    ia, ib = BF.pair_indices(64, style)
    theta = BF.plain_inv_freq(64, 10000.0)
    for pos in (3, 1000):
        z = (x[ia] + 1j * x[ib]) * np.exp(1j * pos * theta)
        y = oracle_mod.rope_rotate(cfg, x, pos)
        assert np.allclose(y[ia], z.real, atol=1e-12) and np.allclose(y[ib], z.imag, atol=1e-12)


@pytest.mark.parametrize("style", ["neox", "interleaved"])
def test_relative_position_identity(oracle_mod, style):
    cfg = rope_cfg(rope_style=style, rope_theta=500000.0, rope_scaling="llama3", factor=8.0,
                   low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192)
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n, t in ((10, 3, 1000), (8192, 0, 17), (5, 5, 30000)):
        a = oracle_mod.rope_rotate(cfg, q, m) @ oracle_mod.rope_rotate(cfg, k, n)
        b = oracle_mod.rope_rotate(cfg, q, m + t) @ oracle_mod.rope_rotate(cfg, k, n + t)
        assert a == pytest.approx(b, rel=1e-9, abs=1e-9)


def test_interleaved_is_permuted_neox(oracle_mod):
    """FreeToken PR #722 'Changes': interleaved RoPE on rows equals NeoX RoPE on the
    un-permuted rows. P sends NeoX index p -> 2p and p + D/2 -> 2p + 1."""
    D = 64
    perm = np.empty(D, dtype=int)
    perm[np.arange(D // 2)] = 2 * np.arange(D // 2)
    perm[np.arange(D // 2) + D // 2] = 2 * np.arange(D // 2) + 1
    rng = np.random.default_rng(4)
    x = rng.standard_normal(D)
    cfg_n = rope_cfg(rope_style="neox", rope_theta=500000.0)
    cfg_i = rope_cfg(rope_style="interleaved", rope_theta=500000.0)
    for pos in (1, 77, 9000):
        x_neox = np.empty(D)
        x_neox[np.arange(D)] = x[perm]          # un-permute: neox slot p holds row perm[p]
        y_neox = oracle_mod.rope_rotate(cfg_n, x_neox, pos)
        y_i = oracle_mod.rope_rotate(cfg_i, x, pos)
        y_back = np.empty(D)
        y_back[perm] = y_neox
        assert np.allclose(y_i, y_back, atol=1e-13)


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_one_row_and_invariants(oracle_mod):
    """Decoder page P1.1: one-row RMSNorm against NumPy; plus the closed forms."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(128)
    w = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    y = oracle_mod.rms_norm(x, w, 1e-6)
    assert np.allclose(y, x / np.sqrt(np.mean(x * x) + 1e-6) * w, rtol=1e-14)
    ones = np.ones(128, dtype=np.float32)
    y1 = oracle_mod.rms_norm(x, ones, 0.0)
    assert np.sqrt(np.mean(y1 * y1)) == pytest.approx(1.0, rel=1e-14)
    for c in (-3.0, 0.25):
        yc = oracle_mod.rms_norm(np.full(64, c), np.ones(64, dtype=np.float32), 1e-6)
        assert np.allclose(yc, np.sign(c) / math.sqrt(1 + 1e-6 / c ** 2), rtol=1e-14)


def test_rmsnorm_weight_offset(oracle_mod):
    """Decoder page P1.1: a weight stored as a delta from one applies as (1 + w);
    a zero delta is the unit-weight norm, and the offset adds x / rms(x)."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal(256)
    w = rng.uniform(-0.5, 0.5, 256).astype(np.float32)
    y = oracle_mod.rms_norm(x, w, 1e-6, 1.0)
    r = np.sqrt(np.mean(x * x) + 1e-6)
    assert np.allclose(y, x / r * (1.0 + w.astype(np.float64)), rtol=1e-14)
    zeros, ones = np.zeros(256, dtype=np.float32), np.ones(256, dtype=np.float32)
    assert np.array_equal(oracle_mod.rms_norm(x, zeros, 1e-6, 1.0), oracle_mod.rms_norm(x, ones, 1e-6, 0.0))
    assert np.allclose(y - oracle_mod.rms_norm(x, w, 1e-6, 0.0), x / r, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------ partial rotary, linear scaling

@pytest.mark.parametrize("style,D,R", [("neox", 64, 32), ("neox", 128, 96), ("interleaved", 64, 16),
                                       ("neox", 256, 64)])
def test_partial_rotary_rotates_the_first_dims_only(oracle_mod, style, D, R):
    """Decoder page P1.5: rotary_dim = head_dim * partial_rotary_factor dims
    rotate, with the frequencies of an R-wide head; the other dims pass as they
    are. Checked against complex multiplication and against the full rotation of
    an R-wide head on the first R dims."""
    base = 10000.0
    cfg = rope_cfg(rope_style=style, head_dim=D, rotary_dim=R, rope_theta=base)
    inv, ms = oracle_mod.rope_inv_freq(cfg)
    theta = base ** (-np.arange(R // 2) * 2.0 / R)
    assert np.allclose(inv[: R // 2], theta, rtol=1e-15) and not inv[R // 2:].any() and ms == 1.0
    rng = np.random.default_rng(7)
    x = rng.standard_normal(D)
    ia, ib = BF.pair_indices(R, style)
    head_r = rope_cfg(rope_style=style, head_dim=R, rope_theta=base)
    for pos in (0, 5, 3001):
        y = oracle_mod.rope_rotate(cfg, x, pos)
        assert np.array_equal(y[R:], x[R:])
        z = (x[ia] + 1j * x[ib]) * np.exp(1j * pos * theta)
        assert np.allclose(y[ia], z.real, atol=1e-12) and np.allclose(y[ib], z.imag, atol=1e-12)
        assert np.array_equal(y[:R], oracle_mod.rope_rotate(head_r, x[:R].copy(), pos))


def test_full_rotary_dim_is_the_default(oracle_mod):
    rng = np.random.default_rng(9)
    x = rng.standard_normal(128)
    for style in ("neox", "interleaved"):
        a = rope_cfg(rope_style=style, head_dim=128, rope_scaling="yarn", factor=32.0, original_max_pos=4096)
        for pos in (1, 70000):
            assert np.array_equal(oracle_mod.rope_rotate(a, x, pos),
                                  oracle_mod.rope_rotate(dict(a, rotary_dim=128), x, pos))


def test_yarn_factor_leaves_pass_through_dims_alone(oracle_mod):
    """The attention factor scales the rotated pairs only (each keeps length
    mscale times its own); dims beyond rotary_dim are copied."""
    cfg = rope_cfg(head_dim=64, rotary_dim=32, rope_scaling="yarn", factor=32.0, original_max_pos=4096,
                   rope_theta=150000.0)
    inv, ms = oracle_mod.rope_inv_freq(cfg)
    assert ms == pytest.approx(0.1 * math.log(32.0) + 1.0, rel=1e-15)
    x = np.random.default_rng(10).standard_normal(64)
    y = oracle_mod.rope_rotate(cfg, x, 999)
    ia, ib = BF.pair_indices(32, "neox")
    assert np.allclose(np.hypot(y[ia], y[ib]), ms * np.hypot(x[ia], x[ib]), rtol=1e-13)
    assert np.array_equal(y[32:], x[32:])


@pytest.mark.parametrize("factor", [8.0, 4.0])
def test_linear_scaling_divides_positions(oracle_mod, factor):
    """Support matrix, gemma3 lane: linear scaling of the global layers. Every
    frequency is divided by the factor, so position f t rotates as position t
    does without scaling (bit for bit: a power-of-two factor scales exactly)."""
    cfg = rope_cfg(head_dim=128, rope_theta=1000000.0, rope_scaling="linear", factor=factor)
    inv, ms = oracle_mod.rope_inv_freq(cfg)
    assert np.array_equal(inv, unscaled(oracle_mod, cfg) / factor) and ms == 1.0
    plain = dict(cfg, rope_scaling="none")
    x = np.random.default_rng(11).standard_normal(128)
    for t in (1, 100, 4096):
        assert np.array_equal(oracle_mod.rope_rotate(cfg, x, int(factor) * t), oracle_mod.rope_rotate(plain, x, t))


# ------------------------------------------------------------------ vq8

def test_vq8_codes_bit_exact_vs_numpy_fp32(oracle_mod):
    g = torch.Generator().manual_seed(6)
    v = torch.randn(500, 64, generator=g).numpy().astype(np.float32)
    v[3] = 0.0                      # all-zero row
    v[4] = np.float32(1e-30)        # tiny values
    v[5, :] = np.linspace(-1, 1, 64, dtype=np.float32)
    codes, scales = oracle_mod.vq8_quantize(v)
    c2, s2 = BF.vq8_numpy(v)
    assert np.array_equal(codes, c2) and np.array_equal(scales.view(np.uint32), s2.view(np.uint32))
    assert np.all(np.abs(codes.astype(int)) <= 127)
    assert scales[3] == 0 and np.all(codes[3] == 0)
    nz = scales > 0
    arg = np.argmax(np.abs(v), axis=1)
    assert np.all(np.abs(codes[np.arange(500), arg][nz]) == 127)
    err = np.abs(codes.astype(np.float64) * scales[:, None] - v)
    assert np.all(err <= scales[:, None] * (0.5 + 1e-6) + 1e-45)


# ------------------------------------------------------------------ attention

def tiny(name="llama31_8b_decode", **kw):
    base = dict(batch=2, seq_len=(0, 40), steps=1)
    base.update(kw)
    return W.config(name, **base)


def test_one_key_cache_returns_v(oracle_mod):
    for kw in (dict(), dict(softcap=5.0), dict(window=1, seq_len=30)):
        cfg = tiny(**kw)
        case = host_case(cfg, lens=[0, 0] if "window" not in kw else [30, 12])
        out, a = run_oracle_step(case, oracle_mod)
        v = W.bits(case["v_new"]).astype(np.float64)
        v = oracle_mod.bf16_to_f64(W.bits(case["v_new"])).reshape(v.shape)
        G = cfg["n_q_heads"] // cfg["n_kv_heads"]
        assert np.allclose(out, np.repeat(v, G, axis=1), rtol=0, atol=1e-15)


def test_one_key_sink_mass_closed_form(oracle_mod):
    """First token (position 0): the rotation is the identity times the YaRN
    multiplier m, the stored key is bf16(m k) (torch's cast), and with one key
    out = v / (1 + exp(sink - s)), s = scale m (q . bf16(m k))."""
    cfg = tiny("gptoss_vq8_sink", batch=3, n_q_heads=8, n_kv_heads=2)
    case = host_case(cfg, lens=[0, 0, 0])
    out, a = run_oracle_step(case, oracle_mod)
    q = case["q"].to(torch.float64).numpy()
    _, ms = oracle_mod.rope_inv_freq(cfg)
    k_st = BF.bf16_round(ms * case["k_new"].to(torch.float64).numpy())
    codes, scales = BF.vq8_numpy(case["v_new"].to(torch.float32).numpy())
    vdq = codes.astype(np.float64) * scales[..., None].astype(np.float64)
    G = 4
    for b in range(3):
        for h in range(8):
            s = ms * (q[b, h] @ k_st[b, h // G]) / math.sqrt(64)
            want = vdq[b, h // G] / (1.0 + math.exp(case["sink"][h].item() - s))
            assert np.allclose(out[b, h], want, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("extra", [dict(), dict(window=7), dict(softcap=3.0), dict(has_sink=True)])
def test_zero_query_gives_mean_of_visible_values(oracle_mod, extra):
    cfg = tiny(**extra)
    case = host_case(cfg, lens=[20, 33])
    case["q"] = torch.zeros_like(case["q"])
    out, a = run_oracle_step(case, oracle_mod)
    G = cfg["n_q_heads"] // cfg["n_kv_heads"]
    for b in range(2):
        n = int(a["seq_lens"][b])
        lo = max(0, n - extra.get("window", 0)) if extra.get("window") else 0
        v = oracle_mod.bf16_to_f64(a["v_cache"][b, :, lo:n]).reshape(cfg["n_kv_heads"], n - lo, -1)
        for h in range(cfg["n_q_heads"]):
            den = (n - lo) + (math.exp(case["sink"][h].item()) if extra.get("has_sink") else 0.0)
            assert np.allclose(out[b, h], v[h // G].sum(0) / den, rtol=1e-12, atol=1e-14)


def test_gqa_mapping_contiguous_groups(oracle_mod):
    cfg = tiny(n_q_heads=8, n_kv_heads=2, kv_dtype="f32", io_dtype="f32")
    case = host_case(cfg, lens=[5, 9])
    for g in range(2):
        case["v_cache"][:, g] = float(g + 1)
    case["v_new"][:, 0] = 1.0
    case["v_new"][:, 1] = 2.0
    out, _ = run_oracle_step(case, oracle_mod)
    assert np.allclose(out[:, :4], 1.0, atol=1e-14) and np.allclose(out[:, 4:], 2.0, atol=1e-14)


def test_window_ignores_keys_outside_it(oracle_mod):
    """Decoder page P1.4: window 8 on a 32-token toy; keys outside the window are
    poisoned with NaN and the output must equal the clean run."""
    fx = GOLD["window_toy"]
    cfg = tiny(window=fx["window"], batch=1)
    clean = host_case(cfg, lens=[fx["toy_tokens"] - 1])
    out_clean, _ = run_oracle_step(clean, oracle_mod)
    dirty = host_case(cfg, lens=[fx["toy_tokens"] - 1])
    n_out = fx["toy_tokens"] - fx["window"]
    dirty["k_cache"][:, :, :n_out] = float("nan")
    dirty["v_cache"][:, :, :n_out] = float("nan")
    out_dirty, _ = run_oracle_step(dirty, oracle_mod)
    assert np.all(np.isfinite(out_dirty)) and np.array_equal(out_clean, out_dirty)
    # a window covering everything equals no window
    big = host_case(tiny(window=10_000, batch=1), lens=[31])
    none = host_case(tiny(batch=1), lens=[31])
    assert np.array_equal(run_oracle_step(big, oracle_mod)[0], run_oracle_step(none, oracle_mod)[0])


def test_softcap_limits(oracle_mod):
    huge = host_case(tiny(softcap=1e30), lens=[25, 3])
    none = host_case(tiny(), lens=[25, 3])
    assert np.allclose(run_oracle_step(huge, oracle_mod)[0], run_oracle_step(none, oracle_mod)[0],
                       rtol=1e-12, atol=1e-14)


def test_split_merge_equals_full_softmax(oracle_mod):
    """A blockwise log-sum-exp merge of partials over any split equals the full
    softmax: pins the combine arithmetic the GPU path uses."""
    cfg = tiny(batch=1, has_sink=True, seq_len=100, n_q_heads=4, n_kv_heads=1)
    cfg = dict(cfg, has_sink=False)
    case = host_case(cfg, lens=[99])
    a = oracle_arrays(case, oracle_mod)
    q_rot = oracle_mod.append(cfg, a["q"], a["k_new"], a["v_new"], None, None, a["k_cache"],
                              a["v_cache"], None, a["seq_lens"])
    kr, vr = a["k_cache"][0, 0], a["v_cache"][0, 0]
    full, lse_full = oracle_mod.attend_range(cfg, q_rot[0, 0], kr, vr, None, 0, 100)
    for cuts in ([0, 100], [0, 64, 100], [0, 1, 2, 50, 99, 100], list(range(0, 101, 7)) + [100]):
        parts = [oracle_mod.attend_range(cfg, q_rot[0, 0], kr, vr, None, lo, hi)
                 for lo, hi in zip(cuts[:-1], cuts[1:]) if hi > lo]
        M = max(l for _, l in parts)
        wts = [math.exp(l - M) for _, l in parts]
        merged = sum(w * o for (o, _), w in zip(parts, wts)) / sum(wts)
        assert np.allclose(merged, full, rtol=1e-12, atol=1e-14)
        assert M + math.log(sum(wts)) == pytest.approx(lse_full, rel=1e-13)


def test_q8_on_representable_rows_is_the_exact_cache(oracle_mod):
    """llamay "The KV cache, in three precisions": q8 stores keys and values as
    int8 codes with a scale per row. Rows that are integers times 2^-6 with a
    largest magnitude of 127 quantise exactly, so attention over a q8 cache of
    them equals attention over the same rows kept in fp32, bit for bit."""
    rng = np.random.default_rng(12)
    D, n = 64, 90
    ck = rng.integers(-127, 128, (n, D)); ck[:, 0] = 127
    cv = rng.integers(-127, 128, (n, D)); cv[:, 5] = -127
    k = (ck * 2.0 ** -6).astype(np.float32)
    v = (cv * 2.0 ** -6).astype(np.float32)
    kq, ks = oracle_mod.vq8_quantize(k)
    vq, vs = oracle_mod.vq8_quantize(v)
    assert np.array_equal(kq, ck.astype(np.int8)) and np.all(ks == np.float32(2.0 ** -6))
    q = rng.standard_normal(D)
    for extra in (dict(), dict(softcap=2.0), dict(window=0, has_sink=True)):
        c8 = rope_cfg(head_dim=D, kv_dtype="q8", **extra)
        c32 = rope_cfg(head_dim=D, kv_dtype="f32", **extra)
        sink = 0.3 if extra.get("has_sink") else None
        o8, l8 = oracle_mod.attend_range(c8, q, kq, vq, vs, 3, n, sink=sink, k_scale_rows=ks)
        o32, l32 = oracle_mod.attend_range(c32, q, k, v, None, 3, n, sink=sink)
        assert np.array_equal(o8, o32) and l8 == l32


# ------------------------------------------------------------------ brute force

GRID = [
    dict(name="llama31_8b_decode", n_q_heads=4, n_kv_heads=4, head_dim=64),
    dict(name="llama31_8b_decode", n_q_heads=8, n_kv_heads=4, head_dim=64, rope_style="interleaved"),
    dict(name="qwen3_8b_ragged", n_q_heads=16, n_kv_heads=4, head_dim=64),
    dict(name="gemma2_9b_swa", n_q_heads=8, n_kv_heads=1, head_dim=64, window=9, layers=None),
    dict(name="gptoss_vq8_sink", n_q_heads=16, n_kv_heads=2, head_dim=64),
    dict(name="llama32_1b_tiny", n_q_heads=8, n_kv_heads=2, head_dim=64),
    dict(name="llama31_8b_decode", n_q_heads=4, n_kv_heads=2, head_dim=128, rope_scaling="none",
         kv_dtype="f32", io_dtype="f32", softcap=2.0, window=13, has_sink=True),
    dict(name="qwen3_8b_ragged", n_q_heads=8, n_kv_heads=2, head_dim=128, rotary_dim=96, norm_offset=True),
    dict(name="llama32_1b_tiny", n_q_heads=8, n_kv_heads=2, head_dim=64, rotary_dim=16),
    dict(name="gptoss_vq8_sink", n_q_heads=8, n_kv_heads=2, head_dim=64, rotary_dim=32),
    dict(name="gemma3_12b_local_global", n_q_heads=4, n_kv_heads=2, head_dim=64, layers=None),
    dict(name="llama31_8b_decode", n_q_heads=8, n_kv_heads=2, head_dim=128, kv_dtype="q8"),
    dict(name="gptoss_vq8_sink", n_q_heads=8, n_kv_heads=2, head_dim=64, kv_dtype="q8", window=11),
    dict(name="qwen3_8b_ragged", n_q_heads=4, n_kv_heads=4, head_dim=64, kv_dtype="q8", io_dtype="f32",
         softcap=3.0),
    dict(name="gemma3_12b_local_global", n_q_heads=4, n_kv_heads=2, head_dim=64,
         layers=[dict(window=9, rope_theta=10000.0, rope_scaling="none")]),
]


def _random_grid(n: int, seed: int) -> list:
    """n feature mixes drawn independently: GQA ratio, head_dim, cache and input
    dtypes, pairing, window, softcap, sink, partial rotary, QK norm (with or
    without the stored-delta offset), each on a workload's own rope scaling."""
    rng = np.random.default_rng(seed)
    names = ["llama31_8b_decode", "qwen3_8b_ragged", "gptoss_vq8_sink", "llama32_1b_tiny", "gemma2_9b_swa",
             "gemma3_12b_local_global"]
    grid = []
    for i in range(n):
        D, Hkv, G = int(rng.choice([64, 128])), int(rng.choice([1, 2, 4])), int(rng.choice([1, 2, 4, 8]))
        spec = dict(name=names[i % len(names)], n_q_heads=G * Hkv, n_kv_heads=Hkv, head_dim=D,
                    kv_dtype=str(rng.choice(["f32", "bf16", "vq8", "q8"])), io_dtype=str(rng.choice(["f32", "bf16"])),
                    rope_style=str(rng.choice(["neox", "interleaved"])), layers=None,
                    window=int(rng.integers(1, 30)) if rng.random() < 0.5 else 0,
                    softcap=float(rng.choice([1.0, 5.0, 30.0])) if rng.random() < 0.4 else 0.0,
                    has_sink=bool(rng.random() < 0.4))
        if rng.random() < 0.4:
            spec["rotary_dim"] = int(rng.choice([D // 4, D // 2]))
        if rng.random() < 0.4:
            spec.update(qk_norm=True, norm_offset=bool(rng.random() < 0.5), norm_w_range=(-0.5, 1.5))
        grid.append(spec)
    return grid


def _step_vs_bruteforce(oracle_mod, spec, lens):
    spec = dict(spec)
    name = spec.pop("name")
    cfg = W.config(name, batch=len(lens), seq_len=(0, 40), steps=1, **spec)
    cfg = W.layer_configs(cfg)[0]
    case = host_case(cfg, lens=lens)
    out, a = run_oracle_step(case, oracle_mod)
    # brute force on fp64 copies of the same stored inputs
    f64 = lambda t: t.to(torch.float64).numpy().copy()
    kv = cfg["kv_dtype"]
    vs = ks = None
    if kv == "q8":
        codes, s = BF.vq8_numpy(case["k_values"].numpy())
        kc, ks = codes.astype(np.float64), s.astype(np.float64)
    else:
        kc = f64(case["k_cache"])
    if kv in ("vq8", "q8"):
        codes, s = BF.vq8_numpy(case["v_values"].numpy())
        vc, vs = codes.astype(np.float64), s.astype(np.float64)
    else:
        vc = f64(case["v_cache"])
    inv, ms = (None, 1.0)
    if cfg.get("rope_scaling", "none") != "none":
        inv, ms = oracle_mod.rope_inv_freq(cfg)
    lens = case["lens"].numpy().copy()
    ref = BF.decode_step(cfg, f64(case["q"]), f64(case["k_new"]), f64(case["v_new"]), kc, vc, vs,
                         lens, None if case["q_norm_w"] is None else case["q_norm_w"].numpy(),
                         None if case["k_norm_w"] is None else case["k_norm_w"].numpy(),
                         None if case["sink"] is None else case["sink"].numpy(), inv, ms, ks)
    assert np.array_equal(lens, a["seq_lens"])
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-11)
    if kv in ("vq8", "q8"):
        assert np.array_equal(a["v_cache"], vc.astype(np.int8))
        assert np.array_equal(a["v_scale"], vs.astype(np.float32))
    if kv == "q8":  # the appended keys' codes and scales: the vq8 rule on the rotated key
        assert np.array_equal(a["k_cache"], kc.astype(np.int8))
        assert np.array_equal(a["k_scale"], ks.astype(np.float32))


@pytest.mark.parametrize("spec", GRID, ids=lambda s: "-".join(f"{k}={v}" for k, v in s.items()))
def test_whole_step_matches_bruteforce(oracle_mod, spec):
    _step_vs_bruteforce(oracle_mod, spec, [0, 17, 40])


@pytest.mark.parametrize("i,spec", list(enumerate(_random_grid(24, seed=11))), ids=[f"mix{i}" for i in range(24)])
def test_random_feature_mixes_match_bruteforce(oracle_mod, i, spec):
    """Seeded random mixes of every feature the step has, at random lengths."""
    lens = [int(x) for x in np.random.default_rng(100 + i).integers(0, 41, size=3)]
    _step_vs_bruteforce(oracle_mod, spec, lens)


CHUNKS = [
    dict(name="llama31_8b_decode", n_q_heads=8, n_kv_heads=2, head_dim=64, q_len=4),
    dict(name="qwen3_8b_ragged", n_q_heads=4, n_kv_heads=4, head_dim=64, q_len=3, window=2),
    dict(name="gemma2_9b_swa", n_q_heads=8, n_kv_heads=1, head_dim=64, q_len=5, softcap=3.0, layers=None,
         window=9, has_sink=True),
    dict(name="llama32_1b_tiny", n_q_heads=8, n_kv_heads=2, head_dim=64, q_len=7, rotary_dim=32),
]


def _random_chunks(n: int, seed: int) -> list:
    """Chunk mixes for the matrix brute force (bf16 and fp32 caches): 2 to 8
    tokens, windows shorter and longer than the chunk, softcap, sink, partial
    rotary, QK norm."""
    rng = np.random.default_rng(seed)
    names = ["llama31_8b_decode", "qwen3_8b_ragged", "gptoss_vq8_sink", "gemma2_9b_swa"]
    grid = []
    for i in range(n):
        D, Hkv, G = int(rng.choice([64, 128])), int(rng.choice([1, 2])), int(rng.choice([1, 2, 4, 8]))
        spec = dict(name=names[i % len(names)], n_q_heads=G * Hkv, n_kv_heads=Hkv, head_dim=D,
                    kv_dtype=str(rng.choice(["f32", "bf16"])), io_dtype=str(rng.choice(["f32", "bf16"])),
                    rope_style=str(rng.choice(["neox", "interleaved"])), layers=None, q_len=int(rng.integers(2, 9)),
                    window=int(rng.integers(1, 12)) if rng.random() < 0.6 else 0,
                    softcap=float(rng.choice([2.0, 20.0])) if rng.random() < 0.4 else 0.0,
                    has_sink=bool(rng.random() < 0.4))
        if rng.random() < 0.4:
            spec["rotary_dim"] = D // 2
        if rng.random() < 0.4:
            spec.update(qk_norm=True, norm_offset=bool(rng.random() < 0.5), norm_w_range=(-0.5, 1.5))
        grid.append(spec)
    return grid


@pytest.mark.parametrize("spec", CHUNKS + _random_chunks(10, seed=12),
                         ids=[f"fixed{i}" for i in range(len(CHUNKS))] + [f"mix{i}" for i in range(10)])
def test_chunk_matches_masked_matrix_bruteforce(oracle_mod, spec):
    """Several tokens per sequence: the oracle takes them as decode steps in order;
    the brute force appends all of them first and masks one logit matrix by each
    token's causal and window limits. The two agree."""
    spec = dict(spec)
    name = spec.pop("name")
    cfg = W.layer_configs(W.config(name, batch=3, seq_len=(0, 40), steps=1, **spec))[0]
    case = host_case(cfg, lens=[0, 17, 40])
    out, a = run_oracle_step(case, oracle_mod)
    T = cfg["q_len"]
    assert out.shape == (3, T, cfg["n_q_heads"], cfg["head_dim"])
    f64 = lambda t: t.to(torch.float64).numpy().copy()
    inv, ms = (None, 1.0)
    if cfg.get("rope_scaling", "none") != "none":
        inv, ms = oracle_mod.rope_inv_freq(cfg)
    lens = case["lens"].numpy().copy()
    ref = BF.chunk_step(cfg, f64(case["q"]), f64(case["k_new"]), f64(case["v_new"]), f64(case["k_cache"]),
                        f64(case["v_cache"]), lens, None if case["q_norm_w"] is None else case["q_norm_w"].numpy(),
                        None if case["k_norm_w"] is None else case["k_norm_w"].numpy(),
                        None if case["sink"] is None else case["sink"].numpy(), inv, ms)
    assert np.array_equal(lens, a["seq_lens"]) and np.array_equal(lens, case["lens"].numpy() + T)
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("mistake", ["not_causal", "window_shortened_by_the_chunk"])
def test_chunk_mask_mistakes_break_the_tolerance(oracle_mod, mistake):
    """Negative controls for the chunk's mask: every token seeing all T new keys
    (no causal limit), or every token's window shortened by T - 1 (the widened
    window of the chunk's key range taken the wrong way), fails the parity bar."""
    cfg = W.layer_configs(W.config("llama31_8b_decode", batch=2, seq_len=(0, 90), n_q_heads=8, n_kv_heads=2,
                                   head_dim=64, q_len=6, window=(12 if mistake != "not_causal" else 0)))[0]
    case = host_case(cfg, lens=[30, 90])
    case["q"] = (case["q"].to(torch.float32) * 3).to(case["q"].dtype)
    good, _ = run_oracle_step(case, oracle_mod)
    f64 = lambda t: t.to(torch.float64).numpy().copy()
    inv, ms = oracle_mod.rope_inv_freq(cfg)
    args = lambda: (f64(case["q"]), f64(case["k_new"]), f64(case["v_new"]), f64(case["k_cache"]),
                    f64(case["v_cache"]), case["lens"].numpy().copy(), None, None, None, inv, ms)
    if mistake == "not_causal":
        wrong = BF.chunk_step(cfg, *args(), causal=False)
    else:
        wrong = BF.chunk_step(dict(cfg, window=12 - (cfg["q_len"] - 1)), *args())
    d = np.abs(good - wrong)
    assert d.max() > TOL_MAX or d.mean() > TOL_MEAN, (mistake, d.max(), d.mean())


def test_interleaved_step_equals_permuted_neox_step(oracle_mod):
    D = 64
    perm = np.concatenate([2 * np.arange(D // 2), 2 * np.arange(D // 2) + 1])  # neox p -> row
    cfg_i = W.config("llama32_1b_tiny", batch=2, seq_len=(0, 30), n_q_heads=8, n_kv_heads=2)
    cfg_n = dict(cfg_i, rope_style="neox")
    case = host_case(cfg_i, lens=[12, 29])
    out_i, _ = run_oracle_step(case, oracle_mod)
    pc = dict(case)
    for key in ("q", "k_new", "k_cache"):
        pc[key] = case[key][..., perm].contiguous()
    pc["cfg"] = cfg_n
    out_n, _ = run_oracle_step(pc, oracle_mod)
    assert np.allclose(out_i, out_n, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ negative controls

def _err(a, b):
    d = np.abs(a - b)
    return d.max(), d.mean()


@pytest.mark.parametrize("mistake", ["drop_sink", "ignore_window", "wrong_pairing", "skip_norm",
                                     "no_softcap", "plain_rope_not_llama3", "no_norm_offset",
                                     "full_rotary_not_partial", "no_linear_scaling", "global_theta_on_local"])
def test_planted_mistakes_break_the_tolerance(oracle_mod, mistake):
    """llamay 'The bound, and why it is the one it is': a bound has teeth only if a
    degraded variant fails it. Each planted mistake must exceed the parity bar on
    the output (2e-3 max / 2e-4 mean) or on the appended key rows (one bf16 ulp)."""
    name, over, key, bad, lens, qmul = {
        "drop_sink": ("gptoss_vq8_sink", dict(n_q_heads=16, n_kv_heads=2), "has_sink", False,
                      [2, 9], 1),
        "ignore_window": ("gemma2_9b_swa", dict(n_q_heads=4, n_kv_heads=2, head_dim=64,
                                               layers=[dict(window=16)]), "window", 0, [150, 199], 1),
        "wrong_pairing": ("llama32_1b_tiny", dict(n_q_heads=8, n_kv_heads=2), "rope_style", "neox",
                          [150, 199], 3),
        "skip_norm": ("qwen3_8b_ragged", dict(n_q_heads=8, n_kv_heads=2), "qk_norm", False,
                      [150, 199], 1),
        "no_softcap": ("gemma2_9b_swa", dict(n_q_heads=4, n_kv_heads=2, head_dim=64, softcap=2.0,
                                            layers=None), "softcap", 0.0, [150, 199], 4),
        "plain_rope_not_llama3": ("llama31_8b_decode", dict(n_q_heads=8, n_kv_heads=2),
                                  "rope_scaling", "none", [8000, 8100], 1),
        "no_norm_offset": ("gemma3_12b_local_global", dict(n_q_heads=8, n_kv_heads=2, layers=None),
                           "norm_offset", False, [150, 199], 1),
        "full_rotary_not_partial": ("qwen3_8b_ragged", dict(n_q_heads=8, n_kv_heads=2, rotary_dim=96),
                                    "rotary_dim", 0, [150, 199], 1),
        "no_linear_scaling": ("gemma3_12b_local_global", dict(n_q_heads=8, n_kv_heads=2, layers=None),
                              "rope_scaling", "none", [150, 199], 1),
        "global_theta_on_local": ("gemma3_12b_local_global", dict(n_q_heads=8, n_kv_heads=2,
                                  layers=[dict(window=1024, rope_theta=10000.0, rope_scaling="none")]),
                                  "rope_theta", 1000000.0, [150, 199], 1),
    }[mistake]
    cfg = W.layer_configs(W.config(name, batch=2, seq_len=(0, max(lens) + 1), steps=1, **over))[0]
    case = host_case(cfg, lens=lens)
    case["q"] = (case["q"].to(torch.float32) * qmul).to(case["q"].dtype)
    good, ga = run_oracle_step(case, oracle_mod)
    wrong, wa = run_oracle_step(dict(case, cfg=dict(cfg, **{key: bad})), oracle_mod)
    mx, mean = _err(good, wrong)
    rows = np.arange(2)
    kg = ga["k_cache"][rows, :, np.array(lens)]
    kw = wa["k_cache"][rows, :, np.array(lens)]
    if kg.dtype == np.uint16:
        kg, kw = BF.bf16_round(oracle_mod.bf16_to_f64(kg)), oracle_mod.bf16_to_f64(kw)
    k_ulps = np.abs(kg - kw) / (np.abs(kg) * 2.0 ** -8 + 1e-30)
    assert mx > TOL_MAX or mean > TOL_MEAN or k_ulps.max() > 1.0, (mistake, mx, mean, k_ulps.max())


@pytest.mark.parametrize("name", ["llama31_8b_decode", "gptoss_vq8_sink", "llama31_8b_q8", "llama31_8b_verify"])
def test_oracle_is_independent_of_its_thread_count(oracle_mod, name):
    """The oracle splits a step over threads by (sequence, head) unit only: one
    thread and eight give the same bits, caches and lengths included."""
    cfg = W.layer_configs(W.config(name, batch=4, seq_len=(1, 300), steps=1))[0]
    lens = [1, 77, 150, 300]
    outs = []
    for n in (1, 8):
        case = host_case(cfg, lens=lens)
        out, a = run_oracle_step(case, oracle_mod, n_threads=n)
        outs.append((out, a))
    (o1, a1), (o8, a8) = outs
    assert np.array_equal(o1, o8)
    for k in ("k_cache", "v_cache", "v_scale", "k_scale", "seq_lens"):
        if a1[k] is not None:
            assert np.array_equal(a1[k], a8[k]), k
