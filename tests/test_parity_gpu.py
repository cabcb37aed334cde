"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on the
same seeded inputs.

The bar: cache-append slots, positions (seq_lens), vq8 codes/scales and the
appended bf16 key rows bit-exact (the GPU rotates in fp32 and recomputes in fp64
the rare element whose fp32 result lies within its error bound of a bf16
rounding boundary, so both sides round the exact value to nearest even); q8 key
codes within one of the oracle's where the rotated key lies within fp32
rounding of a code boundary; outputs max|d| <= 2e-3 and mean|d| <= 2e-4 against
the fp64 oracle (fp32 outputs).
"""
import math

import numpy as np
import pytest
import torch

from gqa_attention_kv_qk_gb300 import binding as B
from gqa_attention_kv_qk_gb300 import workloads as W
from tests.cases import gpu_layer, host_case, oracle_arrays, run_oracle_step

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN = 2e-3, 2e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gqa_attention_kv_qk_gb300 import build
    build.build()


def f64(a):
    if isinstance(a, torch.Tensor):
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def bf16_bits_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def assert_out_close(got, want, what="out", tol_max=TOL_MAX, tol_mean=TOL_MEAN):
    d = np.abs(f64(got) - want)
    assert np.all(np.isfinite(f64(got))), f"{what}: non-finite values"
    assert d.max() <= tol_max and d.mean() <= tol_mean, f"{what}: max {d.max():.3g} mean {d.mean():.3g}"
    return d.max(), d.mean()


ENTRIES = ("split", "fused")


def run_and_compare(oracle_mod, cfg, lens, cap=None, steps=1, fill_unused="zero", check_qrot=True,
                    max_seq_len=None, entry="split"):
    """Run `steps` chained decode steps on both sides and compare everything the
    step writes. entry "split" runs the three step entry points one by one,
    "fused" the whole-step call (one append+partial kernel for bf16 / vq8
    caches, then the combine). Returns the worst (max, mean) output error."""
    case = host_case(cfg, lens=lens, cap=cap, fill_unused=fill_unused)
    a = oracle_arrays(case, oracle_mod)
    layer = gpu_layer(case)
    kv = cfg.get("kv_dtype", "bf16")
    C = lambda name: layer.logical(name)  # logical rows [B][Hkv][cap][...], paged or not
    if kv in ("vq8", "q8"):  # both quantisers on the same fp32 values
        assert np.array_equal(C("v_cache").cpu().numpy(), a["v_cache"])
        assert np.array_equal(C("v_scale").cpu().numpy().view(np.uint32), a["v_scale"].view(np.uint32))
    if kv == "q8":
        assert np.array_equal(C("k_cache").cpu().numpy(), a["k_cache"])
        assert np.array_equal(C("k_scale").cpu().numpy().view(np.uint32), a["k_scale"].view(np.uint32))
    B_, Hq, D = cfg["batch"], cfg["n_q_heads"], cfg["head_dim"]
    T = int(cfg.get("q_len", 1) or 1)  # tokens per sequence and step
    tok = (T,) if T > 1 else ()
    worst = (0.0, 0.0)
    for step in range(steps):
        inp = W.step_inputs(cfg, step)
        pre = a["seq_lens"].copy()
        q_rot = torch.empty((B_, *tok, Hq, D), dtype=torch.float32, device="cuda")
        dev = {k: v.cuda() for k, v in inp.items()}
        if entry == "split":
            layer.append(dev["q"], dev["k_new"], dev["v_new"], q_rot=q_rot)
            layer.partial()
            out = layer.combine().clone()
        else:
            out = layer.step(dev["q"], dev["k_new"], dev["v_new"], q_rot=q_rot).clone()
        torch.cuda.synchronize()
        # the fused kernel's arrival counter is back at zero after every launch, and
        # the combine has written the range-balance tables for this grid
        assert int(layer.ws_tensor[4:8].view(torch.int32).item()) == 0
        lay = layer.layout()
        if lay.kernel == 1:
            hdr = layer.ws_tensor[lay.balance_offset: lay.balance_offset + 12].view(torch.int32).cpu().tolist()
            assert hdr[0] == 0x42414c31 and hdr[1] == lay.n_ctas and hdr[2] >= 1
        qrs, wants = [], []
        for t in range(T):  # a chunk is its tokens' decode steps, in order
            pick = (lambda x: x) if T == 1 else (lambda x: x[:, t])
            qr = oracle_mod.append(cfg, W.bits(pick(inp["q"])).copy(), W.bits(pick(inp["k_new"])).copy(),
                                   W.bits(pick(inp["v_new"])).copy(), a["q_norm_w"], a["k_norm_w"], a["k_cache"],
                                   a["v_cache"], a["v_scale"], a["seq_lens"], a["k_scale"])
            qrs.append(qr)
            wants.append(oracle_mod.attend(cfg, qr, a["sink"], a["k_cache"], a["v_cache"], a["v_scale"],
                                           a["seq_lens"], k_scale=a["k_scale"]))
        qr = qrs[0] if T == 1 else np.stack(qrs, axis=1)
        want = wants[0] if T == 1 else np.stack(wants, axis=1)
        # positions / slots: bit-exact
        assert np.array_equal(layer.seq_lens.cpu().numpy(), a["seq_lens"])
        assert layer.device_status() == 0
        if check_qrot:
            assert np.allclose(q_rot.cpu().numpy(), qr, rtol=2e-5, atol=2e-5)
        # the appended rows
        kc_g, vc_g = C("k_cache"), C("v_cache")
        ks_g, vs_g = C("k_scale"), C("v_scale")
        for b, slot in ((b, int(pre[b]) + t) for b in range(B_) for t in range(T)):
            kg = f64(kc_g[b, :, slot].float())
            if kv == "q8":
                # codes of the rotated key: the GPU rotates in fp32, the oracle in fp64, so a
                # code may differ by one where k / s lies within rounding of a tie; the scale
                # (max |k| / 127) by the fp32 rotation's relative error
                kcg, kco = kg.astype(np.int64), a["k_cache"][b, :, slot].astype(np.int64)
                ksg, kso = f64(ks_g[b, :, slot]), a["k_scale"][b, :, slot].astype(np.float64)
                assert np.abs(kcg - kco).max() <= 1, "q8 key code off by more than one"
                assert (kcg != kco).sum() <= max(2, kco.size // 100), "q8 key codes differ beyond rounding ties"
                assert np.allclose(ksg, kso, rtol=2e-6, atol=0), "q8 key scale beyond fp32 rounding"
                assert np.array_equal(vc_g[b, :, slot].cpu().numpy(), a["v_cache"][b, :, slot])
                assert np.array_equal(vs_g[b, :, slot].cpu().numpy().view(np.uint32),
                                      a["v_scale"][b, :, slot].view(np.uint32))
            elif kv == "f32":
                ko = a["k_cache"][b, :, slot].astype(np.float64)
                assert np.allclose(kg, ko, rtol=1e-5, atol=1e-6)
                assert np.array_equal(vc_g[b, :, slot].cpu().numpy(), a["v_cache"][b, :, slot])
            else:
                kbits = kc_g[b, :, slot].view(torch.int16).cpu().numpy().view(np.uint16)
                assert np.array_equal(kbits, a["k_cache"][b, :, slot]), "an appended key row differs"
                if kv == "bf16":
                    vg = vc_g[b, :, slot].view(torch.int16).cpu().numpy().view(np.uint16)
                    assert np.array_equal(vg, a["v_cache"][b, :, slot])
                else:
                    assert np.array_equal(vc_g[b, :, slot].cpu().numpy(), a["v_cache"][b, :, slot])
                    assert np.array_equal(vs_g[b, :, slot].cpu().numpy().view(np.uint32),
                                          a["v_scale"][b, :, slot].view(np.uint32))
        if layer.page_size:  # pages outside every table row are never written
            used = torch.zeros(layer.n_pages, dtype=torch.bool)
            used[layer.block_table.reshape(-1).long().cpu()] = True
            assert not layer.k_cache[~used.cuda()].float().abs().sum().item()
            assert not layer.v_cache[~used.cuda()].float().abs().sum().item()
        mx, mean = assert_out_close(out, want, f"step {step}")
        worst = (max(worst[0], mx), max(worst[1], mean))
    return worst


# ------------------------------------------------------------------ the workloads, small

SMALL = {
    "llama32_1b_tiny": dict(lens=[256]),
    "llama31_8b_decode": dict(overrides=dict(batch=3, seq_len=1400, steps=3), lens=[700, 1000, 1337]),
    "qwen3_8b_ragged": dict(overrides=dict(batch=5, seq_len=(1, 2100)), lens=[1, 64, 129, 2000, 777]),
    "gemma2_9b_swa": dict(overrides=dict(batch=2, seq_len=5000), lens=[3000, 4999]),
    "gptoss_vq8_sink": dict(overrides=dict(batch=3, seq_len=4096), lens=[100, 1000, 4095]),
    "gemma3_12b_local_global": dict(overrides=dict(batch=3, seq_len=(1, 3000)), lens=[2999, 1023, 5]),
    "llama31_8b_q8": dict(overrides=dict(batch=3, seq_len=1400, steps=3), lens=[700, 1000, 1337]),
    "llama31_8b_paged": dict(overrides=dict(batch=3, seq_len=1400, steps=3), lens=[700, 1000, 1337]),
    "llama31_8b_verify": dict(overrides=dict(batch=3, seq_len=1400, steps=3), lens=[700, 1000, 1337]),
}


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("name", list(SMALL))
def test_workload_parity_small(oracle_mod, name, entry):
    spec = SMALL[name]
    cfg = W.config(name, **spec.get("overrides", {}))
    for layer_cfg in W.layer_configs(cfg):
        run_and_compare(oracle_mod, layer_cfg, spec["lens"], steps=cfg.get("steps", 1), entry=entry)


# ------------------------------------------------------------------ edge cases

EDGE = [
    # (id, workload, overrides, lens)
    ("first-token", "llama31_8b_decode", dict(batch=3, seq_len=200), [0, 0, 63]),
    ("tile-boundaries", "llama31_8b_decode", dict(batch=4, seq_len=300), [63, 64, 127, 255]),
    ("last-slot", "llama31_8b_decode", dict(batch=2, seq_len=255), [255, 10]),
    ("window-1", "gemma2_9b_swa", dict(batch=2, seq_len=500, layers=[dict(window=1)]), [499, 3]),
    ("window-ragged", "gemma2_9b_swa", dict(batch=3, seq_len=1000, layers=[dict(window=100)]), [999, 150, 40]),
    ("window-wider", "gemma2_9b_swa", dict(batch=2, seq_len=300, layers=[dict(window=4096)]), [299, 17]),
    ("softcap-strong", "gemma2_9b_swa", dict(batch=2, seq_len=600, softcap=1.0, layers=None), [599, 200]),
    ("mha-g1", "llama31_8b_decode", dict(batch=2, n_q_heads=8, n_kv_heads=8, seq_len=300), [299, 77]),
    ("g16", "llama31_8b_decode", dict(batch=2, n_q_heads=32, n_kv_heads=2, seq_len=300), [299, 77]),
    ("g32-two-groups", "llama31_8b_decode", dict(batch=2, n_q_heads=32, n_kv_heads=1, seq_len=300), [299, 77]),
    ("d64-bf16", "gptoss_vq8_sink", dict(batch=2, kv_dtype="bf16", seq_len=500), [499, 64]),
    ("d128-vq8", "llama31_8b_decode", dict(batch=2, kv_dtype="vq8", seq_len=500), [499, 64]),
    ("d256-vq8-sink", "gemma2_9b_swa", dict(batch=2, kv_dtype="vq8", has_sink=True, seq_len=500, layers=None),
     [499, 64]),
    ("d64-g16-vq8", "gptoss_vq8_sink", dict(batch=2, n_q_heads=32, n_kv_heads=2, seq_len=300), [299, 5]),
    ("f32-io-bf16-cache", "llama31_8b_decode", dict(batch=2, io_dtype="f32", seq_len=300), [299, 5]),
    ("bf16-io-f32-cache", "llama32_1b_tiny", dict(batch=2, io_dtype="bf16", seq_len=300), [299, 5]),
    ("f32-d256-window", "gemma2_9b_swa", dict(batch=2, kv_dtype="f32", io_dtype="f32", seq_len=300,
                                            layers=[dict(window=50)]), [299, 5]),
    ("yarn-qknorm-interleaved", "gptoss_vq8_sink", dict(batch=2, qk_norm=True, norm_w_range=(0.5, 1.5),
                                                       rope_style="interleaved", seq_len=300), [299, 5]),
    # partial rotary (rotary_dim < head_dim), the (1 + w) norm weight, linear scaling
    ("rotary96-of-128-qknorm", "qwen3_8b_ragged", dict(batch=2, seq_len=300, rotary_dim=96), [299, 5]),
    ("rotary16-of-64-interleaved", "llama32_1b_tiny", dict(batch=2, seq_len=300, rotary_dim=16,
                                                           io_dtype="bf16", kv_dtype="bf16"), [299, 5]),
    ("rotary32-of-64-yarn-vq8", "gptoss_vq8_sink", dict(batch=2, seq_len=300, rotary_dim=32), [299, 5]),
    ("f32-rotary48-norm-offset", "llama32_1b_tiny", dict(batch=2, seq_len=300, rotary_dim=48, qk_norm=True,
                                                         norm_offset=True, norm_w_range=(-0.5, 0.5)), [299, 5]),
    ("d256-rotary64-linear", "gemma3_12b_local_global", dict(batch=2, seq_len=600, rotary_dim=64, layers=None),
     [599, 10]),
    # q8 cache (int8 keys and values) at every head_dim and both head tilings
    ("q8-first-token", "llama31_8b_q8", dict(batch=3, seq_len=200), [0, 1, 63]),
    ("q8-d64-sink-yarn", "gptoss_vq8_sink", dict(batch=2, kv_dtype="q8", seq_len=500), [499, 64]),
    ("q8-d64-g16", "gptoss_vq8_sink", dict(batch=2, kv_dtype="q8", n_q_heads=32, n_kv_heads=2, seq_len=300),
     [299, 5]),
    ("q8-d128-g16-qknorm", "qwen3_8b_ragged", dict(batch=3, kv_dtype="q8", n_q_heads=32, n_kv_heads=2,
                                                   seq_len=(1, 700)), [1, 129, 700]),
    ("q8-d256-window-softcap", "gemma2_9b_swa", dict(batch=2, kv_dtype="q8", seq_len=600,
                                                     layers=[dict(window=100)]), [599, 40]),
    ("q8-f32-io-interleaved", "llama31_8b_q8", dict(batch=2, io_dtype="f32", rope_style="interleaved",
                                                    seq_len=300), [299, 0]),
    ("q8-rotary96-norm-offset", "qwen3_8b_ragged", dict(batch=2, kv_dtype="q8", rotary_dim=96, norm_offset=True,
                                                        norm_w_range=(-0.5, 0.5), seq_len=300), [299, 77]),
    # paged caches: page sizes 16 .. 4096, every cache kind, windows that start mid-page
    ("paged-16-bf16", "llama31_8b_decode", dict(batch=3, seq_len=1000, page_size=16), [999, 64, 0]),
    ("paged-64-vq8-window", "gptoss_vq8_sink", dict(batch=2, seq_len=500, page_size=64, window=100), [499, 64]),
    ("paged-32-vq8-window-37", "gptoss_vq8_sink", dict(batch=2, seq_len=500, page_size=32, window=37), [499, 20]),
    ("paged-16-f32-window-37", "llama32_1b_tiny", dict(batch=2, seq_len=300, page_size=16, window=37), [299, 20]),
    ("paged-16-bf16-window-37", "qwen3_8b_ragged", dict(batch=2, seq_len=(1, 500), page_size=16, window=37),
     [499, 20]),
    ("paged-256-q8", "llama31_8b_q8", dict(batch=2, seq_len=700, page_size=256), [699, 300]),
    ("paged-32-f32", "llama32_1b_tiny", dict(batch=2, seq_len=300, page_size=32), [299, 40]),
    ("paged-128-d256", "gemma2_9b_swa", dict(batch=2, seq_len=600, page_size=128, layers=None), [599, 10]),
    ("paged-4096-d256-window", "gemma2_9b_swa", dict(batch=2, seq_len=5000, page_size=4096,
                                                     layers=[dict(window=4096)]), [4999, 4100]),
    # several tokens per sequence (causal chunks): G x T rows from 2 to 64 per kv head,
    # windows shorter than the chunk, every cache kind, paged, first tokens
    ("chunk2-first-token", "llama31_8b_decode", dict(batch=3, seq_len=200, q_len=2), [0, 1, 63]),
    ("chunk4-g4-d128", "llama31_8b_decode", dict(batch=2, seq_len=500, q_len=4), [499, 60]),
    ("chunk3-mha-window2", "qwen3_8b_ragged", dict(batch=2, n_q_heads=8, n_kv_heads=8, seq_len=(1, 300), q_len=3,
                                                   window=2), [299, 1]),
    ("chunk8-g8-d64-vq8-sink", "gptoss_vq8_sink", dict(batch=2, n_q_heads=16, n_kv_heads=2, seq_len=400, q_len=8),
     [399, 100]),
    ("chunk5-d256-window-softcap", "gemma2_9b_swa", dict(batch=2, seq_len=600, q_len=5, layers=[dict(window=7)]),
     [599, 3]),
    ("chunk6-f32-paged16", "llama32_1b_tiny", dict(batch=2, seq_len=300, q_len=6, page_size=16), [290, 40]),
    ("chunk16-q8-paged64", "llama31_8b_q8", dict(batch=2, seq_len=700, q_len=16, page_size=64), [680, 100]),
    ("chunk64-prefill-g2", "llama31_8b_decode", dict(batch=2, n_q_heads=16, n_kv_heads=8, seq_len=300, q_len=64),
     [200, 0]),
    # prefill chunks: 256 and 1,024 tokens (many 16-row groups per kv head), one from an empty cache
    ("chunk256-prefill-g4", "llama31_8b_decode", dict(batch=2, n_q_heads=8, n_kv_heads=2, seq_len=1400, q_len=256,
                                                     steps=1), [1000, 0]),
    ("chunk1024-prefill-g4", "llama31_8b_decode", dict(batch=1, n_q_heads=8, n_kv_heads=2, seq_len=1100, q_len=1024,
                                                      steps=1), [60]),
    # the query-tiled prefill kernel (128+ rows per kv head on a contiguous bf16 cache):
    # head_dim 64 with a window shorter than the chunk and sinks; softcap with bf16
    # output and a row count that is not a multiple of 128; the same geometry on a
    # paged cache, which takes the split-K partial kernel
    ("chunk128-prefill-d64-window-sink", "gptoss_vq8_sink", dict(batch=2, kv_dtype="bf16", seq_len=700, q_len=128,
                                                                 window=100, steps=1), [500, 3]),
    ("chunk100-prefill-softcap-bf16out", "llama31_8b_decode", dict(batch=2, n_q_heads=12, n_kv_heads=4, seq_len=900,
                                                                   q_len=100, softcap=30.0, out_dtype="bf16",
                                                                   steps=1), [700, 64]),
    ("chunk64-prefill-paged32", "llama31_8b_decode", dict(batch=2, seq_len=400, q_len=64, page_size=32, steps=1),
     [300, 31]),
    # short chunks with two column tiles: new rows that cross a stage or page boundary,
    # two head groups, windows shorter than the chunk; head_dim 256 with one column tile
    ("chunk4-g4-stage-crossing", "llama31_8b_decode", dict(batch=4, seq_len=600, q_len=4), [126, 254, 1, 509]),
    ("chunk3-g8-vq8-two-groups", "llama31_8b_decode", dict(batch=2, n_q_heads=32, n_kv_heads=4, kv_dtype="vq8",
                                                           seq_len=400, q_len=3), [127, 30]),
    ("chunk4-q8-window3", "llama31_8b_q8", dict(batch=2, seq_len=500, q_len=4, window=3), [254, 2]),
    ("chunk2-g8-d64-paged32-vq8", "gptoss_vq8_sink", dict(batch=2, seq_len=500, q_len=2, page_size=32), [31, 400]),
    ("chunk4-d256-g4-window", "gemma2_9b_swa", dict(batch=2, n_q_heads=16, n_kv_heads=4, seq_len=600, q_len=4,
                                                    layers=[dict(window=50)]), [126, 590]),
    ("d64-vq8-norm-offset-local", "gemma3_12b_local_global",
     dict(batch=2, seq_len=600, head_dim=64, kv_dtype="vq8", layers=[dict(window=100, rope_theta=10000.0,
                                                                          rope_scaling="none")]), [599, 40]),
    # chunks whose append takes the row-per-warp kernel (NeoX with rotary_dim / 2 not a
    # multiple of 8): one token per CTA, and the token groups of a 1,280-token step;
    # partial rotary in chunks on the staged append (NeoX with the QK norm, interleaved fp32)
    ("chunk4-rotary36-row-append", "llama31_8b_decode", dict(batch=2, seq_len=500, q_len=4, rotary_dim=36),
     [499, 60]),
    ("chunk640-rotary36-grouped-append", "llama31_8b_decode", dict(batch=2, n_q_heads=8, n_kv_heads=2, seq_len=1400,
                                                                   q_len=640, rotary_dim=36, steps=1), [700, 0]),
    ("chunk4-rotary96-qknorm", "qwen3_8b_ragged", dict(batch=2, seq_len=300, q_len=4, rotary_dim=96), [296, 5]),
    ("chunk3-rotary16-interleaved-f32", "llama32_1b_tiny", dict(batch=2, seq_len=300, q_len=3, rotary_dim=16),
     [290, 5]),
]


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("spec", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(oracle_mod, spec, entry):
    _, name, over, lens = spec
    cfg = W.config(name, **over)
    for layer_cfg in W.layer_configs(cfg):
        run_and_compare(oracle_mod, layer_cfg, lens, entry=entry)


@pytest.mark.parametrize("name,over,T", [
    ("qwen3_8b_ragged", dict(batch=512, n_q_heads=8, n_kv_heads=8, seq_len=(0, 200)), 1),    # QK norm, fused
    ("gptoss_vq8_sink", dict(batch=1024, n_q_heads=8, n_kv_heads=8, seq_len=(0, 200)), 1),   # YaRN multiplier, D=64
    ("qwen3_8b_ragged", dict(batch=64, n_q_heads=8, n_kv_heads=8, seq_len=(0, 200), q_len=16), 16),  # separate append
])
def test_appended_keys_bit_exact_at_scale(oracle_mod, name, over, T):
    """The appended bf16 key rows equal the oracle's bits over ~1M key elements
    per case: about one element in 150 lies within the fp32 path's error bound of
    a bf16 rounding boundary and is recomputed in fp64 (after the last segment in
    the fused kernel, queued per CTA in the staged append of the 16-token step),
    so the fp64 path runs thousands of times here, with and without the QK norm
    and under YaRN's cos / sin multiplier."""
    cfg = W.layer_configs(W.config(name, steps=1, **over))[0]
    lens = [int(x) for x in np.random.default_rng(17).integers(0, 180, size=cfg["batch"])]
    case = host_case(cfg, lens=lens)
    a = oracle_arrays(case, oracle_mod)
    layer = gpu_layer(case)
    inp = W.step_inputs(cfg, 0)
    layer.step(inp["q"].cuda(), inp["k_new"].cuda(), inp["v_new"].cuda())
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    for t in range(T):
        pick = (lambda x: x) if T == 1 else (lambda x: x[:, t])
        oracle_mod.append(cfg, W.bits(pick(inp["q"])).copy(), W.bits(pick(inp["k_new"])).copy(),
                          W.bits(pick(inp["v_new"])).copy(), a["q_norm_w"], a["k_norm_w"], a["k_cache"],
                          a["v_cache"], a["v_scale"], a["seq_lens"], a["k_scale"])
    kg = layer.logical("k_cache").view(torch.int16).cpu().numpy().view(np.uint16)
    Bn = cfg["batch"]
    pos = np.array(lens)[:, None] + np.arange(T)[None, :]          # [B][T]
    got = kg[np.arange(Bn)[:, None], :, pos]                        # [B][T][Hkv][D]
    want = a["k_cache"][np.arange(Bn)[:, None], :, pos]
    assert got.size >= 500_000
    assert np.array_equal(got, want), f"{int((got != want).sum())} of {got.size} key elements differ"


@pytest.mark.parametrize("entry", ENTRIES)
def test_unused_slots_hold_nan(oracle_mod, entry):
    """Slots beyond each sequence hold NaN; masking must keep them out of every
    result, and the fused kernel must replace the loaded NaN row of the new slot."""
    for name, over, lens in (("llama31_8b_decode", dict(batch=3, seq_len=400), [10, 200, 399]),
                             ("gptoss_vq8_sink", dict(batch=2, seq_len=400), [33, 380]),
                             ("gemma2_9b_swa", dict(batch=2, seq_len=400, layers=[dict(window=70)]), [399, 90]),
                             ("qwen3_8b_ragged", dict(batch=3, seq_len=(1, 400)), [0, 127, 128]),
                             # a prefill chunk (the query-tiled kernel): the last key block's value rows
                             # past the sequence's end are NaN in the cache
                             ("llama31_8b_decode", dict(batch=2, n_q_heads=8, n_kv_heads=2, seq_len=400, q_len=64),
                              [10, 300])):
        cfg = W.layer_configs(W.config(name, **over))[0]
        run_and_compare(oracle_mod, cfg, lens, fill_unused="nan", steps=2, entry=entry)


def test_ranges_follow_measured_speed():
    """The tensor-core kernel sizes its ranges by the speeds measured in earlier
    launches on the same workspace: after a few launches the range table differs
    from the uniform split, still covers every stage once, and the slot weights
    are positive."""
    cfg = W.config("llama31_8b_decode", batch=4, seq_len=4000)
    case = host_case(cfg)
    layer = gpu_layer(case)
    dev = {k: case[k].cuda() for k in ("q", "k_new", "v_new")}
    lens0 = layer.seq_lens.clone()
    for _ in range(4):
        layer.seq_lens.copy_(lens0)
        layer.step(dev["q"], dev["k_new"], dev["v_new"], advance_hint=False)
    torch.cuda.synchronize()
    lay = layer.layout()
    ws = layer.ws_tensor
    T = int(ws[lay.prefix_offset: lay.prefix_offset + (cfg["batch"] + 1) * 4].view(torch.int32)[-1].item())
    P = lay.n_ctas
    assert T >= P
    starts = ws[lay.ranges_offset: lay.ranges_offset + (P + 1) * 8].view(torch.int64).cpu().numpy()
    assert starts[0] == 0 and starts[-1] == T and np.all(np.diff(starts) >= 1)
    uniform = np.array([c * T // P for c in range(P + 1)])
    assert not np.array_equal(starts, uniform)
    al = lambda x: -(-x // 256) * 256
    w0 = lay.balance_offset + 256 + al(8 * P) + al(4 * P)
    weight = ws[w0: w0 + 4 * P].view(torch.float32)
    assert bool(torch.all(weight > 0))
    assert layer.device_status() == 0


@pytest.mark.parametrize("entry", ENTRIES)
def test_batch_slices(oracle_mod, entry):
    """More sequences than one launch takes: the step runs as several slices
    (each with its own stage prefix and records), lengths advance in every slice."""
    cfg = W.config("qwen3_8b_ragged", batch=1100, n_q_heads=8, n_kv_heads=2, seq_len=(1, 130))
    lay_batch = B.uaa_get_workspace_layout(B.make_desc(cfg), 1100, 130, 152)
    assert lay_batch.n_slices == 2
    rng = np.random.default_rng(5)
    run_and_compare(oracle_mod, cfg, [int(x) for x in rng.integers(0, 130, size=1100)], cap=256, entry=entry,
                    check_qrot=True)


@pytest.mark.parametrize("entry", ENTRIES)
def test_batch_slices_chunk(oracle_mod, entry):
    """Slices with four tokens per sequence: a slice's queries, new rows, q' rows
    and outputs start q_len rows per sequence further on."""
    cfg = W.config("qwen3_8b_ragged", batch=1100, n_q_heads=8, n_kv_heads=2, seq_len=(1, 130), q_len=4)
    lay_batch = B.uaa_get_workspace_layout(B.make_desc(cfg), 1100, 130, 152, 4)
    assert lay_batch.n_slices == 2
    rng = np.random.default_rng(6)
    run_and_compare(oracle_mod, cfg, [int(x) for x in rng.integers(0, 130, size=1100)], cap=256, entry=entry,
                    check_qrot=True)


def test_bf16_output(oracle_mod):
    cfg = W.config("llama31_8b_decode", batch=2, seq_len=300, out_dtype="bf16")
    case = host_case(cfg, lens=[299, 40])
    a = oracle_arrays(case, oracle_mod)
    layer = gpu_layer(case)
    out = layer.step(case["q"].cuda(), case["k_new"].cuda(), case["v_new"].cuda()).float().cpu().numpy()
    want = oracle_mod.decode_step(cfg, a["q"], a["k_new"], a["v_new"], None, None, None, a["k_cache"],
                                  a["v_cache"], None, a["seq_lens"])
    assert np.all(np.abs(out - want) <= TOL_MAX + np.abs(want) * 2.0 ** -8)


def test_batch_zero_is_a_no_op():
    cfg = W.config("llama31_8b_decode", batch=1, seq_len=10)
    from gqa_attention_kv_qk_gb300.layer import DecodeLayer
    layer = DecodeLayer(cfg, 1, 64)
    args = layer.args(None, None, None)
    args.batch = 0
    assert B.uaa_decode_attn(layer.desc, args, layer.ws, torch.cuda.current_stream(), check=False) == B.UAA_OK


# ------------------------------------------------------------------ device-side checks

def test_capacity_flag_and_no_write(oracle_mod):
    cfg = W.config("llama31_8b_decode", batch=2, seq_len=60)
    case = host_case(cfg, lens=[60, 10], cap=64)
    layer = gpu_layer(case)
    layer.set_lengths([64, 10])  # sequence 0 is full
    before = layer.k_cache.clone()
    args = layer.args(case["q"].cuda(), case["k_new"].cuda(), case["v_new"].cuda(), max_seq_len=62)
    B.uaa_decode_attn(layer.desc, args, layer.ws, torch.cuda.current_stream())
    flags = layer.device_status()
    assert flags & B.UAA_DEVFLAG_CAPACITY
    assert layer.seq_lens.cpu().tolist() == [64, 11]
    assert torch.equal(layer.k_cache[0], before[0])
    assert layer.device_status() == 0  # cleared by the read


@pytest.mark.parametrize("name", ["llama31_8b_decode", "llama32_1b_tiny"])
@pytest.mark.parametrize("entry", ENTRIES)
def test_bad_page_entry_is_flagged_and_nothing_else_changes(oracle_mod, name, entry):
    """Failure detection on the host side of a paged cache: a block-table entry
    outside the pool (one under a visible page, one under the new token's page)
    is read as zeros and never written through; the step sets UAA_DEVFLAG_PAGE,
    the other sequence's output stays exact and no page of the pool changes but
    the other sequence's new slot. Both the tensor-core (bf16) and the CUDA-core
    (fp32) kernels."""
    cfg = W.config(name, batch=2, seq_len=300, page_size=32)
    case = host_case(cfg, lens=[299, 200])
    want, _ = run_oracle_step(case, oracle_mod)
    layer = gpu_layer(case)
    orig = layer.block_table.clone()
    k_before, v_before = layer.k_cache.clone(), layer.v_cache.clone()
    layer.block_table[0, 3] = layer.n_pages + 5   # keys 96 .. 127 of sequence 0
    layer.block_table[0, 299 // 32] = -1          # the page of sequence 0's new token
    q, k, v = case["q"].cuda(), case["k_new"].cuda(), case["v_new"].cuda()
    if entry == "split":
        layer.append(q, k, v)
        layer.partial()
        out = layer.combine()
    else:
        out = layer.step(q, k, v)
    torch.cuda.synchronize()
    assert layer.device_status() & B.UAA_DEVFLAG_PAGE
    assert_out_close(out[1].cpu().numpy(), want[1], "the other sequence")
    # only sequence 1's new slot was written
    slot1 = (int(orig[1, 200 // 32]), 200 % 32)
    for pool, before in ((layer.k_cache, k_before), (layer.v_cache, v_before)):
        diff = (pool.float() != before.float()).flatten(2).any(-1).nonzero().tolist()  # [page, head]
        rows = {(pg, h) for pg, h in diff}
        assert rows <= {(slot1[0], h) for h in range(cfg["n_kv_heads"])}, rows
        changed = (pool[slot1[0]].float() != before[slot1[0]].float()).any(-1).nonzero().tolist()
        assert all(r == slot1[1] for _, r in changed), changed


def test_length_hint_violation_is_flagged_and_results_stay_exact(oracle_mod):
    """max_seq_len only bounds the cache check; a longer sequence is flagged at the
    append, and the stream-K split still covers every key."""
    cfg = W.config("llama31_8b_decode", batch=2, seq_len=3000)
    case = host_case(cfg, lens=[2999, 5])
    a = oracle_arrays(case, oracle_mod)
    layer = gpu_layer(case)
    args = layer.args(case["q"].cuda(), case["k_new"].cuda(), case["v_new"].cuda(), max_seq_len=5)
    B.uaa_decode_attn(layer.desc, args, layer.ws, torch.cuda.current_stream())
    flags = layer.device_status()
    assert flags & B.UAA_DEVFLAG_LEN_HINT
    want = oracle_mod.decode_step(cfg, a["q"], a["k_new"], a["v_new"], None, None, None, a["k_cache"],
                                  a["v_cache"], None, a["seq_lens"])
    assert_out_close(layer.out.cpu(), want)


def test_partial_repeated_without_combine_sets_timeout(oracle_mod):
    """The range slots a tensor-core partial launch claims are freed by its
    combine. A second partial launch before that combine finds every slot taken:
    each of its CTAs returns at once (no wait runs out, nothing hangs) and
    UAA_DEVFLAG_TIMEOUT is raised; once the caller zeroes the workspace, the next
    step matches the oracle again."""
    cfg = W.config("llama31_8b_decode", batch=3, seq_len=1400, steps=1)
    case = host_case(cfg, lens=[1000, 1399, 5])
    layer = gpu_layer(case)
    assert layer.layout().kernel == 1
    dev = {k: case[k].cuda() for k in ("q", "k_new", "v_new")}
    layer.append(dev["q"], dev["k_new"], dev["v_new"])
    layer.partial()
    layer.partial()  # the combine of the first launch never ran
    torch.cuda.synchronize()
    assert layer.device_status() & B.UAA_DEVFLAG_TIMEOUT
    layer.ws_tensor.zero_()
    layer.set_lengths(case["lens"])
    out = layer.step(dev["q"], dev["k_new"], dev["v_new"]).cpu()
    want, a = run_oracle_step(case, oracle_mod)
    assert_out_close(out, want)
    assert np.array_equal(layer.seq_lens.cpu().numpy(), a["seq_lens"])
    assert layer.device_status() == 0


def test_workspace_shared_by_two_geometries(oracle_mod):
    """One workspace serving two descs of different P in turn (head_dim 128 at two
    CTAs per SM, then head_dim 256 at one): the second geometry's balance arrays
    lie over the first's claim words. A launch of the second desc with fewer
    stages than CTAs leaves the slots without work at weight 0 (nothing
    measured, so the next launch splits uniformly) instead of reading stale
    words as rates; both descs match the oracle throughout."""
    c1 = W.config("llama31_8b_decode", batch=4, seq_len=4000, steps=1)
    c2 = W.layer_configs(W.config("gemma2_9b_swa", batch=2, seq_len=300, steps=1, layers=[dict(window=0)]))[0]
    case1, case2 = host_case(c1), host_case(c2, lens=[299, 40])
    L1, L2 = gpu_layer(case1), gpu_layer(case2)
    P1, P2 = L1.layout().n_ctas, L2.layout().n_ctas
    assert P1 != P2 and L1.layout().kernel == 1 and L2.layout().kernel == 1
    nbytes = max(L1.ws_tensor.numel(), L2.ws_tensor.numel())
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for L in (L1, L2):
        L.ws_tensor, L.ws = ws, B.UaaWorkspace(ws.data_ptr(), nbytes)
    d1 = {k: case1[k].cuda() for k in ("q", "k_new", "v_new")}
    d2 = {k: case2[k].cuda() for k in ("q", "k_new", "v_new")}
    want1, _ = run_oracle_step(case1, oracle_mod)
    want2, _ = run_oracle_step(case2, oracle_mod)
    al = lambda x: -(-x // 256) * 256
    for rep in range(2):
        for _ in range(3):
            L1.set_lengths(case1["lens"])
            assert_out_close(L1.step(d1["q"], d1["k_new"], d1["v_new"]).cpu(), want1, "head_dim 128")
        L2.set_lengths(case2["lens"])
        assert_out_close(L2.step(d2["q"], d2["k_new"], d2["v_new"]).cpu(), want2, "head_dim 256")
        torch.cuda.synchronize()
        lay = L2.layout()
        T2 = int(ws[lay.prefix_offset: lay.prefix_offset + 3 * 4].view(torch.int32)[-1].item())
        assert 0 < T2 < P2
        w0 = lay.balance_offset + 256 + al(8 * P2) + al(4 * P2)
        weight = ws[w0: w0 + 4 * P2].view(torch.float32).cpu().numpy()
        cumw = ws[w0 + al(4 * P2): w0 + al(4 * P2) + 4 * (P2 + 1)].view(torch.int32).cpu().numpy()
        assert np.all(weight[T2:] == 0.0), "a slot without work kept a weight"
        assert np.all(cumw == 0), "a launch with unmeasured slots must split uniformly next"
        assert L1.device_status() == 0


@pytest.mark.parametrize("name,over", [("llama31_8b_decode", dict(batch=4, seq_len=4000)),
                                       ("gptoss_vq8_sink", dict(batch=4, seq_len=3000)),
                                       ("llama31_8b_q8", dict(batch=3, seq_len=3000))])
def test_reproducible_desc_gives_equal_bits(oracle_mod, name, over):
    """With reproducible = 1 the tensor-core kernel keeps its ranges uniform
    whatever the slot speeds measured before: the same step repeated on the same
    inputs gives the same bits on every launch, and matches the oracle."""
    cfg = W.config(name, reproducible=True, steps=1, **over)
    case = host_case(cfg)
    layer = gpu_layer(case)
    assert layer.layout().kernel == 1
    dev = {k: case[k].cuda() for k in ("q", "k_new", "v_new")}
    outs = []
    for _ in range(5):
        layer.set_lengths(case["lens"])
        outs.append(layer.step(dev["q"], dev["k_new"], dev["v_new"], advance_hint=False).clone())
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    want, a = run_oracle_step(case, oracle_mod)
    assert_out_close(outs[0].cpu(), want)
    lay = layer.layout()
    ws = layer.ws_tensor
    Bn, P = cfg["batch"], lay.n_ctas
    T = int(ws[lay.prefix_offset: lay.prefix_offset + (Bn + 1) * 4].view(torch.int32)[-1].item())
    n = min(P, T)
    starts = ws[lay.ranges_offset: lay.ranges_offset + (n + 1) * 8].view(torch.int64).cpu().numpy()
    assert np.array_equal(starts, [c * T // n for c in range(n + 1)])
    assert layer.device_status() == 0


@pytest.mark.parametrize("over,lens", [
    (dict(batch=3, seq_len=1500), [1499, 600, 0]),
    (dict(batch=2, seq_len=1100, window=700, softcap=30.0, has_sink=True, qk_norm=True,
          norm_w_range=(0.5, 1.5)), [1099, 1]),
    (dict(batch=2, seq_len=1100, n_q_heads=40, n_kv_heads=4, page_size=64), [1099, 513]),
])
def test_fp32_step_in_one_kernel(oracle_mod, over, lens):
    """The fp32 decode step in one launch with several key splits per unit, merged
    by the split that finishes last (with window, softcap, sink and QK norm; ten
    query heads per kv head, two head groups; paged), over two chained steps."""
    cfg = W.config("llama32_1b_tiny", steps=2, **over)
    lay = B.uaa_get_workspace_layout(B.make_desc(cfg), cfg["batch"], max(lens) + 1, 0)
    assert lay.step_kernels == 1 and lay.step_splits >= 2
    run_and_compare(oracle_mod, cfg, lens, steps=2, entry="fused")


# ------------------------------------------------------------------ split partials

def stream_k_segments(prefix, starts, units, head_groups):
    """The documented stream-K partition: range c holds stages [starts[c],
    starts[c+1]) of the concatenated unit stages (the table the partial kernel
    leaves in the workspace), cut at unit boundaries."""
    import bisect
    T = int(prefix[-1])
    assert starts[0] == 0 and starts[-1] == T and np.all(np.diff(starts) > 0)
    for c in range(len(starts) - 1):
        s, e = int(starts[c]), int(starts[c + 1])
        pos = s
        while pos < e:
            b = bisect.bisect_right(prefix, pos) - 1
            stg = (int(prefix[b + 1]) - int(prefix[b])) // units
            local = pos - int(prefix[b])
            u, st0 = divmod(local, stg)
            n = min(e - pos, stg - st0)
            kvh, hg = divmod(u, head_groups)
            yield dict(cta=c, slot=0 if pos == s else 1, b=b, kvh=kvh, hg=hg, st0=st0, n=n,
                       whole=(st0 == 0 and n == stg))
            pos += n


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("name,over,lens", [
    ("llama31_8b_decode", dict(batch=3, seq_len=3000), [2999, 700, 1]),
    ("gptoss_vq8_sink", dict(batch=2, seq_len=3000), [2999, 130]),
    ("gemma2_9b_swa", dict(batch=2, seq_len=3000, layers=[dict(window=1000)]), [2999, 1500]),
    ("llama32_1b_tiny", dict(batch=1, seq_len=700), [699]),
    ("llama31_8b_decode", dict(batch=2, n_q_heads=32, n_kv_heads=2, seq_len=900), [899, 64]),
])
def test_partial_records_match_oracle_ranges(oracle_mod, name, over, lens, entry):
    """After the append and the partial step (separate, or the fused
    append+partial call): each record equals the oracle's softmax restricted to
    its segment's keys, and each unit finished inside one CTA has its output rows
    (sink included) equal to the full attention."""
    cfg = W.layer_configs(W.config(name, **over))[0]
    case = host_case(cfg, lens=lens)
    a = oracle_arrays(case, oracle_mod)
    layer = gpu_layer(case)
    lay = layer.layout()
    dev = {k: case[k].cuda() for k in ("q", "k_new", "v_new")}
    lens0 = layer.seq_lens.clone()
    stream = torch.cuda.current_stream()
    for rep in range(3):  # from the second launch on, the tensor-core kernel's ranges are weighted
        if rep:  # the combine frees the range slots of the previous partial launch
            B.uaa_decode_attn_combine(layer.desc, layer.args(None, None, None), layer.ws, stream)
        layer.seq_lens.copy_(lens0)
        layer.out.fill_(float("nan"))
        if entry == "split":
            layer.append(dev["q"], dev["k_new"], dev["v_new"])
            layer.partial()
        else:
            layer.append_partial(dev["q"], dev["k_new"], dev["v_new"])
    torch.cuda.synchronize()
    qr = oracle_mod.append(cfg, a["q"], a["k_new"], a["v_new"], a["q_norm_w"], a["k_norm_w"], a["k_cache"],
                           a["v_cache"], a["v_scale"], a["seq_lens"])
    full = oracle_mod.attend(cfg, qr, a["sink"], a["k_cache"], a["v_cache"], a["v_scale"], a["seq_lens"])
    Bn, Hq, D, Hkv = cfg["batch"], cfg["n_q_heads"], cfg["head_dim"], cfg["n_kv_heads"]
    G = Hq // Hkv
    HC, P, mg = lay.heads_per_cta, lay.n_ctas, lay.stage_keys // 64
    hgroups = -(-G // HC)
    ws = layer.ws_tensor
    assert lay.n_slices == 1
    prefix = ws[lay.prefix_offset: lay.prefix_offset + (Bn + 1) * 4].view(torch.int32).cpu().numpy()
    n_ranges = min(P, int(prefix[-1]))
    starts = ws[lay.ranges_offset: lay.ranges_offset + (n_ranges + 1) * 8].view(torch.int64).cpu().numpy()
    rec_lse = ws[lay.rec_lse_offset: lay.rec_lse_offset + 2 * P * HC * 4].view(torch.float32).view(2 * P, HC)
    rec_o = ws[lay.rec_o_offset: lay.rec_o_offset + 2 * P * HC * D * 4].view(torch.float32).view(2 * P, HC, D)
    rec_lse, rec_o = rec_lse.cpu().numpy(), rec_o.cpu().numpy()
    out = layer.out.cpu().numpy()
    W_ = cfg.get("window", 0) or 0
    n_whole = n_rec = 0
    for sg in stream_k_segments(prefix, starts, Hkv * hgroups, hgroups):
        b = sg["b"]
        n = int(a["seq_lens"][b])
        lo = max(0, n - W_) if W_ else 0
        t0 = lo // 64
        j0 = max(lo, (t0 + mg * sg["st0"]) * 64)
        j1 = min(n, (t0 + mg * (sg["st0"] + sg["n"])) * 64)
        heads = [sg["kvh"] * G + sg["hg"] * HC + hc for hc in range(HC) if sg["hg"] * HC + hc < G]
        for hc, h in enumerate(heads):
            if sg["whole"]:
                assert np.max(np.abs(out[b, h] - full[b, h])) <= TOL_MAX
                n_whole += 1
            else:
                g = sg["kvh"]
                sr = None if a["v_scale"] is None else a["v_scale"][b, g]
                o, l_nat = oracle_mod.attend_range(cfg, qr[b, h], a["k_cache"][b, g], a["v_cache"][b, g], sr, j0, j1)
                r = 2 * sg["cta"] + sg["slot"]
                assert np.max(np.abs(rec_o[r, hc] - o)) <= TOL_MAX
                assert abs(rec_lse[r, hc] * math.log(2.0) - l_nat) <= 2e-3 * max(1.0, abs(l_nat))
                n_rec += 1
    assert n_rec > 0  # every case here has units cut between CTAs


# ------------------------------------------------------------------ full size, sampled

FULL = ["llama32_1b_tiny", "llama31_8b_decode", "qwen3_8b_ragged", "gemma2_9b_swa", "gptoss_vq8_sink",
        "gemma3_12b_local_global", "llama31_8b_q8", "llama31_8b_paged", "llama31_8b_verify"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(oracle_mod, name):
    """The workloads at their full sizes, in the launch configuration the benchmark
    times (one fused uaa_decode_attn call per layer); outputs checked on sampled
    (sequence, head) rows, cache writes and lengths checked everywhere."""
    cfg = W.config(name)
    rng = np.random.default_rng(123)
    for layer_cfg in W.layer_configs(cfg):
        case = host_case(layer_cfg)
        layer = gpu_layer(case)
        out = layer.step(case["q"].cuda(), case["k_new"].cuda(), case["v_new"].cuda()).cpu().numpy()
        a = oracle_arrays(case, oracle_mod)
        T = int(layer_cfg.get("q_len", 1) or 1)
        Bn, Hq = layer_cfg["batch"], layer_cfg["n_q_heads"]
        units = sorted({(int(rng.integers(Bn)), int(rng.integers(Hq))) for _ in range(24)} | {(0, 0), (Bn - 1, Hq - 1)})
        for t in range(T):  # token t: appended, then attended, before token t + 1
            pick = (lambda x: x) if T == 1 else (lambda x: np.ascontiguousarray(x[:, t]))
            qr = oracle_mod.append(layer_cfg, pick(a["q"]), pick(a["k_new"]), pick(a["v_new"]), a["q_norm_w"],
                                   a["k_norm_w"], a["k_cache"], a["v_cache"], a["v_scale"], a["seq_lens"], a["k_scale"])
            want = oracle_mod.attend(layer_cfg, qr, a["sink"], a["k_cache"], a["v_cache"], a["v_scale"],
                                     a["seq_lens"], units=units, k_scale=a["k_scale"])
            got = np.stack([(out[b, h] if T == 1 else out[b, t, h]) for b, h in units])
            assert_out_close(got, want, f"{name} token {t}")
        assert np.array_equal(layer.seq_lens.cpu().numpy(), a["seq_lens"])
        assert layer.device_status() == 0
        if layer_cfg["kv_dtype"] in ("vq8", "q8"):
            pre = case["lens"].numpy()
            vc = layer.logical("v_cache")
            for b in range(Bn):
                assert np.array_equal(vc[b, :, pre[b]].cpu().numpy(), a["v_cache"][b, :, pre[b]])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama31_8b_decode", "llama31_8b_q8"])
def test_full_size_64_chained_steps(oracle_mod, name):
    """The Llama-3.1-8B-like workload as the benchmark runs it: 16 sequences from
    8192 cached tokens, 64 consecutive decode steps through the whole-step call
    (fresh q / k / v for every step). Every step's full output against the
    oracle's; after the last step the lengths, all 64 appended key and value rows
    of every (sequence, kv head), and the untouched rows below them."""
    cfg = W.config(name)
    n = cfg["steps"]
    assert n == 64
    case = host_case(cfg)
    a = oracle_arrays(case, oracle_mod)
    kv = cfg["kv_dtype"]
    orig = {k: a[k].copy() for k in ("k_cache", "v_cache")}
    layer = gpu_layer(case)
    L0 = case["lens"].numpy().astype(np.int64)
    assert np.all(L0 == L0[0])
    L = int(L0[0])
    hint = L + n - 1
    for step in range(n):
        inp = W.step_inputs(cfg, step)
        out = layer.step(inp["q"].cuda(), inp["k_new"].cuda(), inp["v_new"].cuda(), max_seq_len=hint).cpu()
        qr = oracle_mod.append(cfg, W.bits(inp["q"]).copy(), W.bits(inp["k_new"]).copy(),
                               W.bits(inp["v_new"]).copy(), a["q_norm_w"], a["k_norm_w"], a["k_cache"],
                               a["v_cache"], a["v_scale"], a["seq_lens"], a["k_scale"])
        want = oracle_mod.attend(cfg, qr, a["sink"], a["k_cache"], a["v_cache"], a["v_scale"], a["seq_lens"],
                                 k_scale=a["k_scale"])
        assert_out_close(out, want, f"{name} step {step}")
        assert np.array_equal(layer.seq_lens.cpu().numpy(), a["seq_lens"])
    assert layer.device_status() == 0
    assert np.all(a["seq_lens"] == L + n)
    new = slice(L, L + n)
    kg = layer.k_cache[:, :, new].cpu()
    if kv == "q8":
        vg = layer.v_cache[:, :, new].cpu().numpy()
        kcg, kco = kg.numpy().astype(np.int64), a["k_cache"][:, :, new].astype(np.int64)
        assert np.abs(kcg - kco).max() <= 1, "q8 key code off by more than one"
        per_row = (kcg != kco).sum(axis=-1)
        assert per_row.max() <= 2 and (kcg != kco).sum() <= kco.size // 100
        ksg = layer.k_scale[:, :, new].cpu().numpy().astype(np.float64)
        assert np.allclose(ksg, a["k_scale"][:, :, new], rtol=2e-6, atol=0)
        assert np.array_equal(vg, a["v_cache"][:, :, new])
        assert np.array_equal(layer.v_scale[:, :, new].cpu().numpy().view(np.uint32),
                              a["v_scale"][:, :, new].view(np.uint32))
        below = (layer.k_cache[:, :, :L].cpu().numpy(), layer.v_cache[:, :, :L].cpu().numpy())
    else:
        assert np.array_equal(kg.view(torch.int16).numpy().view(np.uint16), a["k_cache"][:, :, new]), \
            "an appended key row differs"
        assert np.array_equal(layer.v_cache[:, :, new].view(torch.int16).cpu().numpy().view(np.uint16),
                              a["v_cache"][:, :, new]), "an appended value row differs"
        below = (layer.k_cache[:, :, :L].view(torch.int16).cpu().numpy().view(np.uint16),
                 layer.v_cache[:, :, :L].view(torch.int16).cpu().numpy().view(np.uint16))
    assert np.array_equal(below[0], orig["k_cache"][:, :, :L]), "a cached key row changed"
    assert np.array_equal(below[1], orig["v_cache"][:, :, :L]), "a cached value row changed"
