"""Test cases built from the seeded workload generators.

`host_case` draws one step's inputs and a cache; `oracle_arrays` turns them into
the storage arrays the oracle takes (a vq8 or q8 cache quantised by the oracle's
own quantiser). Nothing here computes any part of the method.
"""
import numpy as np
import torch

from gqa_attention_kv_qk_gb300 import workloads as W


host_case = W.host_case  # seeded inputs and cache (gqa_attention_kv_qk_gb300.workloads)


def oracle_arrays(case: dict, oracle_mod) -> dict:
    """Storage arrays for the oracle (copies: the oracle's append mutates them)."""
    cfg = case["cfg"]
    a = dict(
        q=W.bits(case["q"]).copy(), k_new=W.bits(case["k_new"]).copy(),
        v_new=W.bits(case["v_new"]).copy(),
        seq_lens=case["lens"].numpy().astype(np.int32).copy(),
        q_norm_w=None if case["q_norm_w"] is None else case["q_norm_w"].numpy().copy(),
        k_norm_w=None if case["k_norm_w"] is None else case["k_norm_w"].numpy().copy(),
        sink=None if case["sink"] is None else case["sink"].numpy().copy(),
    )
    kv = cfg.get("kv_dtype")
    if kv == "q8":
        a["k_cache"], a["k_scale"] = oracle_mod.vq8_quantize(case["k_values"].numpy())
    else:
        a["k_cache"], a["k_scale"] = W.bits(case["k_cache"]).copy(), None
    if kv in ("vq8", "q8"):
        codes, scales = oracle_mod.vq8_quantize(case["v_values"].numpy())
        a["v_cache"], a["v_scale"] = codes, scales
    else:
        a["v_cache"], a["v_scale"] = W.bits(case["v_cache"]).copy(), None
    return a


def run_oracle_step(case: dict, oracle_mod, n_threads=None):
    a = oracle_arrays(case, oracle_mod)
    step = oracle_mod.chunk_step if int(case["cfg"].get("q_len", 1) or 1) > 1 else oracle_mod.decode_step
    out = step(case["cfg"], a["q"], a["k_new"], a["v_new"], a["q_norm_w"],
                                 a["k_norm_w"], a["sink"], a["k_cache"], a["v_cache"],
                                 a["v_scale"], a["seq_lens"], n_threads=n_threads, k_scale=a["k_scale"])
    return out, a


# ---------------------------------------------------------------- GPU side

def gpu_layer(case: dict, device="cuda"):
    """A DecodeLayer holding the case's cache (a vq8 / q8 cache is quantised on the device)."""
    from gqa_attention_kv_qk_gb300.layer import DecodeLayer
    return DecodeLayer.for_case(case, device)
