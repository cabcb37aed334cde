"""Brute-force decode step in matrix form, for pinning the oracle on tiny inputs.

Written independently of the oracle: rotations are explicit D x D matrices,
the GQA grouping is numpy repeat, the softmax is one vectorised expression over
the masked logit vector with the sink appended as an extra entry, bf16 storage
uses torch's cast and vq8 uses numpy float32 arithmetic. Only the rotary
frequency table of the scaled variants (llama3, yarn) is taken as an argument;
those tables are pinned separately.
"""
import numpy as np
import torch


def plain_inv_freq(D: int, base: float) -> np.ndarray:
    return np.power(float(base), -np.arange(0, D, 2, dtype=np.float64) / D)


def pair_indices(D: int, style: str):
    half = D // 2
    p = np.arange(half)
    if style == "neox":
        return p, p + half
    return 2 * p, 2 * p + 1


def rotation_matrix(D: int, style: str, inv_freq: np.ndarray, mscale: float, pos: int,
                    rotary_dim: int = 0) -> np.ndarray:
    """Block diagonal: the rotation of the first rotary_dim dims (all of them when
    0), and the identity on the rest."""
    rd = rotary_dim or D
    R = np.eye(D, dtype=np.float64)
    ia, ib = pair_indices(rd, style)
    ang = pos * np.asarray(inv_freq)[: rd // 2]
    c, s = np.cos(ang) * mscale, np.sin(ang) * mscale
    R[ia, ia] = c
    R[ia, ib] = -s
    R[ib, ia] = s
    R[ib, ib] = c
    return R


def rmsnorm_rows(X: np.ndarray, w: np.ndarray, eps: float, w_offset: float = 0.0) -> np.ndarray:
    return X / np.sqrt(np.mean(X * X, axis=-1, keepdims=True) + eps) * (w.astype(np.float64) + w_offset)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def vq8_numpy(v: np.ndarray):
    v = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v), axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(v / s[..., None]).astype(np.float32)
    q = np.where(s[..., None] == 0, np.float32(0), np.clip(q, -127, 127))
    return q.astype(np.int8), s


def chunk_step(cfg: dict, q, k_new, v_new, k_cache, v_cache, seq_lens, q_norm_w=None, k_norm_w=None, sink=None,
               inv_freq=None, mscale=1.0, causal=True):
    """T tokens per sequence in one matrix expression (bf16 and f32 caches): all T
    keys appended at positions L .. L + T - 1 first, then one logit matrix of the
    T Hq query rows against every key, masked by token t's causal (j <= L + t) and
    window (j > L + t - W) limits, softmax per row with the sink as an extra
    column. q [B][T][Hq][D], k_new / v_new [B][T][Hkv][D] fp64; caches mutate.
    Returns out [B][T][Hq][D]."""
    B, T, Hq, D = q.shape
    Hkv = k_new.shape[2]
    G = Hq // Hkv
    style = cfg.get("rope_style", "neox")
    rd = cfg.get("rotary_dim", 0) or D
    off = 1.0 if cfg.get("norm_offset") else 0.0
    if inv_freq is None:
        inv_freq = plain_inv_freq(rd, cfg.get("rope_theta", 10000.0))
    scale = cfg.get("scale", 0.0) or 1.0 / np.sqrt(D)
    kv = cfg.get("kv_dtype", "bf16")
    W = cfg.get("window", 0) or 0
    cap_ = cfg.get("softcap", 0.0) or 0.0
    eps = cfg.get("norm_eps", 1e-6)
    out = np.zeros((B, T, Hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        Qr = np.zeros((T, Hq, D))
        for t in range(T):
            R = rotation_matrix(D, style, inv_freq, mscale, L + t, rd)
            qb, kb = q[b, t].astype(np.float64), k_new[b, t].astype(np.float64)
            if cfg.get("qk_norm"):
                qb, kb = rmsnorm_rows(qb, q_norm_w, eps, off), rmsnorm_rows(kb, k_norm_w, eps, off)
            Qr[t] = qb @ R.T
            kr = kb @ R.T
            if kv == "bf16":
                k_cache[b, :, L + t], v_cache[b, :, L + t] = bf16_round(kr), bf16_round(v_new[b, t])
            else:
                k_cache[b, :, L + t] = kr.astype(np.float32).astype(np.float64)
                v_cache[b, :, L + t] = v_new[b, t].astype(np.float32).astype(np.float64)
        n = L + T
        seq_lens[b] = n
        K = np.repeat(k_cache[b, :, :n], G, axis=0)                      # [Hq][n][D]
        V = np.repeat(v_cache[b, :, :n], G, axis=0)
        S = scale * np.einsum("thd,hjd->thj", Qr, K)                     # [T][Hq][n]
        if cap_ > 0:
            S = cap_ * np.tanh(S / cap_)
        j = np.arange(n)[None, :]
        pos = (L + np.arange(T))[:, None]
        visible = ((j <= pos) if causal else (j < n)) & ((j > pos - W) if W > 0 else True)  # [T][n]
        S = np.where(visible[:, None, :], S, -np.inf)
        if sink is not None:
            z = np.broadcast_to(np.asarray(sink, dtype=np.float64)[None, :, None], (T, Hq, 1))
            S = np.concatenate([S, z], axis=2)
        P = np.exp(S - S.max(axis=2, keepdims=True))
        P = P / P.sum(axis=2, keepdims=True)
        out[b] = np.einsum("thj,hjd->thd", P[:, :, :n], V)
    return out


def decode_step(cfg: dict, q, k_new, v_new, k_cache, v_cache, v_scale, seq_lens,
                q_norm_w=None, k_norm_w=None, sink=None, inv_freq=None, mscale=1.0, k_scale=None):
    """All arrays fp64 (values, codes as float, scales as float). Caches mutate.
    Returns out [B][Hq][D]."""
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    G = Hq // Hkv
    style = cfg.get("rope_style", "neox")
    rd = cfg.get("rotary_dim", 0) or D
    off = 1.0 if cfg.get("norm_offset") else 0.0
    if inv_freq is None:
        inv_freq = plain_inv_freq(rd, cfg.get("rope_theta", 10000.0))
    scale = cfg.get("scale", 0.0) or 1.0 / np.sqrt(D)
    kv = cfg.get("kv_dtype", "bf16")
    W = cfg.get("window", 0) or 0
    cap_ = cfg.get("softcap", 0.0) or 0.0
    out = np.zeros((B, Hq, D))
    for b in range(B):
        pos = int(seq_lens[b])
        R = rotation_matrix(D, style, inv_freq, mscale, pos, rd)
        qb, kb = q[b].astype(np.float64), k_new[b].astype(np.float64)
        if cfg.get("qk_norm"):
            qb = rmsnorm_rows(qb, q_norm_w, cfg.get("norm_eps", 1e-6), off)
            kb = rmsnorm_rows(kb, k_norm_w, cfg.get("norm_eps", 1e-6), off)
        qr = qb @ R.T
        kr = kb @ R.T
        if kv == "bf16":
            kr = bf16_round(kr)
            vb = bf16_round(v_new[b])
        elif kv == "f32":
            kr = kr.astype(np.float32).astype(np.float64)
            vb = v_new[b].astype(np.float32).astype(np.float64)
        elif kv == "q8":
            kcodes, ks = vq8_numpy(kr.astype(np.float32))
            k_scale[b, :, pos] = ks
            kr = kcodes.astype(np.float64)
            codes, s = vq8_numpy(v_new[b].astype(np.float32))
            v_scale[b, :, pos] = s
            vb = codes.astype(np.float64)
        else:
            kr = bf16_round(kr)
            codes, s = vq8_numpy(v_new[b].astype(np.float32))
            v_scale[b, :, pos] = s
            vb = codes.astype(np.float64)
        k_cache[b, :, pos] = kr
        v_cache[b, :, pos] = vb
        seq_lens[b] = pos + 1
        n = pos + 1
        lo = max(0, n - W) if W > 0 else 0
        K = np.repeat(k_cache[b, :, lo:n], G, axis=0)          # [Hq][n'][D]
        V = np.repeat(v_cache[b, :, lo:n], G, axis=0)
        if kv in ("vq8", "q8"):
            V = V * np.repeat(v_scale[b, :, lo:n], G, axis=0)[..., None]
        if kv == "q8":
            K = K * np.repeat(k_scale[b, :, lo:n], G, axis=0)[..., None]
        S = scale * np.einsum("hd,hjd->hj", qr, K)
        if cap_ > 0:
            S = cap_ * np.tanh(S / cap_)
        if sink is not None:
            S = np.concatenate([S, np.asarray(sink, dtype=np.float64)[:, None]], axis=1)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P = P / P.sum(axis=1, keepdims=True)
        out[b] = np.einsum("hj,hjd->hd", P[:, : n - lo], V)
    return out
