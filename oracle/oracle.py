"""ctypes face of the CPU fp64 oracle (liboracle.so).

Test infrastructure: only the tests, the smoke check and the benchmark's
CPU-baseline / reference legs import this module. Arrays are numpy; bf16 data
travels as uint16 bit patterns, vq8 / q8 codes as int8.

A step description is a plain dict with the keys
  n_q_heads n_kv_heads head_dim scale rope_style rope_theta rope_scaling factor
  low_freq_factor high_freq_factor original_max_pos beta_fast beta_slow
  attn_factor qk_norm norm_eps window softcap has_sink kv_dtype io_dtype
  rotary_dim norm_offset
(missing keys take the neutral value: no scaling, no norm, no window, ...).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_STYLE = {"neox": 0, "interleaved": 1}
_SCALING = {"none": 0, "llama3": 1, "yarn": 2, "linear": 3}
_DTYPE = {"f32": 0, "bf16": 1, "vq8": 2, "q8": 3}


class OracleDesc(ctypes.Structure):
    _fields_ = [
        ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("scale", ctypes.c_double),
        ("rope_style", ctypes.c_int), ("rope_theta", ctypes.c_double),
        ("rope_scaling", ctypes.c_int), ("factor", ctypes.c_double),
        ("low_freq_factor", ctypes.c_double), ("high_freq_factor", ctypes.c_double),
        ("original_max_pos", ctypes.c_int), ("beta_fast", ctypes.c_double),
        ("beta_slow", ctypes.c_double), ("attn_factor", ctypes.c_double),
        ("qk_norm", ctypes.c_int), ("norm_eps", ctypes.c_double),
        ("window", ctypes.c_int), ("softcap", ctypes.c_double), ("has_sink", ctypes.c_int),
        ("kv_dtype", ctypes.c_int), ("io_dtype", ctypes.c_int),
        ("rotary_dim", ctypes.c_int), ("norm_offset", ctypes.c_int),
    ]


def make_desc(cfg: dict) -> OracleDesc:
    d = OracleDesc()
    d.n_q_heads = int(cfg["n_q_heads"])
    d.n_kv_heads = int(cfg["n_kv_heads"])
    d.head_dim = int(cfg["head_dim"])
    d.scale = float(cfg.get("scale", 0.0) or 0.0)
    d.rope_style = _STYLE[cfg.get("rope_style", "neox")]
    d.rope_theta = float(cfg.get("rope_theta", 10000.0))
    d.rope_scaling = _SCALING[cfg.get("rope_scaling", "none")]
    d.factor = float(cfg.get("factor", 1.0))
    d.low_freq_factor = float(cfg.get("low_freq_factor", 1.0))
    d.high_freq_factor = float(cfg.get("high_freq_factor", 4.0))
    d.original_max_pos = int(cfg.get("original_max_pos", 8192))
    d.beta_fast = float(cfg.get("beta_fast", 32.0))
    d.beta_slow = float(cfg.get("beta_slow", 1.0))
    d.attn_factor = float(cfg.get("attn_factor", 0.0) or 0.0)
    d.qk_norm = int(bool(cfg.get("qk_norm", False)))
    d.norm_eps = float(cfg.get("norm_eps", 1e-6))
    d.window = int(cfg.get("window", 0) or 0)
    d.softcap = float(cfg.get("softcap", 0.0) or 0.0)
    d.has_sink = int(bool(cfg.get("has_sink", False)))
    d.kv_dtype = _DTYPE[cfg.get("kv_dtype", "bf16")]
    d.io_dtype = _DTYPE[cfg.get("io_dtype", "bf16")]
    d.rotary_dim = int(cfg.get("rotary_dim", 0) or 0)
    d.norm_offset = int(bool(cfg.get("norm_offset", False)))
    return d


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.POINTER
        vp, dp, fp, ip = ctypes.c_void_p, P(ctypes.c_double), P(ctypes.c_float), P(ctypes.c_int32)
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        L.oracle_bf16_from_double.restype = ctypes.c_uint16
        L.oracle_rope_inv_freq.argtypes = [P(OracleDesc), dp, dp]
        L.oracle_rms_norm.argtypes = [dp, fp, ctypes.c_int, ctypes.c_double, ctypes.c_double, dp]
        L.oracle_rope_rotate.argtypes = [P(OracleDesc), dp, ctypes.c_double, ctypes.c_long, dp, dp]
        L.oracle_vq8_quantize_row.argtypes = [fp, ctypes.c_int, P(ctypes.c_int8), fp]
        L.oracle_append.argtypes = [P(OracleDesc), ctypes.c_int, vp, vp, vp, fp, fp, vp, vp, fp, fp,
                                    ctypes.c_int, ip, dp]
        L.oracle_append.restype = ctypes.c_int
        L.oracle_attend_range.argtypes = [P(OracleDesc), dp, vp, vp, fp, fp, ctypes.c_long,
                                          ctypes.c_long, ctypes.c_int, ctypes.c_double, dp, dp]
        L.oracle_attend.argtypes = [P(OracleDesc), ctypes.c_int, dp, fp, vp, vp, fp, fp, ctypes.c_int,
                                    ip, ip, ctypes.c_int, dp, ctypes.c_int]
        L.oracle_decode_step.argtypes = [P(OracleDesc), ctypes.c_int, vp, vp, vp, fp, fp, fp, vp,
                                         vp, fp, fp, ctypes.c_int, ip, dp, ctypes.c_int]
        L.oracle_decode_step.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a, ctype=None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    if ctype is None:
        return ctypes.c_void_p(a.ctypes.data)
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _io_array(x, io_dtype):
    x = np.ascontiguousarray(x)
    want = np.float32 if io_dtype == "f32" else np.uint16
    assert x.dtype == want, f"io array must be {want}, got {x.dtype}"
    return x


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------- elementwise parts

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    f = lib().oracle_bf16_to_double
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([f(int(v)) for v in flat], dtype=np.float64).reshape(np.shape(bits))


def bf16_from_f64(x: np.ndarray) -> np.ndarray:
    f = lib().oracle_bf16_from_double
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.array([f(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(x))


def rope_inv_freq(cfg: dict):
    d = make_desc(cfg)
    out = np.zeros(d.head_dim // 2, dtype=np.float64)
    ms = ctypes.c_double()
    lib().oracle_rope_inv_freq(ctypes.byref(d), _ptr(out, ctypes.c_double), ctypes.byref(ms))
    return out, ms.value


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float, w_offset: float = 0.0) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = np.zeros_like(x)
    lib().oracle_rms_norm(_ptr(x, ctypes.c_double), _ptr(w, ctypes.c_float), x.size, eps,
                          float(w_offset), _ptr(y, ctypes.c_double))
    return y


def rope_rotate(cfg: dict, x: np.ndarray, pos: int) -> np.ndarray:
    d = make_desc(cfg)
    inv, ms = rope_inv_freq(cfg)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros_like(x)
    lib().oracle_rope_rotate(ctypes.byref(d), _ptr(inv, ctypes.c_double), ms, int(pos),
                             _ptr(x, ctypes.c_double), _ptr(y, ctypes.c_double))
    return y


def vq8_quantize(v: np.ndarray):
    """v: float32 [..., D] -> (codes int8 [..., D], scales float32 [...])."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    D = v.shape[-1]
    rows = v.reshape(-1, D)
    codes = np.zeros(rows.shape, dtype=np.int8)
    scales = np.zeros(rows.shape[0], dtype=np.float32)
    L = lib()
    for r in range(rows.shape[0]):
        row = np.ascontiguousarray(rows[r])
        c = np.zeros(D, dtype=np.int8)
        s = ctypes.c_float()
        L.oracle_vq8_quantize_row(_ptr(row, ctypes.c_float), D, _ptr(c, ctypes.c_int8),
                                  ctypes.byref(s))
        codes[r] = c
        scales[r] = s.value
    return codes.reshape(v.shape), scales.reshape(v.shape[:-1])


# ---------------------------------------------------------------- the step

def append(cfg: dict, q, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, v_scale,
           seq_lens, k_scale=None) -> np.ndarray:
    """Append in place (caches, scales and seq_lens mutate). Returns q_rot fp64 [B][Hq][D]."""
    d = make_desc(cfg)
    io = cfg.get("io_dtype", "bf16")
    q, k_new, v_new = (_io_array(a, io) for a in (q, k_new, v_new))
    B = q.shape[0]
    q_rot = np.zeros((B, d.n_q_heads, d.head_dim), dtype=np.float64)
    w_q = None if q_norm_w is None else np.ascontiguousarray(q_norm_w, dtype=np.float32)
    w_k = None if k_norm_w is None else np.ascontiguousarray(k_norm_w, dtype=np.float32)
    if d.qk_norm:
        assert w_q is not None and w_k is not None
    assert seq_lens.dtype == np.int32 and seq_lens.flags["C_CONTIGUOUS"]
    cap = k_cache.shape[2]
    rc = lib().oracle_append(ctypes.byref(d), B, _ptr(q), _ptr(k_new), _ptr(v_new),
                             _ptr(w_q, ctypes.c_float), _ptr(w_k, ctypes.c_float),
                             _ptr(k_cache), _ptr(v_cache), _ptr(v_scale, ctypes.c_float),
                             _ptr(k_scale, ctypes.c_float),
                             cap, _ptr(seq_lens, ctypes.c_int32), _ptr(q_rot, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle append refused: a sequence is at capacity")
    return q_rot


def attend(cfg: dict, q_rot, sink, k_cache, v_cache, v_scale, seq_lens, units=None,
           n_threads=None, k_scale=None) -> np.ndarray:
    """Attention after the append. units: None (all, -> [B][Hq][D]) or list of (b, h)."""
    d = make_desc(cfg)
    q_rot = np.ascontiguousarray(q_rot, dtype=np.float64)
    B = q_rot.shape[0]
    cap = k_cache.shape[2]
    sink_a = None if sink is None else np.ascontiguousarray(sink, dtype=np.float32)
    if d.has_sink:
        assert sink_a is not None
    if units is None:
        u_arr, n_units = None, B * d.n_q_heads
        out = np.zeros((B, d.n_q_heads, d.head_dim), dtype=np.float64)
    else:
        u_arr = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
        n_units = u_arr.shape[0]
        out = np.zeros((n_units, d.head_dim), dtype=np.float64)
    lib().oracle_attend(ctypes.byref(d), B, _ptr(q_rot, ctypes.c_double),
                        _ptr(sink_a, ctypes.c_float), _ptr(k_cache), _ptr(v_cache),
                        _ptr(v_scale, ctypes.c_float), _ptr(k_scale, ctypes.c_float), cap,
                        _ptr(seq_lens, ctypes.c_int32),
                        _ptr(u_arr, ctypes.c_int32), n_units, _ptr(out, ctypes.c_double),
                        int(n_threads or default_threads()))
    return out


def attend_range(cfg: dict, q_row, k_rows, v_rows, scale_rows, j_lo, j_hi, sink=None, k_scale_rows=None):
    """One query row over keys [j_lo, j_hi) of one kv head's rows. -> (o, natural lse)."""
    d = make_desc(cfg)
    q_row = np.ascontiguousarray(q_row, dtype=np.float64)
    o = np.zeros(d.head_dim, dtype=np.float64)
    lse = ctypes.c_double()
    lib().oracle_attend_range(ctypes.byref(d), _ptr(q_row, ctypes.c_double),
                              _ptr(np.ascontiguousarray(k_rows)),
                              _ptr(np.ascontiguousarray(v_rows)),
                              _ptr(None if scale_rows is None else np.ascontiguousarray(scale_rows),
                                   ctypes.c_float),
                              _ptr(None if k_scale_rows is None else np.ascontiguousarray(k_scale_rows),
                                   ctypes.c_float),
                              int(j_lo), int(j_hi), int(sink is not None),
                              float(sink if sink is not None else 0.0), _ptr(o, ctypes.c_double),
                              ctypes.byref(lse))
    return o, lse.value


def chunk_step(cfg: dict, q, k_new, v_new, q_norm_w, k_norm_w, sink, k_cache, v_cache,
               v_scale, seq_lens, n_threads=None, k_scale=None) -> np.ndarray:
    """T tokens per sequence (q [B][T][Hq][D], k_new / v_new [B][T][Hkv][D]): token t
    takes position seq_len + t and attends every key up to its own and no later one
    (causal within the chunk), so the chunk is T decode steps, taken in order. The
    decoder page's absolute-KV-index position (P1.3) fixes where each token sits.
    Returns out [B][T][Hq][D]; caches and seq_lens mutate (seq_lens += T)."""
    T = q.shape[1]
    outs = []
    for t in range(T):
        outs.append(decode_step(cfg, np.ascontiguousarray(q[:, t]), np.ascontiguousarray(k_new[:, t]),
                                np.ascontiguousarray(v_new[:, t]), q_norm_w, k_norm_w, sink, k_cache, v_cache,
                                v_scale, seq_lens, n_threads, k_scale))
    return np.stack(outs, axis=1)


def decode_step(cfg: dict, q, k_new, v_new, q_norm_w, k_norm_w, sink, k_cache, v_cache,
                v_scale, seq_lens, n_threads=None, k_scale=None) -> np.ndarray:
    """append + attend over the whole batch; caches and seq_lens mutate in place."""
    q_rot = append(cfg, q, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, v_scale, seq_lens, k_scale)
    return attend(cfg, q_rot, sink, k_cache, v_cache, v_scale, seq_lens, None, n_threads, k_scale)
