"""ctypes binding of libuaa (include/uaa.h): the same names, argument marshalling only.

Every computation runs in the CUDA library. If libuaa.so has not been built,
loading fails with an error that says so; there is no other implementation to
fall back to.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libuaa.so")

UAA_OK = 0
UAA_ERR_INVALID_ARGUMENT = 1
UAA_ERR_UNSUPPORTED = 2
UAA_ERR_CAPACITY = 3
UAA_ERR_CUDA = 4
UAA_ERR_DEVICE = 5

UAA_DEVFLAG_CAPACITY = 0x1
UAA_DEVFLAG_LEN_HINT = 0x2
UAA_DEVFLAG_TIMEOUT = 0x4
UAA_DEVFLAG_PAGE = 0x8

ROPE_STYLE = {"neox": 0, "interleaved": 1}
ROPE_SCALING = {"none": 0, "llama3": 1, "yarn": 2, "linear": 3}
DTYPE = {"f32": 0, "bf16": 1, "vq8": 2, "q8": 3}


class UaaRopeParams(ctypes.Structure):
    _fields_ = [("style", ctypes.c_int32), ("theta", ctypes.c_double), ("scaling", ctypes.c_int32),
                ("factor", ctypes.c_double), ("low_freq_factor", ctypes.c_double),
                ("high_freq_factor", ctypes.c_double), ("original_max_pos", ctypes.c_int32),
                ("beta_fast", ctypes.c_double), ("beta_slow", ctypes.c_double),
                ("attn_factor", ctypes.c_double)]


class UaaAttnDesc(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("scale", ctypes.c_float), ("rope", UaaRopeParams),
                ("qk_norm", ctypes.c_int32), ("norm_eps", ctypes.c_float), ("window", ctypes.c_int32),
                ("softcap", ctypes.c_float), ("has_sink", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("rotary_dim", ctypes.c_int32),
                ("norm_offset", ctypes.c_int32), ("reproducible", ctypes.c_int32)]


class UaaStepArgs(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("q_norm_w", ctypes.c_void_p),
                ("k_norm_w", ctypes.c_void_p), ("sink", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("cache_capacity", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("max_seq_len", ctypes.c_int32),
                ("out", ctypes.c_void_p), ("q_rot", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("page_size", ctypes.c_int32),
                ("pages_per_seq", ctypes.c_int32), ("n_pages", ctypes.c_int32), ("q_len", ctypes.c_int32)]


class UaaWorkspace(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class UaaWorkspaceLayout(ctypes.Structure):
    _fields_ = [("n_ctas", ctypes.c_int32), ("stage_keys", ctypes.c_int32),
                ("heads_per_cta", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("n_slices", ctypes.c_int32), ("slice_batch", ctypes.c_int32),
                ("step_kernels", ctypes.c_int32), ("step_splits", ctypes.c_int32),
                ("status_offset", ctypes.c_size_t), ("q_rot_offset", ctypes.c_size_t),
                ("prefix_offset", ctypes.c_size_t), ("rec_lse_offset", ctypes.c_size_t),
                ("rec_o_offset", ctypes.c_size_t), ("prefix_stride", ctypes.c_size_t),
                ("rec_lse_stride", ctypes.c_size_t), ("rec_o_stride", ctypes.c_size_t),
                ("ranges_offset", ctypes.c_size_t), ("ranges_stride", ctypes.c_size_t),
                ("owners_offset", ctypes.c_size_t), ("owners_stride", ctypes.c_size_t),
                ("balance_offset", ctypes.c_size_t), ("total_bytes", ctypes.c_size_t)]


class UaaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status
        self.message = message


_lib = None

# (name, restype, argtypes) for every entry point include/uaa.h declares.
_P = ctypes.POINTER
_SIGS = [
    ("uaa_rope_qk_norm_append", ctypes.c_int, [_P(UaaAttnDesc), _P(UaaStepArgs), _P(UaaWorkspace), ctypes.c_void_p]),
    ("uaa_decode_attn_partial", ctypes.c_int, [_P(UaaAttnDesc), _P(UaaStepArgs), _P(UaaWorkspace), ctypes.c_void_p]),
    ("uaa_decode_attn_combine", ctypes.c_int, [_P(UaaAttnDesc), _P(UaaStepArgs), _P(UaaWorkspace), ctypes.c_void_p]),
    ("uaa_decode_attn_append_partial", ctypes.c_int,
     [_P(UaaAttnDesc), _P(UaaStepArgs), _P(UaaWorkspace), ctypes.c_void_p]),
    ("uaa_decode_attn", ctypes.c_int, [_P(UaaAttnDesc), _P(UaaStepArgs), _P(UaaWorkspace), ctypes.c_void_p]),
    ("uaa_workspace_size", ctypes.c_size_t,
     [_P(UaaAttnDesc), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    ("uaa_num_splits", ctypes.c_int32, [_P(UaaAttnDesc), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    ("uaa_get_workspace_layout", ctypes.c_int,
     [_P(UaaAttnDesc), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P(UaaWorkspaceLayout)]),
    ("uaa_vq8_quantize", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
      ctypes.c_void_p]),
    ("uaa_device_status", ctypes.c_int, [_P(UaaWorkspace), ctypes.c_void_p, _P(ctypes.c_uint32)]),
    ("uaa_last_error", ctypes.c_char_p, []),
    ("uaa_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("uaa_abi_version", ctypes.c_int32, []),
    ("uaa_decode_attn_static", ctypes.c_int, [_P(UaaAttnDesc), _P(UaaStepArgs), ctypes.c_void_p]),
]


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libuaa.so is not built ({_LIB_PATH}); run "
                              "`python -m gqa_attention_kv_qk_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(_LIB_PATH)
        for name, res, args in _SIGS:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().uaa_status_string(int(status)).decode()
    except ImportError:
        return f"status {status}"


def last_error() -> str:
    return lib().uaa_last_error().decode()


def _check(status: int, check: bool) -> int:
    if check and status != UAA_OK:
        raise UaaError(status, last_error())
    return status


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        return ctypes.c_void_p(0)
    if hasattr(stream, "cuda_stream"):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ---------------------------------------------------------------- the entry points

def uaa_rope_qk_norm_append(desc, args, ws, stream=None, check=True) -> int:
    return _check(lib().uaa_rope_qk_norm_append(ctypes.byref(desc), ctypes.byref(args), ctypes.byref(ws),
                                                _stream(stream)), check)


def uaa_decode_attn_partial(desc, args, ws, stream=None, check=True) -> int:
    return _check(lib().uaa_decode_attn_partial(ctypes.byref(desc), ctypes.byref(args), ctypes.byref(ws),
                                                _stream(stream)), check)


def uaa_decode_attn_combine(desc, args, ws, stream=None, check=True) -> int:
    return _check(lib().uaa_decode_attn_combine(ctypes.byref(desc), ctypes.byref(args), ctypes.byref(ws),
                                                _stream(stream)), check)


def uaa_decode_attn_append_partial(desc, args, ws, stream=None, check=True) -> int:
    return _check(lib().uaa_decode_attn_append_partial(ctypes.byref(desc), ctypes.byref(args), ctypes.byref(ws),
                                                       _stream(stream)), check)


def uaa_decode_attn(desc, args, ws, stream=None, check=True) -> int:
    return _check(lib().uaa_decode_attn(ctypes.byref(desc), ctypes.byref(args), ctypes.byref(ws),
                                        _stream(stream)), check)


def uaa_workspace_size(desc, batch: int, max_seq_len: int, n_sm: int = 0, q_len: int = 1) -> int:
    return int(lib().uaa_workspace_size(ctypes.byref(desc), batch, max_seq_len, n_sm, q_len))


def uaa_num_splits(desc, batch: int, max_seq_len: int, n_sm: int = 0, q_len: int = 1) -> int:
    return int(lib().uaa_num_splits(ctypes.byref(desc), batch, max_seq_len, n_sm, q_len))


def uaa_get_workspace_layout(desc, batch: int, max_seq_len: int, n_sm: int = 0, q_len: int = 1) -> UaaWorkspaceLayout:
    out = UaaWorkspaceLayout()
    _check(lib().uaa_get_workspace_layout(ctypes.byref(desc), batch, max_seq_len, n_sm, q_len,
                                          ctypes.byref(out)), True)
    return out


def uaa_vq8_quantize(v_ptr: int, v_dtype: int, n_rows: int, head_dim: int, codes_ptr: int, scales_ptr: int,
                     stream=None, check=True) -> int:
    return _check(lib().uaa_vq8_quantize(ctypes.c_void_p(v_ptr), v_dtype, n_rows, head_dim,
                                         ctypes.c_void_p(codes_ptr), ctypes.c_void_p(scales_ptr),
                                         _stream(stream)), check)


def uaa_device_status(ws, stream=None) -> int:
    """Device flags (UAA_DEVFLAG_*) of the workspace; clears them."""
    f = ctypes.c_uint32(0)
    st = lib().uaa_device_status(ctypes.byref(ws), _stream(stream), ctypes.byref(f))
    if st not in (UAA_OK, UAA_ERR_DEVICE):
        raise UaaError(st, last_error())
    return int(f.value)


def uaa_abi_version() -> int:
    return int(lib().uaa_abi_version())


UAA_STATIC_SCRATCH_BYTES = 8 << 20


def uaa_decode_attn_static(desc, args, stream=None, check=True) -> int:
    """uaa_decode_attn for callers that cannot allocate device memory: the scratch
    is the library's built-in UAA_STATIC_SCRATCH_BYTES array (see include/uaa.h)."""
    return _check(lib().uaa_decode_attn_static(ctypes.byref(desc), ctypes.byref(args), _stream(stream)), check)


# ---------------------------------------------------------------- marshalling helpers

def make_desc(cfg: dict) -> UaaAttnDesc:
    """Descriptor from a workload dict (the vocabulary of workloads.CONFIGS)."""
    d = UaaAttnDesc()
    d.n_q_heads = int(cfg["n_q_heads"])
    d.n_kv_heads = int(cfg["n_kv_heads"])
    d.head_dim = int(cfg["head_dim"])
    d.scale = float(cfg.get("scale", 0.0) or 0.0)
    r = d.rope
    r.style = ROPE_STYLE[cfg.get("rope_style", "neox")]
    r.theta = float(cfg.get("rope_theta", 10000.0))
    r.scaling = ROPE_SCALING[cfg.get("rope_scaling", "none")]
    r.factor = float(cfg.get("factor", 1.0))
    r.low_freq_factor = float(cfg.get("low_freq_factor", 1.0))
    r.high_freq_factor = float(cfg.get("high_freq_factor", 4.0))
    r.original_max_pos = int(cfg.get("original_max_pos", 8192))
    r.beta_fast = float(cfg.get("beta_fast", 32.0))
    r.beta_slow = float(cfg.get("beta_slow", 1.0))
    r.attn_factor = float(cfg.get("attn_factor", 0.0) or 0.0)
    d.qk_norm = int(bool(cfg.get("qk_norm", False)))
    d.norm_eps = float(cfg.get("norm_eps", 1e-6))
    d.window = int(cfg.get("window", 0) or 0)
    d.softcap = float(cfg.get("softcap", 0.0) or 0.0)
    d.has_sink = int(bool(cfg.get("has_sink", False)))
    d.kv_dtype = DTYPE[cfg.get("kv_dtype", "bf16")]
    d.io_dtype = DTYPE[cfg.get("io_dtype", "bf16")]
    d.out_dtype = DTYPE[cfg.get("out_dtype", "f32")]
    d.rotary_dim = int(cfg.get("rotary_dim", 0) or 0)
    d.norm_offset = int(bool(cfg.get("norm_offset", False)))
    d.reproducible = int(bool(cfg.get("reproducible", False)))
    return d


def ptr(t) -> int:
    """Device address of a tensor (0 for None)."""
    return 0 if t is None else int(t.data_ptr())
