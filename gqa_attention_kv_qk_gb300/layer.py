"""DecodeLayer: one attention layer's KV cache and workspace on a CUDA device.

PyTorch allocates the device memory and supplies the stream; every step of the
method runs in libuaa through the C ABI (binding.py). This is the call a user
makes: build the layer, load or grow its cache, then `step(q, k_new, v_new)`.
"""
from __future__ import annotations

import torch

from . import binding as B
from . import workloads as W

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _require_cuda(device):
    if not torch.cuda.is_available():
        raise RuntimeError("DecodeLayer needs a CUDA device; libuaa has no CPU implementation")
    return torch.device(device)


class DecodeLayer:
    """page_size: store the caches as pools of pages of that many positions;
    block_table ([batch][capacity / page_size] int32, default: sequence b takes
    pages b P .. b P + P - 1) maps each sequence's logical pages to pool pages, of
    which there are n_pages (default: just enough). max_q_len: the most tokens per
    sequence one step takes (q, k_new, v_new of shape [B][T][H][D]); the
    workspace is sized for it."""

    def __init__(self, cfg: dict, batch: int, capacity: int, device="cuda", page_size=None, block_table=None,
                 n_pages=None, max_q_len=1):
        self.cfg = dict(cfg)
        self.device = _require_cuda(device)
        self.batch = int(batch)
        self.capacity = int(capacity)
        self.desc = B.make_desc(cfg)
        Hq, Hkv, D = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
        kv = cfg.get("kv_dtype", "bf16")
        dev = self.device
        self.page_size = int(page_size or 0)
        if self.page_size:
            if capacity % self.page_size:
                raise ValueError(f"capacity {capacity} is not a multiple of page_size {self.page_size}")
            self.pages_per_seq = capacity // self.page_size
            if block_table is None:
                block_table = torch.arange(batch * self.pages_per_seq, dtype=torch.int32).reshape(batch, -1)
            self.block_table = torch.as_tensor(block_table, dtype=torch.int32).to(dev).contiguous()
            assert self.block_table.shape == (batch, self.pages_per_seq)
            self.n_pages = int(n_pages or batch * self.pages_per_seq)
            rows = (self.n_pages, Hkv, self.page_size)  # pools of pages
        else:
            self.pages_per_seq = self.n_pages = 0
            self.block_table = None
            rows = (batch, Hkv, capacity)
        kdt = torch.float32 if kv == "f32" else torch.bfloat16
        if kv == "q8":
            self.k_cache = torch.zeros((*rows, D), dtype=torch.int8, device=dev)
            self.k_scale = torch.zeros(rows, dtype=torch.float32, device=dev)
        else:
            self.k_cache = torch.zeros((*rows, D), dtype=kdt, device=dev)
            self.k_scale = None
        if kv in ("vq8", "q8"):
            self.v_cache = torch.zeros((*rows, D), dtype=torch.int8, device=dev)
            self.v_scale = torch.zeros(rows, dtype=torch.float32, device=dev)
        else:
            self.v_cache = torch.zeros((*rows, D), dtype=kdt, device=dev)
            self.v_scale = None
        self.seq_lens = torch.zeros((batch,), dtype=torch.int32, device=dev)
        self.max_len_hint = 0
        self.out = torch.empty((batch, Hq, D), dtype=_TORCH_DTYPE[cfg.get("out_dtype", "f32")], device=dev)
        self._outs = {1: self.out}  # per tokens-per-step count: [B][Hq][D], or [B][T][Hq][D]
        self.q_len = 1              # tokens per sequence of the current step
        self.max_q_len = int(max_q_len)
        self.q_norm_w = self.k_norm_w = self.sink = None
        # workspace sized for the longest allowed sequence; zeroed once (status word)
        nbytes = B.uaa_workspace_size(self.desc, batch, capacity - 1, 0, self.max_q_len)
        if nbytes == 0:
            raise B.UaaError(B.UAA_ERR_UNSUPPORTED, B.last_error())
        self.ws_tensor = torch.zeros((nbytes,), dtype=torch.uint8, device=dev)
        self.ws = B.UaaWorkspace(self.ws_tensor.data_ptr(), nbytes)

    @classmethod
    def for_case(cls, case: dict, device="cuda") -> "DecodeLayer":
        """A layer holding a host case of workloads.host_case (a vq8 / q8 cache is
        quantised on the device); a paged workload gets a pool with spare pages,
        assigned in seeded random order."""
        cfg = case["cfg"]
        ps = int(cfg.get("page_size", 0) or 0)
        T = int(cfg.get("q_len", 1) or 1)
        if ps:
            P = case["cap"] // ps
            n_pages = cfg["batch"] * P + max(2, cfg["batch"])
            layer = cls(cfg, cfg["batch"], case["cap"], device, page_size=ps,
                        block_table=W.block_table(cfg, P, n_pages), n_pages=n_pages, max_q_len=T)
        else:
            layer = cls(cfg, cfg["batch"], case["cap"], device, max_q_len=T)
        k = case["k_values"] if cfg.get("kv_dtype") == "q8" else case["k_cache"]
        v = case["v_values"] if cfg.get("kv_dtype") in ("vq8", "q8") else case["v_cache"]
        layer.load_cache(k, v, case["lens"])
        layer.set_params(case["q_norm_w"], case["k_norm_w"], case["sink"])
        return layer

    # ------------------------------------------------------------ state
    def set_params(self, q_norm_w=None, k_norm_w=None, sink=None):
        to = lambda t: None if t is None else t.to(device=self.device, dtype=torch.float32).contiguous()
        self.q_norm_w, self.k_norm_w, self.sink = to(q_norm_w), to(k_norm_w), to(sink)

    def _to_pool(self, logical, pool):
        """Logical rows [B][Hkv][cap][...] into a pool [n_pages][Hkv][page_size][...]."""
        Bn, Hkv, ps, P = self.batch, logical.shape[1], self.page_size, self.pages_per_seq
        rest = tuple(logical.shape[3:])
        x = logical.reshape(Bn, Hkv, P, ps, *rest).transpose(1, 2).reshape(Bn * P, Hkv, ps, *rest)
        pool.index_copy_(0, self.block_table.reshape(-1).long(), x.to(device=pool.device, dtype=pool.dtype))

    def logical(self, name: str):
        """A cache tensor ("k_cache", "v_cache", "k_scale", "v_scale") as logical
        rows [B][Hkv][cap][...] (a gathered copy for a paged layer)."""
        t = getattr(self, name)
        if t is None or not self.page_size:
            return t
        Bn, P, ps = self.batch, self.pages_per_seq, self.page_size
        x = t.index_select(0, self.block_table.reshape(-1).long())
        Hkv, rest = x.shape[1], tuple(x.shape[3:])
        return x.reshape(Bn, P, Hkv, ps, *rest).transpose(1, 2).reshape(Bn, Hkv, P * ps, *rest)

    def load_cache(self, k, v, lens):
        """Copy host caches (logical rows [B][Hkv][cap][D]) in. For a vq8 layer `v`
        holds fp32 values, and for a q8 layer `k` too, quantised on the device by
        uaa_vq8_quantize (the append's own rule)."""
        D = self.cfg["head_dim"]
        s = torch.cuda.current_stream(self.device)

        def put(vals, cache, scales):
            if scales is not None:  # codes and scales of the logical rows, then into place
                vals = vals.to(device=self.device, dtype=torch.float32).contiguous()
                codes = torch.empty(vals.shape, dtype=torch.int8, device=self.device)
                sc = torch.empty(vals.shape[:-1], dtype=torch.float32, device=self.device)
                B.uaa_vq8_quantize(vals.data_ptr(), B.DTYPE["f32"], vals.numel() // D, D, codes.data_ptr(),
                                   sc.data_ptr(), s)
                pairs = ((codes, cache), (sc, scales))
            else:
                pairs = ((vals, cache),)
            for src, dst in pairs:
                if self.page_size:
                    self._to_pool(src.to(self.device), dst)
                else:
                    dst.copy_(src)

        put(k, self.k_cache, self.k_scale)
        put(v, self.v_cache, self.v_scale)
        lens = torch.as_tensor(lens, dtype=torch.int32)
        self.seq_lens.copy_(lens)
        self.max_len_hint = int(lens.max()) if lens.numel() else 0

    def set_lengths(self, lens):
        lens = torch.as_tensor(lens, dtype=torch.int32)
        self.seq_lens.copy_(lens)
        self.max_len_hint = int(lens.max()) if lens.numel() else 0

    # ------------------------------------------------------------ calls
    def out_for(self, q_len: int):
        """The layer's output rows for steps of q_len tokens per sequence."""
        o = self._outs.get(q_len)
        if o is None:
            o = self._outs[q_len] = torch.empty((self.batch, q_len, *self.out.shape[1:]), dtype=self.out.dtype,
                                                device=self.device)
        return o

    def _begin(self, q):
        """Tokens per sequence of a step's q ([B][Hq][D] or [B][T][Hq][D])."""
        T = int(q.shape[1]) if q.dim() == 4 else 1
        if T > self.max_q_len:
            raise ValueError(f"{T} tokens per sequence, the layer was built for max_q_len={self.max_q_len}")
        self.q_len = T
        return T

    def args(self, q, k_new, v_new, max_seq_len=None, q_rot=None, out=None) -> B.UaaStepArgs:
        """The step's argument struct (a copy of one built once per distinct set of pointers)."""
        msl = self.max_len_hint if max_seq_len is None else int(max_seq_len)
        if out is None:
            out = self.out_for(self.q_len)
        key = (B.ptr(q), B.ptr(k_new), B.ptr(v_new), msl, B.ptr(q_rot), B.ptr(out), self.q_len)
        cache = self.__dict__.setdefault("_args_cache", {})
        a = cache.get(key)
        if a is None:
            if len(cache) > 64:
                cache.clear()
            a = cache[key] = self._build_args(q, k_new, v_new, msl, q_rot, out)
        return B.UaaStepArgs.from_buffer_copy(a)  # a copy: callers may change fields

    def _build_args(self, q, k_new, v_new, max_seq_len, q_rot, out) -> B.UaaStepArgs:
        a = B.UaaStepArgs()
        a.batch = self.batch
        a.q, a.k_new, a.v_new = B.ptr(q), B.ptr(k_new), B.ptr(v_new)
        a.q_norm_w, a.k_norm_w, a.sink = B.ptr(self.q_norm_w), B.ptr(self.k_norm_w), B.ptr(self.sink)
        a.k_cache, a.v_cache, a.v_scale = B.ptr(self.k_cache), B.ptr(self.v_cache), B.ptr(self.v_scale)
        a.cache_capacity = self.capacity
        a.seq_lens = B.ptr(self.seq_lens)
        a.max_seq_len = max_seq_len
        a.out = B.ptr(self.out if out is None else out)
        a.q_rot = B.ptr(q_rot)
        a.k_scale = B.ptr(self.k_scale)
        a.q_len = self.q_len
        if self.page_size:
            a.block_table = B.ptr(self.block_table)
            a.page_size, a.pages_per_seq, a.n_pages = self.page_size, self.pages_per_seq, self.n_pages
        return a

    def step(self, q, k_new, v_new, stream=None, max_seq_len=None, advance_hint=True, q_rot=None, out=None):
        """One step (append, split-K partials, combine) on `stream` for q of one token
        per sequence ([B][Hq][D]) or T tokens ([B][T][Hq][D], causal within the
        chunk); the output rows ([B][Hq][D] or [B][T][Hq][D]) go to `out` if given."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        T = self._begin(q)
        want = self.out_for(T)
        if out is not None:
            assert out.shape == want.shape and out.dtype == want.dtype and out.is_contiguous()
        B.uaa_decode_attn(self.desc, self.args(q, k_new, v_new, max_seq_len, q_rot=q_rot, out=out), self.ws, s)
        if advance_hint and max_seq_len is None:
            self.max_len_hint += T
        return want if out is None else out

    def append(self, q, k_new, v_new, stream=None, q_rot=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        self._begin(q)
        B.uaa_rope_qk_norm_append(self.desc, self.args(q, k_new, v_new, q_rot=q_rot), self.ws, s)

    def append_partial(self, q, k_new, v_new, stream=None, q_rot=None):
        """Steps 1 and 2 (one fused kernel for bf16 / vq8 / q8 caches and one token);
        follow with combine()."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        self._begin(q)
        B.uaa_decode_attn_append_partial(self.desc, self.args(q, k_new, v_new, q_rot=q_rot), self.ws, s)

    def partial(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        B.uaa_decode_attn_partial(self.desc, self.args(None, None, None), self.ws, s)

    def combine(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        B.uaa_decode_attn_combine(self.desc, self.args(None, None, None), self.ws, s)
        self.max_len_hint += self.q_len
        return self.out_for(self.q_len)

    def layout(self, max_seq_len=None) -> B.UaaWorkspaceLayout:
        return B.uaa_get_workspace_layout(self.desc, self.batch,
                                          self.max_len_hint if max_seq_len is None else max_seq_len, 0, self.q_len)

    def device_status(self, stream=None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return B.uaa_device_status(self.ws, s)
