"""Host-side tests of the C ABI: the library loads and exports every entry point
include/uaa.h declares, descriptors outside the supported ranges are refused with
a message naming the fact, and the split geometry is consistent. No call here
reaches a GPU: every refusal returns before the first CUDA call, and the geometry
queries take an explicit SM count."""
import ctypes
import os
import re

import pytest

from gqa_attention_kv_qk_gb300 import binding as B
from gqa_attention_kv_qk_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "uaa.h")


@pytest.fixture(scope="module")
def L():
    from gqa_attention_kv_qk_gb300 import build
    build.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(uaa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_entry_point_is_exported(L):
    names = declared_functions()
    assert "uaa_decode_attn" in names and len(names) >= 12
    for n in names:
        assert hasattr(L, n), f"{n} declared in uaa.h but not exported"
    bound = {s[0] for s in B._SIGS}
    assert bound == set(names), "binding and header disagree"
    assert B.uaa_abi_version() == 11


def good_desc(**kw):
    cfg = W.config("llama31_8b_decode")
    cfg.update(kw)
    return B.make_desc(cfg)


def fake_args(**kw):
    a = B.UaaStepArgs()
    a.batch = 2
    for f in ("q", "k_new", "v_new", "k_cache", "v_cache", "seq_lens", "out", "v_scale", "q_norm_w",
              "k_norm_w", "sink"):
        setattr(a, f, 0x10000)  # aligned, never dereferenced: every case fails before any launch
    a.cache_capacity = 128
    a.max_seq_len = 64
    a.q_rot = None
    for k, v in kw.items():
        setattr(a, k, v)
    return a


WS = B.UaaWorkspace(0x20000, 1 << 30)


@pytest.mark.parametrize("kw,status,fact", [
    (dict(head_dim=96), B.UAA_ERR_UNSUPPORTED, "head_dim=96"),
    (dict(head_dim=32), B.UAA_ERR_UNSUPPORTED, "head_dim=32"),
    (dict(n_q_heads=30), B.UAA_ERR_UNSUPPORTED, "n_q_heads=30"),
    (dict(n_kv_heads=0), B.UAA_ERR_UNSUPPORTED, "n_kv_heads=0"),
    (dict(window=-1), B.UAA_ERR_UNSUPPORTED, "window=-1"),
    (dict(softcap=-2.0), B.UAA_ERR_UNSUPPORTED, "softcap=-2"),
    (dict(rope_theta=0.0), B.UAA_ERR_UNSUPPORTED, "rope.theta=0"),
    (dict(rope_scaling="llama3", factor=0.5), B.UAA_ERR_UNSUPPORTED, "llama3"),
    (dict(rope_scaling="yarn", beta_fast=1.0, beta_slow=32.0), B.UAA_ERR_UNSUPPORTED, "yarn"),
    (dict(rope_scaling="linear", factor=0.0), B.UAA_ERR_UNSUPPORTED, "linear"),
    (dict(rotary_dim=31), B.UAA_ERR_UNSUPPORTED, "rotary_dim=31"),
    (dict(rotary_dim=130), B.UAA_ERR_UNSUPPORTED, "rotary_dim=130"),
    (dict(rotary_dim=-2), B.UAA_ERR_UNSUPPORTED, "rotary_dim=-2"),
])
def test_descriptor_refusals_name_the_fact(L, kw, status, fact):
    st = B.uaa_decode_attn(good_desc(**kw), fake_args(), WS, None, check=False)
    assert st == status
    assert fact in B.last_error()


def test_enum_refusals(L):
    d = good_desc()
    d.kv_dtype = 7
    assert B.uaa_decode_attn(d, fake_args(), WS, None, check=False) == B.UAA_ERR_UNSUPPORTED
    assert "kv_dtype=7" in B.last_error()
    d = good_desc()
    d.norm_offset = 2
    assert B.uaa_decode_attn(d, fake_args(), WS, None, check=False) == B.UAA_ERR_UNSUPPORTED
    assert "norm_offset=2" in B.last_error()
    d = good_desc()
    d.reproducible = 3
    assert B.uaa_decode_attn(d, fake_args(), WS, None, check=False) == B.UAA_ERR_UNSUPPORTED
    assert "reproducible=3" in B.last_error()
    d = good_desc()
    d.rope.scaling = 9
    assert B.uaa_decode_attn(d, fake_args(), WS, None, check=False) == B.UAA_ERR_UNSUPPORTED
    assert "rope.scaling=9" in B.last_error()
    d = good_desc()
    d.rope.style = 3
    assert B.uaa_decode_attn(d, fake_args(), WS, None, check=False) == B.UAA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,status,fact", [
    (dict(q=None), B.UAA_ERR_INVALID_ARGUMENT, "q is NULL"),
    (dict(k_cache=0x10001), B.UAA_ERR_INVALID_ARGUMENT, "k_cache is not 16-byte aligned"),
    (dict(seq_lens=None), B.UAA_ERR_INVALID_ARGUMENT, "seq_lens is NULL"),
    (dict(max_seq_len=128), B.UAA_ERR_CAPACITY, "does not fit cache_capacity=128"),
    (dict(cache_capacity=130), B.UAA_ERR_INVALID_ARGUMENT, "cache_capacity=130"),
    (dict(batch=-1), B.UAA_ERR_INVALID_ARGUMENT, "batch=-1"),
])
def test_argument_refusals(L, kw, status, fact):
    st = B.uaa_decode_attn(good_desc(), fake_args(**kw), WS, None, check=False)
    assert st == status
    assert fact in B.last_error()


@pytest.mark.parametrize("kw,status,fact", [
    (dict(block_table=0x10000, page_size=24, pages_per_seq=8, n_pages=16), B.UAA_ERR_UNSUPPORTED, "page_size=24"),
    (dict(block_table=0x10000, page_size=8, pages_per_seq=16, n_pages=16), B.UAA_ERR_UNSUPPORTED, "page_size=8"),
    (dict(block_table=0x10000, page_size=16, pages_per_seq=3, n_pages=16), B.UAA_ERR_INVALID_ARGUMENT,
     "pages_per_seq=3"),
    (dict(block_table=0x10000, page_size=16, pages_per_seq=8, n_pages=0), B.UAA_ERR_INVALID_ARGUMENT, "n_pages=0"),
    (dict(block_table=0x10008, page_size=16, pages_per_seq=8, n_pages=16), B.UAA_ERR_INVALID_ARGUMENT,
     "block_table is not 16-byte aligned"),
])
def test_paging_refusals(L, kw, status, fact):
    """A paged cache needs a power-of-two page size in [16, 4096] and a capacity of
    whole pages (cache_capacity 128 here)."""
    a = fake_args(cache_capacity=128, max_seq_len=64, **kw)
    assert B.uaa_decode_attn(good_desc(), a, WS, None, check=False) == status
    assert fact in B.last_error()


@pytest.mark.parametrize("kv", ["vq8", "q8"])
def test_int8_caches_refuse_16_key_pages(L, kv):
    a = fake_args(cache_capacity=128, max_seq_len=64, block_table=0x10000, page_size=16, pages_per_seq=8,
                  n_pages=16, k_scale=0x10000)
    assert B.uaa_decode_attn(good_desc(kv_dtype=kv), a, WS, None, check=False) == B.UAA_ERR_UNSUPPORTED
    assert "page_size=16 is below 32" in B.last_error()


def test_sink_flag_without_pointer_is_refused(L):
    st = B.uaa_decode_attn(good_desc(has_sink=True), fake_args(sink=None), WS, None, check=False)
    assert st == B.UAA_ERR_UNSUPPORTED and "sink is NULL while has_sink=1" in B.last_error()
    st = B.uaa_decode_attn(good_desc(qk_norm=True), fake_args(q_norm_w=None), WS, None, check=False)
    assert st == B.UAA_ERR_INVALID_ARGUMENT and "q_norm_w" in B.last_error()


def test_vq8_quantize_refusals(L):
    assert B.uaa_vq8_quantize(0x10000, 0, 4, 96, 0x10000, 0x10000, None, check=False) == B.UAA_ERR_UNSUPPORTED
    assert B.uaa_vq8_quantize(0x10000, 2, 4, 64, 0x10000, 0x10000, None, check=False) == B.UAA_ERR_UNSUPPORTED
    assert B.uaa_vq8_quantize(0x10001, 0, 4, 64, 0x10000, 0x10000, None, check=False) == B.UAA_ERR_INVALID_ARGUMENT
    assert B.uaa_vq8_quantize(0, 0, 0, 64, 0, 0, None, check=False) == B.UAA_OK  # nothing to do


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_workspace_layout_is_consistent(L, name):
    for layer in W.layer_configs(W.config(name)):
        d = B.make_desc(layer)
        batch = layer["batch"]
        longest = W.capacity(layer, extra=layer.get("steps", 1)) - 1
        for n_sm in (1, 20, 152):
            lay = B.uaa_get_workspace_layout(d, batch, longest, n_sm)
            kernel = 0 if layer["kv_dtype"] == "f32" else 1
            per_sm = 4 if kernel == 0 else (1 if layer["head_dim"] == 256 else 2)
            assert lay.kernel == kernel and lay.n_ctas == n_sm * per_sm
            d64 = kernel == 1 and layer["head_dim"] == 64
            int8 = layer["kv_dtype"] in ("vq8", "q8")
            want = (256 if int8 else 128) if d64 else (128 if layer["kv_dtype"] == "q8" else 64)
            assert lay.stage_keys == want
            assert lay.n_slices == -(-batch // lay.slice_batch) and lay.slice_batch <= 1024
            Hq, D, HC, P = layer["n_q_heads"], layer["head_dim"], lay.heads_per_cta, lay.n_ctas
            assert lay.prefix_offset >= lay.q_rot_offset + batch * Hq * D * 4
            assert lay.prefix_stride >= (lay.slice_batch + 1) * 4
            assert lay.rec_lse_offset >= lay.prefix_offset + lay.n_slices * lay.prefix_stride
            assert lay.rec_lse_stride >= 2 * P * HC * 4
            assert lay.rec_o_offset >= lay.rec_lse_offset + lay.n_slices * lay.rec_lse_stride
            assert lay.rec_o_stride >= 2 * P * HC * D * 4
            assert lay.balance_offset == 256  # fixed: the learned range weights survive a batch change
            assert lay.q_rot_offset >= lay.balance_offset + 256 + 8 * P + 4 * (3 * P + 1)
            assert lay.ranges_offset >= lay.rec_o_offset + lay.n_slices * lay.rec_o_stride
            assert lay.ranges_stride >= (P + 1) * 8
            assert lay.owners_offset >= lay.ranges_offset + lay.n_slices * lay.ranges_stride
            units = layer["n_kv_heads"] * -(-(Hq // layer["n_kv_heads"]) // HC)
            assert lay.owners_stride >= lay.slice_batch * units * 8
            assert lay.total_bytes >= lay.owners_offset + lay.n_slices * lay.owners_stride
            assert B.uaa_workspace_size(d, batch, longest, n_sm) == lay.total_bytes
            assert B.uaa_num_splits(d, batch, longest, n_sm) == P
            for off in (lay.q_rot_offset, lay.prefix_offset, lay.rec_lse_offset, lay.rec_o_offset,
                        lay.ranges_offset, lay.owners_offset, lay.balance_offset):
                assert off % 256 == 0


def test_large_batches_are_sliced(L):
    d = B.make_desc(W.config("llama31_8b_decode"))
    lay = B.uaa_get_workspace_layout(d, 2500, 100, 152)
    assert (lay.slice_batch, lay.n_slices) == (1024, 3)


def test_large_chunked_batches_are_sliced(L):
    """Slices with several tokens per sequence: the same 1024-sequence slices, and
    the q' region holds every slice's q_len rows per sequence (slice s starts
    1024 q_len Hq rows in)."""
    cfg = W.config("llama31_8b_decode")
    d = B.make_desc(cfg)
    for T in (2, 4):
        lay = B.uaa_get_workspace_layout(d, 2500, 100, 152, q_len=T)
        assert (lay.slice_batch, lay.n_slices) == (1024, 3)
        assert lay.prefix_offset - lay.q_rot_offset >= 2500 * T * cfg["n_q_heads"] * cfg["head_dim"] * 4


@pytest.mark.parametrize("name,kv", [("llama31_8b_decode", "bf16"), ("gptoss_vq8_sink", "vq8"),
                                     ("llama31_8b_decode", "q8"), ("gemma2_9b_swa", "bf16"),
                                     ("llama32_1b_tiny", "f32")])
def test_chunk_geometry(L, name, kv):
    """Steps of q_len tokens: a unit's rows are the q_len G (token, head) pairs of
    a kv head, 8 or 16 to a unit (8 at head_dim 256 and on the CUDA-core kernel);
    two 8-row tiles run one CTA per SM; the q' region holds q_len rows per
    sequence; a workspace sized for q_len serves every smaller q_len."""
    cfg = W.layer_configs(W.config(name, kv_dtype=kv, io_dtype="f32" if kv == "f32" else "bf16"))[0]
    d = B.make_desc(cfg)
    G = cfg["n_q_heads"] // cfg["n_kv_heads"]
    sizes = []
    for T in (1, 2, 4, 16, 64):
        lay = B.uaa_get_workspace_layout(d, 8, 1000, 152, q_len=T)
        rows = T * G
        # 128 rows or more per kv head on a bf16 cache at head_dim 64 / 128: the
        # query-tiled prefill kernel (append + prefill, no combine; a paged cache of
        # the same geometry takes the partial kernel, whose geometry is still reported)
        prefill = kv == "bf16" and cfg["head_dim"] in (64, 128) and rows >= 128
        assert lay.kernel == (2 if prefill else (0 if kv == "f32" else 1))
        assert lay.step_kernels == (2 if prefill or (kv != "f32" and T == 1) else (1 if lay.step_splits else 3))
        tc = lay.kernel in (1, 2)
        wide = tc and cfg["head_dim"] != 256 and rows > 8
        assert lay.heads_per_cta == (16 if wide else 8)
        if tc:  # keys per ring stage: two 16-key groups per warp where keys are cheap or rows many
            D = cfg["head_dim"]
            want = (256 if kv in ("vq8", "q8") else 128) if D == 64 else (128 if kv == "q8" or (wide and D == 128)
                                                                         else 64)
            assert lay.stage_keys == want, (T, lay.stage_keys, want)
        assert lay.n_ctas == 152 * (4 if lay.kernel == 0 else (1 if cfg["head_dim"] == 256 or wide else 2))
        assert lay.prefix_offset - lay.q_rot_offset >= 8 * T * cfg["n_q_heads"] * cfg["head_dim"] * 4
        sizes.append(B.uaa_workspace_size(d, 8, 1000, 152, q_len=T))
        assert sizes[-1] == lay.total_bytes
    assert B.uaa_workspace_size(d, 8, 1000, 152, q_len=2000) == 0  # beyond the largest chunk
    # a larger chunk never needs less workspace, so one sized for q_len serves the smaller ones
    assert sizes == sorted(sizes)


def test_chunk_capacity_refusal(L):
    a = fake_args(cache_capacity=128, max_seq_len=120, q_len=16)
    assert B.uaa_decode_attn(good_desc(), a, WS, None, check=False) == B.UAA_ERR_CAPACITY
    assert "16 new token(s) does not fit cache_capacity=128" in B.last_error()


def test_geometry_query_refuses_bad_desc(L):
    assert B.uaa_workspace_size(good_desc(head_dim=48), 4, 100, 152) == 0
    assert B.uaa_num_splits(good_desc(n_q_heads=9), 4, 100, 152) == 0
    assert "n_q_heads=9" in B.last_error()


def test_status_strings(L):
    for s, name in ((0, "UAA_OK"), (1, "UAA_ERR_INVALID_ARGUMENT"), (2, "UAA_ERR_UNSUPPORTED"),
                    (3, "UAA_ERR_CAPACITY"), (4, "UAA_ERR_CUDA"), (5, "UAA_ERR_DEVICE")):
        assert B.status_string(s) == name


def test_struct_sizes_match_the_header(L, tmp_path):
    """Compile a probe against include/uaa.h and compare sizeof/offsetof with ctypes."""
    import subprocess
    src = tmp_path / "probe.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "uaa.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(uaa_attn_desc), sizeof(uaa_step_args),'
        ' sizeof(uaa_workspace), sizeof(uaa_workspace_layout), offsetof(uaa_attn_desc, out_dtype),'
        ' offsetof(uaa_attn_desc, norm_offset),'
        ' offsetof(uaa_step_args, q_rot), offsetof(uaa_workspace_layout, total_bytes));'
        ' printf("%zu\\n", offsetof(uaa_attn_desc, reproducible)); return 0;}\n')
    exe = tmp_path / "probe"
    r = subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include", str(src),
                        "-o", str(exe)], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("no C compiler / CUDA headers for the probe: " + r.stderr[:200])
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    want = [ctypes.sizeof(B.UaaAttnDesc), ctypes.sizeof(B.UaaStepArgs), ctypes.sizeof(B.UaaWorkspace),
            ctypes.sizeof(B.UaaWorkspaceLayout), B.UaaAttnDesc.out_dtype.offset, B.UaaAttnDesc.norm_offset.offset,
            B.UaaStepArgs.q_rot.offset,
            B.UaaWorkspaceLayout.total_bytes.offset, B.UaaAttnDesc.reproducible.offset]
    assert got == want
