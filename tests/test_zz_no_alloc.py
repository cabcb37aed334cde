"""uaa_decode_attn_static: the decode step for callers that cannot allocate device
memory themselves (a plugin whose host framework owns every device allocation,
or a serving loop that must not block on the allocator). Its scratch is the
library's built-in array, so the caller passes only inputs and outputs.

It is checked through the C ABI against uaa_decode_attn (caller workspace) on
two calls in a row, within the parity tolerance of the other GPU tests. This
file is collected last so that a stop-at-first-failure run has already run
everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

from gqa_attention_kv_qk_gb300 import binding as B
from gqa_attention_kv_qk_gb300 import workloads as W
from tests.cases import gpu_layer, host_case

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN = 2e-3, 2e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gqa_attention_kv_qk_gb300 import build
    build.build()


@pytest.mark.parametrize("name,over,lens", [
    ("llama31_8b_decode", dict(batch=3, seq_len=700), [699, 300, 5]),
    ("gptoss_vq8_sink", dict(batch=2, seq_len=500), [499, 77]),
    ("llama31_8b_q8", dict(batch=2, seq_len=300), [299, 30]),
    ("llama31_8b_verify", dict(batch=2, seq_len=400, page_size=64), [390, 77]),
])
def test_static_scratch_matches_workspace_entry(name, over, lens):
    cfg = W.config(name, **over)
    case = host_case(cfg, lens=lens)
    with_ws = gpu_layer(case)
    no_alloc = gpu_layer(case)
    stream = torch.cuda.current_stream()
    for step in range(2):  # two calls in a row: the shared scratch keeps the previous contents
        inp = {k: v.cuda() for k, v in W.step_inputs(cfg, step).items()}
        T = with_ws._begin(inp["q"])
        no_alloc._begin(inp["q"])
        B.uaa_decode_attn(with_ws.desc, with_ws.args(inp["q"], inp["k_new"], inp["v_new"]), with_ws.ws, stream)
        B.uaa_decode_attn_static(no_alloc.desc, no_alloc.args(inp["q"], inp["k_new"], inp["v_new"]), stream)
        with_ws.max_len_hint += T
        no_alloc.max_len_hint += T
        torch.cuda.synchronize()
        want = with_ws.out_for(T).double().cpu().numpy()
        got = no_alloc.out_for(T).double().cpu().numpy()
        d = np.abs(got - want)
        assert np.all(np.isfinite(got))
        assert d.max() <= TOL_MAX and d.mean() <= TOL_MEAN, (step, d.max(), d.mean())
        assert torch.equal(with_ws.seq_lens, no_alloc.seq_lens)
        assert torch.equal(with_ws.k_cache, no_alloc.k_cache)
        assert torch.equal(with_ws.v_cache, no_alloc.v_cache)


def test_static_scratch_refuses_steps_beyond_its_size():
    cfg = W.config("llama31_8b_decode", batch=512, n_q_heads=64, n_kv_heads=8)
    desc = B.make_desc(cfg)
    need = B.uaa_workspace_size(desc, 512, 32767, 0)
    assert need > B.UAA_STATIC_SCRATCH_BYTES
    args = B.UaaStepArgs()
    args.batch = 512
    args.max_seq_len = 32767
    args.cache_capacity = 32768
    st = B.uaa_decode_attn_static(desc, args, torch.cuda.current_stream(), check=False)
    assert st == B.UAA_ERR_INVALID_ARGUMENT
    msg = B.last_error()
    assert str(need) in msg and str(B.UAA_STATIC_SCRATCH_BYTES) in msg
