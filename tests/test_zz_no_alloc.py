"""The allocation-free decode entry point against the workspace one.

pa_paged_decode_attn_noalloc exists for callers that cannot allocate device
memory where decode runs -- for example a plugin whose host program owns every
device allocation, or a serving loop that must never call cudaMalloc because
it synchronises the device.  Instead of a caller workspace it uses a fixed
scratch array inside the library, shared by every call on the device.

This file is collected last so that a stop-at-first-failure run has already
run everything else; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import workloads as W
from _helpers import assert_attention_close, npy

pytestmark = pytest.mark.gpu
MAX_SPLITS = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


def _step(seed, lens):
    st = W.make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=2, size=32768,
                            page_size=16, seed=seed, layer=1, max_ctx=4096, device="cuda")
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, st.k_new, st.v_new, st.loc)
    return st


def test_noalloc_matches_workspace_entry_point_twice():
    # Two calls in a row with different batches and lengths: the second call
    # must not see the first call's partials or merge tickets.  The first
    # batch has requests long enough to be split, so the merge path runs.
    for seed, lens in ((11, [4000, 17, 900]), (12, [1, 2500, 64, 3000, 5, 1024])):
        st = _step(seed, lens)
        B, Hq, D = st.q.shape
        ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, Hq, 8, D, MAX_SPLITS))
        ref = torch.full_like(st.q, float("nan"))
        api.pa_paged_decode_attn(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                 st.kv.req_pool_indices, st.kv.seq_lens, st.scale, ws, MAX_SPLITS, ref)
        got = torch.full_like(st.q, float("nan"))
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        api.pa_paged_decode_attn_noalloc(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                         st.kv.req_pool_indices, st.kv.seq_lens, st.scale, MAX_SPLITS, got,
                                         error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert api.pa_get_error(ws) == 0
        assert_attention_close(npy(got.float()), npy(ref.float()).astype(np.float64),
                               f"no-alloc decode vs workspace decode, seed {seed}")


def test_noalloc_rejects_batches_beyond_its_array():
    st = _step(13, [64] * 20)   # 20 requests x 64 splits x 32 heads x 130 floats > 16 MiB
    out = torch.empty_like(st.q)
    with pytest.raises(api.PaError) as e:
        api.pa_paged_decode_attn_noalloc(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                         st.kv.req_pool_indices, st.kv.seq_lens, st.scale, MAX_SPLITS, out)
    assert e.value.status == 5   # PA_ERR_WORKSPACE
