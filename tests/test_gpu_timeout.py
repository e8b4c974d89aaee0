"""The kernels' bounded pipeline waits, driven to give up.

Every wait in the decode and prefill kernels has a time limit, after which
the CTA sets PA_DEVERR_TIMEOUT, lets the copies and tensor-core work it has
issued finish, frees its tensor memory and exits.  The host's wait-limit hook
set to 0 makes every such wait give up at once, so these tests drive that
abort path with no fault and no hang: each call must return, report the bit,
and the next call on the same (re-initialised) workspace must be correct.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import workloads as W
from _helpers import assert_attention_close, bits, npy

pytestmark = pytest.mark.gpu
DEVERR_TIMEOUT = 0x10


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()
    yield
    api.pa_set_wait_timeout_ns(api.WAIT_TIMEOUT_DEFAULT_NS)


def _expire_every_wait(call):
    """Run `call` with every bounded wait giving up at once."""
    api.pa_set_wait_timeout_ns(0)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        api.pa_set_wait_timeout_ns(api.WAIT_TIMEOUT_DEFAULT_NS)


def test_decode_wait_timeout_reports_and_recovers():
    lens = [3000, 40, 1100]
    st = W.make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=1, size=8192,
                            page_size=16, seed=91, max_ctx=3100, device="cuda")
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, st.k_new, st.v_new, st.loc)
    kb, vb = oracle.kv_store(kb0, vb0, st.layer, bits(st.k_new), bits(st.v_new), npy(st.loc))
    B, Hq, D = st.q.shape
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, Hq, 8, D, 64))
    out = torch.full_like(st.q, float("nan"))

    def call():
        api.pa_paged_decode_attn(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                 st.kv.req_pool_indices, st.kv.seq_lens, st.scale, ws, 64, out)
    _expire_every_wait(call)
    assert api.pa_get_error(ws) & DEVERR_TIMEOUT
    # an aborted call may leave merge counters behind: re-initialise, then
    # the same call is correct
    api.pa_workspace_init(ws)
    call()
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    ref = oracle.decode(bits(st.q), kb, vb, st.layer, npy(st.kv.req_to_token), npy(st.kv.req_pool_indices),
                        npy(st.kv.seq_lens), st.scale)
    assert_attention_close(npy(out.float()), ref, "decode after an aborted call")


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_wait_timeout_reports_and_recovers(fp8):
    new, pre = [300, 77, 1000], [500, 0, 64]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=32, n_kv_heads=8, head_dim=128,
                              size=8192, page_size=16, seed=92, device="cuda")
    kb0, vb0 = bits(pb.kv.k_buf), bits(pb.kv.v_buf)
    kb, vb = oracle.kv_store(kb0, vb0, pb.layer, bits(pb.k_new), bits(pb.v_new), npy(pb.loc))
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes())
    out = torch.full_like(pb.q, float("nan"))
    args = (pb.qo_indptr, pb.kv_indptr, pb.kv.req_to_token, pb.kv.req_pool_indices, pb.scale)
    if fp8:
        n_layers, size, Hkv, D = pb.kv.k_buf.shape
        ks = torch.full((n_layers, Hkv), 4.5 / 448, dtype=torch.float32, device="cuda")
        vs = ks.clone()
        k8 = torch.zeros((n_layers, size, Hkv, D), dtype=torch.uint8, device="cuda")
        v8 = torch.zeros_like(k8)
        every = torch.arange(size, dtype=torch.int32, device="cuda")
        api.pa_kv_store_fp8(k8, v8, pb.layer, pb.kv.k_buf[pb.layer], pb.kv.v_buf[pb.layer], every, ks, vs)
        api.pa_kv_store_fp8(k8, v8, pb.layer, pb.k_new, pb.v_new, pb.loc, ks, vs)
        kh, vh = oracle.kv_store_fp8(np.zeros(k8.shape, np.uint8), np.zeros(v8.shape, np.uint8), pb.layer,
                                     kb[pb.layer], vb[pb.layer], npy(every), npy(ks), npy(vs))

        def call():
            api.pa_paged_prefill_attn_fp8(pb.q, k8, v8, pb.layer, *args, ks, vs, ws, out)
    else:
        api.pa_kv_store(pb.kv.k_buf, pb.kv.v_buf, pb.layer, pb.k_new, pb.v_new, pb.loc)

        def call():
            api.pa_paged_prefill_attn(pb.q, pb.kv.k_buf, pb.kv.v_buf, pb.layer, *args, ws, out)
    _expire_every_wait(call)
    assert api.pa_get_error(ws) & DEVERR_TIMEOUT
    words = ws.view(torch.int32)
    assert int(words[16]) == 0 and int(words[32]) == 0     # the work queue is back at zero
    api.pa_workspace_init(ws)
    call()
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    host = (npy(pb.qo_indptr), npy(pb.kv_indptr), npy(pb.kv.req_to_token), npy(pb.kv.req_pool_indices), pb.scale)
    if fp8:
        ref = oracle.prefill_fp8(bits(pb.q), kh, vh, pb.layer, *host, npy(ks), npy(vs))
    else:
        ref = oracle.prefill(bits(pb.q), kb, vb, pb.layer, *host)
    assert_attention_close(npy(out.float()), ref, f"prefill after an aborted call (fp8={fp8})")
