"""dattn_decode_noalloc: the fused decode with the library's fixed scratch array.

Some callers cannot allocate device memory: a plugin or custom op given only its input and
output pointers, code under a framework allocator that owns all device memory, or a
latency-critical path that cannot risk cudaMalloc's implicit synchronisation. For them the
library keeps its decode scratch in a static 8 MiB device array. This test checks that two
calls in a row through that entry point match the workspace-based dattn_decode, and the
oracle's full softmax attention, within the parity tolerance used everywhere else. Between
the calls the query changes, and the shared scratch must not carry state from one call to
the next: a stale merge counter would leave heads unmerged and fail the oracle check. It runs alone in a fresh process
as well as after the rest of the suite, which is why pytest collects it last.
"""
import ctypes

import pytest
import torch

from _util import assert_out_close, check_dense

pytestmark = pytest.mark.gpu


def _lib():
    import split_kv_decode_distattention_gb300 as dattn
    dattn.load_library()
    return dattn


@pytest.mark.parametrize("splits", [0, 37])
def test_noalloc_decode_matches_workspace_decode_on_two_calls(splits):
    dattn = _lib()
    from split_kv_decode_distattention_gb300 import workloads as W
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("noalloc", B=4, Hq=16, Hkv=4, d=128, P=16, lens=[5000, 1234, 77, 3000],
                  seed=17)
    cache = PagedCache(case, "cuda")
    ws = cache.workspace(num_splits=splits)
    for call in range(2):
        q = case.q(call, "cuda")
        ref = torch.empty(case.B, case.Hq, case.d, device="cuda")
        ref_m = torch.empty(case.B, case.Hq, device="cuda")
        ref_e = torch.empty_like(ref_m)
        cache.decode(q, ref, ws, m_g=ref_m, e_g=ref_e, num_splits=splits)
        out = torch.full_like(ref, float("nan"))
        m_g = torch.full_like(ref_m, float("nan"))
        e_g = torch.full_like(ref_e, float("nan"))
        dattn.dattn_decode_noalloc(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                                   cache.seq_lens, out, m_g=m_g, e_g=e_g, num_splits=splits,
                                   dev_err=cache.dev_err)
        torch.cuda.synchronize()
        assert int(cache.dev_err.item()) == 0
        assert_out_close(out.cpu().numpy(), ref.cpu().numpy(), f"call {call}")
        assert torch.allclose(m_g, ref_m, rtol=1e-5, atol=0)
        assert torch.allclose(e_g, ref_e, rtol=1e-4, atol=0)
        check_dense(case, q, case.lens, out, m_g, e_g, "cuda", what=f"noalloc call {call}")


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    dattn = _lib()
    lib = dattn.load_library()
    bt = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    lay = dattn.KVLayout(64, 8, 128, 16, bt)
    p = ctypes.c_void_p(256)  # never dereferenced: the size check fails first
    # 4096 requests x 8 KV heads x group 8 needs far more than 8 MiB of scratch
    st = lib.dattn_decode_noalloc(ctypes.byref(lay.c), p, p, p, 4096, 64, 0.1, p, None, 0, p,
                                  None, None, None, None)
    assert dattn.dattn_status_string(st) == "DATTN_ERR_WORKSPACE"
