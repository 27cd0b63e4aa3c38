"""vlc_attn_fwd_noalloc: the forward call for callers that cannot allocate device memory.

Such callers (code running inside another runtime's execution hook where allocating
is forbidden, or services whose device-memory budget is fixed at start-up) cannot hand
the library a workspace; this entry point keeps its scratch in a static device array.
The test calls it through the C ABI twice in a row, on two different packs, and checks
each result against vlc_attn_fwd (which takes a workspace) with the parity tolerances.
It lives in its own file so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from variable_length_causal_gb300 import synth

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as vlc

    return vlc.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _run_both(lib, lens, H, d, seed):
    import variable_length_causal_gb300 as vlc

    dev = torch.device("cuda:0")
    w = synth.custom_workload(lens, H, d)
    q, k, v = (t.to(dev) for t in synth.make_tensors(w, seed=seed))
    cu = torch.from_numpy(w.cu).to(dev)
    o_ref, lse_ref = vlc.varlen_attn_fwd(q, k, v, cu, w.max_seqlen)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((H, w.total), float("nan"), device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    st = lib.vlc_attn_fwd_noalloc(_p(q), _p(k), _p(v), _p(cu), w.nseg, w.total, H, d, w.max_seqlen,
                                  0.0, 10000.0, _p(o), _p(lse), _p(err), stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    eo = (o.float() - o_ref.float()).abs()
    el = (lse - lse_ref).abs()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert eo.max().item() <= O_MAX and eo.mean().item() <= O_MEAN
    assert el.max().item() <= LSE_MAX


def test_noalloc_matches_workspace_forward_twice(lib):
    _run_both(lib, [300, 5, 129, 1, 640], 4, 128, seed=31)
    _run_both(lib, [77, 1000, 3], 2, 64, seed=32)


def test_noalloc_rejects_oversize_and_reports_bad_cu(lib):
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    x = torch.zeros(16, 1, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 16, device=dev)
    cu = torch.tensor([0, 16], dtype=torch.int32, device=dev)
    # a segment so long that its RoPE table alone exceeds the static array
    big = 1 << 20
    assert lib.vlc_attn_fwd_noalloc(_p(x), _p(x), _p(x), _p(cu), 1, big, 1, 128, big, 0.0, 10000.0,
                                    _p(x), _p(lse), None, stream) == 4
    # invalid cu_seqlens: reported through err_out, outputs untouched
    bad = torch.tensor([0, 10, 16], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.full_like(x, 3.0)
    assert lib.vlc_attn_fwd_noalloc(_p(x), _p(x), _p(x), _p(bad), 2, 16, 1, 128, 9, 0.0, 10000.0,
                                    _p(o), _p(lse), _p(err), stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) & 0x8
    assert bool((o == 3.0).all())
