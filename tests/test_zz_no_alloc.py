"""vlc_attn_fwd_noalloc: the forward call for callers that cannot allocate device memory.

Such callers (code running inside another runtime's execution hook where allocating
is forbidden, or services whose device-memory budget is fixed at start-up) cannot hand
the library a workspace; this entry point keeps its scratch in a static device array.
The tests call it through the C ABI twice in a row, on two different packs, and check
each result against vlc_attn_fwd (which takes a workspace) with the parity tolerances;
one pack (with a segment of more than 2048 keys) has a whole forward workspace that fits
in the static array, so k is rotated once inside it, and that result is also checked
against the fp64 oracle.  The file sits last in pytest's collection order.
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


def _run_both(lib, lens, H, d, seed, check_oracle=False):
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
    if check_oracle:
        import oracle

        o_or, lse_or = oracle.attn_fwd(q.cpu(), k.cpu(), v.cpu(), w.cu)
        eo = np.abs(o.float().cpu().numpy() - o_or)
        assert eo.max() <= O_MAX and eo.mean() <= O_MEAN
        assert np.abs(lse.cpu().numpy() - lse_or).max() <= LSE_MAX
    return w


def test_noalloc_matches_workspace_forward_twice(lib):
    _run_both(lib, [300, 5, 129, 1, 640], 4, 128, seed=31)
    _run_both(lib, [77, 1000, 3], 2, 64, seed=32)


def test_noalloc_long_segment_rotated_k_in_scratch(lib):
    # a 2300-key segment: the whole forward workspace (rotated copy of k included) fits in
    # the static array, so the long segment's k is rotated once into it, as vlc_attn_fwd does
    lens, H, d = [2300, 40, 700], 2, 128
    total = sum(lens)
    full = lib.vlc_workspace_bytes(len(lens), total, H, d, max(lens), 0)
    assert 0 < full <= (8 << 20)
    _run_both(lib, lens, H, d, seed=33, check_oracle=True)
    _run_both(lib, lens, H, d, seed=34, check_oracle=True)


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
    # unsupported shapes give the status vlc_attn_fwd gives: a segment longer than the
    # library's limit, an unsupported head dimension
    too_long = (1 << 20) + 1
    assert lib.vlc_attn_fwd_noalloc(_p(x), _p(x), _p(x), _p(cu), 1, 16, 1, 128, too_long, 0.0, 10000.0,
                                    _p(x), _p(lse), None, stream) == 3
    assert lib.vlc_attn_fwd_noalloc(_p(x), _p(x), _p(x), _p(cu), 1, 16, 1, 96, 16, 0.0, 10000.0,
                                    _p(x), _p(lse), None, stream) == 3
    # invalid cu_seqlens: reported through err_out, outputs untouched
    bad = torch.tensor([0, 10, 16], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.full_like(x, 3.0)
    assert lib.vlc_attn_fwd_noalloc(_p(x), _p(x), _p(x), _p(bad), 2, 16, 1, 128, 9, 0.0, 10000.0,
                                    _p(o), _p(lse), _p(err), stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) & 0x8
    assert bool((o == 3.0).all())
