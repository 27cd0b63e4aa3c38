"""The failure path of the bounded waits, exercised without faulting or hanging a GPU.

Every mbarrier wait inside the attention kernels is bounded.  When one expires the
kernel raises VLC_DEVERR_TIMEOUT in the workspace's error word, waits (bounded) for
its own copies and MMAs in flight, frees its tensor memory and returns; the later
kernels of the call do nothing.  Here the wait limit is shortened to 1 microsecond
(vlc_set_wait_limit_us), so waits expire in the middle of normal work -- nothing is
broken on purpose -- and the test checks that each call returns promptly with
VLC_ERR_TIMEOUT, and that normal calls on the same stream afterwards match the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from variable_length_causal_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module")
def vlc():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as m

    m.load_library()
    return m


def _pack():
    w = synth.custom_workload([700, 129, 1500, 64, 300, 1024, 5, 2000], 4, 128)
    q, k, v, g = synth.make_tensors(w, seed=91, with_grad=True)
    return w, q, k, v, g


def test_expired_waits_report_timeout_then_calls_recover(vlc):
    w, q, k, v, g = _pack()
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cu = torch.from_numpy(w.cu).to(DEV)
    wsf = vlc.new_workspace(w.nseg, w.total, w.H, w.d, w.max_seqlen, False, DEV)
    wsb = vlc.new_workspace(w.nseg, w.total, w.H, w.d, w.max_seqlen, True, DEV)
    o = torch.empty_like(qd)
    lse = torch.empty((w.H, w.total), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    try:
        vlc.set_wait_limit_us(1)
        for form in ("fused", "rotated"):
            t0 = time.perf_counter()
            if form == "fused":
                vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, out=o, lse=lse, workspace=wsf, check=False)
            else:
                qr, kr = vlc.rope_qk(qd, kd, cu, w.max_seqlen)
                vlc.varlen_attn_fwd(qr, kr, vd, cu, w.max_seqlen, out=o, lse=lse, workspace=wsf, check=False,
                                    qk_rotated=True)
            st, bits = vlc.get_error(wsf)
            assert time.perf_counter() - t0 < 10.0
            assert st == vlc.binding.VLC_ERR_TIMEOUT and bits & vlc.binding.DEVERR_TIMEOUT, (form, st, bits)
        # a valid forward result, then a backward whose waits expire
        vlc.set_wait_limit_us(0)
        o, lse = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen)
        vlc.set_wait_limit_us(1)
        t0 = time.perf_counter()
        vlc.varlen_attn_bwd(gd, qd, kd, vd, o, lse, cu, w.max_seqlen, workspace=wsb, check=False)
        st, bits = vlc.get_error(wsb)
        assert time.perf_counter() - t0 < 10.0
        assert st == vlc.binding.VLC_ERR_TIMEOUT and bits & vlc.binding.DEVERR_TIMEOUT, (st, bits)
    finally:
        vlc.set_wait_limit_us(0)
    # the default limit again: the same stream and workspaces give correct results
    o2, lse2 = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, workspace=wsf)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.cu)
    e = np.abs(o2.float().cpu().numpy() - o_ref)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3
    assert np.abs(lse2.cpu().numpy() - lse_ref).max() <= 1e-3
    grads = vlc.varlen_attn_bwd(gd, qd, kd, vd, o2, lse2, cu, w.max_seqlen, workspace=wsb)
    ref = oracle.attn_bwd(g, q, k, v, w.cu)
    for a, b in zip(grads, ref):
        assert np.abs(a.float().cpu().numpy() - b).max() <= 5e-2
