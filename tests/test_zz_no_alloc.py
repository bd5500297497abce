"""The allocation-free decode entry point, called through the C ABI.

nc_attn_decode_noalloc serves callers that cannot hand the library any
device memory -- a serving loop that must not call cudaMalloc between tokens
because it synchronises the whole device, or a host program that owns all
device memory itself.  It keeps its scratch in a fixed array inside the
library, so these tests check that two calls in a row (sharing that array)
each give what the ordinary workspace-based nc_attn_decode gives, and that a
problem too big for the array is refused before anything runs.

This file sorts last so that, in a run that stops at the first failure,
every other test has already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

EPS, BASE = workloads.EPS, workloads.ROPE_BASE
MAX_ABS = 1e-2  # the decode tolerance used by the parity tests


@pytest.fixture(scope="module")
def nc():
    import causal_attention_rope_nc_b300 as m
    return m


def _call_noalloc(nc, q, k_new, v_new, kcache, vcache, lens, out):
    """Raw C-ABI call with device pointers, on the current stream."""
    B, Tcap, H, D = kcache.shape
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = nc.lib.nc_attn_decode_noalloc(p(q), p(k_new), p(v_new), p(kcache), p(vcache), p(lens), p(out),
                                       B, H, D, Tcap, EPS, BASE,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0, nc.lib.nc_strerror(rc)


def test_oversize_problem_is_refused(nc):
    """Needs no GPU: the size check runs before any CUDA call."""
    fake = ctypes.c_void_p(4096)
    # 64 streams x capacity 32768 x 16 heads: far more partials than 16 MiB
    rc = nc.lib.nc_attn_decode_noalloc(fake, None, None, fake, fake, fake, fake, 64, 16, 128, 32768,
                                       EPS, BASE, None)
    assert rc == nc.NC_ETOOLARGE


@pytest.mark.gpu
def test_two_calls_match_the_workspace_decode(nc):
    """Each path gets its own copy of the caches, so the slot that the second
    call writes (the new token's normalised, rotated key and its value) is
    compared too, not only the outputs."""
    w = workloads.D20_DECODE
    assert nc.workspace_size(nc.NC_OP_DECODE, w.B, w.Tcap, w.H, w.D) <= 16 << 20
    lens, q, k_raw, v = workloads.decode_workload_inputs(w)
    kcache = nc.qk_norm_rope(k_raw.cuda(), eps=EPS, rope_base=BASE)
    vcache = v.cuda()
    qd = q.cuda()
    # second call: other lengths and a new token written into the cache
    lens2 = torch.flip(lens, [0]).contiguous()
    idx = (lens2 - 1).long()
    k_new = k_raw[torch.arange(w.B), idx].contiguous().cuda()
    v_new = v[torch.arange(w.B), idx].contiguous().cuda()
    bi, pi = torch.arange(w.B, device="cuda"), idx.cuda()
    for ln, kn, vn in ((lens, None, None), (lens2, k_new, v_new)):
        ld = ln.cuda()
        kc_ws, vc_ws = kcache.clone(), vcache.clone()
        kc_na, vc_na = kcache.clone(), vcache.clone()
        if kn is not None:  # the slot to be written holds zeros in both copies
            for t in (kc_ws, vc_ws, kc_na, vc_na):
                t[bi, pi] = 0
        ref = nc.attn_decode(qd, kc_ws, vc_ws, ld, k_new=kn, v_new=vn, eps=EPS, rope_base=BASE)
        out = torch.empty_like(ref)
        _call_noalloc(nc, qd, kn, vn, kc_na, vc_na, ld, out)
        torch.cuda.synchronize()
        assert nc.device_status() == 0
        err = float((out.float() - ref.float()).abs().max())
        assert err <= MAX_ABS, err
        assert bool(torch.isfinite(out.float()).all())
        if kn is not None:
            assert torch.equal(kc_na[bi, pi], kc_ws[bi, pi])
            assert torch.equal(vc_na[bi, pi], vc_ws[bi, pi])
            assert bool((vc_na[bi, pi] == v_new).all())
        assert torch.equal(kc_na, kc_ws) and torch.equal(vc_na, vc_ws)
