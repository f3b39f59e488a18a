"""moe_route_static: routing without a workspace.

Some callers cannot allocate device memory -- a host framework that owns
every allocation, a region where cudaMalloc is not allowed, a fixed memory
plan -- so they cannot hand moe_route its workspace.  moe_route_static keeps
that scratch in a fixed device array inside the library instead.  These
tests call it through the C ABI and compare it with moe_route (which uses a
caller-provided workspace) on two calls in a row with different inputs: the
array is shared and keeps the previous call's contents, so the second call
must not be affected by what the first left behind.

Collected last on purpose (file name), so a failure here comes after every
other test has run; it also passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

from mixture_experts_ffn_02_gb300 import binding, synth
from mixture_experts_ffn_02_gb300.binding import Layer, MoETensors

pytestmark = pytest.mark.gpu

def _route_with_workspace(s, L, norm, bias, valid):
    lay = Layer.create(s, norm_topk=norm)
    lay.bufs.update(logits=L, bias=bias, valid=valid)
    lay.route()
    torch.cuda.synchronize()
    assert lay.status() == 0
    return lay


def _route_static(lib, cfg, s, L, bias, valid):
    dev = L.device
    out = dict(topk_idx=torch.full((s.T, s.k), -7, dtype=torch.int32, device=dev),
               gates=torch.full((s.T, s.k), 9.0, device=dev),
               counts=torch.full((s.E,), -1, dtype=torch.int32, device=dev),
               f=torch.full((s.E,), 9.0, device=dev), p=torch.full((s.E,), 9.0, device=dev),
               aux=torch.full((4,), 9.0, device=dev))
    t = MoETensors(logits=L.data_ptr(), bias=None if bias is None else bias.data_ptr(),
                   valid=None if valid is None else valid.data_ptr(),
                   **{k: v.data_ptr() for k, v in out.items()})
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    rc = lib.moe_route_static(ctypes.byref(cfg), ctypes.byref(t),
                              ctypes.c_void_p(status.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, binding.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    return out


def _same(ref_lay, out):
    """Same kernel, same grid, same inputs: the same bytes, bit for bit."""
    b = ref_lay.bufs
    for n in ("topk_idx", "counts", "gates", "f", "p"):
        assert torch.equal(out[n], b[n]), n
    assert torch.equal(out["aux"][:1], b["aux"][:1])


@pytest.mark.parametrize("cfg_id,T,norm,pad", [(2, 32768, 1, 0), (3, 65536, 1, 5243),
                                               (4, 16384, 1, 0), (5, 32768, 0, 0),
                                               (1, 256, 1, 0)])
def test_static_route_matches_workspace_route_twice(cfg_id, T, norm, pad):
    lib = binding.load()
    s = synth.scaled(synth.shape(cfg_id), T=T, T_real=None)
    cfg = binding.config(s, norm_topk=norm)
    bias = synth.selection_bias(s)
    bias = None if bias is None else bias.cuda()
    valid = None
    if pad:
        valid = torch.ones(T, dtype=torch.uint8)
        valid[T - pad:] = 0
        valid = valid.cuda()
    for call, seed in enumerate((11, 12)):        # two calls in a row, new inputs
        L = synth.random_logits(T, s.E, seed=seed + cfg_id).cuda()
        ref = _route_with_workspace(s, L, norm, bias, valid)
        out = _route_static(lib, cfg, s, L, bias, valid)
        _same(ref, out)


def test_static_route_widest_router_fits():
    """The route grid is capped at what the fixed scratch holds (for moe_route
    too), so even the widest router (E = 256) at a large T runs through the
    static entry point and matches the workspace route."""
    lib = binding.load()
    s = synth.MoEShape("wide", T=65536, d=64, E=256, k=8, H=64, n_shared=0, H_shared=0)
    cfg = binding.config(s)
    L = synth.random_logits(s.T, s.E, seed=5).cuda()
    ref = _route_with_workspace(s, L, 1, None, None)
    out = _route_static(lib, cfg, s, L, None, None)
    _same(ref, out)


def test_static_route_allocates_nothing():
    """The call itself allocates no device memory: after a first call (which
    resolves the scratch address and loads the kernel), the free device
    memory the driver reports and torch's reserved pool are the same before
    and after a second call, whose outputs match the workspace route."""
    lib = binding.load()
    s = synth.scaled(synth.shape(2), T=32768, T_real=None)
    cfg = binding.config(s)
    L = synth.random_logits(s.T, s.E, seed=21).cuda()
    ref = _route_with_workspace(s, L, 1, None, None)
    _route_static(lib, cfg, s, L, None, None)              # set-up call
    dev = L.device
    out = dict(topk_idx=torch.empty((s.T, s.k), dtype=torch.int32, device=dev),
               gates=torch.empty((s.T, s.k), device=dev),
               counts=torch.empty((s.E,), dtype=torch.int32, device=dev),
               f=torch.empty((s.E,), device=dev), p=torch.empty((s.E,), device=dev),
               aux=torch.empty((4,), device=dev))
    t = MoETensors(logits=L.data_ptr(), **{k: v.data_ptr() for k, v in out.items()})
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    rc = lib.moe_route_static(ctypes.byref(cfg), ctypes.byref(t),
                              ctypes.c_void_p(status.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert rc == 0, binding.STATUS.get(rc, rc)
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_reserved() == reserved0
    assert int(status[0]) == 0
    _same(ref, out)
