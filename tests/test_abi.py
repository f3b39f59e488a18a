"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every function `include/moe.h` declares, and its host-side queries (shape
rules, row capacity, workspace size) behave as documented.  No kernel runs."""
import ctypes
import os
import re

import pytest

from mixture_experts_ffn_02_gb300 import binding, build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clib():
    build.build()
    return binding.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(moe_\w+)\s*\(", src, re.M)))


# the calls of the layer's problem statement: router logits, routing,
# dispatch, the experts, the combine, forward and backward, plus the
# workspace query, the status read and the error messages
BOUNDARY = ["moe_workspace_bytes", "moe_router_logits", "moe_route", "moe_permute",
            "moe_expert_ffn", "moe_combine", "moe_forward", "moe_backward", "moe_get_status",
            "moe_strerror"]


def test_header_declares_the_abi():
    names = declared_functions()
    for n in BOUNDARY + ["moe_expert_gate_up", "moe_expert_down", "moe_shared_ffn",
                         "moe_router_route", "moe_shared_ffn_combine"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(clib):
    for n in declared_functions():
        assert hasattr(clib, n), n
    assert set(declared_functions()) <= set(binding.SIGNATURES)


def test_abi_version_and_messages(clib):
    assert clib.moe_abi_version() == 6
    for code in range(10):
        assert clib.moe_strerror(code)
    assert b"unknown" in clib.moe_strerror(99)


def cfg(**kw):
    base = dict(T=256, d=64, E=4, k=2, H=128, n_shared=1, H_shared=128, norm_topk=1,
                aux_coef=0.01, z_coef=0.0)
    base.update(kw)
    return binding.MoEConfig(**base)


@pytest.mark.parametrize("bad", [dict(T=0), dict(d=100), dict(H=96), dict(k=0), dict(k=5),
                                 dict(E=257, k=2), dict(E=64, k=33), dict(n_shared=-1),
                                 dict(H_shared=100), dict(T=2 ** 30, k=8),
                                 dict(z_coef=float("nan"))])
def test_shape_rules(clib, bad):
    assert clib.moe_check_config(ctypes.byref(cfg(**bad))) == 2


def test_valid_configs(clib):
    for s in synth.SHAPES.values():
        assert clib.moe_check_config(ctypes.byref(binding.config(s))) == 0
    assert clib.moe_check_config(None) == 1


def test_row_capacity_bounds_every_padded_layout(clib):
    c = cfg(T=1000, E=8, k=2)
    r = ctypes.c_int64()
    assert clib.moe_row_capacity(ctypes.byref(c), ctypes.byref(r)) == 0
    assert r.value == (1000 * 2 + 127 * 8) // 128 * 128
    # worst case: every expert's count is 1 more than a multiple of 128
    counts = [129] * 7 + [2000 - 129 * 7]
    assert sum((n + 127) // 128 * 128 for n in counts) <= r.value


def test_workspace_grows_with_training(clib):
    c = binding.config(synth.shape(5))
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert clib.moe_workspace_bytes(ctypes.byref(c), 0, ctypes.byref(a)) == 0
    assert clib.moe_workspace_bytes(ctypes.byref(c), 1, ctypes.byref(b)) == 0
    assert 0 < a.value < b.value


def test_entry_points_reject_bad_arguments_without_touching_the_gpu(clib):
    c = cfg()
    t = binding.MoETensors()
    # NULL workspace is reported before any device work
    for name in ["moe_forward", "moe_route", "moe_permute", "moe_combine"]:
        rc = getattr(clib, name)(ctypes.byref(c), ctypes.byref(t), None, 0, None)
        assert rc in (4, 5, 6), (name, rc)   # workspace, or no CUDA device here
    bad = cfg(d=65)
    assert clib.moe_forward(ctypes.byref(bad), ctypes.byref(t), None, 0, None) == 2


def test_struct_layouts_match_the_header():
    """The binding's ctypes structures have the header's field order."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for struct, cls in (("moe_config", binding.MoEConfig), ("moe_tensors", binding.MoETensors),
                        ("moe_grads", binding.MoEGrads),
                        ("moe_mx_tensors", binding.MoEMxTensors)):
        body = re.search(r"typedef struct " + struct + r" \{(.*?)\} " + struct, src, re.S).group(1)
        names = re.findall(r"\b(\w+)\s*;", body)
        assert names == [f[0] for f in cls._fields_], struct


def test_mx_sizes_and_shape_rule(clib):
    """MXFP8 buffers: codes keep the bf16 tensors' element counts, one scale
    byte per 32 values in 512-byte atoms; a d or H off the tile grid is a
    shape error (d must be a multiple of 256 and H of 128; the tiny 64-wide
    layer has no MX path)."""
    s = synth.shape(2)
    c = binding.config(s)
    sizes = (ctypes.c_size_t * binding.MOE_MX_FIELDS)()
    assert clib.moe_mx_sizes(ctypes.byref(c), sizes) == 0
    R = ctypes.c_int64()
    assert clib.moe_row_capacity(ctypes.byref(c), ctypes.byref(R)) == 0
    E, d, H, R = s.E, s.d, s.H, R.value
    Hs, Tp = s.n_shared * s.H_shared, (s.T + 127) // 128 * 128
    assert list(sizes) == [E * 2 * H * d, E * 2 * H * d // 32, E * d * H, E * d * H // 32,
                           R * d, R * d // 32, R * H, R * H // 32,
                           2 * Hs * d, 2 * Hs * d // 32, d * Hs, d * Hs // 32,
                           Tp * d, Tp * d // 32, Tp * Hs, Tp * Hs // 32,
                           # the training step's: transposed weights, d_out, d_gu
                           E * d * 2 * H, E * d * 2 * H // 32, E * H * d, E * H * d // 32,
                           R * d, R * d // 32, R * 2 * H, R * 2 * H // 32, R * 2 * H * 2]
    c5 = binding.config(synth.shape(5))              # no shared expert: its buffers are 0
    assert clib.moe_mx_sizes(ctypes.byref(c5), sizes) == 0
    assert list(sizes)[8:16] == [0] * 8 and min(list(sizes)[16:]) > 0
    tiny = binding.config(synth.shape(1))
    assert clib.moe_mx_sizes(ctypes.byref(tiny), sizes) == 2
    t = binding.MoETensors()
    m = binding.MoEMxTensors()
    assert clib.moe_mx_forward(ctypes.byref(tiny), ctypes.byref(t), ctypes.byref(m), None, 0,
                               None) == 2
    assert clib.moe_mx_forward_train(ctypes.byref(tiny), ctypes.byref(t), ctypes.byref(m),
                                     None, 0, None) == 2
    gr = binding.MoEGrads()
    assert clib.moe_mx_backward(ctypes.byref(tiny), ctypes.byref(t), ctypes.byref(m),
                                ctypes.byref(gr), None, 0, None) == 2


def test_debug_build_exports_the_abi():
    """The checking variant (device bounds checks, MOE_DEBUG_BOUNDS) builds,
    exports every declared symbol and says which build it is."""
    dbg = binding.load(debug=True)
    for n in declared_functions():
        assert hasattr(dbg, n), n
    assert dbg.moe_debug_bounds() == 1
    assert binding.load().moe_debug_bounds() == 0
    assert b"debug bounds" in dbg.moe_strerror(10)
