"""Thin Python binding of the C ABI in ``include/moe.h``.

Argument marshalling only: torch allocates device memory and supplies the
stream; every step of the layer runs in the CUDA kernels of
``_build/libmoe_gb300.so``.  There is no fallback: if the library is missing
or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import build as _build

c_int32 = ctypes.c_int32
c_float = ctypes.c_float
c_void_p = ctypes.c_void_p

MOE_ROW_ALIGN = 128

STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_NULL", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_ALIGN",
    4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE", 7: "MOE_ERR_TIMEOUT",
    8: "MOE_ERR_INDEX", 9: "MOE_ERR_NONFINITE", 10: "MOE_ERR_BOUNDS",
}


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", c_int32), ("d", c_int32), ("E", c_int32), ("k", c_int32),
                ("H", c_int32), ("n_shared", c_int32), ("H_shared", c_int32),
                ("norm_topk", c_int32), ("aux_coef", c_float), ("z_coef", c_float)]


TENSOR_FIELDS = ["x", "Wr", "bias", "valid", "W_gu", "W_down", "Ws_gu", "Ws_down",
                 "logits", "topk_idx", "gates", "counts", "f", "p", "aux", "router_stats",
                 "offsets", "row_offsets", "perm", "inv", "x_perm",
                 "ab", "h", "out_perm", "s_ab", "s_h", "s_out", "y"]
GRAD_FIELDS = ["dY", "dx", "dWr", "dW_gu", "dW_down", "dWs_gu", "dWs_down", "d_logits"]


class MoETensors(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in TENSOR_FIELDS]


class MoEGrads(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in GRAD_FIELDS]


MOE_MX_FIELDS = 25
MX_FIELDS = ["W_gu_q", "W_gu_s", "W_down_q", "W_down_s", "x_q", "x_s", "h_q", "h_s",
             "Ws_gu_q", "Ws_gu_s", "Ws_down_q", "Ws_down_s", "xt_q", "xt_s", "hs_q", "hs_s",
             "W_gu_tq", "W_gu_ts", "W_down_tq", "W_down_ts", "dout_q", "dout_s", "dgu_q",
             "dgu_s", "ab16"]
MX_TRAIN_FIELDS = MX_FIELDS[16:]


class MoEMxTensors(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in MX_FIELDS]


_STEP = [ctypes.POINTER(MoEConfig), ctypes.POINTER(MoETensors), c_void_p, ctypes.c_size_t,
         c_void_p]
_MX_STEP = [ctypes.POINTER(MoEConfig), ctypes.POINTER(MoETensors),
            ctypes.POINTER(MoEMxTensors), c_void_p, ctypes.c_size_t, c_void_p]
SIGNATURES = {
    "moe_abi_version": (ctypes.c_int, []),
    "moe_debug_bounds": (ctypes.c_int, []),
    "moe_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_check_config": (ctypes.c_int, [ctypes.POINTER(MoEConfig)]),
    "moe_row_capacity": (ctypes.c_int, [ctypes.POINTER(MoEConfig),
                                        ctypes.POINTER(ctypes.c_int64)]),
    "moe_workspace_bytes": (ctypes.c_int, [ctypes.POINTER(MoEConfig), ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_size_t)]),
    "moe_get_status": (ctypes.c_int, [c_void_p, c_void_p, ctypes.POINTER(ctypes.c_int)]),
    "moe_workspace_offsets": (ctypes.c_int, [ctypes.POINTER(MoEConfig),
                                             ctypes.POINTER(ctypes.c_size_t)]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [c_void_p, ctypes.c_uint64, c_void_p]),
    "moe_router_logits": (ctypes.c_int, _STEP),
    "moe_route": (ctypes.c_int, _STEP),
    "moe_router_route": (ctypes.c_int, _STEP),
    "moe_permute": (ctypes.c_int, _STEP),
    "moe_expert_gate_up": (ctypes.c_int, _STEP),
    "moe_expert_down": (ctypes.c_int, _STEP),
    "moe_shared_ffn": (ctypes.c_int, _STEP),
    "moe_combine": (ctypes.c_int, _STEP),
    "moe_shared_ffn_combine": (ctypes.c_int, _STEP),
    "moe_expert_ffn": (ctypes.c_int, _STEP),
    "moe_forward": (ctypes.c_int, _STEP),
    "moe_backward": (ctypes.c_int, [ctypes.POINTER(MoEConfig), ctypes.POINTER(MoETensors),
                                    ctypes.POINTER(MoEGrads), c_void_p, ctypes.c_size_t,
                                    c_void_p]),
    "moe_route_static": (ctypes.c_int, [ctypes.POINTER(MoEConfig), ctypes.POINTER(MoETensors),
                                        c_void_p, c_void_p]),
    "moe_mx_sizes": (ctypes.c_int, [ctypes.POINTER(MoEConfig), ctypes.POINTER(ctypes.c_size_t)]),
    "moe_mx_quantize_weights": (ctypes.c_int, [ctypes.POINTER(MoEConfig),
                                               ctypes.POINTER(MoETensors),
                                               ctypes.POINTER(MoEMxTensors), c_void_p]),
    "moe_mx_permute": (ctypes.c_int, _MX_STEP),
    "moe_mx_expert_gate_up": (ctypes.c_int, _MX_STEP),
    "moe_mx_expert_down": (ctypes.c_int, _MX_STEP),
    "moe_mx_shared_ffn": (ctypes.c_int, _MX_STEP),
    "moe_mx_forward": (ctypes.c_int, _MX_STEP),
    "moe_mx_forward_train": (ctypes.c_int, _MX_STEP),
    "moe_mx_backward": (ctypes.c_int, [ctypes.POINTER(MoEConfig), ctypes.POINTER(MoETensors),
                                       ctypes.POINTER(MoEMxTensors), ctypes.POINTER(MoEGrads),
                                       c_void_p, ctypes.c_size_t, c_void_p]),
    "moe_route_partials": (ctypes.c_int, [ctypes.POINTER(MoEConfig), ctypes.POINTER(MoETensors),
                                          c_void_p, c_void_p]),
    "moe_route_finalize": (ctypes.c_int, [ctypes.POINTER(MoEConfig), ctypes.POINTER(MoETensors),
                                          c_void_p, c_void_p]),
}

_LIB = None
_LIB_DEBUG = None


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


def load(path: str | None = None, build_if_missing: bool = False,
         debug: bool | None = None) -> ctypes.CDLL:
    """Load the shared library (no fallback: raises if it is absent).  With
    ``debug`` (default: the environment variable MOE_DEBUG_BOUNDS=1) the
    variant with device bounds checks, built on demand."""
    global _LIB, _LIB_DEBUG
    if debug is None:
        debug = os.environ.get("MOE_DEBUG_BOUNDS") == "1"
    cached = _LIB_DEBUG if debug else _LIB
    if cached is not None and path is None:
        return cached
    p = path or (_build.LIB_DEBUG if debug else _build.LIB)
    if debug and path is None and not os.path.exists(p):
        _build.build(debug=True)
    if not os.path.exists(p):
        if build_if_missing:
            _build.build()
        else:
            raise RuntimeError(f"MoE CUDA library not built: {p} (run build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        if debug:
            _LIB_DEBUG = lib
        else:
            _LIB = lib
    return lib


def check(code: int, where: str):
    if code != 0:
        raise MoEError(code, where)


def config(shape, **over) -> MoEConfig:
    """MoEConfig from a synth.MoEShape (or anything with the same fields)."""
    c = MoEConfig(T=shape.T, d=shape.d, E=shape.E, k=shape.k, H=shape.H,
                  n_shared=shape.n_shared, H_shared=shape.H_shared,
                  norm_topk=shape.norm_topk, aux_coef=shape.aux_coef,
                  z_coef=getattr(shape, "z_coef", 0.0))
    for k_, v in over.items():
        setattr(c, k_, v)
    return c


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream():
    import torch
    return c_void_p(torch.cuda.current_stream().cuda_stream)


@dataclass
class Layer:
    """One MoE layer call's device buffers (torch) and the library handle."""
    cfg: MoEConfig
    training: bool
    bufs: dict
    grads: dict
    ws: object
    lib: ctypes.CDLL
    mx: dict = None

    @classmethod
    def create(cls, shape, training: bool = False, device: str = "cuda", lib=None,
               gather: bool = False, **over):
        """Device buffers for one layer.  gather=True (inference only) leaves
        x_perm out: the permute then copies no rows and the gate/up GEMM
        gathers them from x."""
        import torch
        if gather and training:
            raise ValueError("the backward needs x_perm: gather=True is for inference")
        lib = lib or load()
        cfg = config(shape, **over)
        check(lib.moe_check_config(ctypes.byref(cfg)), "moe_check_config")
        rows = ctypes.c_int64()
        check(lib.moe_row_capacity(ctypes.byref(cfg), ctypes.byref(rows)), "moe_row_capacity")
        R = rows.value
        wsb = ctypes.c_size_t()
        check(lib.moe_workspace_bytes(ctypes.byref(cfg), int(training), ctypes.byref(wsb)),
              "moe_workspace_bytes")
        T, d, E, k, H = cfg.T, cfg.d, cfg.E, cfg.k, cfg.H
        Hs = cfg.n_shared * cfg.H_shared
        bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
        dev = torch.device(device)

        def z(*s, dt):
            return torch.empty(*s, dtype=dt, device=dev)

        b = dict(logits=z(T, E, dt=f32), topk_idx=z(T, k, dt=i32), gates=z(T, k, dt=f32),
                 counts=z(E, dt=i32), f=z(E, dt=f32), p=z(E, dt=f32), aux=z(4, dt=f32),
                 router_stats=z(8, dt=f32),
                 offsets=z(E + 1, dt=i32), row_offsets=z(E + 1, dt=i32), perm=z(R, dt=i32),
                 inv=z(T * k, dt=i32), x_perm=None if gather else z(R, d, dt=bf),
                 h=z(R, H, dt=bf),
                 out_perm=z(R, d, dt=bf), y=z(T, d, dt=bf),
                 ab=z(R, 2 * H, dt=bf) if training else None,
                 s_h=z(T, Hs, dt=bf) if Hs else None,
                 s_out=z(T, d, dt=f32) if Hs else None,
                 s_ab=z(T, 2 * Hs, dt=bf) if (Hs and training) else None)
        g = {}
        if training:
            g = dict(dx=z(T, d, dt=bf), dWr=z(d, E, dt=f32), dW_gu=z(E, 2 * H, d, dt=bf),
                     dW_down=z(E, d, H, dt=bf), d_logits=z(T, E, dt=f32),
                     dWs_gu=z(2 * Hs, d, dt=bf) if Hs else None,
                     dWs_down=z(d, Hs, dt=bf) if Hs else None)
        ws = torch.zeros(max(wsb.value, 16), dtype=torch.uint8, device=dev)
        return cls(cfg=cfg, training=training, bufs=b, grads=g, ws=ws, lib=lib)

    @property
    def R_cap(self) -> int:
        return self.bufs["perm"].shape[0]

    def set_inputs(self, x, Wr, W_gu, W_down, Ws_gu=None, Ws_down=None, bias=None,
                   valid=None):
        self.bufs.update(x=x, Wr=Wr, W_gu=W_gu, W_down=W_down, Ws_gu=Ws_gu, Ws_down=Ws_down,
                         bias=bias, valid=valid)

    def tensors(self) -> MoETensors:
        return MoETensors(**{n: _ptr(self.bufs.get(n)) for n in TENSOR_FIELDS})

    def grad_struct(self, dY) -> MoEGrads:
        d = {n: _ptr(self.grads.get(n)) for n in GRAD_FIELDS if n != "dY"}
        return MoEGrads(dY=_ptr(dY), **d)

    def _step(self, name):
        t = self.tensors()
        fn = getattr(self.lib, name)
        check(fn(ctypes.byref(self.cfg), ctypes.byref(t), c_void_p(self.ws.data_ptr()),
                 self.ws.numel(), _stream()), name)

    def router_logits(self): self._step("moe_router_logits")
    def route(self): self._step("moe_route")
    def router_route(self): self._step("moe_router_route")
    def permute(self): self._step("moe_permute")
    def gate_up(self): self._step("moe_expert_gate_up")
    def down(self): self._step("moe_expert_down")
    def shared(self): self._step("moe_shared_ffn")
    def combine(self): self._step("moe_combine")
    def shared_combine(self): self._step("moe_shared_ffn_combine")
    def expert_ffn(self): self._step("moe_expert_ffn")
    def forward(self): self._step("moe_forward")

    def step(self, dY=None, timed=None):
        """One pass of the layer, call by call: moe_router_route, moe_permute,
        moe_expert_gate_up, moe_expert_down, moe_shared_ffn_combine (the
        combine in the shared expert's down GEMM, or the combine kernel when
        there is no shared expert), then moe_backward if dY is given.  The
        same kernels in the same order as moe_forward + moe_backward.
        ``timed(name, fn)``, if given, runs each call (to bracket it with
        events); names: router_route, permute, gate_up, down, combine
        (shared_combine with a shared expert), backward."""
        run = timed or (lambda name, fn: fn())
        run("router_route", self.router_route)
        run("permute", self.permute)
        run("gate_up", self.gate_up)
        run("down", self.down)
        if self.cfg.n_shared > 0:
            run("shared_combine", self.shared_combine)
        else:
            run("combine", self.combine)
        if dY is not None:
            run("backward", lambda: self.backward(dY))

    def backward(self, dY):
        t = self.tensors()
        g = self.grad_struct(dY)
        check(self.lib.moe_backward(ctypes.byref(self.cfg), ctypes.byref(t), ctypes.byref(g),
                                    c_void_p(self.ws.data_ptr()), self.ws.numel(), _stream()),
              "moe_backward")

    # ---- MXFP8 routed experts (inference)
    def mx_alloc(self):
        """Device buffers of moe_mx_tensors (sizes from moe_mx_sizes); the
        training step's eight only on a training layer."""
        import torch
        sizes = (ctypes.c_size_t * len(MX_FIELDS))()
        check(self.lib.moe_mx_sizes(ctypes.byref(self.cfg), sizes), "moe_mx_sizes")
        dev = self.ws.device
        self.mx = {n: (torch.empty(int(sz), dtype=torch.uint8, device=dev)
                       if sz and (self.training or n not in MX_TRAIN_FIELDS) else None)
                   for n, sz in zip(MX_FIELDS, sizes)}
        return self.mx

    def mx_tensors(self) -> MoEMxTensors:
        return MoEMxTensors(**{n: _ptr(self.mx.get(n)) for n in MX_FIELDS})

    def _mx_step(self, name):
        t = self.tensors()
        m = self.mx_tensors()
        fn = getattr(self.lib, name)
        check(fn(ctypes.byref(self.cfg), ctypes.byref(t), ctypes.byref(m),
                 c_void_p(self.ws.data_ptr()), self.ws.numel(), _stream()), name)

    def mx_quantize_weights(self):
        t = self.tensors()
        m = self.mx_tensors()
        check(self.lib.moe_mx_quantize_weights(ctypes.byref(self.cfg), ctypes.byref(t),
                                               ctypes.byref(m), _stream()),
              "moe_mx_quantize_weights")

    def mx_permute(self): self._mx_step("moe_mx_permute")
    def mx_gate_up(self): self._mx_step("moe_mx_expert_gate_up")
    def mx_down(self): self._mx_step("moe_mx_expert_down")
    def mx_shared(self): self._mx_step("moe_mx_shared_ffn")
    def mx_forward(self): self._mx_step("moe_mx_forward")
    def mx_forward_train(self): self._mx_step("moe_mx_forward_train")

    def mx_step(self, dY):
        """One MXFP8 training step: moe_mx_forward_train then moe_mx_backward
        (the weight codes from mx_quantize_weights)."""
        self.mx_forward_train()
        self.mx_backward(dY)

    def mx_backward(self, dY):
        t = self.tensors()
        m = self.mx_tensors()
        gr = self.grad_struct(dY)
        check(self.lib.moe_mx_backward(ctypes.byref(self.cfg), ctypes.byref(t), ctypes.byref(m),
                                       ctypes.byref(gr), c_void_p(self.ws.data_ptr()),
                                       self.ws.numel(), _stream()), "moe_mx_backward")

    def route_partials(self, sums):
        """This rank's routing sums into ``sums`` ([2E+1] float64, device)."""
        t = self.tensors()
        check(self.lib.moe_route_partials(ctypes.byref(self.cfg), ctypes.byref(t),
                                          c_void_p(sums.data_ptr()), _stream()),
              "moe_route_partials")

    def route_finalize(self, sums):
        """Global f, p, aux from sums added over the data-parallel ranks."""
        t = self.tensors()
        check(self.lib.moe_route_finalize(ctypes.byref(self.cfg), ctypes.byref(t),
                                          c_void_p(sums.data_ptr()), _stream()),
              "moe_route_finalize")

    def intermediates(self) -> dict:
        """Views of the backward's stored intermediates in the workspace
        (moe_workspace_offsets): d_out [R][d] bf16, d_gu [R][2H] bf16,
        dx_perm [R][d] bf16, and ds_gu [T][2Hs] bf16 with a shared expert."""
        import torch
        if not self.training:
            raise ValueError("only a training workspace holds the backward's intermediates")
        off = (ctypes.c_size_t * 4)()
        check(self.lib.moe_workspace_offsets(ctypes.byref(self.cfg), off),
              "moe_workspace_offsets")
        R, d, H = self.R_cap, self.cfg.d, self.cfg.H
        Hs = self.cfg.n_shared * self.cfg.H_shared

        def view(o, n, dt, shape):
            nb = n * torch.empty((), dtype=dt).element_size()
            return self.ws[o:o + nb].view(dt).view(*shape)
        out = dict(d_out=view(off[0], R * d, torch.bfloat16, (R, d)),
                   d_gu=view(off[1], R * 2 * H, torch.bfloat16, (R, 2 * H)),
                   dx_perm=view(off[2], R * d, torch.bfloat16, (R, d)))
        if Hs:
            out["ds_gu"] = view(off[3], self.cfg.T * 2 * Hs, torch.bfloat16,
                                (self.cfg.T, 2 * Hs))
        return out

    def status(self) -> int:
        out = ctypes.c_int()
        check(self.lib.moe_get_status(c_void_p(self.ws.data_ptr()), _stream(),
                                      ctypes.byref(out)), "moe_get_status")
        return out.value


def to_device(inputs: dict, device="cuda") -> dict:
    """Copy the synth.make_inputs() CPU tensors to the device."""
    out = {}
    for k_, v in inputs.items():
        out[k_] = v.to(device) if hasattr(v, "to") and v is not None and k_ != "shape" else v
    return out
