"""Python binding of the NVFP4 routed-expert MoE layer library (libnvfp4moe.so).

The functions below carry the C ABI's names and only marshal arguments:
torch tensors become device pointers (``data_ptr()``), streams become
``cudaStream_t`` handles, and every step of the layer runs in the library's
CUDA kernels.  There is no fallback: if the library has not been built, the
import fails with an error that says so.

Layouts and the meaning of every argument are documented in include/moe.h.
"""
import ctypes
import os

import torch

from . import build as _build

_LIB = None

MOE_OK = 0
MOE_ERR_INVALID_ARGUMENT = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_OUT_OF_MEMORY = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_PARTIAL_OVERFLOW = 6

# every entry point declared in include/moe.h
EXPORTED = (
    "moe_status_string", "moe_workspace_bytes", "moe_packed_weight_bytes", "moe_layer_create",
    "moe_quantize_act", "moe_quantize_weights", "moe_forward", "moe_layer_status", "moe_destroy",
    "moe_layer_set_trace", "moe_kernel_launches", "moe_forward_noalloc", "moe_stack_forward",
    "moe_selftest_bounded_waits", "moe_layer_set_resident",
)

MOE_FLAG_MULTI_KERNEL = 1

# bytes of the device scratch array behind moe_forward_noalloc (include/moe.h)
MOE_NOALLOC_SCRATCH_BYTES = 4 << 20

MOE_STEP_NONE = 0
MOE_STEP_ROUTER = 1
MOE_STEP_QUANT = 3
MOE_STEP_PERMUTE = 4
MOE_STEP_GATEUP = 5
MOE_STEP_DOWN = 6


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class LayerDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("h_tensor_scale", ctypes.c_float), ("route_keep", ctypes.c_int32)]


class NVFP4(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p)]


class Debug(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("logits", "idx", "weights", "counts", "offsets", "perm", "inv", "hq", "hs",
                 "xq_codes", "xq_scales", "xq_tensor_scale", "phase_ns")]


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str = None) -> ctypes.CDLL:
    """Load the library (once).  Raises if it is missing: there is no fallback."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or lib_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with nvfp4_routed_expert_gb300.build.build() "
                          "(nvcc for sm_103a); the layer has no non-CUDA implementation")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    st = ctypes.c_int
    lib.moe_status_string.argtypes = [st]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_workspace_bytes.argtypes = [ctypes.POINTER(LayerDesc)]
    lib.moe_workspace_bytes.restype = sz
    lib.moe_packed_weight_bytes.argtypes = [ctypes.POINTER(LayerDesc)]
    lib.moe_packed_weight_bytes.restype = sz
    lib.moe_layer_create.argtypes = [ctypes.POINTER(LayerDesc), vp, vp, ctypes.POINTER(NVFP4),
                                     ctypes.POINTER(NVFP4), ctypes.POINTER(NVFP4), vp, vp,
                                     ctypes.POINTER(vp)]
    lib.moe_layer_create.restype = st
    lib.moe_quantize_act.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
    lib.moe_quantize_act.restype = st
    lib.moe_quantize_weights.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
    lib.moe_quantize_weights.restype = st
    lib.moe_forward.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, ctypes.POINTER(Debug), vp]
    lib.moe_forward.restype = st
    lib.moe_layer_status.argtypes = [vp, vp]
    lib.moe_layer_status.restype = st
    lib.moe_destroy.argtypes = [vp]
    lib.moe_destroy.restype = None
    lib.moe_layer_set_resident.argtypes = [vp, vp]
    lib.moe_layer_set_resident.restype = st
    lib.moe_layer_set_trace.argtypes = [vp, ctypes.c_int, vp, vp]
    lib.moe_layer_set_trace.restype = st
    lib.moe_kernel_launches.argtypes = []
    lib.moe_kernel_launches.restype = ctypes.c_uint64
    lib.moe_forward_noalloc.argtypes = [vp, vp, i32, vp, vp, vp, vp]
    lib.moe_forward_noalloc.restype = st
    lib.moe_stack_forward.argtypes = [ctypes.POINTER(vp), i32, vp, i32, vp, ctypes.POINTER(vp), vp,
                                      vp]
    lib.moe_stack_forward.restype = st
    lib.moe_selftest_bounded_waits.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.moe_selftest_bounded_waits.restype = st
    _LIB = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def make_desc(hidden, num_experts, top_k, inter, max_tokens, h_tensor_scale=2.0 ** -6, flags=0,
              route_keep=0):
    return LayerDesc(hidden, num_experts, top_k, inter, max_tokens, flags, h_tensor_scale, route_keep)


def moe_workspace_bytes(desc: LayerDesc) -> int:
    return load().moe_workspace_bytes(ctypes.byref(desc))


def moe_packed_weight_bytes(desc: LayerDesc) -> int:
    return load().moe_packed_weight_bytes(ctypes.byref(desc))


def moe_quantize_weights(w, codes, scales, tensor_scale, stream=None):
    """w fp32 [M][rows][cols] -> codes uint8 [M][rows][cols/2], scales [M][rows][cols/16],
    tensor_scale fp32 [M]."""
    m, rows, cols = w.shape
    _check(load().moe_quantize_weights(_ptr(w), m, rows, cols, _ptr(codes), _ptr(scales),
                                       _ptr(tensor_scale), _stream(stream)), "moe_quantize_weights")


def quantize_weights(w, stream=None):
    """Allocate and fill the NVFP4 form of fp32 weights [M][rows][cols]."""
    m, rows, cols = w.shape
    codes = torch.empty(m, rows, cols // 2, dtype=torch.uint8, device=w.device)
    scales = torch.empty(m, rows, cols // 16, dtype=torch.uint8, device=w.device)
    ts = torch.empty(m, dtype=torch.float32, device=w.device)
    moe_quantize_weights(w, codes, scales, ts, stream)
    return codes, scales, ts


class Layer:
    """Owns a moe_layer handle and the tensors it borrows."""

    def __init__(self, desc: LayerDesc, router_w, router_bias, gate, up, down, stream=None):
        self.desc = desc
        self._keep = (router_w, router_bias, gate, up, down)
        nv = [NVFP4(_ptr(c), _ptr(s), _ptr(t)) for (c, s, t) in (gate, up, down)]
        nbytes = moe_packed_weight_bytes(desc)
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=router_w.device) if nbytes else None
        handle = ctypes.c_void_p()
        _check(load().moe_layer_create(ctypes.byref(desc), _ptr(router_w), _ptr(router_bias),
                                       ctypes.byref(nv[0]), ctypes.byref(nv[1]), ctypes.byref(nv[2]),
                                       _ptr(self.packed), _stream(stream), ctypes.byref(handle)),
               "moe_layer_create")
        self.handle = handle

    def workspace(self, device=None):
        n = moe_workspace_bytes(self.desc)
        return torch.empty(n, dtype=torch.uint8, device=device or self._keep[0].device)

    def close(self):
        if self.handle:
            load().moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_layer_create(desc, router_w, router_bias, gate, up, down, stream=None) -> Layer:
    return Layer(desc, router_w, router_bias, gate, up, down, stream)


def moe_quantize_act(layer: Layer, x, codes, scales, tensor_scale, workspace, stream=None):
    _check(load().moe_quantize_act(layer.handle, _ptr(x), x.shape[0], _ptr(codes), _ptr(scales),
                                   _ptr(tensor_scale), _ptr(workspace), _stream(stream)),
           "moe_quantize_act")


def moe_forward(layer: Layer, x, y, workspace, xq=None, residual=None, x_next=None, debug=None,
                stream=None, tokens=None):
    """xq: None or (codes, scales, tensor_scale); debug: None or a dict of device tensors
    keyed like moe_debug."""
    dbg = None
    if debug is not None:
        dbg = Debug(*[_ptr(debug.get(n)) for n, _ in Debug._fields_])
    xc, xs, xt = xq if xq is not None else (None, None, None)
    n = x.shape[0] if tokens is None else tokens
    _check(load().moe_forward(layer.handle, _ptr(x), _ptr(xc), _ptr(xs), _ptr(xt), n,
                              _ptr(residual), _ptr(y), _ptr(x_next), _ptr(workspace),
                              ctypes.byref(dbg) if dbg is not None else None, _stream(stream)),
           "moe_forward")


def moe_forward_noalloc(layer: Layer, x, y, residual=None, x_next=None, stream=None,
                        tokens=None):
    """moe_forward without a workspace: the library's own device scratch array
    is used, so the call allocates nothing (see include/moe.h for its limits)."""
    n = x.shape[0] if tokens is None else tokens
    _check(load().moe_forward_noalloc(layer.handle, _ptr(x), n, _ptr(residual), _ptr(y),
                                      _ptr(x_next), _stream(stream)), "moe_forward_noalloc")


def moe_stack_forward(layers, x, x_out, workspace, ys=None, stream=None, tokens=None):
    """Decode (1..8 tokens) through a stack of layers in one kernel launch:
    x_{l+1} = bf16(x_l + y_l); `ys` is None or a list of fp32 [T][H] tensors
    (entries may be None) that receive each layer's y."""
    n = len(layers)
    handles = (ctypes.c_void_p * n)(*[l.handle.value for l in layers])
    y_arr = None
    if ys is not None:
        y_arr = (ctypes.c_void_p * n)(*[_ptr(y) for y in ys])
    t = x.shape[0] if tokens is None else tokens
    _check(load().moe_stack_forward(handles, n, _ptr(x), t, _ptr(x_out), y_arr, _ptr(workspace),
                                    _stream(stream)), "moe_stack_forward")


def moe_layer_set_resident(layer: Layer, resident):
    """Route-tail skip: the uint8 device tensor [E] of experts never skipped
    (nonzero = resident), or None; the tensor is kept alive with the layer."""
    layer._resident = resident
    _check(load().moe_layer_set_resident(layer.handle, _ptr(resident)), "moe_layer_set_resident")


def moe_layer_status(layer: Layer, stream=None) -> int:
    return load().moe_layer_status(layer.handle, _stream(stream))


def moe_layer_set_trace(layer: Layer, step: int, start_event=None, end_event=None):
    """Record torch.cuda.Event start/end around `step` in every later forward."""
    se = start_event.cuda_event if start_event is not None else None
    ee = end_event.cuda_event if end_event is not None else None
    _check(load().moe_layer_set_trace(layer.handle, step, se, ee), "moe_layer_set_trace")


MOE_SELFTEST_SCRATCH_BYTES = 8192


def moe_selftest_bounded_waits(scratch, stream=None):
    """Run the library's wait self-test (see include/moe.h); returns the two
    device status words; raises MoeError if the waits did not run out and report."""
    words = (ctypes.c_uint32 * 2)()
    _check(load().moe_selftest_bounded_waits(_ptr(scratch), words, _stream(stream)),
           "moe_selftest_bounded_waits")
    return int(words[0]), int(words[1])


def moe_kernel_launches() -> int:
    return int(load().moe_kernel_launches())


def moe_destroy(layer: Layer):
    layer.close()
