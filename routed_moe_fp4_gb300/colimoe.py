"""Python binding of libcolimoe.so: the C ABI of include/colimoe.h under the same names.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels. torch
provides device memory and streams. There is no CPU fallback: if the library is missing or the
device is not a GB300, the calls raise.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libcolimoe.so")

COLI_OK = 0
COLI_ERR_INVALID_ARG = -1
COLI_ERR_UNSUPPORTED_ARCH = -2
COLI_ERR_OUT_OF_MEMORY = -3
COLI_ERR_CUDA = -4
COLI_FFN_AUTO, COLI_FFN_GEMV, COLI_FFN_GEMM_MXF4 = 0, 1, 2
COLI_DENSE_AUTO, COLI_DENSE_CUDA_CORES, COLI_DENSE_TENSOR = 0, 1, 2

EXPORTED = ("coli_moe_create", "coli_moe_forward", "coli_moe_forward_host", "coli_moe_destroy",
            "coli_moe_last_error", "coli_moe_set_ffn_path", "coli_moe_debug_routing",
            "coli_moe_last_launch_count", "coli_moe_last_ffn_path", "coli_moe_set_profiling", "coli_moe_stage_times",
            "coli_moe_device_error", "coli_moe_set_wait_limit", "coli_moe_route_static",
            "coli_bank_create", "coli_bank_destroy", "coli_moe_forward_banked", "coli_bank_set_copy_blocks",
            "coli_bank_state", "coli_dense_create", "coli_dense_forward", "coli_dense_destroy",
            "coli_dense_last_error", "coli_dense_device_error", "coli_dense_set_path", "coli_dense_last_path",
            "coli_moe_forward_nvfp4", "coli_moe_test_alloc_failure")
COLI_STAGES = 5
STAGE_NAMES = ("router", "permute", "ffn_gate_up", "ffn_down", "combine")


class coli_moe_config(C.Structure):
    _fields_ = [("num_experts", C.c_int32), ("hidden", C.c_int32), ("inter", C.c_int32),
                ("shared_inter", C.c_int32), ("max_tokens", C.c_int32), ("max_top_k", C.c_int32)]


class coli_mxfp4_experts(C.Structure):
    _fields_ = [("gate_up_codes", C.c_void_p), ("gate_up_scales", C.c_void_p),
                ("down_codes", C.c_void_p), ("down_scales", C.c_void_p)]


class coli_nvfp4_experts(C.Structure):
    _fields_ = [("gate_up_codes", C.c_void_p), ("gate_up_scales", C.c_void_p), ("gate_up_global", C.c_void_p),
                ("down_codes", C.c_void_p), ("down_scales", C.c_void_p), ("down_global", C.c_void_p)]


class coli_moe_routing(C.Structure):
    _fields_ = [("scores", C.c_void_p), ("idx", C.c_void_p), ("weights", C.c_void_p), ("cnt", C.c_void_p),
                ("off", C.c_void_p), ("src_token", C.c_void_p), ("inv_row", C.c_void_p)]


class ColiError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"colimoe error {code}: {msg}")
        self.code = code


_lib: Optional[C.CDLL] = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Loads the library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m routed_moe_fp4_gb300.build` "
                           "(nvcc, sm_103a); there is no fallback implementation")
    lib = C.CDLL(path)
    vp = C.c_void_p
    lib.coli_moe_create.argtypes = [C.POINTER(coli_moe_config), vp, C.POINTER(vp)]
    lib.coli_moe_create.restype = C.c_int
    fwd_args = [vp, vp, C.c_int32, vp, vp, C.POINTER(coli_mxfp4_experts), C.POINTER(coli_mxfp4_experts),
                C.c_int32, vp]
    lib.coli_moe_forward.argtypes = fwd_args
    lib.coli_moe_forward.restype = C.c_int
    lib.coli_moe_forward_host.argtypes = fwd_args
    lib.coli_moe_forward_host.restype = C.c_int
    lib.coli_moe_destroy.argtypes = [vp]
    lib.coli_moe_destroy.restype = None
    lib.coli_moe_last_error.argtypes = [vp]
    lib.coli_moe_last_error.restype = C.c_char_p
    lib.coli_moe_set_ffn_path.argtypes = [vp, C.c_int32]
    lib.coli_moe_set_ffn_path.restype = C.c_int
    lib.coli_moe_debug_routing.argtypes = [vp, C.POINTER(coli_moe_routing)]
    lib.coli_moe_debug_routing.restype = C.c_int
    lib.coli_moe_last_launch_count.argtypes = [vp]
    lib.coli_moe_last_launch_count.restype = C.c_int32
    lib.coli_moe_last_ffn_path.argtypes = [vp]
    lib.coli_moe_last_ffn_path.restype = C.c_int32
    lib.coli_moe_set_wait_limit.argtypes = [vp, C.c_int64]
    lib.coli_moe_set_wait_limit.restype = C.c_int
    lib.coli_moe_set_profiling.argtypes = [vp, C.c_int32]
    lib.coli_moe_set_profiling.restype = C.c_int
    lib.coli_moe_stage_times.argtypes = [vp, C.POINTER(C.c_float)]
    lib.coli_moe_stage_times.restype = C.c_int
    lib.coli_moe_device_error.argtypes = [vp, C.POINTER(C.c_int32)]
    lib.coli_moe_device_error.restype = C.c_int
    lib.coli_moe_route_static.argtypes = [vp, C.c_int32, C.c_int32, vp, vp, C.c_int32, C.c_int32, vp, vp, vp]
    lib.coli_moe_route_static.restype = C.c_int
    lib.coli_bank_create.argtypes = [vp, C.c_int32, C.POINTER(coli_mxfp4_experts), C.POINTER(vp)]
    lib.coli_bank_create.restype = C.c_int
    lib.coli_bank_destroy.argtypes = [vp]
    lib.coli_bank_destroy.restype = None
    lib.coli_moe_forward_banked.argtypes = [vp, vp, vp, C.c_int32, vp, vp, C.POINTER(coli_mxfp4_experts),
                                            C.c_int32, vp]
    lib.coli_moe_forward_banked.restype = C.c_int
    lib.coli_bank_set_copy_blocks.argtypes = [vp, C.c_int32]
    lib.coli_bank_set_copy_blocks.restype = C.c_int
    lib.coli_bank_state.argtypes = [vp, vp, vp, vp, vp, vp]
    lib.coli_bank_state.restype = C.c_int
    lib.coli_moe_forward_nvfp4.argtypes = [vp, vp, C.c_int32, vp, vp, C.POINTER(coli_nvfp4_experts),
                                           C.POINTER(coli_nvfp4_experts), C.c_int32, vp]
    lib.coli_moe_forward_nvfp4.restype = C.c_int
    lib.coli_dense_create.argtypes = [C.c_int32, C.c_int32, vp, C.POINTER(vp)]
    lib.coli_dense_create.restype = C.c_int
    lib.coli_dense_forward.argtypes = [vp, vp, C.c_int32, C.c_int32, vp, vp, C.c_int32, vp]
    lib.coli_dense_forward.restype = C.c_int
    lib.coli_dense_destroy.argtypes = [vp]
    lib.coli_dense_destroy.restype = None
    lib.coli_dense_last_error.argtypes = [vp]
    lib.coli_dense_last_error.restype = C.c_char_p
    lib.coli_dense_device_error.argtypes = [vp, C.POINTER(C.c_int32)]
    lib.coli_dense_device_error.restype = C.c_int
    lib.coli_dense_set_path.argtypes = [vp, C.c_int32]
    lib.coli_dense_set_path.restype = C.c_int
    lib.coli_dense_last_path.argtypes = [vp]
    lib.coli_dense_last_path.restype = C.c_int
    lib.coli_moe_test_alloc_failure.argtypes = [C.POINTER(coli_moe_config), C.c_int32, C.POINTER(C.c_int32),
                                                C.POINTER(C.c_int32)]
    lib.coli_moe_test_alloc_failure.restype = C.c_int
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    """Device/host address of a torch tensor, numpy array or int (None stays None). The library
    reads every array as dense rows, so a strided view is refused rather than misread."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("the library takes contiguous row-major tensors; pass .contiguous()")
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        if not t.flags["C_CONTIGUOUS"]:
            raise ValueError("the library takes C-contiguous arrays; pass np.ascontiguousarray(a)")
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _check(h, rc: int) -> int:
    if rc != COLI_OK:
        raise ColiError(rc, coli_moe_last_error(h))
    return rc


# ---- the ABI under its own names --------------------------------------------------------

def coli_moe_last_error(h=None) -> str:
    return load().coli_moe_last_error(h).decode()


def coli_moe_create(cfg: coli_moe_config, cuda_stream=None) -> C.c_void_p:
    """cuda_stream: a torch.cuda.Stream, a raw cudaStream_t int, or None (default stream)."""
    lib = load()
    st = getattr(cuda_stream, "cuda_stream", cuda_stream)
    out = C.c_void_p()
    rc = lib.coli_moe_create(C.byref(cfg), st, C.byref(out))
    _check(None, rc)
    return out


def coli_moe_forward(h, x_bf16, T: int, router_w, router_bias, packed_experts: coli_mxfp4_experts,
                     shared_expert: Optional[coli_mxfp4_experts], top_k: int, out_bf16) -> int:
    rc = load().coli_moe_forward(h, _ptr(x_bf16), T, _ptr(router_w), _ptr(router_bias), C.byref(packed_experts),
                                 C.byref(shared_expert) if shared_expert is not None else None, top_k,
                                 _ptr(out_bf16))
    return _check(h, rc)


def coli_moe_forward_host(h, x_bf16_host, T: int, router_w, router_bias, packed_experts: coli_mxfp4_experts,
                          shared_expert: Optional[coli_mxfp4_experts], top_k: int, out_bf16_host) -> int:
    rc = load().coli_moe_forward_host(h, _ptr(x_bf16_host), T, _ptr(router_w), _ptr(router_bias),
                                      C.byref(packed_experts),
                                      C.byref(shared_expert) if shared_expert is not None else None, top_k,
                                      _ptr(out_bf16_host))
    return _check(h, rc)


def coli_moe_destroy(h) -> None:
    load().coli_moe_destroy(h)


def coli_moe_set_ffn_path(h, path: int) -> int:
    return _check(h, load().coli_moe_set_ffn_path(h, path))


def coli_moe_debug_routing(h, dst: coli_moe_routing) -> int:
    return _check(h, load().coli_moe_debug_routing(h, C.byref(dst)))


def coli_moe_last_launch_count(h) -> int:
    return load().coli_moe_last_launch_count(h)


def coli_moe_last_ffn_path(h) -> int:
    return load().coli_moe_last_ffn_path(h)


def coli_moe_set_wait_limit(h, ns: int) -> int:
    return _check(h, load().coli_moe_set_wait_limit(h, ns))


def coli_moe_set_profiling(h, enable: bool) -> int:
    return _check(h, load().coli_moe_set_profiling(h, int(bool(enable))))


def coli_moe_device_error(h) -> int:
    """Device error code of the forwards since the last call (0 = none); clears it."""
    code = C.c_int32()
    _check(h, load().coli_moe_device_error(h, C.byref(code)))
    return code.value


def coli_moe_stage_times(h) -> dict:
    """Stage durations (ms) of the last profiled forward, by stage name."""
    buf = (C.c_float * COLI_STAGES)()
    _check(h, load().coli_moe_stage_times(h, buf))
    return dict(zip(STAGE_NAMES, [float(v) for v in buf]))


def coli_moe_test_alloc_failure(cfg: coli_moe_config, fail_at: int):
    """Runs create's workspace allocation on a host allocator failing at allocation `fail_at`;
    returns (return code, allocations attempted, blocks still allocated after the cleanup)."""
    n, live = C.c_int32(0), C.c_int32(0)
    rc = load().coli_moe_test_alloc_failure(C.byref(cfg), fail_at, C.byref(n), C.byref(live))
    return rc, n.value, live.value


def coli_moe_route_static(x_bf16, T: int, H: int, router_w, router_bias, E: int, top_k: int, idx_out,
                          weights_out, cuda_stream=None) -> int:
    """Routing into caller buffers with no device allocation (see include/colimoe.h)."""
    st = getattr(cuda_stream, "cuda_stream", cuda_stream)
    rc = load().coli_moe_route_static(_ptr(x_bf16), T, H, _ptr(router_w), _ptr(router_bias), E, top_k,
                                      _ptr(idx_out), _ptr(weights_out), st)
    return _check(None, rc)


def coli_bank_create(h, slots: int, host_experts: coli_mxfp4_experts) -> C.c_void_p:
    out = C.c_void_p()
    _check(h, load().coli_bank_create(h, slots, C.byref(host_experts), C.byref(out)))
    return out


def coli_bank_destroy(bank) -> None:
    load().coli_bank_destroy(bank)


def coli_moe_forward_banked(h, bank, x_bf16, T: int, router_w, router_bias,
                            shared_expert: Optional[coli_mxfp4_experts], top_k: int, out_bf16) -> int:
    sh = C.byref(shared_expert) if shared_expert is not None else None
    return _check(h, load().coli_moe_forward_banked(h, bank, _ptr(x_bf16), T, _ptr(router_w), _ptr(router_bias),
                                                    sh, top_k, _ptr(out_bf16)))


def coli_bank_set_copy_blocks(h, bank, blocks: int) -> int:
    return _check(h, load().coli_bank_set_copy_blocks(bank, blocks))


def coli_bank_state(h, bank, E: int, S: int) -> dict:
    """The bank's state as numpy arrays (synchronises the handle's stream)."""
    import numpy as np
    st = dict(slot_of=np.zeros(E, np.int32), expert_in=np.zeros(S, np.int32), usage=np.zeros(E, np.uint32),
              last_use=np.zeros(S, np.int32), stats=np.zeros(3, np.int64))
    _check(h, load().coli_bank_state(bank, *[st[k].ctypes.data for k in
                                            ("slot_of", "expert_in", "usage", "last_use", "stats")]))
    return st


# ---- convenience: device-resident inputs of a workload -----------------------------------

class DeviceExperts:
    """MXFP4 expert arrays copied to the device, with the struct the ABI takes."""

    def __init__(self, host, device="cuda"):
        import torch
        self.tensors = [torch.from_numpy(a).to(device) for a in
                        (host.gate_up_codes, host.gate_up_scales, host.down_codes, host.down_scales)]
        self.struct = coli_mxfp4_experts(*[t.data_ptr() for t in self.tensors])

    @property
    def nbytes(self) -> int:
        return sum(t.numel() for t in self.tensors)


class MoELayer:
    """A handle plus device copies of one workload's weights (router, experts, shared)."""

    def __init__(self, inputs, max_tokens: Optional[int] = None, stream=None, device="cuda"):
        import torch
        wl = inputs.workload
        self.wl = wl
        self.top_k = wl.top_k
        self.router_w = torch.from_numpy(inputs.router_w).to(device)
        self.router_b = None if inputs.router_b is None else torch.from_numpy(inputs.router_b).to(device)
        self.experts = DeviceExperts(inputs.experts, device)
        self.shared = DeviceExperts(inputs.shared, device) if inputs.shared is not None else None
        cfg = coli_moe_config(wl.E, wl.H, wl.I, wl.I_s if inputs.shared is not None else 0,
                              max_tokens or max(wl.T, 1), wl.top_k)
        self.stream = stream
        self.h = coli_moe_create(cfg, stream)

    def forward(self, x, out, T: Optional[int] = None) -> None:
        T = x.shape[0] if T is None else T
        coli_moe_forward(self.h, x, T, self.router_w, self.router_b, self.experts.struct,
                         self.shared.struct if self.shared is not None else None, self.top_k, out)

    def forward_host(self, x_host, out_host, T: Optional[int] = None) -> None:
        T = x_host.shape[0] if T is None else T
        coli_moe_forward_host(self.h, x_host, T, self.router_w, self.router_b, self.experts.struct,
                              self.shared.struct if self.shared is not None else None, self.top_k, out_host)

    def set_ffn_path(self, path: int) -> None:
        coli_moe_set_ffn_path(self.h, path)

    def routing(self, T: int):
        """Routing of the last forward as numpy arrays."""
        import numpy as np
        wl = self.wl
        k, E = self.top_k, wl.E
        rows = T * k + (T if self.shared is not None else 0)
        r = dict(scores=np.zeros((T, E), np.float32), idx=np.zeros((T, k), np.int32),
                 weights=np.zeros((T, k), np.float32), cnt=np.zeros(E + 1, np.int32),
                 off=np.zeros(E + 2, np.int32), src_token=np.zeros(rows, np.int32),
                 inv_row=np.zeros((T, k), np.int32))
        dst = coli_moe_routing(*[r[n].ctypes.data for n in
                                 ("scores", "idx", "weights", "cnt", "off", "src_token", "inv_row")])
        coli_moe_debug_routing(self.h, dst)
        return r

    def set_profiling(self, enable: bool) -> None:
        coli_moe_set_profiling(self.h, enable)

    def stage_times(self) -> dict:
        return coli_moe_stage_times(self.h)

    def device_error(self) -> int:
        return coli_moe_device_error(self.h)

    def launches(self) -> int:
        return coli_moe_last_launch_count(self.h)

    def set_wait_limit(self, ns: int) -> None:
        """Limit of the FP4 path's barrier waits in ns (0 = default); a test hook for the failure path."""
        coli_moe_set_wait_limit(self.h, ns)

    def ffn_path(self) -> int:
        """The FFN path the last forward ran (COLI_FFN_*)."""
        return coli_moe_last_ffn_path(self.h)

    def close(self) -> None:
        for b in list(getattr(self, "_banks", [])):
            b.close()
        if self.h:
            coli_moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def coli_moe_forward_nvfp4(h, x_bf16, T: int, router_w, router_bias, packed_experts: coli_nvfp4_experts,
                           shared_expert: Optional[coli_nvfp4_experts], top_k: int, out_bf16) -> int:
    sh = C.byref(shared_expert) if shared_expert is not None else None
    return _check(h, load().coli_moe_forward_nvfp4(h, _ptr(x_bf16), T, _ptr(router_w), _ptr(router_bias),
                                                   C.byref(packed_experts), sh, top_k, _ptr(out_bf16)))


class DeviceNvExperts:
    """NVFP4 expert arrays (synthetic.NVFP4Experts) copied to the device, with the ABI struct."""

    def __init__(self, host, device="cuda"):
        import torch
        self.tensors = [torch.from_numpy(a).to(device) for a in
                        (host.gate_up_codes, host.gate_up_scales, host.gate_up_global,
                         host.down_codes, host.down_scales, host.down_global)]
        self.struct = coli_nvfp4_experts(*[t.data_ptr() for t in self.tensors])


class NvMoELayer(MoELayer):
    """MoELayer over NVFP4 experts: forward() runs coli_moe_forward_nvfp4."""

    def __init__(self, inputs, max_tokens: Optional[int] = None, stream=None, device="cuda"):
        import torch
        wl = inputs.workload
        self.wl = wl
        self.top_k = wl.top_k
        self.router_w = torch.from_numpy(inputs.router_w).to(device)
        self.router_b = None if inputs.router_b is None else torch.from_numpy(inputs.router_b).to(device)
        self.experts = DeviceNvExperts(inputs.experts, device)
        self.shared = DeviceNvExperts(inputs.shared, device) if inputs.shared is not None else None
        cfg = coli_moe_config(wl.E, wl.H, wl.I, wl.I_s if inputs.shared is not None else 0,
                              max_tokens or max(wl.T, 1), wl.top_k)
        self.stream = stream
        self.h = coli_moe_create(cfg, stream)

    def forward(self, x, out, T: Optional[int] = None) -> None:
        T = x.shape[0] if T is None else T
        coli_moe_forward_nvfp4(self.h, x, T, self.router_w, self.router_b, self.experts.struct,
                               self.shared.struct if self.shared is not None else None, self.top_k, out)


class HostExperts:
    """MXFP4 expert arrays in page-locked host memory (the device reads them over the host link)."""

    def __init__(self, host):
        import torch
        self.tensors = [torch.from_numpy(a).pin_memory() for a in
                        (host.gate_up_codes, host.gate_up_scales, host.down_codes, host.down_scales)]
        self.struct = coli_mxfp4_experts(*[t.data_ptr() for t in self.tensors])


class ExpertBank:
    """A bank of device slots over a layer's experts held in page-locked host memory."""

    def __init__(self, layer: "MoELayer", slots: int, host_experts: HostExperts):
        self.layer, self.slots, self.host = layer, slots, host_experts
        self.b = coli_bank_create(layer.h, slots, host_experts.struct)
        if not hasattr(layer, "_banks"):
            layer._banks = []
        layer._banks.append(self)

    def forward(self, x, out, T: Optional[int] = None) -> None:
        L = self.layer
        T = x.shape[0] if T is None else T
        coli_moe_forward_banked(L.h, self.b, x, T, L.router_w, L.router_b,
                                L.shared.struct if L.shared is not None else None, L.top_k, out)

    def set_copy_blocks(self, blocks: int) -> None:
        coli_bank_set_copy_blocks(self.layer.h, self.b, blocks)

    def state(self) -> dict:
        return coli_bank_state(self.layer.h, self.b, self.layer.wl.E, self.slots)

    def close(self) -> None:
        if self.b:
            coli_bank_destroy(self.b)
            self.b = None
            self.layer._banks.remove(self)


# ---- FP8 dense projection -----------------------------------------------------------------

def coli_dense_last_error(d=None) -> str:
    return load().coli_dense_last_error(d).decode()


def _dcheck(d, rc: int) -> int:
    if rc != COLI_OK:
        raise ColiError(rc, coli_dense_last_error(d))
    return rc


def coli_dense_create(max_tokens: int, max_k: int, cuda_stream=None) -> C.c_void_p:
    st = getattr(cuda_stream, "cuda_stream", cuda_stream)
    out = C.c_void_p()
    _dcheck(None, load().coli_dense_create(max_tokens, max_k, st, C.byref(out)))
    return out


def coli_dense_forward(d, x_bf16, T: int, K: int, w_e4m3, w_scale, N: int, out_bf16) -> int:
    return _dcheck(d, load().coli_dense_forward(d, _ptr(x_bf16), T, K, _ptr(w_e4m3), _ptr(w_scale), N,
                                                _ptr(out_bf16)))


def coli_dense_destroy(d) -> None:
    load().coli_dense_destroy(d)


def coli_dense_device_error(d) -> int:
    code = C.c_int32(0)
    _dcheck(d, load().coli_dense_device_error(d, C.byref(code)))
    return code.value


def coli_dense_set_path(d, path: int) -> int:
    return _dcheck(d, load().coli_dense_set_path(d, path))


def coli_dense_last_path(d) -> int:
    return load().coli_dense_last_path(d)


class DenseLayer:
    """A dense handle plus device copies of one FP8 projection's weights (E4M3 codes, block scales)."""

    def __init__(self, inputs, max_tokens: Optional[int] = None, stream=None, device="cuda"):
        import torch
        wl = inputs.workload
        self.wl = wl
        self.w = torch.from_numpy(inputs.w).to(device)
        self.w_scale = torch.from_numpy(inputs.w_scale).to(device)
        self.stream = stream
        self.d = coli_dense_create(max_tokens or max(wl.T, 1), wl.K, stream)

    def forward(self, x, out, T: Optional[int] = None) -> None:
        T = x.shape[0] if T is None else T
        coli_dense_forward(self.d, x, T, self.wl.K, self.w, self.w_scale, self.wl.N, out)

    def set_path(self, path: int) -> None:
        coli_dense_set_path(self.d, path)

    def last_path(self) -> int:
        return coli_dense_last_path(self.d)

    def device_error(self) -> int:
        return coli_dense_device_error(self.d)

    def close(self) -> None:
        if self.d:
            coli_dense_destroy(self.d)
            self.d = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
