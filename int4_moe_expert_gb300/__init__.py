"""Python binding of the GB300 int4 routed-MoE FFN library (libmoe_gb300.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/moe.h.  PyTorch supplies device
memory and streams.  There is no CPU fallback: if the library is not built,
loading fails loudly.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

import numpy as np

__all__ = [
    "MOE_OK", "MOE_ERR_INVALID", "MOE_ERR_CUDA", "MOE_ERR_NOMEM", "MOE_ERR_UNSUPPORTED",
    "MOE_FLAG_PRENORM_RESIDUAL", "MOE_FLAG_TRACE", "MOE_FLAG_CUDA_CORES", "MOE_SCORE_SIGMOID", "MOE_SCORE_SOFTMAX", "MOE_FORMAT_INT4", "MOE_FORMAT_INT8", "MOE_FORMAT_G64", "MOE_TRACE_SLOTS", "moe_trace_read", "MoeError", "MoeConfig", "MoeWeights", "MoeLayer",
    "lib", "library_path", "moe_init", "moe_forward", "moe_forward_debug", "moe_forward_host",
    "moe_destroy", "moe_last_error", "moe_workspace_bytes", "moe_abi_version",
    "moe_profile_start", "moe_profile_read", "moe_route_noalloc", "moe_device_error",
    "moe_debug_stall_next_call",
    "moe_debug_check",
    "moe_debug_set_topk",
    "moe_debug_check_result",
    "MOE_FLAG_DEBUG_CHECKS",
    "MOE_DEVICE_ERR_GRID",
    "MOE_DEVICE_ERR_CHECK",
    "MOE_DEVICE_ERR_TC",
    "moe_uses_streaming_decode", "moe_streaming_decode_max_tokens", "moe_uses_tensor_cores",
]

MOE_OK, MOE_ERR_INVALID, MOE_ERR_CUDA, MOE_ERR_NOMEM, MOE_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
MOE_FLAG_PRENORM_RESIDUAL = 1
MOE_FLAG_TRACE = 2
MOE_FLAG_CUDA_CORES = 4
MOE_FLAG_DEBUG_CHECKS = 8
MOE_DEVICE_ERR_GRID, MOE_DEVICE_ERR_CHECK, MOE_DEVICE_ERR_TC = 8, 16, 32
MOE_TRACE_SLOTS = 64
MOE_SCORE_SIGMOID, MOE_SCORE_SOFTMAX = 0, 1
MOE_FORMAT_INT4, MOE_FORMAT_INT8, MOE_FORMAT_G64 = 0, 1, 2
_STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_CUDA", 3: "MOE_ERR_NOMEM",
           4: "MOE_ERR_UNSUPPORTED"}

_PKG = Path(__file__).resolve().parent
_LIB_PATH = _PKG / "libmoe_gb300.so"
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)}: {msg}")
        self.status = status


class MoeConfig(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_experts", C.c_int32), ("top_k", C.c_int32),
                ("moe_inter", C.c_int32), ("n_shared", C.c_int32), ("shared_inter", C.c_int32),
                ("n_group", C.c_int32), ("norm_topk", C.c_int32), ("routed_scale", C.c_float),
                ("rms_eps", C.c_float), ("flags", C.c_uint32), ("topk_group", C.c_int32),
                ("score_func", C.c_int32), ("expert_format", C.c_int32), ("shared_format", C.c_int32),
                ("ep_size", C.c_int32), ("ep_rank", C.c_int32)]


class MoeWeights(C.Structure):
    _fields_ = [("router_w", C.c_void_p), ("router_bias", C.c_void_p),
                ("expert_slab", C.POINTER(C.c_void_p)), ("expert_scale", C.POINTER(C.c_void_p)),
                ("shared_slab", C.c_void_p), ("shared_scale", C.c_void_p)]


def library_path() -> Path:
    return _LIB_PATH


def lib():
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(str(_LIB_PATH))
        vp, i32 = C.c_void_p, C.c_int32
        L.moe_init.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights), i32, C.POINTER(vp)]
        L.moe_init.restype = C.c_int
        L.moe_forward.argtypes = [vp, vp, i32, vp, vp]
        L.moe_forward.restype = C.c_int
        L.moe_forward_debug.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
        L.moe_forward_debug.restype = C.c_int
        L.moe_forward_host.argtypes = [vp, vp, i32, vp, vp]
        L.moe_forward_host.restype = C.c_int
        L.moe_destroy.argtypes = [vp]
        L.moe_destroy.restype = C.c_int
        L.moe_last_error.restype = C.c_char_p
        L.moe_workspace_bytes.argtypes = [C.POINTER(MoeConfig), i32]
        L.moe_workspace_bytes.restype = C.c_size_t
        L.moe_abi_version.restype = i32
        L.moe_profile_start.argtypes = [vp, i32]
        L.moe_profile_start.restype = C.c_int
        L.moe_profile_read.argtypes = [vp, C.POINTER(i32), C.POINTER(C.c_float)]
        L.moe_profile_read.restype = C.c_int
        L.moe_device_error.argtypes = [vp, C.POINTER(C.c_uint32)]
        L.moe_device_error.restype = C.c_int
        L.moe_debug_stall_next_call.argtypes = [vp]
        L.moe_debug_stall_next_call.restype = C.c_int
        L.moe_debug_check.argtypes = [vp, C.c_int32]
        L.moe_debug_check.restype = C.c_int
        L.moe_debug_set_topk.argtypes = [vp, C.c_int32, C.c_int32]
        L.moe_debug_set_topk.restype = C.c_int
        L.moe_debug_check_result.argtypes = [vp, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
        L.moe_debug_check_result.restype = C.c_int
        L.moe_uses_streaming_decode.argtypes = [vp]
        L.moe_uses_streaming_decode.restype = i32
        L.moe_streaming_decode_max_tokens.argtypes = [vp]
        L.moe_streaming_decode_max_tokens.restype = i32
        L.moe_uses_tensor_cores.argtypes = [vp]
        L.moe_uses_tensor_cores.restype = i32
        L.moe_route_noalloc.argtypes = [C.POINTER(MoeConfig), vp, vp, vp, i32, vp, vp, vp]
        L.moe_route_noalloc.restype = C.c_int
        L.moe_trace_read.argtypes = [vp, vp, i32, C.POINTER(i32)]
        L.moe_trace_read.restype = C.c_int
        _lib = L
    return _lib


def moe_last_error() -> str:
    return lib().moe_last_error().decode(errors="replace")


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where, moe_last_error())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_workspace_bytes(cfg: MoeConfig, max_tokens: int) -> int:
    return lib().moe_workspace_bytes(C.byref(cfg), max_tokens)


def moe_init(cfg: MoeConfig, weights: MoeWeights, max_tokens: int) -> int:
    h = C.c_void_p()
    _check(lib().moe_init(C.byref(cfg), C.byref(weights), max_tokens, C.byref(h)), "moe_init")
    return h.value


def moe_forward(handle: int, x, T: int, y, stream=None) -> None:
    _check(lib().moe_forward(handle, _ptr(x), T, _ptr(y), _stream_handle(stream)), "moe_forward")


def moe_forward_debug(handle: int, x, T: int, y, topk_idx, topk_w, expert_counts=None,
                      stream=None) -> None:
    _check(lib().moe_forward_debug(handle, _ptr(x), T, _ptr(y), _ptr(topk_idx), _ptr(topk_w),
                                   _ptr(expert_counts), _stream_handle(stream)),
           "moe_forward_debug")


def moe_forward_host(handle: int, x_host, T: int, y_host, stream=None) -> None:
    _check(lib().moe_forward_host(handle, _ptr(x_host), T, _ptr(y_host), _stream_handle(stream)),
           "moe_forward_host")


MOE_PROFILE_STAGES = 4
PROFILE_STAGE_NAMES = ("router", "gate_up", "down", "combine")


def moe_profile_start(handle: int, max_calls: int) -> None:
    _check(lib().moe_profile_start(handle, max_calls), "moe_profile_start")


def moe_profile_read(handle: int):
    """-> (n_calls, {stage name: mean ms})"""
    n = C.c_int32()
    ms = (C.c_float * MOE_PROFILE_STAGES)()
    _check(lib().moe_profile_read(handle, C.byref(n), ms), "moe_profile_read")
    return n.value, dict(zip(PROFILE_STAGE_NAMES, list(ms)))


MOE_ROUTE_NOALLOC_MAX_TOKENS = 8
MOE_ROUTE_NOALLOC_MAX_EXPERTS = 1024


def moe_route_noalloc(cfg: MoeConfig, router_w, router_bias, x, T: int, topk_idx, topk_w,
                      stream=None) -> None:
    """Router + top-k without any device allocation by the library (its
    scratch is a fixed static device array); see moe.h.  All tensors are
    caller-owned device memory."""
    status = lib().moe_route_noalloc(C.byref(cfg), _ptr(router_w), _ptr(router_bias), _ptr(x), T,
                                     _ptr(topk_idx), _ptr(topk_w), _stream_handle(stream))
    if status != MOE_OK:
        raise MoeError(status, "moe_route_noalloc", "rejected (see moe.h for the limits)")


def moe_device_error(handle: int, check: bool = True) -> int:
    """Device error flags since the last check (0 = none); raises if any, unless
    check is False (the flags are then returned; the handle is reset either way)."""
    f = C.c_uint32()
    st = lib().moe_device_error(handle, C.byref(f))
    if check or st != MOE_ERR_CUDA or f.value == 0:
        _check(st, "moe_device_error")
    return f.value


def moe_debug_check(handle: int, T: int) -> None:
    """Run the routing/bucket checks over the handle's last call of T tokens."""
    _check(lib().moe_debug_check(handle, T), "moe_debug_check")


def moe_debug_set_topk(handle: int, pair: int, expert: int) -> None:
    """Overwrite one top-K index of the workspace (test hook for the checks)."""
    _check(lib().moe_debug_set_topk(handle, pair, expert), "moe_debug_set_topk")


def moe_debug_check_result(handle: int):
    """(failing pair, check code) of the last failed check, (-1, 0) if none."""
    pair, code = C.c_int32(0), C.c_int32(0)
    _check(lib().moe_debug_check_result(handle, C.byref(pair), C.byref(code)), "moe_debug_check_result")
    return pair.value, code.value


def moe_debug_stall_next_call(handle: int) -> None:
    """Make the next T == 1 call on the decode kernel time out (tests of the bounded waits)."""
    _check(lib().moe_debug_stall_next_call(handle), "moe_debug_stall_next_call")


def moe_uses_streaming_decode(handle: int) -> bool:
    return bool(lib().moe_uses_streaming_decode(handle))


def moe_streaming_decode_max_tokens(handle: int) -> int:
    """Calls of up to this many tokens run one single-kernel decode step per token (0: none)."""
    return int(lib().moe_streaming_decode_max_tokens(handle))


def moe_uses_tensor_cores(handle: int) -> bool:
    return bool(lib().moe_uses_tensor_cores(handle))


def moe_destroy(handle: int) -> None:
    _check(lib().moe_destroy(handle), "moe_destroy")


def make_config(H, E, K, I, n_shared=0, I_shared=0, routed_scale=1.0, norm_topk=1,
                prenorm_residual=False, rms_eps=1e-5, n_group=1, trace=False, topk_group=1,
                score_func=0, cuda_cores=False, expert_format=0, shared_format=0, ep_size=1,
                ep_rank=0, debug_checks=False) -> MoeConfig:
    flags = ((MOE_FLAG_PRENORM_RESIDUAL if prenorm_residual else 0) | (MOE_FLAG_TRACE if trace else 0) |
             (MOE_FLAG_CUDA_CORES if cuda_cores else 0) | (MOE_FLAG_DEBUG_CHECKS if debug_checks else 0))
    return MoeConfig(H, E, K, I, n_shared, I_shared if n_shared else 0, n_group, norm_topk,
                     float(routed_scale), float(rms_eps), flags, topk_group, score_func,
                     expert_format, shared_format, ep_size, ep_rank)


def moe_trace_read(handle: int, capacity_blocks: int = 1024):
    """Timeline of the last decode call (handle made with trace=True): a uint64
    numpy array [blocks, MOE_TRACE_SLOTS] of global-timer nanoseconds, 0 where
    a point was not reached (slot meanings in include/moe.h)."""
    out = np.zeros((capacity_blocks, MOE_TRACE_SLOTS), dtype=np.uint64)
    n = C.c_int32(0)
    _check(lib().moe_trace_read(handle, out.ctypes.data, capacity_blocks, C.byref(n)), "moe_trace_read")
    return out[:min(n.value, capacity_blocks)]


class MoeLayer:
    """One MoE layer resident on the current CUDA device.

    Uploads host arrays (router [E,H] f32, bias [E] f32, slabs [E, nbytes] u8,
    scales [E, 2I+H] f32, optional shared slab/scale) into device tensors it
    owns, and holds a library handle that borrows them.  expert_rows (optional)
    maps each expert to a row of slabs/scales, so experts may share storage; a
    None entry passes NULL for that expert (one another expert-parallel rank
    computes).
    """

    def __init__(self, cfg: MoeConfig, router_w, router_b, slabs, scales, sh_slab=None,
                 sh_scale=None, max_tokens: int = 1, device=None, expert_rows=None):
        import torch
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.cfg = cfg
        self.max_tokens = max_tokens

        def up(a, dtype):
            if a is None:
                return None
            if isinstance(a, torch.Tensor):
                return a.to(device=dev, dtype=dtype).contiguous()
            return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dtype)

        self.router_w = up(router_w, torch.float32)
        self.router_b = up(router_b, torch.float32)
        self.slabs = up(slabs, torch.uint8)
        self.scales = up(scales, torch.float32)
        self.sh_slab = up(sh_slab, torch.uint8)
        self.sh_scale = up(sh_scale, torch.float32)
        E = cfg.n_experts
        sp = self.slabs.data_ptr()
        cp = self.scales.data_ptr()
        sb = self.slabs.stride(0)
        cb = self.scales.stride(0) * 4
        rows = list(range(E)) if expert_rows is None else list(expert_rows)   # expert -> row
        self._slab_ptrs = (C.c_void_p * E)(*[None if r is None else sp + r * sb for r in rows])
        self._scale_ptrs = (C.c_void_p * E)(*[None if r is None else cp + r * cb for r in rows])
        self.weights = MoeWeights(_ptr(self.router_w), _ptr(self.router_b),
                                  C.cast(self._slab_ptrs, C.POINTER(C.c_void_p)),
                                  C.cast(self._scale_ptrs, C.POINTER(C.c_void_p)),
                                  _ptr(self.sh_slab), _ptr(self.sh_scale))
        self.handle = moe_init(cfg, self.weights, max_tokens)

    def forward(self, x, y=None, stream=None):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        moe_forward(self.handle, x, T, y, stream)
        return y

    def forward_debug(self, x, stream=None, counts=False):
        import torch
        T = x.shape[0]
        y = torch.empty_like(x)
        idx = torch.empty((T, self.cfg.top_k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.cfg.top_k), dtype=torch.float32, device=x.device)
        cnt = torch.empty(self.cfg.n_experts, dtype=torch.int32, device=x.device) if counts else None
        moe_forward_debug(self.handle, x, T, y, idx, w, cnt, stream)
        return (y, idx, w, cnt) if counts else (y, idx, w)

    def forward_host(self, x_host: np.ndarray, y_host: np.ndarray | None = None, stream=None):
        x_host = np.ascontiguousarray(x_host, dtype=np.float32)
        if y_host is None:
            y_host = np.empty_like(x_host)
        moe_forward_host(self.handle, x_host, x_host.shape[0], y_host, stream)
        return y_host

    def close(self):
        if getattr(self, "handle", None):
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
