"""CPU oracle for the int4 routed-MoE FFN step -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It wraps ``moe_oracle.c`` (plain C, double
precision) through ctypes; the GPU library never loads it and shares no code
with it.  Every function cites, in the C source, the page passage it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "moe_oracle.c"
_LIB_PATH = _HERE / "liboracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile the oracle with gcc (-O2, OpenMP over independent output rows)."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < max(
            _SRC.stat().st_mtime, (_HERE / "moe_oracle.h").stat().st_mtime):
        tmp = _LIB_PATH.with_suffix(".so.tmp%d" % os.getpid())
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Cfg(C.Structure):
    _fields_ = [("H", C.c_int), ("E", C.c_int), ("K", C.c_int), ("I", C.c_int),
                ("n_shared", C.c_int), ("I_shared", C.c_int), ("n_group", C.c_int),
                ("norm_topk", C.c_int), ("prenorm_residual", C.c_int),
                ("routed_scale", C.c_double), ("rms_eps", C.c_double),
                ("topk_group", C.c_int), ("score_func", C.c_int),
                ("expert_format", C.c_int), ("shared_format", C.c_int)]


SCORE_SIGMOID, SCORE_SOFTMAX = 0, 1
FORMAT_INT4, FORMAT_INT8, FORMAT_G64 = 0, 1, 2


class Layer(C.Structure):
    _fields_ = [("router_w", C.c_void_p), ("router_b", C.c_void_p),
                ("slab", C.POINTER(C.c_void_p)), ("scale", C.POINTER(C.c_void_p)),
                ("sh_slab", C.c_void_p), ("sh_scale", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(str(_LIB_PATH))
        vp, ip = C.c_void_p, C.c_int
        L.oracle_unpack_int4.argtypes = [vp, ip, vp]
        L.oracle_quantize_int4.argtypes = [vp, ip, ip, vp, vp]
        L.oracle_silu.argtypes = [C.c_double]
        L.oracle_silu.restype = C.c_double
        L.oracle_rmsnorm.argtypes = [vp, ip, C.c_double, vp]
        L.oracle_expert.argtypes = [ip, ip, vp, vp, vp, vp, vp]
        L.oracle_expert_fmt.argtypes = [ip, ip, ip, vp, vp, vp, vp, vp]
        L.oracle_quantize_int8.argtypes = [vp, ip, ip, vp, vp]
        L.oracle_route.argtypes = [C.POINTER(Cfg), vp, vp, vp, vp, vp, vp, vp]
        L.oracle_route.restype = ip
        L.oracle_weights_for.argtypes = [C.POINTER(Cfg), vp, vp, vp, vp]
        L.oracle_weights_for.restype = ip
        L.oracle_moe_token.argtypes = [C.POINTER(Cfg), C.POINTER(Layer), vp, vp, vp, vp, vp, vp]
        L.oracle_moe_token.restype = ip
        L.oracle_moe_forward.argtypes = [C.POINTER(Cfg), C.POINTER(Layer), vp, ip, vp, vp, vp, vp]
        L.oracle_moe_forward.restype = ip
        L.oracle_threads.restype = ip
        L.oracle_set_threads.argtypes = [ip]
        L.oracle_set_threads.restype = None
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def make_cfg(H, E, K, I, n_shared=0, I_shared=0, routed_scale=1.0, norm_topk=1,
             prenorm_residual=0, rms_eps=1e-5, n_group=1, topk_group=1,
             score_func=SCORE_SIGMOID, expert_format=FORMAT_INT4,
             shared_format=FORMAT_INT4) -> Cfg:
    return Cfg(H, E, K, I, n_shared, I_shared, n_group, norm_topk, prenorm_residual,
               float(routed_scale), float(rms_eps), topk_group, score_func, expert_format,
               shared_format)


def cfg_from_workload(wl) -> Cfg:
    return make_cfg(wl.H, wl.E, wl.K, wl.I, wl.n_shared, wl.I_shared, wl.routed_scale,
                    wl.norm_topk, int(wl.prenorm_residual), wl.rms_eps, wl.n_group,
                    wl.topk_group, wl.score_func, wl.expert_format, wl.shared_format)


def unpack_int4(row: np.ndarray, n: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    q = np.zeros(n, dtype=np.int32)
    lib().oracle_unpack_int4(_p(row), n, _p(q))
    return q


def quantize_int4(w: np.ndarray):
    w = np.ascontiguousarray(w, dtype=np.float32)
    O, I = w.shape
    q4 = np.zeros((O, (I + 1) // 2), dtype=np.uint8)
    s = np.zeros(O, dtype=np.float32)
    lib().oracle_quantize_int4(_p(w), O, I, _p(q4), _p(s))
    return q4, s


def quantize_int8(w: np.ndarray):
    w = np.ascontiguousarray(w, dtype=np.float32)
    O, I = w.shape
    q = np.zeros((O, I), dtype=np.int8)
    s = np.zeros(O, dtype=np.float32)
    lib().oracle_quantize_int8(_p(w), O, I, _p(q), _p(s))
    return q, s


def silu(v: float) -> float:
    return lib().oracle_silu(float(v))


def rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    lib().oracle_rmsnorm(_p(x), x.size, float(eps), _p(out))
    return out


def expert(H: int, I: int, slab: np.ndarray, scale: np.ndarray, x: np.ndarray,
           fmt: int = FORMAT_INT4):
    slab = np.ascontiguousarray(slab, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float64)
    d = np.zeros(H, dtype=np.float64)
    h = np.zeros(I, dtype=np.float64)
    lib().oracle_expert_fmt(H, I, int(fmt), _p(slab), _p(scale), _p(x), _p(d), _p(h))
    return d, h


def route(cfg: Cfg, router_w: np.ndarray, router_b: np.ndarray, x: np.ndarray):
    """Returns (idx[K], w[K], margin, scores[3, E])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    idx = np.zeros(cfg.K, dtype=np.int32)
    w = np.zeros(cfg.K, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    sc = np.zeros(3 * cfg.E, dtype=np.float64)
    rw = np.ascontiguousarray(router_w, dtype=np.float32)
    rb = np.ascontiguousarray(router_b, dtype=np.float32)
    rc = lib().oracle_route(C.byref(cfg), _p(rw), _p(rb), _p(x), _p(idx), _p(w), _p(m), _p(sc))
    if rc != 0:
        raise ValueError("oracle_route: invalid config")
    return idx, w, float(m[0]), sc.reshape(3, cfg.E)


def weights_for(cfg: Cfg, router_w: np.ndarray, x: np.ndarray, idx) -> np.ndarray:
    """Routing weights the oracle gives a given selection idx[K] of token x (its
    router input, already pre-normed where the layer asks for it)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    rw = np.ascontiguousarray(router_w, dtype=np.float32)
    ii = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.zeros(cfg.K, dtype=np.float64)
    rc = lib().oracle_weights_for(C.byref(cfg), _p(rw), _p(x), _p(ii), _p(w))
    if rc != 0:
        raise ValueError("oracle_weights_for: invalid config or selection")
    return w


class LayerRef:
    """Keeps the numpy arrays alive behind an oracle_layer struct."""

    def __init__(self, cfg: Cfg, router_w, router_b, slabs, scales, sh_slab=None, sh_scale=None):
        self.cfg = cfg
        self.router_w = np.ascontiguousarray(router_w, dtype=np.float32)
        self.router_b = np.ascontiguousarray(router_b, dtype=np.float32)
        self.slabs = [None if s is None else np.ascontiguousarray(s, dtype=np.uint8) for s in slabs]
        self.scales = [None if s is None else np.ascontiguousarray(s, dtype=np.float32) for s in scales]
        self.sh_slab = None if sh_slab is None else np.ascontiguousarray(sh_slab, dtype=np.uint8)
        self.sh_scale = None if sh_scale is None else np.ascontiguousarray(sh_scale, dtype=np.float32)
        E = cfg.E
        self._slab_ptrs = (C.c_void_p * E)(*[_p(s) for s in self.slabs])
        self._scale_ptrs = (C.c_void_p * E)(*[_p(s) for s in self.scales])
        self.struct = Layer(_p(self.router_w), _p(self.router_b),
                            C.cast(self._slab_ptrs, C.POINTER(C.c_void_p)),
                            C.cast(self._scale_ptrs, C.POINTER(C.c_void_p)),
                            _p(self.sh_slab), _p(self.sh_scale))

    @classmethod
    def from_inputs(cls, cfg: Cfg, li, experts=None):
        """From a synth.LayerInputs; ``experts`` limits which routed experts are visible."""
        ids = set(range(cfg.E)) if experts is None else set(int(e) for e in experts)
        slabs = [li.slabs[e] if e in ids else None for e in range(cfg.E)]
        scales = [li.scales[e] if e in ids else None for e in range(cfg.E)]
        return cls(cfg, li.router_w, li.router_b, slabs, scales, li.sh_slab, li.sh_scale)

    def token(self, x: np.ndarray, forced_idx=None):
        """One token -> (y[H] float64, idx[K], w[K], margin)."""
        cfg = self.cfg
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.zeros(cfg.H, dtype=np.float64)
        idx = np.zeros(cfg.K, dtype=np.int32)
        w = np.zeros(cfg.K, dtype=np.float64)
        m = np.zeros(1, dtype=np.float64)
        fi = None if forced_idx is None else np.ascontiguousarray(forced_idx, dtype=np.int32)
        rc = lib().oracle_moe_token(C.byref(cfg), C.byref(self.struct), _p(x), _p(fi),
                                    _p(y), _p(idx), _p(w), _p(m))
        if rc != 0:
            raise ValueError("oracle_moe_token failed (%d)" % rc)
        return y, idx, w, float(m[0])

    def forward(self, x: np.ndarray):
        """x[T, H] float32 -> (y[T,H] float64, idx[T,K], w[T,K], margin[T])."""
        cfg = self.cfg
        x = np.ascontiguousarray(x, dtype=np.float32)
        T = x.shape[0]
        y = np.zeros((T, cfg.H), dtype=np.float64)
        idx = np.zeros((T, cfg.K), dtype=np.int32)
        w = np.zeros((T, cfg.K), dtype=np.float64)
        m = np.zeros(T, dtype=np.float64)
        rc = lib().oracle_moe_forward(C.byref(cfg), C.byref(self.struct), _p(x), T,
                                      _p(y), _p(idx), _p(w), _p(m))
        if rc != 0:
            raise ValueError("oracle_moe_forward failed (%d)" % rc)
        return y, idx, w, m


def threads() -> int:
    return lib().oracle_threads()


def set_threads(n: int) -> None:
    """OpenMP threads of the following oracle calls (timing on one core)."""
    lib().oracle_set_threads(int(n))
