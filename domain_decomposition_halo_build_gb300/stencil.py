"""ctypes binding of the 2-D stencil halo workload of libhalo.so
(include/stencil.h), argument marshalling only: the exchange and the sweeps
run in the library's CUDA kernels; PyTorch provides device memory and streams.
No CPU fallback."""
from __future__ import annotations

import ctypes

from . import halo

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_P = ctypes.POINTER

SIGNATURES = {
    "stencil_setup": (ctypes.c_int, [_i32, _i32, _i32, _P(_vp)]),
    "stencil_layout": (ctypes.c_int, [_vp, _P(_i32), _P(_i32), _P(_i32), _P(_i64), _P(_i64)]),
    "stencil_exchange": (ctypes.c_int, [_vp, _vp, _vp]),
    "stencil_sweep": (ctypes.c_int, [_vp, _vp, _vp, _vp]),
    "stencil_sweep_fused": (ctypes.c_int, [_vp, _vp, _vp, _vp]),
    "stencil_iterate": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp]),
    "stencil_status": (ctypes.c_int, [_vp, _vp]),
    "stencil_destroy": (None, [_vp]),
}

_bound = False


def load_library():
    global _bound
    lib = halo.load_library()
    if not _bound:
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _bound = True
    return lib


class StencilPlan:
    """px x py blocks of n x n cells; fields are flat float32 CUDA tensors of
    ``total_floats`` elements in the layout of include/stencil.h."""

    def __init__(self, px: int, py: int, n: int):
        self._lib = load_library()
        h = _vp()
        halo._check(self._lib.stencil_setup(int(px), int(py), int(n), ctypes.byref(h)), "stencil_setup")
        self._h = h
        self.px, self.py, self.n = int(px), int(py), int(n)
        pitch, rows, col0 = _i32(), _i32(), _i32()
        tile, total = _i64(), _i64()
        halo._check(self._lib.stencil_layout(h, ctypes.byref(pitch), ctypes.byref(rows),
                                             ctypes.byref(col0), ctypes.byref(tile),
                                             ctypes.byref(total)), "stencil_layout")
        self.pitch, self.rows, self.col0 = pitch.value, rows.value, col0.value
        self.tile_floats, self.total_floats = tile.value, total.value

    def _field(self, t):
        import torch
        return halo._dev_ptr(t, torch.float32, (self.total_floats,))

    def empty(self, device="cuda"):
        import torch
        return torch.zeros(self.total_floats, dtype=torch.float32, device=device)

    def exchange(self, field, stream=None):
        halo._check(self._lib.stencil_exchange(self._h, self._field(field),
                                               halo._stream_handle(stream)), "stencil_exchange")

    def sweep(self, src, dst, stream=None):
        halo._check(self._lib.stencil_sweep(self._h, self._field(src), self._field(dst),
                                            halo._stream_handle(stream)), "stencil_sweep")

    def sweep_fused(self, src, dst, stream=None):
        halo._check(self._lib.stencil_sweep_fused(self._h, self._field(src), self._field(dst),
                                                  halo._stream_handle(stream)),
                    "stencil_sweep_fused")

    def iterate(self, a, b, iterations, stream=None):
        """stencil_iterate: `iterations` fused iterations in one launch; the
        result is in a (even count) or b (odd)."""
        halo._check(self._lib.stencil_iterate(self._h, self._field(a), self._field(b),
                                              int(iterations), halo._stream_handle(stream)),
                    "stencil_iterate")
        return a if iterations % 2 == 0 else b

    def status(self, stream=None) -> int:
        return self._lib.stencil_status(self._h, halo._stream_handle(stream))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.stencil_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
