"""CPU oracle for the eighth-shell halo exchange -- TEST INFRASTRUCTURE.

The oracle is a plain sequential C implementation (``halo_oracle.c``) of what
the halo build, the coordinate exchange and the force reduction compute, written
from the page "Redesigning GROMACS Halo Exchange: Improving Strong Scaling with
GPU-initiated NVSHMEM" (section 3 and Algorithms 1, 3, 4, 6).  It shares no
code with the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s ``cpu_baseline`` / ``--impl reference`` legs may import it; the
library itself never does.

Parity status of each function: every function is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (closed forms of the pulse structure, a direct
geometric construction of every domain's halo, brute-force pair coverage on
tiny inputs, hand-worked golden examples, exact force conservation and the
per-atom closed form with integer-valued forces) and by the planted-mistake
tests in ``tests/test_oracle_mutants.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "halo_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

OK, EINVAL, EPULSES, EDOMAIN, ENOMEM = 0, -1, -2, -3, -4

CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC"]


def build_oracle(src: str = SOURCE, out: str = LIBRARY, force: bool = False) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc (plain C11).

    With OpenMP where the compiler has it (only the optional host threads of
    the two exchanges use it); without, the same source builds sequential."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    r = subprocess.run(["gcc", *CFLAGS, "-fopenmp", "-o", tmp, src, "-lm"], capture_output=True)
    if r.returncode != 0:
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__("oracle_setup failed with code %d" % code)
        self.code = code


def _f32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _i32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _i64p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _bind(lib):
    vp = ctypes.c_void_p
    lib.oracle_setup.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int),
                                 ctypes.c_float, ctypes.POINTER(ctypes.c_float),
                                 ctypes.POINTER(ctypes.c_int32), ctypes.c_int64,
                                 ctypes.POINTER(vp)]
    lib.oracle_setup.restype = ctypes.c_int
    lib.oracle_setup_ex.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int),
                                    ctypes.c_float, ctypes.POINTER(ctypes.c_float),
                                    ctypes.POINTER(ctypes.c_int32), ctypes.c_int64, ctypes.c_int,
                                    ctypes.POINTER(vp)]
    lib.oracle_setup_ex.restype = ctypes.c_int
    lib.oracle_free.argtypes = [vp]
    lib.oracle_free.restype = None
    lib.oracle_num_domains.argtypes = [vp]
    lib.oracle_num_domains.restype = ctypes.c_int
    lib.oracle_num_pulses.argtypes = [vp]
    lib.oracle_num_pulses.restype = ctypes.c_int
    lib.oracle_pulses.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    lib.oracle_pulses.restype = None
    lib.oracle_n_local_total.argtypes = [vp]
    lib.oracle_n_local_total.restype = ctypes.c_int64
    lib.oracle_layout.argtypes = [vp, ctypes.POINTER(ctypes.c_int64),
                                  ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    lib.oracle_layout.restype = None
    lib.oracle_pulse_info.argtypes = [vp, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_float)]
    lib.oracle_pulse_info.restype = ctypes.c_int
    lib.oracle_index_map.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]
    lib.oracle_index_map.restype = ctypes.c_int
    for name in ("oracle_local_coords", "oracle_exchange_x", "oracle_exchange_f"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, ctypes.POINTER(ctypes.c_float)]
        fn.restype = None
    lib.oracle_set_threads.argtypes = [vp, ctypes.c_int]
    lib.oracle_set_threads.restype = None
    lib.oracle_openmp.argtypes = []
    lib.oracle_openmp.restype = ctypes.c_int
    lib.oracle_local_to_global.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.oracle_local_to_global.restype = None
    lib.oracle_load_home.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    lib.oracle_load_home.restype = None
    return lib


_LIBS: dict = {}


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library at ``path``."""
    if path is None:
        path = build_oracle()
    path = os.path.abspath(path)
    if path not in _LIBS:
        _LIBS[path] = _bind(ctypes.CDLL(path))
    return _LIBS[path]


@dataclass
class PulseInfo:
    send_domain: int
    recv_domain: int
    send_size: int
    split: int
    dep_offset: int
    atom_offset: int
    coord_shift: np.ndarray


class Oracle:
    """One oracle plan: the setup result plus the two exchanges.

    All arrays use the dense local layout: domain D's slots start at
    ``base[D]`` and hold ``[home atoms in input order | halo of pulse 0 |
    ... | halo of pulse P-1]``.
    """

    def __init__(self, box, grid, rc, xyz, dom, lib=None, prune=False):
        """``prune``: keep a forwarded candidate only if it lies within rc of
        the receiver's home box over all dims where it is beyond it (corner
        pruning; off by default, the page's one-dimensional slabs)."""
        self.lib = lib if lib is not None else load()
        self.prune = bool(prune)
        self.box = np.ascontiguousarray(box, dtype=np.float32)
        self.grid = np.ascontiguousarray(grid, dtype=np.int32)
        self.rc = float(np.float32(rc))
        xyz = np.ascontiguousarray(xyz, dtype=np.float32).reshape(-1, 3)
        dom = np.ascontiguousarray(dom, dtype=np.int32)
        self.n_atoms = xyz.shape[0]
        h = ctypes.c_void_p()
        code = self.lib.oracle_setup_ex(_f32p(self.box), self.grid.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                        ctypes.c_float(self.rc), _f32p(xyz), _i32p(dom),
                                        ctypes.c_int64(self.n_atoms), 1 if self.prune else 0,
                                        ctypes.byref(h))
        if code != OK:
            raise OracleError(code)
        self._h = h
        self.n_domains = self.lib.oracle_num_domains(h)
        self.n_pulses = self.lib.oracle_num_pulses(h)
        per_dim = np.zeros(3, np.int32)
        dims = np.zeros(max(self.n_pulses, 1), np.int32)
        self.lib.oracle_pulses(h, _i32p(per_dim), _i32p(dims))
        self.pulses_per_dim = per_dim
        self.pulse_dim = dims[: self.n_pulses].copy()
        self.n_local_total = int(self.lib.oracle_n_local_total(h))
        self.base = np.zeros(self.n_domains, np.int64)
        self.n_home = np.zeros(self.n_domains, np.int32)
        self.n_local = np.zeros(self.n_domains, np.int32)
        self.lib.oracle_layout(h, _i64p(self.base), _i32p(self.n_home), _i32p(self.n_local))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self.lib.oracle_free(h)
            self._h = None

    # -- plan queries ----------------------------------------------------------
    def pulse(self, s: int, p: int) -> PulseInfo:
        info = np.zeros(6, np.int32)
        shift = np.zeros(3, np.float32)
        if self.lib.oracle_pulse_info(self._h, s, p, _i32p(info), _f32p(shift)) != OK:
            raise IndexError((s, p))
        return PulseInfo(*[int(v) for v in info], shift)

    def index_map(self, s: int, p: int) -> np.ndarray:
        n = self.pulse(s, p).send_size
        out = np.zeros(max(n, 1), np.int32)
        self.lib.oracle_index_map(self._h, s, p, _i32p(out))
        return out[:n].copy()

    def local_coords(self) -> np.ndarray:
        out = np.zeros((self.n_local_total, 3), np.float32)
        self.lib.oracle_local_coords(self._h, _f32p(out))
        return out

    def local_to_global(self) -> np.ndarray:
        out = np.zeros(self.n_local_total, np.int32)
        self.lib.oracle_local_to_global(self._h, _i32p(out))
        return out

    def load_home(self, global_xyz) -> np.ndarray:
        g = np.ascontiguousarray(global_xyz, dtype=np.float32).reshape(-1, 3)
        out = np.zeros((self.n_local_total, 3), np.float32)
        self.lib.oracle_load_home(self._h, _f32p(g), _f32p(out))
        return out

    # -- exchanges (in place on a dense local array) ----------------------------
    def set_threads(self, threads: int) -> None:
        """Run the senders of each pulse on ``threads`` OpenMP threads (1: none)."""
        self.lib.oracle_set_threads(self._h, int(threads))

    @property
    def openmp(self) -> bool:
        """Whether this oracle build has OpenMP (else set_threads has no effect)."""
        return bool(self.lib.oracle_openmp())

    def exchange_x(self, local: np.ndarray) -> np.ndarray:
        assert local.dtype == np.float32 and local.flags.c_contiguous
        assert local.shape == (self.n_local_total, 3)
        self.lib.oracle_exchange_x(self._h, _f32p(local))
        return local

    def exchange_f(self, local: np.ndarray) -> np.ndarray:
        assert local.dtype == np.float32 and local.flags.c_contiguous
        assert local.shape == (self.n_local_total, 3)
        self.lib.oracle_exchange_f(self._h, _f32p(local))
        return local
