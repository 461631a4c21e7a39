"""Run by tests/test_gpu_debug_build.py in a child process whose HALO_LIBRARY
points at the bounds-checking build: every mode's exchanges (and the home
copies) on several systems, with and without corner pruning, must report no
HALO_EBOUNDS and still match the oracle bit for bit."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from domain_decomposition_halo_build_gb300 import halo, synth  # noqa: E402
from gpu_adaptor import GpuPlan  # noqa: E402


def bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def main():
    import torch
    assert halo.LIBRARY.endswith("libhalo_debug.so"), halo.LIBRARY
    problems = [synth.WORKLOADS[n] for n in ("water24k_2x4x8", "water48k_2x2x2", "water1M_4x4x4")]
    checked = 0
    for w in problems:
        xyz, dom = synth.system(w)
        for prune in (False, True):
            o = oracle.Oracle(w.box, w.grid, w.rc, xyz, dom, prune=prune)
            g = GpuPlan(w.box, w.grid, w.rc, xyz, dom, prune=prune)
            want_x = o.load_home(xyz)
            o.exchange_x(want_x)
            f0 = synth.forces(o.n_local_total, seed=3)
            want_f = f0.copy()
            o.exchange_f(want_f)
            for mode in ("fused", "stepwise", "flat", "staged"):
                g.plan.set_mode(mode)
                loc = g.plan.load_home(g.xyz_d)
                g.plan.exchange_x(loc)
                f = torch.from_numpy(f0).cuda()
                g.plan.exchange_f(f)
                back = g.plan.store_home(f)
                code = g.plan.status()
                assert code == halo.OK, (w.name, prune, mode, code)
                assert np.array_equal(bits(loc.cpu().numpy()), bits(want_x)), (w.name, prune, mode)
                assert np.array_equal(bits(f.cpu().numpy()), bits(want_f)), (w.name, prune, mode)
                assert back.shape == (w.n_atoms, 3)
                checked += 1
            g.close()
    print("debug build ok: %d plan/mode combinations" % checked)


if __name__ == "__main__":
    main()
