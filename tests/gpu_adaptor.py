"""Adaptor that gives a library plan (through the C ABI) the interface of
oracle.Oracle, so the same checks run on both.  Host numpy in, host numpy
out; the computation itself runs in libhalo.so's kernels."""
from __future__ import annotations

import numpy as np


class GpuPlan:
    def __init__(self, box, grid, rc, xyz, dom, device="cuda:0", prune=False):
        import torch
        from domain_decomposition_halo_build_gb300 import halo
        self.torch = torch
        self.device = device
        self.xyz_d = torch.from_numpy(np.ascontiguousarray(xyz, np.float32).reshape(-1, 3)).to(device)
        self.dom_d = torch.from_numpy(np.ascontiguousarray(dom, np.int32)).to(device)
        self.plan = halo.HaloPlan(box, grid, rc, self.xyz_d, self.dom_d, prune=prune)
        self.prune = bool(prune)
        p = self.plan
        self.box, self.grid, self.rc = p.box, p.grid, p.rc
        self._sync()

    def _sync(self):
        p = self.plan
        self.n_domains, self.n_pulses = p.n_domains, p.n_pulses
        self.pulses_per_dim, self.pulse_dim = p.pulses_per_dim, p.pulse_dim
        self.n_atoms, self.n_local_total = p.n_atoms, p.n_local_total
        self.base, self.n_home, self.n_local = p.base, p.n_home, p.n_local

    def rebuild(self, xyz, dom):
        torch = self.torch
        self.xyz_d = torch.from_numpy(np.ascontiguousarray(xyz, np.float32)).to(self.device)
        self.dom_d = torch.from_numpy(np.ascontiguousarray(dom, np.int32)).to(self.device)
        self.plan.rebuild(self.xyz_d, self.dom_d)
        self._sync()

    class _Info:
        def __init__(self, i):
            self.send_domain = i.send_domain
            self.recv_domain = i.recv_domain
            self.send_size = i.send_size
            self.split = i.split
            self.dep_offset = i.dep_offset
            self.atom_offset = i.atom_offset
            self.coord_shift = np.asarray(list(i.coord_shift), np.float32)

    def pulse(self, s, p):
        return self._Info(self.plan.pulse(s, p))

    def index_map(self, s, p):
        return self.plan.index_map(s, p)

    def local_to_global(self):
        out = self.plan.local_to_global()
        self.torch.cuda.synchronize()
        return out.cpu().numpy()

    def load_home(self, xyz):
        g = self.torch.from_numpy(np.ascontiguousarray(xyz, np.float32)).to(self.device)
        out = self.plan.load_home(g)
        self.torch.cuda.synchronize()
        return out.cpu().numpy()

    def local_coords(self):
        loc = self.plan.load_home(self.xyz_d)
        self.plan.exchange_x(loc)
        self.torch.cuda.synchronize()
        return loc.cpu().numpy()

    def exchange_x(self, local):
        t = self.torch.from_numpy(local).to(self.device)
        self.plan.exchange_x(t)
        self.check_status()
        local[...] = t.cpu().numpy()
        return local

    def exchange_f(self, local):
        t = self.torch.from_numpy(local).to(self.device)
        self.plan.exchange_f(t)
        self.check_status()
        local[...] = t.cpu().numpy()
        return local

    def check_status(self):
        code = self.plan.status()
        assert code == 0, "device error %d" % code

    def close(self):
        self.plan.close()
