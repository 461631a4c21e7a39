"""Planted mistakes: each mutant is the oracle with one plausible error
(wrong direction, sign, index, order, bound ...), compiled on the CPU.  The
pins of tests/pins.py must reject every one of them; a mutant they accept
would mean the pins cannot tell that mistake from the right answer."""
import os
import tempfile

import pytest

import oracle
import pins
from domain_decomposition_halo_build_gb300 import synth

MUTANTS = {
    "direction_reversed": (
        "rc3[d] = (c[d] - 1 + o->grid[d]) % o->grid[d];",
        "rc3[d] = (c[d] + 1) % o->grid[d];"),
    "shift_sign": (
        "o->shift[3 * sp + d] = box[d];",
        "o->shift[3 * sp + d] = -box[d];"),
    "shift_on_top_sender": (
        "if (c[d] == 0) o->shift[3 * sp + d]",
        "if (c[d] == o->grid[d] - 1) o->shift[3 * sp + d]"),
    "threshold_upper_face": (
        "(double)c[d] * (double)box[d] /",
        "(double)(c[d] + 1) * (double)box[d] /"),
    "threshold_without_cutoff_rounding": (
        "(double)rc);",
        "(double)rc * 0.999);"),
    "forwarded_pulse_takes_all": (
        "cand_lo[s] = (k == 0) ? 0 : prev_start[s];",
        "cand_lo[s] = 0;"),
    "first_pulse_home_only": (
        "cand_hi[s] = (int32_t)o->xyz[s].n;",
        "cand_hi[s] = (k == 0) ? o->n_home[s] : (int32_t)o->xyz[s].n;"),
    "predicate_not_strict": (
        "if (o->xyz[s].v[3 * (int64_t)i + d] < thr &&",
        "if (o->xyz[s].v[3 * (int64_t)i + d] <= thr &&"),
    "split_off_by_one": (
        "if (m->v[j] < o->n_home[s]) nsplit++;",
        "if (m->v[j] <= o->n_home[s]) nsplit++;"),
    "pulse_order_xyz": (
        "for (int d = 2; d >= 0; d--) {",
        "for (int d = 0; d < 3; d++) {"),
    "pulse_count_floor": (
        "p = (int)ceil((double)rc / w);",
        "p = (int)floor((double)rc / w); if (p < 1) p = 1;"),
    "exchange_x_drops_shift": (
        "dst[3 * i + e] = src[3 * (int64_t)m->v[i] + e] + sh[e];",
        "dst[3 * i + e] = src[3 * (int64_t)m->v[i] + e];"),
    "forces_forward_order": (
        "for (int p = P - 1; p >= 0; p--)",
        "for (int p = 0; p < P; p++)"),
    "forces_reversed_pairing": (
        "own[3 * (int64_t)m->v[i] + e] + halo[3 * i + e];",
        "own[3 * (int64_t)m->v[i] + e] + halo[3 * (m->n - 1 - i) + e];"),
    "forces_wrong_halo_slice": (
        "const float *halo = local + 3 * (o->base[r] + o->atom_offset[sp]);",
        "const float *halo = local + 3 * (o->base[r] + o->n_home[r]);"),
    "corner_distance_from_upper_face": (
        "const double lo_d = (double)c[d] * (double)o->box[d] / (double)o->grid[d];",
        "const double lo_d = (double)(c[d] + 1) * (double)o->box[d] / (double)o->grid[d];"),
    "corner_ignores_path_dims": (
        "r2 = r2 + u * u;",
        "r2 = r2 + 0.0 * u * u;"),
    "corner_path_dims_lower_face": (
        "const double hi_e = (double)(c[e] + 1) * (double)o->box[e] / (double)o->grid[e];",
        "const double hi_e = (double)c[e] * (double)o->box[e] / (double)o->grid[e];"),
    "corner_path_not_inherited": (
        "ivec_push(&o->disp[r], o->disp[s].v[m->v[j]] | (1 << d))",
        "ivec_push(&o->disp[r], (1 << d))"),
    "control_comment_only": (
        "/* dense layout: base[D] = sum of local sizes of lower domain ids */",
        "/* dense layout (unchanged code; only this comment differs) */"),
}
# the last entry is a control that changes nothing: it must PASS the pins
CONTROL = "control_comment_only"


def _build_mutant(tmp, name):
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, ("mutation anchor not unique", name)
    path = os.path.join(tmp, name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return oracle.build_oracle(path, os.path.join(tmp, "lib_" + name + ".so"), force=True)


def _run_pins(lib):
    def make(box, grid, rc, xyz, dom, prune=False):
        return oracle.Oracle(box, grid, rc, xyz, dom, lib=lib, prune=prune)

    for ex in pins.EXAMPLES:
        pins.check_example(make, pins.load_example(ex))
    struct = pins.load_pulse_structure()
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    o = make(w.box, w.grid, w.rc, xyz, dom)
    pins.check_pulse_structure(o, struct[w.name])
    pins.check_maps(o)
    pins.check_geometric(o, xyz, dom)
    pins.check_load_and_exchange_x(o, xyz)
    pins.check_forces_integer(o)
    for box, grid, rc, n in [((3.0, 2.6, 2.2), (3, 2, 2), 0.6, 300),
                             ((4.0, 4.0, 4.0), (1, 2, 5), 1.1, 300)]:
        xyz, dom = synth.custom_system(n, box, grid, seed=11)
        o = make(box, grid, rc, xyz, dom)
        pins.check_pair_coverage(o, xyz, dom)
        pins.check_forces_integer(o)
    # corner pruning: the direct construction, pair coverage and the forces
    w = synth.WORKLOADS["water24k_2x4x8"]
    xyz, dom = synth.system(w)
    o = make(w.box, w.grid, w.rc, xyz, dom, prune=True)
    pins.check_maps(o)
    pins.check_geometric(o, xyz, dom)
    pins.check_forces_integer(o)
    box, grid, rc = (3.0, 2.6, 2.2), (3, 2, 2), 0.6
    xyz, dom = synth.custom_system(300, box, grid, seed=11)
    o = make(box, grid, rc, xyz, dom, prune=True)
    pins.check_pair_coverage(o, xyz, dom)


@pytest.fixture(scope="module")
def tmpdir_mut():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", sorted(k for k in MUTANTS if k != CONTROL))
def test_pins_reject_mutant(tmpdir_mut, name):
    lib = oracle.load(_build_mutant(tmpdir_mut, name))
    with pytest.raises((AssertionError, oracle.OracleError, IndexError)):
        _run_pins(lib)


def test_pins_accept_control(tmpdir_mut):
    """A semantically neutral edit passes, so the rejections above are caused by
    the planted mistakes and not by the mutation harness."""
    lib = oracle.load(_build_mutant(tmpdir_mut, CONTROL))
    _run_pins(lib)
