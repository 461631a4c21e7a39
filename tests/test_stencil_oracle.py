"""The stencil oracle against hand-worked examples, exact fixed points and the
decomposition identity (no GPU), and planted mistakes that the pins must
reject."""
import importlib.util
import os
import tempfile

import pytest

import stencil_pins
from oracle import stencil as S


def test_jacobi_hand_example():
    stencil_pins.check_jacobi_golden(S)


def test_harmonic_fields_are_fixed_points():
    stencil_pins.check_fixed_points(S)


def test_exchange_hand_example():
    stencil_pins.check_exchange_golden(S)


def test_decomposition_identity():
    stencil_pins.check_decomposition(S)


def test_layout_sizes():
    assert S.pitch(4) == 12 and S.tile_floats(4) == 6 * 12
    assert S.pitch(512) % 4 == 0  # every row starts 16-byte aligned


MUTANTS = {
    "exchange_sends_second_row_up": (
        "dst[ty - 1, tx][n + 1, COL0:COL0 + n] = t[1, COL0:COL0 + n]",
        "dst[ty - 1, tx][n + 1, COL0:COL0 + n] = t[2, COL0:COL0 + n]"),
    "exchange_columns_swapped": (
        "dst[ty, tx - 1][1:n + 1, COL0 + n] = t[1:n + 1, COL0]",
        "dst[ty, tx - 1][1:n + 1, COL0 + n] = t[1:n + 1, COL0 + n - 1]"),
    "exchange_skips_last_block_row": (
        "if ty < py - 1:  # block below",
        "if ty < py - 2:  # block below"),
    "sweep_north_twice": (
        "ns = a[:-2, 1:-1] + a[2:, 1:-1]",
        "ns = a[:-2, 1:-1] + a[:-2, 1:-1]"),
    "sweep_weight": (
        "b[1:-1, 1:-1] = (ns + we) * q",
        "b[1:-1, 1:-1] = (ns + we) * np.float32(0.2)"),
    "to_tiles_west_ghost_shifted": (
        "t[1:n + 1, COL0 - 1] = blk[1:n + 1, 0]",
        "t[1:n + 1, COL0 - 1] = blk[0:n, 0]"),
    "tile_sweep_reads_centre_for_west": (
        "we = t[1:n + 1, COL0 - 1:COL0 + n - 1] + t[1:n + 1, COL0 + 1:COL0 + n + 1]",
        "we = t[1:n + 1, COL0:COL0 + n] + t[1:n + 1, COL0 + 1:COL0 + n + 1]"),
    "control_comment_only": (
        "# first block column inside a tile row",
        "# (unchanged code; only this comment differs)"),
}
CONTROL = "control_comment_only"


def _mutant(name, tmp):
    src = open(S.__file__).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, ("mutation anchor not unique", name)
    path = os.path.join(tmp, "stencil_%s.py" % name)
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("stencil_" + name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(k for k in MUTANTS if k != CONTROL))
def test_pins_reject_mutant(name):
    with tempfile.TemporaryDirectory() as tmp:
        mod = _mutant(name, tmp)
        with pytest.raises(AssertionError):
            stencil_pins.run_all(mod)


def test_pins_accept_control():
    with tempfile.TemporaryDirectory() as tmp:
        stencil_pins.run_all(_mutant(CONTROL, tmp))
