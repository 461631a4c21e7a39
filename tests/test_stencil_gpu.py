"""The 2-D stencil halo workload on the GPU (through the C ABI) against the
stencil oracle: whole fields compared bit-exactly (padding and ghost corners
included, which no call may touch)."""
import numpy as np
import pytest

from oracle import stencil as S

pytestmark = pytest.mark.gpu

# (px, py, n): single block, 1-D grids both ways, 2-D grids, several column
# blocks with a ragged last one (n/4 > 128), ragged row bands (n % 16 != 0)
GRIDS = [(1, 1, 4), (2, 1, 4), (1, 3, 8), (3, 1, 12), (2, 2, 4), (2, 4, 8), (3, 2, 36),
         (2, 2, 520), (4, 2, 1000), (1, 2, 2048)]
SENTINEL = np.float32(3.5)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def make_field(px, py, n, seed):
    rng = np.random.default_rng(seed)
    a = rng.random((py * n + 2, px * n + 2)).astype(np.float32)
    f = S.to_tiles(a, px, py, n)
    f[unused(px, py, n)] = SENTINEL
    return a, f


def unused(px, py, n):
    m = np.ones((py, px, n + 2, S.pitch(n)), bool)
    c0 = S.COL0
    m[:, :, 1:n + 1, c0 - 1:c0 + n + 1] = False
    m[:, :, 0, c0:c0 + n] = False
    m[:, :, n + 1, c0:c0 + n] = False
    return m.reshape(-1)


def inner_ghosts(px, py, n):
    import stencil_pins
    return stencil_pins.inner_ghost_mask(S, px, py, n)


def bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def plan_for(px, py, n):
    from domain_decomposition_halo_build_gb300 import stencil
    p = stencil.StencilPlan(px, py, n)
    assert p.total_floats == px * py * S.tile_floats(n)
    assert (p.pitch, p.col0) == (S.pitch(n), S.COL0)
    return p


@pytest.mark.parametrize("px,py,n", GRIDS)
def test_exchange(px, py, n):
    import torch
    a, f = make_field(px, py, n, seed=n + px)
    f[inner_ghosts(px, py, n)] = -9.0
    want = S.exchange_tiles(f, px, py, n)
    p = plan_for(px, py, n)
    d = torch.from_numpy(f).cuda()
    p.exchange(d)
    np.testing.assert_array_equal(bits(d.cpu().numpy()), bits(want))


@pytest.mark.parametrize("px,py,n", GRIDS)
def test_sweep_and_fused(px, py, n):
    import torch
    a, fin = make_field(px, py, n, seed=2 * n + py)
    rng = np.random.default_rng(7)
    fout = rng.random(fin.shape).astype(np.float32)   # garbage everywhere ...
    fout[unused(px, py, n)] = SENTINEL
    border = np.zeros_like(a)
    border[0, :], border[-1, :], border[:, 0], border[:, -1] = a[0, :], a[-1, :], a[:, 0], a[:, -1]
    mb = __import__("stencil_pins").matrix_border_mask(S, px, py, n)
    fout[mb] = S.to_tiles(border, px, py, n)[mb]      # ... but the fixed border
    p = plan_for(px, py, n)
    din = torch.from_numpy(fin).cuda()
    for fused, want in ((False, S.jacobi_tiles(fin, fout, px, py, n)),
                        (True, S.fused_step(fin, fout, px, py, n))):
        dout = torch.from_numpy(fout).cuda()
        (p.sweep_fused if fused else p.sweep)(din, dout)
        np.testing.assert_array_equal(bits(dout.cpu().numpy()), bits(want), err_msg="fused=%s" % fused)
    if not (px == 1 and py == 1):
        # the fused step equals a sweep followed by an exchange of the result
        d1 = torch.from_numpy(fout).cuda()
        p.sweep(din, d1)
        p.exchange(d1)
        d2 = torch.from_numpy(fout).cuda()
        p.sweep_fused(din, d2)
        assert torch.equal(d1, d2)


@pytest.mark.parametrize("px,py,n", [(2, 4, 8), (3, 2, 36), (4, 2, 1000)])
def test_iterations_match_whole_matrix_sweeps(px, py, n):
    """Ten fused iterations (two fields, alternating) give the tile field of ten
    Jacobi sweeps of the whole matrix; so do ten sweep + exchange pairs."""
    import torch
    a, f = make_field(px, py, n, seed=11)
    want = S.to_tiles(S.jacobi_global(a, 10), px, py, n)
    want[unused(px, py, n)] = SENTINEL
    p = plan_for(px, py, n)
    for fused in (True, False):
        cur = torch.from_numpy(f).cuda()
        nxt = cur.clone()
        for _ in range(10):
            if fused:
                p.sweep_fused(cur, nxt)
            else:
                p.sweep(cur, nxt)
                p.exchange(nxt)
            cur, nxt = nxt, cur
        np.testing.assert_array_equal(bits(cur.cpu().numpy()), bits(want), err_msg="fused=%s" % fused)


def test_bench_size_fused_step():
    """The largest bench configuration's shape class: 2 x 4 blocks of 4096^2
    (134M cells), one fused step, compared whole."""
    import torch
    px, py, n = 2, 4, 4096
    a, f = make_field(px, py, n, seed=5)
    p = plan_for(px, py, n)
    din = torch.from_numpy(f).cuda()
    dout = din.clone()
    p.sweep_fused(din, dout)
    want = S.fused_step(f, f, px, py, n)
    np.testing.assert_array_equal(bits(dout.cpu().numpy()), bits(want))


def test_bad_arguments():
    import torch
    from domain_decomposition_halo_build_gb300 import halo
    p = plan_for(2, 2, 8)
    d = torch.zeros(p.total_floats, device="cuda")
    with pytest.raises(halo.HaloError):
        p.sweep(d, d)                       # in == out
    with pytest.raises(ValueError):
        p.exchange(torch.zeros(p.total_floats + 4, device="cuda"))


@pytest.mark.parametrize("px,py,n", [(1, 1, 4), (2, 4, 8), (3, 2, 36), (2, 2, 520), (4, 2, 1000)])
@pytest.mark.parametrize("iterations", [0, 1, 2, 5])
def test_iterate_in_one_launch(px, py, n, iterations):
    """stencil_iterate: that many fused iterations in one cooperative launch
    (grid-wide barriers between them) give the tile field of that many sweeps
    of the whole matrix, in a for an even count and in b for an odd one."""
    import torch
    a, f = make_field(px, py, n, seed=iterations + 7)
    want = S.to_tiles(S.jacobi_global(a, iterations), px, py, n)
    want[unused(px, py, n)] = SENTINEL
    p = plan_for(px, py, n)
    da = torch.from_numpy(f).cuda()
    db = da.clone()
    res = p.iterate(da, db, iterations)
    assert p.status() == 0
    assert (res is da) == (iterations % 2 == 0)
    np.testing.assert_array_equal(bits(res.cpu().numpy()), bits(want))


def test_iterate_matches_separate_fused_launches():
    """Twelve iterations in one launch and twelve fused launches agree bit for
    bit on the bench's 2 x 4 grid of blocks."""
    import torch
    px, py, n = 2, 4, 512
    a, f = make_field(px, py, n, seed=21)
    p = plan_for(px, py, n)
    da, db = torch.from_numpy(f).cuda(), torch.from_numpy(f).cuda()
    one = p.iterate(da, db, 12)
    cur, nxt = torch.from_numpy(f).cuda(), torch.from_numpy(f).cuda()
    for _ in range(12):
        p.sweep_fused(cur, nxt)
        cur, nxt = nxt, cur
    assert p.status() == 0
    assert torch.equal(one, cur)
