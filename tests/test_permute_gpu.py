"""wp_permute on the GPU against the oracle: bit-exact (gpu)."""
import itertools

import numpy as np
import pytest
import torch

from oracle import permute as opm
from oracle import plan as op

pytestmark = pytest.mark.gpu

LAYOUTS = (op.CANONICAL, op.REGULAR, op.SHIFTED)


@pytest.fixture(scope="module")
def vds():
    import __graft_entry__
    __graft_entry__.build()
    import video_dit_shifted_gb300 as m
    return m


def _bits(t):
    return t.view(torch.int16).cpu().numpy() if t.element_size() == 2 else t.view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("grid", [(2, 45, 80, 1, 3, 3), (3, 7, 11, 2, 2, 3), (1, 1, 1, 1, 1, 1),
                                  (21, 45, 80, 4, 3, 3), (33, 6, 4, 4, 1, 2)])
@pytest.mark.parametrize("width,dtype", [(8, torch.bfloat16), (2560, torch.bfloat16), (36, torch.float32)])
def test_all_layout_pairs_bit_exact(vds, grid, width, dtype):
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    src = torch.randn((N, width), device="cuda").to(dtype)
    for a, b in itertools.product(LAYOUTS, LAYOUTS):
        dst = torch.full_like(src, float("nan"))
        vds.permute(plan, src, dst, a, b)
        ia, ib = op.layout_tables(*grid, a)[1], op.layout_tables(*grid, b)[1]
        assert np.array_equal(_bits(dst), opm.permute_rows(_bits(src), ia, ib)), (a, b)
    plan.close()


def test_strided_rows_and_round_trip(vds):
    grid = (5, 45, 80, 4, 3, 3)
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    big = torch.randn((N, 3, 512), device="cuda").to(torch.bfloat16)
    src = big[:, 1]                                  # row stride 3*512 elements
    out = torch.zeros((N, 600), device="cuda", dtype=torch.bfloat16)
    dst = out[:, 40:552]                             # 80-byte offset, stride 1200 B
    vds.permute(plan, src, dst, op.REGULAR, op.SHIFTED)
    ir, isf = op.layout_tables(*grid, op.REGULAR)[1], op.layout_tables(*grid, op.SHIFTED)[1]
    assert np.array_equal(_bits(dst.contiguous()), opm.permute_rows(_bits(src.contiguous()), ir, isf))
    assert torch.count_nonzero(out[:, :40]) == 0 and torch.count_nonzero(out[:, 552:]) == 0
    back = torch.empty((N, 512), device="cuda", dtype=torch.bfloat16)
    vds.permute(plan, dst, back, op.SHIFTED, op.REGULAR)
    assert torch.equal(back, src)
    plan.close()


def test_in_place_is_rejected(vds):
    plan = vds.Plan(2, 45, 80, 1, 3, 3, device="cuda")
    x = torch.zeros((plan.N, 64), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(vds.wp.WpError) as e:
        vds.permute(plan, x, x, op.REGULAR, op.SHIFTED)
    assert e.value.code == 1
    plan.close()


SWEEP = [(T, H, W, 4, 3, 3) for (H, W) in ((45, 80), (68, 120), (90, 160)) for T in (5, 21, 30)]


@pytest.mark.parametrize("grid", SWEEP)
def test_sweep_full_size(vds, grid):
    """[N, 2560] bf16 rows at the re-layout sweep sizes, both directions:
    every destination row equals the source row the oracle's id tables name
    (dst[q] = src[pos_src[ids_dst[q]]], the gather done on the device from
    the oracle's index table), and the round trip is the identity."""
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    g = torch.Generator(device="cuda").manual_seed(grid[0] * 1000 + grid[1])
    src = torch.randn((N, 2560), device="cuda", generator=g).to(torch.bfloat16)
    shf = torch.empty_like(src)
    back = torch.empty_like(src)
    vds.permute(plan, src, shf, op.REGULAR, op.SHIFTED)
    vds.permute(plan, shf, back, op.SHIFTED, op.REGULAR)
    ir, isf = op.layout_tables(*grid, op.REGULAR)[1], op.layout_tables(*grid, op.SHIFTED)[1]
    r2s = torch.from_numpy(opm.inverse(ir)[isf]).cuda()      # shifted row q <- regular row r2s[q]
    s2r = torch.from_numpy(opm.inverse(isf)[ir]).cuda()
    assert torch.equal(shf, src[r2s])
    assert torch.equal(back, shf[s2r])
    assert torch.equal(back, src)
    plan.close()


def _random_cases(n, seed=23):
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        grid = (rng.randint(1, 5), rng.randint(1, 50), rng.randint(1, 70),
                rng.randint(1, 4), rng.randint(1, 4), rng.randint(1, 4))
        if min(op.window_size(*grid)) < 1:
            continue
        pair = rng.sample([op.CANONICAL, op.REGULAR, op.SHIFTED], 2)
        out.append((grid, tuple(pair), 8 * rng.randint(1, 300)))
    return out


@pytest.mark.parametrize("grid,pair,width", _random_cases(10))
def test_random_grids_bit_exact(vds, grid, pair, width):
    """Seeded random grids, window counts, layout pairs and row widths (16 B
    to 4.8 KB of int16): every row equals the oracle's permutation."""
    src_l, dst_l = pair
    plan = vds.Plan(*grid, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(sum(grid) + width)
    src = torch.randint(-2 ** 15, 2 ** 15, (plan.N, width), dtype=torch.int16, device="cuda", generator=g)
    dst = torch.empty_like(src)
    vds.permute(plan, src, dst, src_l, dst_l)
    torch.cuda.synchronize()
    ids = {l: op.layout_tables(*grid, l)[1] for l in pair}
    want = opm.permute_rows(src.cpu().numpy(), ids[src_l], ids[dst_l])
    assert np.array_equal(dst.cpu().numpy(), want)
    plan.close()
