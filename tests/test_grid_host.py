"""The kernels' work-order and tile-range helpers (fa_kernels.h), run on the
host through a small harness compiled with nvcc (CPU only)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("grid") / "grid_check")
    subprocess.run([nvcc, "-std=c++17", "-arch=sm_103a", "-o", exe,
                    os.path.join(HERE, "grid_check.cu")], check=True, capture_output=True)

    def run(*args):
        out = subprocess.run([exe, *map(str, args)], check=True, capture_output=True, text=True)
        return [list(map(int, line.split())) for line in out.stdout.splitlines()]
    return run


@pytest.mark.parametrize("BH,tiles,group", [(1, 1, 1), (7, 3, 2), (16, 8, 5), (64, 4, 76),
                                            (33, 16, 16), (5, 9, 1)])
def test_decode_grid_is_a_bijection_in_group_order(harness, BH, tiles, group):
    """Every (head, tile rank) appears once; heads come in groups of `group`
    (the last one shorter); inside a group the rank varies slowest, so every
    head's rank r is scheduled before any head's rank r + 1."""
    pos = harness("d", BH, tiles, group)
    assert sorted(map(tuple, pos)) == [(h, r) for h in range(BH) for r in range(tiles)]
    for L, (bh, rank) in enumerate(pos):
        g = bh // group
        gh = min(group, BH - g * group)
        assert L == g * group * tiles + rank * gh + (bh - g * group)


@pytest.mark.parametrize("nkv,coff", [(1, 0), (8, 0), (8, 128), (9, 100), (64, 7168), (5, 1)])
def test_first_query_tile_is_the_first_that_sees_the_key_tile(harness, nkv, coff):
    """Query i sees key j iff j <= i + coff.  The first query tile of key
    tile kt is the lowest 128-row tile holding a row that sees key kt*128."""
    for kt, t in enumerate(r[0] for r in harness("f", nkv, coff)):
        first_row = max(0, kt * 128 - coff)
        assert t == first_row // 128
        assert all(i + coff < kt * 128 for i in range(0, t * 128))  # earlier tiles see nothing


def test_head_group_and_persistence_rule(harness):
    for BH, tiles, sms in ((1024, 4, 152), (16, 64, 152), (3, 1, 152), (500, 7, 148)):
        g = harness("h", BH, tiles, sms)[0][0]
        assert 1 <= g <= BH and g == min(BH, max(1, -(-2 * sms // tiles)))
    rule = lambda c, s, t: harness("p", c, s, t)[0][0]
    assert rule(0, 0, 64) == 1 and rule(1, 0, 16) == 1 and rule(1, 0, 17) == 0
    assert rule(0, 1, 4) == 0 and rule(1, 1, 4) == 0
