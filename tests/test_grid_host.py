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


@pytest.mark.parametrize("BH,tiles", [(1, 2), (3, 32), (40, 64), (7, 18)])
def test_decode_pair_units_cover_every_item_with_equal_causal_work(harness, BH, tiles):
    """Item 2u + s is key tile j (s = 0) or tiles-1-j (s = 1) of head
    u / (tiles/2), j = u mod tiles/2: every (head, tile) appears once, and
    under a square causal mask (key tile kt sees tiles - kt query tiles) every
    unit sees tiles + 1 query tiles."""
    pos = harness("u", BH, tiles)
    assert sorted(map(tuple, pos)) == [(h, r) for h in range(BH) for r in range(tiles)]
    for u in range(BH * tiles // 2):
        (h0, r0), (h1, r1) = pos[2 * u], pos[2 * u + 1]
        assert h0 == h1 == u // (tiles // 2) and r0 == u % (tiles // 2) and r1 == tiles - 1 - r0
        assert (tiles - r0) + (tiles - r1) == tiles + 1


def test_pair_launch_rule(harness):
    """Causal, dense and square only; tile counts between the persistent
    rule's limit (16) and the kernel's maximum, even; units at least one per
    SM and filling the last wave of CTAs to 95 % or more."""
    rule = lambda *a: harness("l", *a)[0][0]
    # the long causal bench shape: 128 heads x 64 key tiles, 4096 units on 152 SMs (27 waves, 99.8 %)
    assert rule(1, 0, 1, 64, 128 * 64, 152, 64) == 1
    assert rule(0, 0, 1, 64, 128 * 64, 152, 64) == 0       # not causal
    assert rule(1, 1, 1, 64, 128 * 64, 152, 64) == 0       # block-sparse
    assert rule(1, 0, 0, 64, 128 * 64, 152, 64) == 0       # query and key lengths differ
    assert rule(1, 0, 1, 16, 4096 * 16, 152, 64) == 0      # the persistent rule covers it
    assert rule(1, 0, 1, 63, 128 * 63, 152, 64) == 0       # odd tile count
    assert rule(1, 0, 1, 128, 64 * 128, 152, 64) == 0      # beyond the kernel's maximum
    assert rule(1, 0, 1, 128, 64 * 128, 152, 128) == 1
    assert rule(1, 0, 1, 32, 16 * 32, 152, 64) == 0        # 256 units: 2 waves, 84 % full
    assert rule(1, 0, 1, 32, 8 * 32, 152, 64) == 0         # 128 units: fewer than SMs
    assert rule(1, 0, 1, 32, 128 * 32, 152, 64) == 1       # 2048 units: 14 waves, 96 % full
