"""The FP4 GEMM's tile layout, simulated on the CPU: every tile the permutation lays out and the
kernel decodes stays inside the buffers, and the tiles cover every row once.

This mirrors the n-tile records of the permutation (tiles of `ntile` and 2 * `ntile` rows over the
touched groups, {first row, group | rows << 16}) and the kernel's decode of tile t into (n-tile
t / m_tiles, m-tile t % m_tiles), for the tile sizes each launch uses, and checks the predicate the
bounds-checked build (-DCOLI_BOUNDS_CHECK) evaluates before it would skip a tile. The GPU side of
the same check is tests/test_bounds_check_gpu.py.
"""
import numpy as np
import pytest

BM = 128


def records(cnt, ntile):
    """Small and large n-tile records over the touched groups, in group order."""
    off = np.concatenate([[0], np.cumsum(cnt)])
    small, large = [], []
    for g, c in enumerate(cnt):
        for size, out in ((ntile, small), (2 * ntile, large)):
            for r in range(-(-c // size)):
                out.append((off[g] + r * size, g, min(size, c - r * size)))
    return small, large


def check_launch(recs, E, rows, m_tiles, gate_up, I, I_s, H, big, bh_max):
    covered = {}
    for t in range(len(recs) * m_tiles):
        row0, g, n = recs[t // m_tiles]
        mt = t % m_tiles
        Ig = I_s if g == E else I
        valid = (mt * BM < Ig) if gate_up else True
        if not valid:
            continue
        mrows = 2 * BM if (big and not gate_up) else BM
        bad = (g > E or n < 1 or n > bh_max or row0 < 0 or row0 + n > rows or
               (mt * BM + BM > Ig if gate_up else mt * mrows + mrows > H))
        assert not bad, (t, row0, g, n, mt)
        for r in range(row0, row0 + n):
            covered[(r, mt)] = covered.get((r, mt), 0) + 1
    # every (row, m-tile of its group) exactly once
    assert all(v == 1 for v in covered.values())


@pytest.mark.parametrize("E,H,I,I_s,T,k,skew", [
    (256, 4096, 2048, 2048, 8, 8, 0.0),      # decode
    (256, 4096, 2048, 2048, 512, 8, 0.0),    # prefill
    (256, 7168, 2048, 2048, 4096, 8, 1.1),   # skewed (Zipf)
    (32, 7168, 2048, 2048, 1024, 8, 0.0),    # reduced skewed
    (8, 512, 256, 384, 200, 2, 0.0),         # big tiles, wider shared expert
    (6, 768, 384, 128, 400, 3, 0.5),         # big tiles, narrower shared expert
    (16, 384, 128, 128, 37, 3, 0.0),         # ragged
    (1, 256, 128, 0, 4, 1, 0.0),             # one expert, no shared expert
])
def test_tiles_stay_in_bounds(E, H, I, I_s, T, k, skew):
    rng = np.random.default_rng(E * 7 + T)
    if skew > 0:
        p = (np.arange(E) + 1.0) ** -skew
        p /= p.sum()
    else:
        p = np.full(E, 1.0 / E)
    cnt = np.zeros(E, np.int64)
    for _ in range(T):                           # top-k distinct experts per token
        cnt[rng.choice(E, size=min(k, E), replace=False, p=p)] += 1
    cnt = list(cnt) + ([T] if I_s else [])      # group E: the shared expert, T rows
    rows = T * k + (T if I_s else 0)
    I_max = max(I, I_s)
    big = T * k >= 48 * E and H % 256 == 0
    ntile = 24 if big else 16
    small, large = records(cnt, ntile)
    gu32 = big or T * k >= 16 * E
    gate_up_recs = large if gu32 else small
    bh_gu = 48 if big else (32 if gu32 else 16)
    check_launch(gate_up_recs, E, rows, -(-I_max // BM), True, I, I_s, H, big, bh_gu)
    check_launch(large, E, rows, H // (2 * BM) if big else H // BM, False, I, I_s, H, big, 48 if big else 32)
    # a planted mistake is caught: a record one row past the end
    bad = list(large)
    row0, g, n = bad[-1]
    bad[-1] = (row0 + 1, g, n)
    with pytest.raises(AssertionError):
        check_launch(bad, E, rows, H // (2 * BM) if big else H // BM, False, I, I_s, H, big, 48 if big else 32)


EPI_WARPS = 8
BN_GATE_UP = 16


def h_counter_increments(recs, E, m_tiles, I, I_s):
    """Per group: the raises the gate/up launch makes (every epilogue warp, once per valid tile)."""
    inc = [0] * (E + 1)
    for t in range(len(recs) * m_tiles):
        row0, g, n = recs[t // m_tiles]
        Ig = I_s if g == E else I
        if (t % m_tiles) * BM < Ig:
            inc[g] += EPI_WARPS
    return inc


def h_counter_target(c, Ig):
    """What the down launch's producer waits for: the group's 16-row gate/up tiles x its m-tiles x
    the epilogue warps."""
    return EPI_WARPS * (-(-c // BN_GATE_UP)) * (-(-Ig // BM))


@pytest.mark.parametrize("E,I,I_s,T,k", [
    (256, 2048, 2048, 8, 8),      # decode
    (256, 2048, 2048, 4, 8),      # four tokens
    (256, 2048, 2048, 63, 8),     # the largest token count of the mode
    (64, 2048, 1024, 40, 6),      # narrower shared expert
    (12, 512, 1024, 21, 3),       # wider shared expert
    (16, 384, 0, 30, 2),          # no shared expert
])
def test_h_counter_targets_match_the_gate_up_raises(E, I, I_s, T, k):
    """The down launch of a few-token forward starts on a group once its counter reaches the target:
    that target must equal the raises the gate/up launch makes for the group, or the down launch
    would wait until its limit (too high) or read h early (too low)."""
    rng = np.random.default_rng(E + 31 * T)
    cnt = np.zeros(E, np.int64)
    for _ in range(T):
        cnt[rng.choice(E, size=min(k, E), replace=False)] += 1
    cnt = list(cnt) + ([T] if I_s else [])
    small, _ = records(cnt, BN_GATE_UP)
    I_max = max(I, I_s)
    inc = h_counter_increments(small, E, -(-I_max // BM), I, I_s)
    for g, c in enumerate(cnt):
        if c == 0:
            continue
        Ig = I_s if g == E else I
        assert inc[g] == h_counter_target(c, Ig), (g, c, inc[g])
    # a planted mistake is caught: counting m-tiles of the widest intermediate size for every group
    # (it differs for the group whose intermediate size is the smaller one)
    if I_s and -(-I // BM) != -(-I_s // BM):
        narrow = E if I_s < I else next(g for g, c in enumerate(cnt[:E]) if c)
        assert inc[narrow] != EPI_WARPS * (-(-cnt[narrow] // BN_GATE_UP)) * (-(-I_max // BM))
