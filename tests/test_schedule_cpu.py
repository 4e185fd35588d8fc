"""The backward's tile schedules, checked on the host (no GPU): every dZ, dX
and dW tile is handed out exactly once, the split schedule keeps each wave's
dZ tiles in a launch before its dX/dW launch, and in the fused schedule every
tile that waits (dX on its dZ rows, dW on its dZ column, a later wave's dZ on
the previous wave's readers of its buffer slot) only waits on tiles with an
earlier ticket, which is what rules out a deadlock of the persistent launch."""
import numpy as np
import pytest

DZ, DX, DW, DX2, DZ2, DW2 = 0, 1, 2, 3, 4, 5


def narrow(u):
    """Units as (kind, wave, a, b) 256 x 256 tiles; a wide dX tile (kind 3,
    512-column hidden tile b) counts as the dX tiles 2b and 2b + 1, a wide dZ
    tile (kind 4, first vocabulary tile b) as the dZ tiles b and b + 1, a wide
    dW tile (kind 5) as the dW tiles 2b and 2b + 1."""
    out = []
    for _, k, w, a, b in u.tolist():
        if k == DX2:
            out += [(DX, w, a, 2 * b), (DX, w, a, 2 * b + 1)]
        elif k == DZ2:
            out += [(DZ, w, a, b), (DZ, w, a, b + 1)]
        elif k == DW2:
            out += [(DW, w, a, 2 * b), (DW, w, a, 2 * b + 1)]
        else:
            out.append((k, w, a, b))
    return sorted(out)


@pytest.fixture(scope="module")
def flp():
    from entropy_loss_gb300 import build, flp
    build.build()
    flp.load()
    return flp


def cdiv(a, b):
    return -(-a // b)


def workspace_for(flp, M, H, V, chunk):
    """Smallest workspace whose split-schedule wave holds `chunk` rows."""
    lo, hi = 0, 1 << 42
    while lo < hi:
        mid = (lo + hi) // 2
        try:
            rows = flp.backward_plan(M, H, V, mid, "split")[0]
        except flp.FlpError:
            rows = 0
        if rows >= min(chunk, cdiv(M, 128) * 128):
            hi = mid
        else:
            lo = mid + 1
    return lo


def expected_units(M, H, V, chunk):
    Vt, Nh = cdiv(V, 256), cdiv(H, 256)
    out = []
    for w, r0 in enumerate(range(0, M, chunk)):
        Mt = cdiv(min(chunk, M - r0), 256)
        out += [(DZ, w, m, v) for m in range(Mt) for v in range(Vt)]
        out += [(DX, w, m, h) for m in range(Mt) for h in range(Nh)]
        out += [(DW, w, v, h) for v in range(Vt) for h in range(Nh)]
    return sorted(out)


SHAPES = [
    # M, H, V, wave rows, pairs
    (256, 256, 4096, 8192, 76),
    (4096, 4096, 131072, 8192, 76),
    (4096, 4096, 131072, 8192, 1),
    (4096, 4096, 131072, 2048, 74),
    (20001, 4096, 128257, 20096, 76),
    (20001, 4096, 128257, 4096, 76),
    (32768, 5120, 152064, 8192, 76),
    (8192, 2048, 151936, 8192, 76),
    (700, 136, 2100, 256, 2),
    (300, 200, 3001, 256, 76),
    (5000, 64, 1000, 512, 5),
    (1, 8, 1, 128, 76),
    (32768, 64, 1000, 256, 76),   # 128 waves: the fused segment table spans three launches
]


@pytest.mark.parametrize("schedule", ["split", "fused"])
@pytest.mark.parametrize("M,H,V,chunk,pairs", SHAPES)
def test_every_tile_exactly_once(flp, schedule, M, H, V, chunk, pairs):
    ws = workspace_for(flp, M, H, V, chunk)
    rows, waves, used = flp.backward_plan(M, H, V, ws, schedule)
    assert used == schedule
    u = flp.backward_schedule(M, H, V, ws, schedule, pairs)
    assert narrow(u) == expected_units(M, H, V, rows)
    assert waves == cdiv(M, rows)
    # dX tiles (and the split schedule's dW tiles) are wide exactly when H
    # spans an even number of 256-column tiles
    kinds = set(u[:, 1].tolist())
    if cdiv(H, 256) % 2 == 0:
        assert DX2 in kinds and DX not in kinds
        assert (DW2 in kinds and DW not in kinds) if schedule == "split" else (DW in kinds and DW2 not in kinds)
    else:
        assert DX in kinds and DX2 not in kinds and DW2 not in kinds


@pytest.mark.parametrize("M,H,V,chunk,pairs", SHAPES)
def test_split_schedule_orders_phases_by_launch(flp, M, H, V, chunk, pairs):
    ws = workspace_for(flp, M, H, V, chunk)
    rows, waves, _ = flp.backward_plan(M, H, V, ws, "split")
    u = flp.backward_schedule(M, H, V, ws, "split", pairs)
    launch, kind, wave = u[:, 0], u[:, 1], u[:, 2]
    assert launch.max() + 1 == 2 * waves
    for li in range(2 * waves):
        sel = launch == li
        assert np.all(wave[sel] == li // 2)
        if li % 2 == 0:
            # wide dZ tiles; a 256-column one only for an odd last vocabulary tile
            assert np.all(np.isin(kind[sel], (DZ, DZ2)))
            narrow_dz = u[sel & (kind == DZ)]
            assert np.all(narrow_dz[:, 4] == cdiv(V, 256) - 1) and cdiv(V, 256) % 2 == (len(narrow_dz) > 0)
        else:
            assert not np.any(np.isin(kind[sel], (DZ, DZ2)))
            # the long dX tiles first, the short dW tiles fill the tail
            k = np.where(kind[sel] == DX2, DX, np.where(kind[sel] == DW2, DW, kind[sel]))
            assert np.all(np.diff(k) >= 0)


@pytest.mark.parametrize("M,H,V,chunk,pairs", SHAPES)
def test_fused_waits_only_on_earlier_tickets(flp, M, H, V, chunk, pairs):
    ws = workspace_for(flp, M, H, V, chunk)
    rows, waves, used = flp.backward_plan(M, H, V, ws, "fused")
    assert used == "fused"
    u = flp.backward_schedule(M, H, V, ws, "fused", pairs)
    kind, wave, a, b = u[:, 1].copy(), u[:, 2], u[:, 3], u[:, 4]
    kind[kind == DX2] = DX  # a wide dX tile waits and signals like a dX tile
    pos = np.arange(len(u))
    Vt, Nh, Mt_full = cdiv(V, 256), cdiv(H, 256), cdiv(rows, 256)
    last_dz_row = np.full((waves, Mt_full), -1)
    last_dz_col = np.full((waves, Vt), -1)
    last_dx_row = np.full((waves, Mt_full), -1)
    last_dw_col = np.full((waves, Vt), -1)
    s = kind == DZ
    np.maximum.at(last_dz_row, (wave[s], a[s]), pos[s])
    np.maximum.at(last_dz_col, (wave[s], b[s]), pos[s])
    s = kind == DX
    np.maximum.at(last_dx_row, (wave[s], a[s]), pos[s])
    s = kind == DW
    np.maximum.at(last_dw_col, (wave[s], a[s]), pos[s])
    # dX on every dZ tile of its rows, dW on every dZ tile of its column
    s = kind == DX
    assert np.all(last_dz_row[wave[s], a[s]] < pos[s])
    s = kind == DW
    assert np.all(last_dz_col[wave[s], a[s]] < pos[s])
    # a later wave's dZ tile after the previous wave's readers of its slot,
    # a later wave's dW add after the previous wave's
    s = (kind == DZ) & (wave > 0)
    assert np.all(last_dx_row[wave[s] - 1, a[s]] < pos[s])
    assert np.all(last_dw_col[wave[s] - 1, b[s]] < pos[s])
    s = (kind == DW) & (wave > 0)
    assert np.all(last_dw_col[wave[s] - 1, a[s]] < pos[s])


def test_fused_schedule_splits_into_launches_when_the_table_overflows(flp):
    """Up to 160 segments fit one launch's table; more waves start another
    launch, at a wave boundary (a wave never spans two launches)."""
    M, H, V = 32768, 64, 1000
    ws = workspace_for(flp, M, H, V, 256)
    u = flp.backward_schedule(M, H, V, ws, "fused", 76)
    launch, wave = u[:, 0], u[:, 2]
    assert launch.max() + 1 == 3
    assert np.all(np.diff(launch) >= 0)
    for w in np.unique(wave):
        assert len(np.unique(launch[wave == w])) == 1


def test_fused_interleaves_dw_with_the_dz_sweep(flp):
    """At the headline shape a large share of the dW tiles is handed out
    during the dZ sweep, a few columns behind it, and the dX tiles are
    followed by enough dW tiles to even out their end (the wide dX tiles are
    long, so that tail holds over half of the dW tiles)."""
    M, H, V = 4096, 4096, 131072
    ws = workspace_for(flp, M, H, V, M)
    u = flp.backward_schedule(M, H, V, ws, "fused", 76)
    kind = u[:, 1].copy()
    kind[kind == DX2] = DX
    last_dz = np.nonzero(kind == DZ)[0].max()
    first_dx = np.nonzero(kind == DX)[0].min()
    last_dx = np.nonzero(kind == DX)[0].max()
    dw_pos = np.nonzero(kind == DW)[0]
    assert (dw_pos < last_dz).sum() > 0.3 * len(dw_pos)
    assert first_dx > last_dz
    # wide dX tiles: twice the K blocks' work per tile
    assert (dw_pos > last_dx).sum() >= 2 * 76 * (131072 // 64) // (4096 // 64)


def test_auto_takes_vsplit_for_short_row_waves(flp):
    """Row waves below 2048 rows (and below M) run the vocabulary split when
    the workspace holds its fp32 dX scratch and a 256-column dZ chunk."""
    M, H, V = 4096, 4096, 131072
    for rows, want in ((1024, "vsplit"), (512, "vsplit"), (2048, "split"), (4096, "split")):
        ws = workspace_for(flp, M, H, V, rows)
        assert flp.backward_plan(M, H, V, ws, "auto")[2] == want, rows
    # 128-row waves: 32 MiB does not hold the 64 MiB dX scratch
    ws = workspace_for(flp, M, H, V, 128)
    assert flp.backward_plan(M, H, V, ws, "auto")[:3] == (128, 32, "split")


def test_plan_picks_and_rejects(flp):
    M, H, V = 5000, 64, 1000
    # a 384-row wave is a multiple of 128 but not 256: fused waves round down
    ws = workspace_for(flp, M, H, V, 384)
    assert flp.backward_plan(M, H, V, ws, "split")[0] == 384
    assert flp.backward_plan(M, H, V, ws, "fused")[0] == 256
    # auto runs the split schedule (the faster one on GB300)
    for rows in (384, 512, M):
        ws = workspace_for(flp, M, H, V, rows)
        assert flp.backward_plan(M, H, V, ws, "auto") == flp.backward_plan(M, H, V, ws, "split")
        assert flp.backward_plan(M, H, V, ws, "auto")[2] == "split"
    ws = workspace_for(flp, M, H, V, M)
    assert flp.backward_plan(M, H, V, ws, "fused")[:3] == (cdiv(M, 128) * 128, 1, "fused")
    # 128 rows of dZ: split only (no room for the vocabulary-split plan either)
    ws = workspace_for(flp, M, H, V, 128)
    assert flp.backward_plan(M, H, V, ws, "auto")[2] == "split"
    with pytest.raises(flp.FlpError) as e:
        flp.backward_plan(M, H, V, ws, "fused")
    assert e.value.status == flp.FLP_ERR_UNSUPPORTED
    with pytest.raises(flp.FlpError) as e:
        flp.backward_plan(M, H, V, 1024, "auto")
    assert e.value.status == flp.FLP_ERR_WORKSPACE


def workspace_for_vsplit(flp, M, H, V, cols):
    """Smallest workspace whose vocabulary-split chunks hold `cols` columns."""
    lo, hi = 0, 1 << 42
    while lo < hi:
        mid = (lo + hi) // 2
        try:
            _, waves, _ = flp.backward_plan(M, H, V, mid, "vsplit")
            ok = waves <= cdiv(cdiv(V, 256) * 256, cols)
        except flp.FlpError:
            ok = False
        if ok:
            hi = mid
        else:
            lo = mid + 1
    return lo


@pytest.mark.parametrize("M,H,V,cols", [
    (4096, 4096, 131072, 32768), (4096, 4096, 131072, 256), (300, 200, 3001, 1024),
    (20001, 4096, 128257, 8192), (1, 8, 1, 256), (700, 512, 2100, 768),
])
def test_vsplit_schedule(flp, M, H, V, cols):
    """All rows in one wave; per vocabulary chunk a dZ launch then a dX + dW
    launch; every dZ and dW tile once, each chunk's dX tiles once per chunk."""
    ws = workspace_for_vsplit(flp, M, H, V, cols)
    rows, chunks, used = flp.backward_plan(M, H, V, ws, "vsplit")
    assert used == "vsplit" and rows >= M and chunks == cdiv(cdiv(V, 256) * 256, cols)
    u = flp.backward_schedule(M, H, V, ws, "vsplit", 76)
    launch = u[:, 0]
    assert launch.max() + 1 == 2 * chunks
    Vt, Nh, Mt = cdiv(V, 256), cdiv(H, 256), cdiv(M, 256)
    per = cols // 256
    seen_dz, seen_dw, seen_dx = [], [], []
    for c in range(chunks):
        dz = u[launch == 2 * c]
        gm = u[launch == 2 * c + 1]
        assert np.all(np.isin(dz[:, 1], (DZ, DZ2))) and not np.any(np.isin(gm[:, 1], (DZ, DZ2)))
        vts = set(range(c * per, min(Vt, (c + 1) * per)))
        dzn = narrow(dz)
        assert {v for _, _, _, v in dzn} == vts          # the chunk's vocabulary tiles
        is_dw = np.isin(gm[:, 1], (DW, DW2))
        dwn = narrow(gm[is_dw])
        assert {v for _, _, v, _ in dwn} == vts
        seen_dz += [(m, v) for _, _, m, v in dzn]
        seen_dw += [(v, h) for _, _, v, h in dwn]
        dx = narrow(gm[~is_dw])
        assert sorted(dx) == sorted((DX, 0, m, h) for m in range(Mt) for h in range(Nh))
    assert sorted(seen_dz) == sorted((m, v) for m in range(Mt) for v in range(Vt))
    assert sorted(seen_dw) == sorted((v, h) for v in range(Vt) for h in range(Nh))


def test_vsplit_workspace_limits(flp):
    M, H, V = 4096, 4096, 131072
    # no room for the fp32 dX scratch, then no room for 256 columns of dZ
    with pytest.raises(flp.FlpError) as e:
        flp.backward_plan(M, H, V, 32 << 20, "vsplit")
    assert e.value.status == flp.FLP_ERR_WORKSPACE
    with pytest.raises(flp.FlpError) as e:
        flp.backward_plan(M, H, V, (64 << 20) + (1 << 20), "vsplit")
    assert e.value.status == flp.FLP_ERR_WORKSPACE
    # a 1 GiB workspace: 64 MiB of fp32 dX scratch, the rest (less a few KiB
    # of header and counters) as 4096-row dZ chunks of whole 256-column tiles
    rows, chunks, _ = flp.backward_plan(M, H, V, 1 << 30, "vsplit")
    cols = ((1 << 30) - (64 << 20) - 8192) // (4096 * 2) // 256 * 256
    assert rows == 4096 and chunks == cdiv(131072, cols)
