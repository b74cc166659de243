"""The cascade kernel's item order, read from the library's host-only diagnostic
(anvil_schedule_runs; no GPU needed).  The kernel only needs every phase of a matrix to
come after the phases it reads (its completion counters enforce the waits, and the walk
progresses because an item only waits for lower-numbered items); these tests check that
property and that every tile of every phase of every matrix appears exactly once, for
the bench's three banks, calls with many matrices, and other map counts.  The
normalisation X / d is not a phase of the cascade: it runs before it, in its own kernel."""
import math

import pytest

anvil = pytest.importorskip("polynomial_matrix_whitening_gb300.anvil")

GRAM, GRAM_NORM, SQPOLY, XUPDATE, XUPDATE_OUT = range(5)


def phase_ops(nmaps):
    ops = [GRAM_NORM]
    for k in range(nmaps):
        if k > 0:
            ops.append(GRAM)
        ops.append(SQPOLY)
        ops.append(XUPDATE_OUT if k == nmaps - 1 else XUPDATE)
    return ops


def tiles(op, m, n):
    T, ntl = math.ceil(min(m, n) / 256), math.ceil(max(m, n) / 256)
    return T * (T + 1) // 2 if op in (GRAM, GRAM_NORM, SQPOLY) else T * ntl


def check_order(shapes, nmaps):
    runs = anvil.schedule_runs(shapes, nmaps)
    ops = phase_ops(nmaps)
    # runs tile the item range in order
    item = 0
    first, last = {}, {}
    for r in runs:
        assert r["begin"] == item
        assert r["op"] == ops[r["phase"]]
        g, m, n = shapes[r["bank"]]
        assert r["tiles"] == tiles(r["op"], m, n)
        assert r["nmat"] >= 1 and 0 <= r["mat0"] and r["mat0"] + r["nmat"] <= g
        for i in range(r["mat0"], r["mat0"] + r["nmat"]):
            key = (r["phase"], r["bank"], i)
            assert key not in first, f"segment {key} listed twice"
            first[key] = item
            item += r["tiles"]
            last[key] = item - 1
    # every segment once
    want = sum(g * tiles(op, m, n) for (g, m, n) in shapes for op in ops)
    assert item == want
    assert len(first) == len(ops) * sum(g for g, _, _ in shapes)
    # every phase after the phase before it (which it reads, or which read the buffer it
    # overwrites)
    for (p, q, i), f in first.items():
        if p > 0:
            assert last[(p - 1, q, i)] < f
    return runs


BENCH = [(22, 256, 768), (22, 768, 768), (22, 2816, 768)]


@pytest.mark.parametrize("shapes,nmaps", [
    (BENCH, 6),
    (BENCH, 1),
    (BENCH, 16),
    ([(1, 1, 1)], 6),
    ([(3, 130, 300), (2, 300, 130), (1, 520, 520)], 6),
    ([(200, 24, 16), (120, 8, 40), (80, 20, 20)], 6),
    ([(500, 24, 16), (300, 8, 40), (200, 20, 20)], 6),
    ([(4, 1000, 264)] * 8, 3),
], ids=["bench", "bench_1map", "bench_16maps", "1x1", "ragged", "400_mats", "1000_mats", "8_banks"])
def test_item_order_respects_dependencies(shapes, nmaps):
    check_order(shapes, nmaps)


def test_order_is_phase_major_heaviest_bank_first():
    """The bench's order: phase by phase, and within a phase the banks heaviest first
    (the 22 x 2816 x 768 bank, whose tiles are the longest, opens every phase)."""
    runs = check_order(BENCH, 6)
    phases = [r["phase"] for r in runs]
    assert phases == sorted(phases)
    starts = {}
    for r in runs:
        starts.setdefault(r["phase"], r["bank"])
    assert set(starts.values()) == {2}
    for shapes in ([(500, 24, 16), (300, 8, 40), (200, 20, 20)], [(4, 1000, 264)] * 8):
        phases = [r["phase"] for r in check_order(shapes, 6)]
        assert phases == sorted(phases)


def test_invalid_arguments():
    with pytest.raises(anvil.AnvilError):
        anvil.schedule_runs(BENCH, 0)
    with pytest.raises(anvil.AnvilError):
        anvil.schedule_runs(BENCH, anvil.MAX_MAPS + 1)
    with pytest.raises(anvil.AnvilError):
        anvil.schedule_runs([(0, 4, 4)], 6)
