"""The host page allocator: the oracle's model pinned to a worked example and
to its invariants, and the library's lnk_pager checked against the model
operation by operation on seeded random sequences.  Host code only (no GPU)."""
import numpy as np
import pytest

from oracle import pager as opager

UNMAPPED = -1


def _lib_pager():
    lnk = pytest.importorskip("paged_kv_gqa_row_gb300")
    return lnk


def _worked_example(make, err_code):
    """A sequence whose outcome follows from the allocator's rules by hand:
    lowest free page first, fork shares pages, the first write into a shared
    page moves the writer to a fresh page (copy), release frees at count 0."""
    pg = make(8, 4, 4)
    pg.reserve(0, 150)                         # 150 positions -> 3 pages: 0, 1, 2
    assert [list(r) for r in pg.table()][0] == [0, 1, 2, UNMAPPED]
    pg.fork(0, 1, 150)                         # row 1 shares 0, 1, 2
    pg.fork(0, 2, 100)                         # row 2 shares 0, 1
    assert [pg.refcount(p) for p in range(4)] == [3, 3, 2, 0]
    assert pg.free_pages() == 5
    copies = pg.prepare_append([1, 2, 0], [150, 100, 150])
    # row 1 writes into page 2 (count 2): moved to page 3; row 2 writes into
    # page 1 (count 3): moved to page 4; row 0 then owns page 2 alone
    assert copies == [(2, 3), (1, 4)]
    t = [list(r) for r in pg.table()]
    assert t[0] == [0, 1, 2, UNMAPPED] and t[1] == [0, 1, 3, UNMAPPED] and t[2] == [0, 4, UNMAPPED, UNMAPPED]
    assert [pg.refcount(p) for p in range(8)] == [3, 2, 1, 1, 1, 0, 0, 0]
    pg.release(0)                              # page 2 reaches 0 and is free again
    assert pg.free_pages() == 4 and pg.refcount(2) == 0
    assert pg.prepare_append([3], [0]) == []   # lowest free page is 2
    assert [list(r) for r in pg.table()][3] == [2, UNMAPPED, UNMAPPED, UNMAPPED]
    assert err_code(lambda: pg.reserve(3, 300)) == "ERANGE"   # 300 > 4 pages x 64
    pg.reserve(3, 256)
    assert [list(r) for r in pg.table()][3] == [2, 5, 6, 7] and pg.free_pages() == 0
    before = [list(r) for r in pg.table()]
    assert err_code(lambda: pg.prepare_append([1], [200])) == "ENOSPACE"
    assert [list(r) for r in pg.table()] == before             # a failed call changes nothing
    assert err_code(lambda: pg.fork(0, 3, 10)) == "EINVAL"     # row 3 is not empty
    for r in range(4):
        pg.release(r)
    assert pg.free_pages() == 8 and all(pg.refcount(p) == 0 for p in range(8))


def _oracle_err(fn):
    try:
        fn()
    except opager.PagerError as e:
        return e.code
    return None


def _lib_err(fn):
    lnk = _lib_pager()
    try:
        fn()
    except lnk.LnkError as e:
        return {1: "EINVAL", 2: "ERANGE", 6: "ENOSPACE"}.get(e.status, str(e.status))
    return None


def test_oracle_pager_worked_example():
    _worked_example(opager.Pager, _oracle_err)


def test_library_pager_worked_example():
    lnk = _lib_pager()
    _worked_example(lnk.Pager, _lib_err)


def _invariants(pg):
    counts = [0] * pg.num_pages
    for r in pg.table():
        for e in r:
            if e != UNMAPPED:
                counts[e] += 1
    assert counts == [pg.refcount(p) for p in range(pg.num_pages)]
    assert pg.free_pages() == sum(1 for c in counts if c == 0)


def _random_ops(rng, num_rows, ppr, n_ops):
    ops = []
    for _ in range(n_ops):
        kind = rng.choice(["reserve", "fork", "append", "append", "release"], p=[0.2, 0.2, 0.25, 0.2, 0.15])
        if kind == "reserve":
            ops.append(("reserve", int(rng.integers(-1, num_rows + 1)), int(rng.integers(-5, ppr * 64 + 40))))
        elif kind == "fork":
            ops.append(("fork", int(rng.integers(0, num_rows)), int(rng.integers(0, num_rows)),
                        int(rng.integers(-2, ppr * 64 + 10))))
        elif kind == "append":
            n = int(rng.integers(0, 7))
            rows = rng.integers(-1 if rng.random() < 0.1 else 0, num_rows, size=n)
            pos = rng.integers(-3, ppr * 64 + (20 if rng.random() < 0.1 else 0), size=n)
            ops.append(("append", rows.tolist(), pos.tolist()))
        else:
            ops.append(("release", int(rng.integers(0, num_rows))))
    return ops


def _apply(pg, op, err):
    kind = op[0]
    if kind == "reserve":
        return err(lambda: pg.reserve(op[1], op[2]))
    if kind == "fork":
        return err(lambda: pg.fork(op[1], op[2], op[3]))
    if kind == "append":
        out = {}

        def call():
            out["copies"] = pg.prepare_append(op[1], op[2])
        e = err(call)
        return e if e else out["copies"]
    return err(lambda: pg.release(op[1]))


@pytest.mark.parametrize("seed", [1, 2, 3, 4, 5])
def test_oracle_pager_invariants(seed):
    rng = np.random.default_rng(seed)
    pg = opager.Pager(24, 6, 5)
    for op in _random_ops(rng, 6, 5, 400):
        _apply(pg, op, _oracle_err)
        _invariants(pg)


@pytest.mark.parametrize("seed", [11, 12, 13, 14, 15, 16])
def test_library_pager_matches_oracle(seed):
    lnk = _lib_pager()
    rng = np.random.default_rng(seed)
    num_pages, num_rows, ppr = [(24, 6, 5), (7, 4, 3), (64, 8, 9)][seed % 3]
    want, got = opager.Pager(num_pages, num_rows, ppr), lnk.Pager(num_pages, num_rows, ppr)
    for i, op in enumerate(_random_ops(rng, num_rows, ppr, 500)):
        a = _apply(want, op, _oracle_err)
        b = _apply(got, op, _lib_err)
        assert a == b, (i, op, a, b)
        assert np.array_equal(np.asarray(want.table(), dtype=np.int32), got.table()), (i, op)
        assert want.free_pages() == got.free_pages()
    assert [want.refcount(p) for p in range(num_pages)] == [got.refcount(p) for p in range(num_pages)]


def test_library_pager_argument_errors():
    lnk = _lib_pager()
    with pytest.raises(lnk.LnkError):
        lnk.Pager(0, 1, 1)
    pg = lnk.Pager(4, 2, 2)
    assert pg.refcount(-1) == -1 and pg.refcount(4) == -1
    with pytest.raises(lnk.LnkError):
        pg.fork(0, 0, 10)
    with pytest.raises(lnk.LnkError):
        pg.release(2)


class _HighestFirst(opager.Pager):
    def _take(self):
        page = max(self.free)
        self.free.remove(page)
        self.count[page] = 1
        return page


class _NoCopyOnWrite(opager.Pager):
    def prepare_append(self, rows, positions):
        copies = []
        for row, pos in zip(rows, positions):
            if pos >= 0 and self.rows[row][pos // 64] == opager.UNMAPPED:
                self.rows[row][pos // 64] = self._take()
        return copies


class _CopyKeepsCount(opager.Pager):
    def prepare_append(self, rows, positions):
        copies = super().prepare_append(rows, positions)
        for old, _ in copies:
            self.count[old] += 1  # forgets that the writer left the old page
        return copies


@pytest.mark.parametrize("cls", [_HighestFirst, _NoCopyOnWrite, _CopyKeepsCount])
def test_worked_example_catches_planted_mistakes(cls):
    with pytest.raises(AssertionError):
        _worked_example(cls, _oracle_err)
