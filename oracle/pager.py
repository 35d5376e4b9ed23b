"""Host page allocator model for the oracle (test infrastructure only).

A plain-Python statement of the allocator the library's lnk_pager implements,
used to check it operation by operation.

Source: "Mistral 7B Instruct v0.3", Entries table (prefill_paged: each token
attends over its row's pages up to its position -- chunks, shared prefixes).
The pages do not say how pages are handed out; the reading taken is the
plainest allocator that lets rows share the pages of a common prefix:

  * free pages are handed out lowest page number first;
  * a page's count is the number of table entries that map it;
  * fork(src, dst, n): the empty row dst maps src's first ceil(n / 64) pages;
  * prepare_append(rows, positions): before the tokens are written, the first
    token of the batch writing into a logical page maps a fresh page if the
    entry is unmapped, or, if the page is mapped by other entries too, maps a
    fresh page instead and records (old, new) for a copy of the contents;
  * release(row): the row's entries are unmapped; a page whose count reaches
    zero is free again.
  * A call that fails (bad row, position past the table row, too few free
    pages) changes nothing.
"""
PAGE_SIZE = 64
UNMAPPED = -1


class PagerError(Exception):
    def __init__(self, code: str):
        super().__init__(code)
        self.code = code  # "EINVAL", "ERANGE" or "ENOSPACE"


class Pager:
    def __init__(self, num_pages: int, num_rows: int, pages_per_row: int):
        if num_pages <= 0 or num_rows <= 0 or pages_per_row <= 0:
            raise PagerError("EINVAL")
        self.num_pages, self.num_rows, self.pages_per_row = num_pages, num_rows, pages_per_row
        self.rows = [[UNMAPPED] * pages_per_row for _ in range(num_rows)]
        self.count = [0] * num_pages
        self.free = set(range(num_pages))

    # -- helpers --
    def _take(self) -> int:
        page = min(self.free)
        self.free.remove(page)
        self.count[page] = 1
        return page

    def _check_row(self, row):
        if not 0 <= row < self.num_rows:
            raise PagerError("EINVAL")

    # -- operations --
    def reserve(self, row: int, length: int):
        self._check_row(row)
        if length < 0:
            raise PagerError("EINVAL")
        if length > self.pages_per_row * PAGE_SIZE:
            raise PagerError("ERANGE")
        n = -(-length // PAGE_SIZE)
        missing = [lp for lp in range(n) if self.rows[row][lp] == UNMAPPED]
        if len(missing) > len(self.free):
            raise PagerError("ENOSPACE")
        for lp in missing:
            self.rows[row][lp] = self._take()

    def fork(self, src: int, dst: int, length: int):
        self._check_row(src)
        self._check_row(dst)
        if src == dst or length <= 0:
            raise PagerError("EINVAL")
        if length > self.pages_per_row * PAGE_SIZE:
            raise PagerError("ERANGE")
        n = -(-length // PAGE_SIZE)
        if any(e != UNMAPPED for e in self.rows[dst]):
            raise PagerError("EINVAL")
        if any(self.rows[src][lp] == UNMAPPED for lp in range(n)):
            raise PagerError("EINVAL")
        for lp in range(n):
            page = self.rows[src][lp]
            self.rows[dst][lp] = page
            self.count[page] += 1

    def prepare_append(self, rows, positions):
        tokens = [(int(r), int(p)) for r, p in zip(rows, positions)]
        for row, pos in tokens:  # every token is checked before anything changes
            if pos < 0:
                continue
            self._check_row(row)
            if pos >= self.pages_per_row * PAGE_SIZE:
                raise PagerError("ERANGE")
        saved = ([list(r) for r in self.rows], list(self.count), set(self.free))
        copies, done = [], set()
        try:
            for row, pos in tokens:
                if pos < 0:
                    continue
                lp = pos // PAGE_SIZE
                if (row, lp) in done:
                    continue
                done.add((row, lp))
                page = self.rows[row][lp]
                if page == UNMAPPED:
                    if not self.free:
                        raise PagerError("ENOSPACE")
                    self.rows[row][lp] = self._take()
                elif self.count[page] > 1:
                    if not self.free:
                        raise PagerError("ENOSPACE")
                    new = self._take()
                    self.count[page] -= 1
                    self.rows[row][lp] = new
                    copies.append((page, new))
        except PagerError:
            self.rows, self.count, self.free = saved
            raise
        return copies

    def release(self, row: int):
        self._check_row(row)
        for lp, page in enumerate(self.rows[row]):
            if page != UNMAPPED:
                self.count[page] -= 1
                if self.count[page] == 0:
                    self.free.add(page)
                self.rows[row][lp] = UNMAPPED

    def table(self):
        return [list(r) for r in self.rows]

    def free_pages(self) -> int:
        return len(self.free)

    def refcount(self, page: int) -> int:
        return self.count[page] if 0 <= page < self.num_pages else -1
