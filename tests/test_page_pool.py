"""The host-side page pool (mla_pool_*): page ids for block tables, reference
counted prefix sharing with copy-on-fork of a partial page, eviction of the
pages before a position. Host only: these run without a GPU."""
import random
import threading

import pytest

NO_PAGES, INVALID = -8, -1


@pytest.fixture(scope="module")
def M():
    import mla_latent_kv_80_b300 as M
    return M


def table_row(pool, seq):
    return pool.block_table()[seq].tolist()


def test_fork_shares_full_pages_and_copies_the_partial_one(M):
    pool = M.PagePool(num_pages=32, page_size=16, max_seqs=4, max_pages_per_seq=12)
    a = pool.new_seq()
    pool.reserve(a, 100)                      # 7 pages, handed out from page 0
    assert table_row(pool, a)[:8] == [0, 1, 2, 3, 4, 5, 6, -1]
    b = pool.fork(a, 100)                     # pages 0-5 full and shared, page 6 holds 4 tokens
    rb = table_row(pool, b)
    assert rb[:6] == [0, 1, 2, 3, 4, 5] and rb[6] == 7 and rb[7] == -1
    assert [pool.page_refs(p) for p in range(8)] == [2, 2, 2, 2, 2, 2, 1, 1]
    src, dst = pool.take_copies()
    assert src.tolist() == [6] and dst.tolist() == [7]
    assert pool.take_copies()[0].numel() == 0  # the queue was emptied
    assert pool.seq_info(b) == (100, 0)
    # Appending to the child allocates its own pages; the parent's stay as they were.
    pool.reserve(b, 150)                      # ten pages: indices 7-9 are new
    assert table_row(pool, b)[7:11] == [8, 9, 10, -1] and table_row(pool, a)[6:8] == [6, -1]
    assert pool.free_pages() == 32 - 11


def test_page_aligned_fork_queues_no_copy(M):
    pool = M.PagePool(num_pages=16, page_size=16, max_seqs=2, max_pages_per_seq=8)
    a = pool.new_seq()
    pool.reserve(a, 64)
    b = pool.fork(a, 64)
    assert table_row(pool, b)[:5] == [0, 1, 2, 3, -1]
    assert pool.take_copies()[0].numel() == 0


def test_eviction_releases_pages_only_when_no_sequence_holds_them(M):
    pool = M.PagePool(num_pages=32, page_size=16, max_seqs=4, max_pages_per_seq=12)
    a = pool.new_seq()
    pool.reserve(a, 100)
    b = pool.fork(a, 96)
    free0 = pool.free_pages()
    pool.evict_before(a, 40)                  # pages 0 and 1 hold only positions < 40
    assert table_row(pool, a)[:3] == [-1, -1, 2]
    assert pool.seq_info(a) == (100, 40)
    assert pool.free_pages() == free0         # b still holds pages 0 and 1
    assert pool.page_refs(0) == 1 and pool.page_refs(1) == 1
    pool.free_seq(b)
    # b's references to pages 0-5 are gone: 0 and 1 return, 2-5 stay with a
    assert pool.free_pages() == free0 + 2
    assert [pool.page_refs(p) for p in range(7)] == [0, 0, 1, 1, 1, 1, 1]
    pool.evict_before(a, 10 ** 6)             # beyond the reserved length: everything it had
    assert pool.seq_info(a) == (100, 100)
    assert all(p == -1 for p in table_row(pool, a)[:6])


def test_exhaustion_and_bad_arguments_leave_the_pool_unchanged(M):
    pool = M.PagePool(num_pages=4, page_size=16, max_seqs=2, max_pages_per_seq=8)
    a = pool.new_seq()
    pool.reserve(a, 48)
    with pytest.raises(M.MlaError) as e:
        pool.reserve(a, 100)                  # 7 pages > 4
    assert e.value.code == NO_PAGES
    assert pool.free_pages() == 1 and table_row(pool, a)[:4] == [0, 1, 2, -1]
    b = pool.new_seq()
    with pytest.raises(M.MlaError) as e:
        pool.new_seq()                        # two sequence slots
    assert e.value.code == NO_PAGES
    with pytest.raises(M.MlaError) as e:
        pool.reserve(b, 16 * 9)               # more pages than a table row holds
    assert e.value.code == INVALID
    with pytest.raises(M.MlaError) as e:
        pool.fork(a, 49)                      # more than the parent holds
    assert e.value.code == INVALID
    pool.free_seq(b)
    with pytest.raises(M.MlaError) as e:
        pool.free_seq(b)                      # already free
    assert e.value.code == INVALID


class Model:
    """Plain restatement of the pool's rules, for the randomized comparison."""

    def __init__(self, n, ps, S, P):
        self.ps, self.P = ps, P
        self.refs = [0] * n
        self.free = list(range(n - 1, -1, -1))
        self.rows = [None] * S
        self.cap = [0] * S
        self.start = [0] * S

    def take(self):
        pg = self.free.pop()
        self.refs[pg] = 1
        return pg

    def drop(self, pg):
        if pg >= 0:
            self.refs[pg] -= 1
            if self.refs[pg] == 0:
                self.free.append(pg)

    def new_seq(self):
        for s, r in enumerate(self.rows):
            if r is None:
                self.rows[s], self.cap[s], self.start[s] = [-1] * self.P, 0, 0
                return s
        return None

    def reserve(self, s, n):
        need = -(-n // self.ps)
        if need > self.P:
            return INVALID
        have = -(-self.cap[s] // self.ps)
        missing = sum(1 for i in range(have, need) if self.rows[s][i] < 0)
        if missing > len(self.free):
            return NO_PAGES
        for i in range(have, need):
            if self.rows[s][i] < 0:
                self.rows[s][i] = self.take()
        self.cap[s] = max(self.cap[s], n)
        return 0

    def fork(self, a, k):
        if k > self.cap[a]:
            return INVALID, None
        full, part = k // self.ps, k % self.ps != 0
        if part and not self.free:
            return NO_PAGES, None
        c = self.new_seq()
        if c is None:
            return NO_PAGES, None
        for i in range(full):
            self.rows[c][i] = self.rows[a][i]
            if self.rows[a][i] >= 0:
                self.refs[self.rows[a][i]] += 1
        if part:
            self.rows[c][full] = self.take()
        self.cap[c], self.start[c] = k, min(self.start[a], k)
        return 0, c

    def evict(self, s, pos):
        pos = min(pos, self.cap[s])
        for i in range(pos // self.ps):
            self.drop(self.rows[s][i])
            self.rows[s][i] = -1
        self.start[s] = max(self.start[s], pos)

    def free_seq(self, s):
        for pg in self.rows[s]:
            self.drop(pg)
        self.rows[s] = None


def test_random_operations_follow_the_rules(M):
    n, ps, S, P = 40, 16, 6, 10
    pool = M.PagePool(n, ps, S, P)
    ref = Model(n, ps, S, P)
    rng = random.Random(11)
    for _ in range(600):
        live = [s for s, r in enumerate(ref.rows) if r is not None]
        op = rng.choice(["new", "reserve", "fork", "evict", "free"])
        if op == "new" or not live:
            s = ref.new_seq()
            if s is None:
                with pytest.raises(M.MlaError):
                    pool.new_seq()
            else:
                assert pool.new_seq() == s
        elif op == "reserve":
            s, k = rng.choice(live), rng.randrange(0, P * ps + 20)
            rc = ref.reserve(s, k)
            if rc:
                with pytest.raises(M.MlaError) as e:
                    pool.reserve(s, k)
                assert e.value.code == rc
            else:
                pool.reserve(s, k)
        elif op == "fork":
            a = rng.choice(live)
            k = rng.randrange(0, ref.cap[a] + 1)
            rc, c = ref.fork(a, k)
            if rc:
                with pytest.raises(M.MlaError):
                    pool.fork(a, k)
            else:
                assert pool.fork(a, k) == c
        elif op == "evict":
            s = rng.choice(live)
            pos = rng.randrange(0, ref.cap[s] + ps + 1)
            ref.evict(s, pos)
            pool.evict_before(s, pos)
        else:
            s = rng.choice(live)
            ref.free_seq(s)
            pool.free_seq(s)
        pool.take_copies()
        t = pool.block_table()
        for s, r in enumerate(ref.rows):
            if r is not None:
                assert t[s].tolist() == r
                assert pool.seq_info(s) == (ref.cap[s], ref.start[s])
        assert pool.free_pages() == len(ref.free)
        assert [pool.page_refs(p) for p in range(n)] == ref.refs


def test_concurrent_sequences_keep_the_pool_consistent(M):
    pool = M.PagePool(num_pages=4000, page_size=16, max_seqs=64, max_pages_per_seq=64)
    errors = []

    def worker(k):
        try:
            for i in range(30):
                s = pool.new_seq()
                L = 16 * (1 + (k + i) % 20)
                pool.reserve(s, L)
                c = pool.fork(s, min(L, 16 * ((k + i) % 3) + 5))
                pool.evict_before(s, 16)
                pool.free_seq(c)
                pool.free_seq(s)
        except Exception as exc:  # pragma: no cover
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors
    assert pool.free_pages() == 4000
