"""The native host block manager (pkv_bm_*) against a plain Python model of
the pages' allocator, on random operation sequences (CPU only):

* free list and reference counts ("KV Cache & PagedAttention", section 4);
* prefix sharing of whole blocks from position 0, keyed here by the exact
  token history itself (the native one keys by a chained hash and checks
  the tokens: the two must agree) ("gpu_paged_kv_cache", "Prefix sharing,
  reference counts, and copy-on-write"; "PagedAttention internals", 04);
* copy-on-write of a shared tail; LRU eviction of unreferenced cached
  blocks, referenced blocks never evicted (section 04); a watermark of
  blocks admissions may not take; swap out / in bookkeeping
  ("gpu_paged_kv_cache", "Reclaiming memory: swap versus recompute")."""
import numpy as np
import pytest

import paged_kv_cache_112_gb300 as pkv
from paged_kv_cache_112_gb300 import build as pkv_build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        pkv_build.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    pkv.load()


class Model:
    """Reference allocator, written for clarity: the same policy as the native
    one (free list popped from the end, freed blocks pushed there; evictable
    cached blocks in least-recently-released order)."""

    def __init__(self, nb, bs, wm):
        self.nb, self.bs, self.wm = nb, bs, wm
        self.ref = [0] * nb
        self.key = [None] * nb          # cached block -> its history key
        self.free = list(range(nb - 1, -1, -1))
        self.evictable = []             # front = least recently released
        self.cache = {}                 # history key -> block
        self.seqs = {}                  # id -> dict(table, tokens, extra, swapped)
        self.count = dict(prompt_tokens=0, prompt_tokens_cached=0, evictions=0, cow_copies=0, swap_outs=0,
                          refusals=0)

    def avail(self):
        return len(self.free) + len(self.evictable)

    def _take(self):
        if self.free:
            b = self.free.pop()
        elif self.evictable:
            b = self.evictable.pop(0)
            self.count["evictions"] += 1
            del self.cache[self.key[b]]
            self.key[b] = None
        else:
            return None
        self.ref[b] = 1
        return b

    def _add_ref(self, b):
        if self.ref[b] == 0 and self.key[b] is not None:
            self.evictable.remove(b)
        self.ref[b] += 1

    def _drop_ref(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            (self.evictable if self.key[b] is not None else self.free).append(b)

    def _register(self, s, i):
        key = (s["extra"], tuple(s["tokens"][: (i + 1) * self.bs]))
        b = s["table"][i]
        if self.key[b] is not None or key in self.cache:
            return
        self.key[b] = key
        self.cache[key] = b

    def add(self, sid, tokens, extra):
        if sid in self.seqs:
            return "invalid", None
        B = self.bs
        hits = []
        for i in range(len(tokens) // B):
            b = self.cache.get((extra, tuple(tokens[: (i + 1) * B])))
            if b is None:
                break
            hits.append(b)
        need = -(-len(tokens) // B) - len(hits)
        hit_evictable = sum(1 for b in hits if self.ref[b] == 0)
        if need > self.avail() - hit_evictable - self.wm:
            self.count["refusals"] += 1
            return "oob", None
        s = dict(table=[], tokens=list(tokens), extra=extra, swapped=False)
        for b in hits:
            self._add_ref(b)
            s["table"].append(b)
        for _ in range(need):
            s["table"].append(self._take())
        cached = len(hits) * B
        self.count["prompt_tokens"] += len(tokens)
        self.count["prompt_tokens_cached"] += cached
        slots = [-1 if t < cached else s["table"][t // B] * B + t % B for t in range(len(tokens))]
        for i in range(len(hits), len(tokens) // B):
            self._register(s, i)
        self.seqs[sid] = s
        return cached, slots

    def fork(self, parent, child):
        if parent not in self.seqs or self.seqs[parent]["swapped"] or child in self.seqs:
            return "invalid"
        p = self.seqs[parent]
        for b in p["table"]:
            self._add_ref(b)
        self.seqs[child] = dict(table=list(p["table"]), tokens=list(p["tokens"]), extra=p["extra"], swapped=False)
        return "ok"

    def append(self, sid, tok):
        s = self.seqs.get(sid)
        if s is None or s["swapped"]:
            return "invalid"
        B, pos = self.bs, len(s["tokens"])
        cow = None
        if pos % B == 0:
            b = self._take()
            if b is None:
                self.count["refusals"] += 1
                return "oob"
            s["table"].append(b)
        else:
            tail = s["table"][pos // B]
            if self.ref[tail] > 1:
                b = self._take()
                if b is None:
                    self.count["refusals"] += 1
                    return "oob"
                self._drop_ref(tail)
                s["table"][pos // B] = b
                cow = (tail, b)
                self.count["cow_copies"] += 1
        s["tokens"].append(tok)
        slot = s["table"][pos // B] * B + pos % B
        if (pos + 1) % B == 0:
            self._register(s, pos // B)
        return slot, cow

    def free_seq(self, sid):
        s = self.seqs.pop(sid, None)
        if s is None:
            return "invalid"
        if not s["swapped"]:
            for b in reversed(s["table"]):
                self._drop_ref(b)
        return "ok"

    def swap_out(self, sid):
        s = self.seqs.get(sid)
        if s is None or s["swapped"]:
            return "invalid"
        blocks = list(s["table"])
        for b in reversed(blocks):
            self._drop_ref(b)
        s["table"], s["swapped"] = [], True
        self.count["swap_outs"] += 1
        return blocks

    def swap_in(self, sid):
        s = self.seqs.get(sid)
        if s is None or not s["swapped"]:
            return "invalid"
        n = -(-len(s["tokens"]) // self.bs)
        if n > self.avail() - self.wm:
            self.count["refusals"] += 1
            return "oob"
        s["table"] = [self._take() for _ in range(n)]
        s["swapped"] = False
        for i in range(len(s["tokens"]) // self.bs):
            self._register(s, i)
        return s["table"]

    def swap_in_cached(self, sid):
        s = self.seqs.get(sid)
        if s is None or not s["swapped"]:
            return "invalid"
        B = self.bs
        hits = []
        for i in range(len(s["tokens"]) // B):
            b = self.cache.get((s["extra"], tuple(s["tokens"][: (i + 1) * B])))
            if b is None:
                break
            hits.append(b)
        n = -(-len(s["tokens"]) // B)
        need = n - len(hits)
        if need > self.avail() - sum(1 for b in hits if self.ref[b] == 0) - self.wm:
            self.count["refusals"] += 1
            return "oob"
        for b in hits:
            self._add_ref(b)
        s["table"] = hits + [self._take() for _ in range(need)]
        s["swapped"] = False
        for i in range(len(hits), len(s["tokens"]) // B):
            self._register(s, i)
        return s["table"], [0] * len(hits) + [1] * need


def _same_state(bm, m):
    assert bm.available_blocks == m.avail()
    assert bm.cached_blocks == len(m.cache)
    assert [bm.refcount(b) for b in range(m.nb)] == m.ref
    for sid, s in m.seqs.items():
        assert bm.seq_len(sid) == len(s["tokens"])
        if not s["swapped"]:
            assert bm.block_table(sid).tolist() == s["table"]
    # conservation: every reference is a table entry of a resident sequence
    assert sum(m.ref) == sum(len(s["table"]) for s in m.seqs.values())
    live = {b for b in range(m.nb) if m.ref[b] > 0}
    assert live.isdisjoint(m.free) and live.isdisjoint(m.evictable)
    assert len(live) + len(m.free) + len(m.evictable) == m.nb
    # operating signals: gauges from the model's state, counters kept beside it
    resident = [s for s in m.seqs.values() if not s["swapped"]]
    fill = [0] * m.nb
    for s in resident:
        for j, b in enumerate(s["table"]):
            fill[b] = max(fill[b], min(m.bs, len(s["tokens"]) - j * m.bs))
    want = dict(num_blocks=m.nb, block_size=m.bs, blocks_free=len(m.free), blocks_cached_unreferenced=len(m.evictable),
                blocks_referenced=len(live), blocks_cached=len(m.cache), slots_holding_tokens=sum(fill),
                sequences_resident=len(resident), sequences_swapped=len(m.seqs) - len(resident),
                table_entries=sum(len(s["table"]) for s in resident),
                max_blocks_per_sequence=max((len(s["table"]) for s in resident), default=0), **m.count)
    assert bm.stats() == want


def _call(fn, *a):
    try:
        return fn(*a)
    except pkv.OutOfBlocks:
        return "oob"
    except pkv.PkvError:
        return "invalid"


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(seed):
    rng = np.random.default_rng(seed)
    nb, bs, wm = int(rng.choice([24, 40])), int(rng.choice([4, 8, 16])), int(rng.integers(0, 4))
    bm, m = pkv.BlockManager(nb, bs, wm), Model(nb, bs, wm)
    system = [int(x) for x in rng.integers(0, 50, size=3 * bs)]  # a shared "system prompt"
    next_id = 0
    for _ in range(400):
        op = rng.choice(["add", "add", "append", "append", "append", "fork", "free", "swap_out", "swap_in",
                         "swap_in_cached", "bad"])
        ids = list(m.seqs)
        if op == "add":
            n_sys = int(rng.integers(0, 4)) * bs - int(rng.integers(0, 2))
            tail = [int(x) for x in rng.integers(0, 50, size=int(rng.integers(0, 2 * bs)))]
            toks = system[: max(0, n_sys)] + tail
            extra = int(rng.integers(0, 2))
            want = m.add(next_id, toks, extra)
            got = _call(bm.add_sequence, next_id, toks, extra)
            if isinstance(want[0], str):
                assert got == want[0]
                m.seqs.pop(next_id, None)
            else:
                assert got[0] == want[0] and got[1].tolist() == want[1]
            next_id += 1
        elif op == "append" and ids:
            sid = int(rng.choice(ids))
            tok = int(rng.integers(0, 50))
            want = m.append(sid, tok)
            got = _call(bm.append, sid, tok)
            assert got == want, (got, want)
        elif op == "fork" and ids:
            parent = int(rng.choice(ids))
            want = m.fork(parent, next_id)
            got = _call(bm.fork, parent, next_id)
            assert (got is None and want == "ok") or got == want
            next_id += 1
        elif op == "free" and ids:
            sid = int(rng.choice(ids))
            assert _call(bm.free, sid) is None and m.free_seq(sid) == "ok"
        elif op == "swap_out" and ids:
            sid = int(rng.choice(ids))
            want = m.swap_out(sid)
            got = _call(bm.swap_out, sid)
            assert (got == want) if isinstance(want, str) else got.tolist() == want
        elif op == "swap_in" and ids:
            sid = int(rng.choice(ids))
            want = m.swap_in(sid)
            got = _call(bm.swap_in, sid)
            assert (got == want) if isinstance(want, str) else got.tolist() == want
        elif op == "swap_in_cached" and ids:
            sid = int(rng.choice(ids))
            want = m.swap_in_cached(sid)
            got = _call(bm.swap_in_cached, sid)
            if isinstance(want, str):
                assert got == want
            else:
                assert got[0].tolist() == want[0] and got[1].tolist() == want[1]
        elif op == "bad":
            assert _call(bm.append, 10 ** 9, 1) == "invalid"
            assert _call(bm.fork, 10 ** 9, 10 ** 9 + 1) == "invalid"
        _same_state(bm, m)


def test_prefix_hit_needs_the_same_history_and_key():
    B = 4
    bm = pkv.BlockManager(16, B)
    a = list(range(10))
    assert bm.add_sequence(1, a)[0] == 0
    cached, slots = bm.add_sequence(2, a[:9])  # two whole blocks of the same history
    assert cached == 8 and (slots[:8] == -1).all() and slots[8] >= 0
    assert bm.block_table(2)[:2].tolist() == bm.block_table(1)[:2].tolist()
    assert bm.add_sequence(3, a, extra_key=7)[0] == 0          # another adapter: no sharing
    assert bm.add_sequence(4, [99] + a[1:])[0] == 0             # differs in block 0: nothing shared
    assert bm.add_sequence(5, a[:4] + [77, 5, 6, 7, 8])[0] == 4  # block 1 differs: only block 0 shared
    assert bm.add_sequence(6, a[4:])[0] == 0                   # same tokens, not from position 0


def test_copy_on_write_of_a_forked_tail():
    B = 4
    bm = pkv.BlockManager(8, B)
    bm.add_sequence(1, [1, 2, 3, 4, 5, 6])  # block 1 half full
    bm.fork(1, 2)
    t1 = bm.block_table(1)
    assert bm.refcount(int(t1[1])) == 2
    slot, cow = bm.append(2, 9)  # the child writes first: it copies
    t2 = bm.block_table(2)
    assert cow == (int(t1[1]), int(t2[1])) and slot == t2[1] * B + 2
    assert bm.refcount(int(t1[1])) == 1 and bm.refcount(int(t2[1])) == 1
    slot, cow = bm.append(1, 8)  # the parent's block is its own again: no copy
    assert cow is None and slot == t1[1] * B + 2


def test_lru_eviction_spares_referenced_blocks():
    B = 4
    bm = pkv.BlockManager(6, B)
    bm.add_sequence(1, [1] * 8)          # blocks for [1]*4, [1]*8 cached
    bm.add_sequence(2, [2] * 8)
    bm.free(1)                           # sequence 1's blocks: evictable, released first
    assert bm.available_blocks == 4 and bm.cached_blocks == 4
    bm.add_sequence(3, [3] * 12)         # needs 3: takes the 2 free ones, then evicts sequence 1's oldest
    assert bm.cached_blocks == 4 + 3 - 1
    assert bm.add_sequence(4, [2] * 8)[0] == 8  # sequence 2's blocks were referenced: still cached
    with pytest.raises(pkv.OutOfBlocks):
        bm.add_sequence(5, [5] * 20)


def test_watermark_reserves_blocks_for_appends():
    B = 4
    bm = pkv.BlockManager(4, B, watermark_blocks=1)
    bm.add_sequence(1, [1] * 12)  # 3 blocks: all but the watermark
    with pytest.raises(pkv.OutOfBlocks):
        bm.add_sequence(2, [2])
    assert bm.append(1, 5)[0] == bm.block_table(1)[3] * B  # an append may take the reserve


def test_c_abi_guards():
    lib = pkv.load()
    assert not lib.pkv_bm_create(0, 16, 0) and not lib.pkv_bm_create(8, 16, 9)
    assert not lib.pkv_bm_create(2, 2 ** 30, 0)  # 2^31 slots: beyond int32
    edge = lib.pkv_bm_create(1, 2 ** 31 - 1, 0)  # the largest slot count that fits
    assert edge
    lib.pkv_bm_destroy(edge)
    assert lib.pkv_bm_available_blocks(None) == -pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_bm_free_sequence(None, 1) == -pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_bm_get_stats(None, None) == -pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_bm_decode_step(None, None, None, 1, None, None, None, 4, -1, None) == -pkv.PKV_ERR_INVALID_ARG
    bm = pkv.BlockManager(4, 16)
    assert lib.pkv_bm_get_stats(bm._h, None) == -pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_bm_decode_step(bm._h, None, None, 0, None, None, None, 0, -1, None) == 0  # empty batch
    assert lib.pkv_bm_decode_step(bm._h, None, None, 1, None, None, None, 4, -1, None) == -pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError):
        bm.add_sequence(1, [1, 2])
        bm.add_sequence(1, [3])  # duplicate id
    with pytest.raises(pkv.PkvError):
        bm.swap_in(1)  # not swapped out
    with pytest.raises(pkv.PkvError):
        bm.block_table(99)
    bm.swap_out(1)
    with pytest.raises(pkv.PkvError):
        bm.append(1, 5)  # swapped out: no appends until swap_in
    assert bm.swap_in(1).size == 1 and bm.append(1, 5)[0] >= 0


def test_concurrent_threads_keep_the_books():
    """Four threads drive one manager at once (ctypes releases the GIL for
    each call, so the C++ runs in parallel behind the manager's mutex).  The
    threads share system prompts, so they hit, share and evict one another's
    cached blocks.  Afterwards every block's refcount equals the number of
    table rows that hold it, and the free and evictable lists hold exactly the
    unreferenced blocks; freeing everything returns the whole pool."""
    import threading

    B, NB = 16, 96
    bm = pkv.BlockManager(NB, B, watermark_blocks=2)
    prompts = [[int(x) for x in np.random.default_rng(p).integers(0, 50, size=3 * B)] for p in range(3)]
    live = {}
    errors = []

    def worker(w):
        rng = np.random.default_rng(1000 + w)
        mine = {}  # id -> (tokens, swapped)
        next_id = w * 1_000_000
        try:
            for _ in range(1500):
                op = rng.integers(0, 6)
                ids = sorted(mine)
                try:
                    if op == 0 or not ids:
                        p = prompts[rng.integers(0, 3)]
                        toks = p[: rng.integers(1, len(p) + 1)] + [int(x) for x in rng.integers(0, 50, rng.integers(0, 9))]
                        bm.add_sequence(next_id, toks)
                        mine[next_id] = (toks, False)
                        next_id += 1
                    elif op == 1:
                        sid = ids[rng.integers(0, len(ids))]
                        toks, sw = mine[sid]
                        if not sw:
                            tok = int(rng.integers(0, 50))
                            bm.append(sid, tok)
                            mine[sid] = (toks + [tok], False)
                    elif op == 2:
                        sid = ids[rng.integers(0, len(ids))]
                        toks, sw = mine[sid]
                        if not sw:
                            bm.fork(sid, next_id)
                            mine[next_id] = (list(toks), False)
                            next_id += 1
                    elif op == 3:
                        sid = ids[rng.integers(0, len(ids))]
                        bm.free(sid)
                        del mine[sid]
                    elif op == 4:
                        sid = ids[rng.integers(0, len(ids))]
                        toks, sw = mine[sid]
                        if sw:
                            bm.swap_in(sid)
                        else:
                            bm.swap_out(sid)
                        mine[sid] = (toks, not sw)
                    else:
                        sid = ids[rng.integers(0, len(ids))]
                        toks, sw = mine[sid]
                        assert bm.seq_len(sid) == len(toks)
                        if not sw:
                            assert len(bm.block_table(sid)) == -(-len(toks) // B)
                except pkv.OutOfBlocks:
                    pass
            live.update(mine)
        except Exception as e:  # surfaced in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(w,)) for w in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    holders = np.zeros(NB, dtype=np.int64)
    for sid, (toks, sw) in live.items():
        assert bm.seq_len(sid) == len(toks)
        if not sw:
            table = bm.block_table(sid)
            assert len(table) == -(-len(toks) // B)
            np.add.at(holders, table, 1)
    refs = np.array([bm.refcount(b) for b in range(NB)])
    assert np.array_equal(refs, holders)
    assert bm.available_blocks == int(np.sum(refs == 0))
    for sid in live:
        bm.free(sid)
    assert bm.available_blocks == NB


def _books(bm, ids, nb):
    """Everything observable about a manager's state for `ids`."""
    return ([bm.seq_len(i) for i in ids], [bm.block_table(i).tolist() for i in ids],
            [bm.refcount(b) for b in range(nb)], bm.available_blocks, bm.cached_blocks)


def test_decode_step_equals_appends_one_by_one():
    """pkv_bm_decode_step over a batch gives the slots, copy-on-write pairs,
    tables and lengths of the same appends made one call at a time, on a twin
    manager, through admissions with prefix hits, forks (parallel samples
    whose shared tails get copied) and frees."""
    B, NB = 16, 200
    a, b = pkv.BlockManager(NB, B), pkv.BlockManager(NB, B)
    rng = np.random.default_rng(7)
    system = [int(x) for x in rng.integers(0, 100, size=2 * B + 5)]
    live, next_id = [], 0
    for step in range(120):
        if step % 10 == 0 and len(live) < 12:  # admit one, fork another
            toks = system + [int(x) for x in rng.integers(0, 100, size=rng.integers(0, 20))]
            for m in (a, b):
                m.add_sequence(next_id, toks)
            live.append(next_id)
            parent = live[int(rng.integers(0, len(live)))]
            for m in (a, b):
                m.fork(parent, next_id + 1)
            live.append(next_id + 1)
            next_id += 2
        if step % 17 == 16 and len(live) > 4:
            gone = live.pop(int(rng.integers(0, len(live))))
            for m in (a, b):
                m.free(gone)
        batch = [i for i in live if rng.random() < 0.8]
        if not batch:
            continue
        toks = [int(x) for x in rng.integers(0, 100, size=len(batch))]
        width = max(-(-(a.seq_len(i) + 1) // B) for i in batch) + int(rng.integers(0, 3))
        slots, lens, tables, pairs = a.decode_step(batch, toks, width)
        want_pairs = []
        for i, (sid, t) in enumerate(zip(batch, toks)):
            slot, cow = b.append(sid, t)
            assert slots[i] == slot
            if cow:
                want_pairs.append(cow)
            assert lens[i] == b.seq_len(sid)
            row = b.block_table(sid)
            assert tables[i, : len(row)].tolist() == row.tolist() and np.all(tables[i, len(row):] == -1)
        assert pairs.tolist() == [list(p) for p in want_pairs]
    assert _books(a, live, NB) == _books(b, live, NB)


def test_decode_step_sibling_tails_copy_once():
    """Two samples forked from one sequence share its partial tail: in one
    batch the first copies it on write, the second then owns it and appends
    in place (one pair)."""
    B = 16
    bm = pkv.BlockManager(16, B)
    bm.add_sequence(1, list(range(20)))
    bm.fork(1, 2)
    tail = int(bm.block_table(1)[1])
    slots, lens, tables, pairs = bm.decode_step([1, 2], [5, 6], 2)
    assert pairs.shape == (1, 2) and pairs[0, 0] == tail and pairs[0, 1] != tail
    assert tables[0, 1] == pairs[0, 1] and tables[1, 1] == tail
    assert slots.tolist() == [int(pairs[0, 1]) * B + 4, tail * B + 4] and lens.tolist() == [21, 21]
    assert bm.refcount(tail) == 1


def test_decode_step_is_all_or_nothing():
    B, NB = 16, 4
    bm = pkv.BlockManager(NB, B)
    bm.add_sequence(1, list(range(16)))       # one full block: its next token needs a fresh one
    bm.add_sequence(2, list(range(100, 132)))  # two full blocks
    bm.fork(2, 3)
    before = _books(bm, [1, 2, 3], NB)
    assert bm.available_blocks == 1
    with pytest.raises(pkv.OutOfBlocks):  # three fresh blocks wanted, one left
        bm.decode_step([1, 2, 3], [7, 8, 9], 4)
    assert _books(bm, [1, 2, 3], NB) == before
    assert bm.stats()["refusals"] == 1
    for bad in (dict(ids=[1, 1], toks=[1, 2], w=4),   # repeated sequence
                dict(ids=[1, 9], toks=[1, 2], w=4),   # unknown sequence
                dict(ids=[2], toks=[1], w=2)):        # row too narrow after the append (3 blocks)
        with pytest.raises(pkv.PkvError):
            bm.decode_step(bad["ids"], bad["toks"], bad["w"])
        assert _books(bm, [1, 2, 3], NB) == before
    bm.swap_out(3)
    with pytest.raises(pkv.PkvError):  # swapped out
        bm.decode_step([3], [1], 4)
    slots, lens, tables, pairs = bm.decode_step([1], [7], 4, pad_value=0)
    assert lens.tolist() == [17] and pairs.shape == (0, 2) and tables[0, 2:].tolist() == [0, 0]
    s0, l0, t0, p0 = bm.decode_step([], [], 4)
    assert s0.size == 0 and p0.shape == (0, 2)


def test_swap_in_reuses_cached_prefix_blocks():
    """A preempted sequence sharing a system prompt: on resume its prompt
    blocks are still cached (another sequence holds them), so only its
    private blocks come back from the host; once nobody holds the prompt and
    its blocks are evicted, everything comes back from the host."""
    B = 16
    bm = pkv.BlockManager(12, B)
    system = list(range(1000, 1000 + 3 * B))
    bm.add_sequence(1, system + [1, 2, 3])
    bm.add_sequence(2, system + [4, 5, 6, 7])
    shared = bm.block_table(2)[:3].tolist()
    out = bm.swap_out(2)
    assert out.tolist()[:3] == shared and len(out) == 4
    blocks, from_host = bm.swap_in_cached(2)
    assert blocks[:3].tolist() == shared and from_host.tolist() == [0, 0, 0, 1]
    assert [bm.refcount(b) for b in shared] == [2, 2, 2]
    # nobody else holds the prompt and the pool is reused.  free(1) releases its table back to front,
    # so prompt block 0 is the most recently released: taking 11 of the 12 blocks evicts blocks 2 and
    # 1 of the prompt but not block 0, which is still a hit; the chain stops at block 1's miss.
    bm.swap_out(2)
    bm.free(1)
    bm.add_sequence(3, list(range(5000, 5000 + 11 * B)))
    bm.free(3)
    blocks, from_host = bm.swap_in_cached(2)
    assert blocks[0] == shared[0] and from_host.tolist() == [0, 1, 1, 1]
    # all twelve blocks taken: nothing of the prompt is left, everything comes from the host
    bm.swap_out(2)
    bm.add_sequence(4, list(range(7000, 7000 + 12 * B)))
    bm.free(4)
    blocks, from_host = bm.swap_in_cached(2)
    assert from_host.tolist() == [1, 1, 1, 1]
    st = bm.stats()
    assert st["swap_outs"] == 3 and st["evictions"] >= 3


def test_pool_blocks_matches_the_pages_sizing():
    """pkv_pool_blocks against the pages' printed pool ("PagedAttention
    internals", 05: an 8B-class model, 32 layers x 8 KV heads x 128 x fp16,
    2 MiB blocks of 16 tokens, 54 GiB of KV -> 27,648 blocks) and against the
    oracle's closed forms on drawn sizes; FP8 pools add a K and a V scale per
    layer and KV head."""
    import oracle.sizing as Z

    GiB = 2 ** 30
    assert pkv.pool_blocks(54 * GiB, 32, 16, 8, 128) == 27648
    assert pkv.pool_blocks(2 * 2 ** 20 - 1, 32, 16, 8, 128) == 0
    rng = np.random.default_rng(3)
    for _ in range(200):
        L, B, H, D, eb = (int(rng.integers(1, 100)), int(rng.choice([8, 16, 32, 64])), int(rng.integers(1, 17)),
                          int(rng.choice([64, 128, 256])), int(rng.choice([1, 2, 4])))
        budget = int(rng.integers(0, 300 * GiB))
        assert pkv.pool_blocks(budget, L, B, H, D, eb) == Z.pool_blocks(budget, Z.block_bytes(L, H, D, eb, B))
    # FP8: one-layer pool of the 8B-class row, 16-token blocks: 32 KiB of codes + 8 heads x 2 scales x 4 B
    assert pkv.pool_blocks(10 * (32768 + 64), 1, 16, 8, 128, elem_bytes=1, with_scales=True) == 10
    with pytest.raises(pkv.PkvError):
        pkv.pool_blocks(GiB, 0, 16, 8, 128)


def test_recompute_preemption_with_the_history():
    """Preemption by recompute: swap out without moving anything, resume with
    swap_in_cached, and recompute exactly the tokens of the from_host blocks
    (their slots from the new table) from the kept history; the shared prompt
    blocks come back from the prefix cache."""
    B = 16
    bm = pkv.BlockManager(16, B)
    system = list(range(500, 500 + 2 * B))
    bm.add_sequence(1, system)
    toks = system + [1, 2, 3, 4, 5]
    bm.add_sequence(2, toks)
    for t in (6, 7):
        bm.append(2, t)
    history = toks + [6, 7]
    assert bm.tokens(2).tolist() == history
    bm.swap_out(2)  # recompute: nothing is copied
    assert bm.tokens(2).tolist() == history  # kept while swapped out
    blocks, from_host = bm.swap_in_cached(2)
    assert from_host.tolist() == [0, 0, 1]
    redo = [t for t in range(len(history)) if from_host[t // B]]
    slots = [int(blocks[t // B]) * B + t % B for t in redo]
    assert redo == list(range(2 * B, len(history))) and len(set(slots)) == len(slots)
    assert bm.block_table(2).tolist() == blocks.tolist()
    assert bm.tokens(1).tolist() == system
    with pytest.raises(pkv.PkvError):
        bm.tokens(99)
