"""Models of the mbarrier protocols of the forward kernels, run under random
interleavings on the CPU.

Each kernel role (TMA producer, MMA issuers, softmax groups) becomes a
generator that yields the barrier waits it makes in the kernel's order;
MMAs and TMA copies complete asynchronously, in issue order per source; an
mbarrier keeps the hardware's phase/parity rule (a parity wait is satisfied
once the barrier's phase parity differs from the one asked for).  A run
checks that no schedule deadlocks and that the facts the kernels rely on
hold (a stage is refilled only after every reader released it, O is read
before the next p v overwrites it, epilogues run in tile order, narrow rows
are widened from the copy that landed for that block, in place in its
stage or from the NVFP4 staging tile before it is refilled).  A timeout on
the GPU would only show such a race as a flag; the model finds it without
one.

Covered: k_fwd's decode phase (a 3-stage K/V ring, two MMA issuers, one
for S^T and one for O^T, 16-bit caches and widened ones, whose narrow rows land in the
stage and are widened in place), its KV-stationary phase (16-bit, FP8
widened in place, NVFP4 through a staging tile) and k_dense.
The dense model without the wait that an empty tile makes before it
publishes O reproduces the race that wait removes (o_full completing twice
ahead of the softmax group's parity wait).
"""
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase = name, count, 0, 0
    def arrive(self):
        self.pending += 1
        assert self.pending <= self.count, self.name
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1
    def ready(self, parity):
        return (self.phase & 1) != parity


def run_fwd_kv_stationary(items, seed, kind="16"):
    """items: list of tile counts (1..4) of the items this CTA claims.
    kind: "16" (16-bit caches), "fp8" (e4m3 rows land in the item's own
    stage and are widened in place) or "fp4" (NVFP4 rows land in one
    staging tile, widened into the stage)."""
    widened_kind = kind != "16"
    rnd = random.Random(seed)
    B = {}
    def bar(n, c=1): B[n] = Bar(n, c)
    for i in range(2):
        bar(f"kv_full{i}"); bar(f"kv_empty{i}", 4)  # 2 issuers + 2 groups (256 threads)
        bar(f"q_full{i}"); bar(f"s_full{i}"); bar(f"p_full{i}"); bar(f"o_full{i}")
    bar("epi_turn0"); bar("epi_turn1"); bar("done", 2)
    bar("stg_full0"); bar("stg_full1"); bar("stg_empty")
    staging = [None]
    widened = {}
    info = [None, None]
    stage_item = [None, None]
    stage_raw = [None, None]        # the item whose narrow rows landed in the stage (fp8)
    stage_readers = {}
    pending = {}
    def later(src, cb): pending.setdefault(src, []).append(cb)
    # ground truth
    q_buf = {0: None, 1: None}      # tile whose q is in group g's buffer (landed)
    S = {0: None, 1: None}          # ('S'|'P', tile)
    O = {0: None, 1: None}          # ('pending'|'done'|'read', tile)
    epi_done = []
    claim = [0]

    def producer():
        it = claim[0]; claim[0] += 1
        n = 0
        while True:
            st, use = n & 1, n >> 1
            yield ("wait", B[f"kv_empty{st}"], (use & 1) ^ 1)
            if n >= 2:
                assert stage_readers.get(n - 2, 0) == 4, ("stage reused early", n)
            if it >= len(items):
                info[st] = (0, n)
                B[f"stg_full{st}" if widened_kind else f"kv_full{st}"].arrive()
                return
            nxt = claim[0]; claim[0] += 1
            info[st] = (items[it], n)
            if kind == "fp8":
                def raw_land(st=st, n=n):
                    stage_raw[st] = n
                    B[f"stg_full{st}"].arrive()
                later(f"tma_kv{st}", raw_land)
            elif kind == "fp4":
                yield ("wait", B["stg_empty"], (n & 1) ^ 1)
                assert n == 0 or widened.get(n - 1), ("staging overwritten before widening", n)
                def stg_land(st=st, n=n):
                    staging[0] = n
                    B[f"stg_full{st}"].arrive()
                later("tma_stg", stg_land)
            else:
                def land(st=st, n=n):
                    stage_item[st] = n
                    B[f"kv_full{st}"].arrive()
                later(f"tma_kv{st}", land)
            it = nxt
            n += 1
            yield None

    def issuer(g):
        n, j, jprev = 0, 0, -1
        while True:
            st = n & 1
            yield ("wait", B[f"kv_full{st}"], (n >> 1) & 1)
            nt, item_n = info[st]
            if nt == 0:
                break
            assert stage_item[st] == item_n
            for t in range(nt):
                if (j & 1) == g:
                    yield ("wait", B[f"q_full{g}"], (j >> 1) & 1)
                    assert q_buf[g] == j, ("q not this tile's", q_buf[g], j)
                    if jprev >= 0:
                        yield ("wait", B[f"o_full{g}"], (jprev >> 1) & 1)
                    # S overwritten: P of jprev must have been consumed by PV(jprev)
                    def qk(g=g, j=j):
                        S[g] = ("S", j)
                        B[f"s_full{g}"].arrive()
                    later(f"mma{g}", qk)
                    yield ("wait", B[f"p_full{g}"], (j >> 1) & 1)
                    assert S[g] == ("P", j)
                    # PV overwrites O (accumulate = 0 at ks = 0): O of jprev must have been read
                    assert jprev < 0 or O[g] == ("read", jprev), ("O overwritten before epilogue", O[g], jprev)
                    O[g] = ("pending", j)
                    def pv(g=g, j=j):
                        O[g] = ("done", j)
                        B[f"o_full{g}"].arrive()
                    later(f"mma{g}", pv)
                    jprev = j
                j += 1
            def rel(st=st, item_n=item_n):
                stage_readers[item_n] = stage_readers.get(item_n, 0) + 1
                B[f"kv_empty{st}"].arrive()
            later(f"mma{g}", rel)
            n += 1
        later(f"mma{g}", lambda: B["done"].arrive())
        yield ("wait", B["done"], 0)

    def softmax(g):
        n, j, pend_j, n_epi = 0, 0, -1, 0
        def epilogue():
            nonlocal n_epi
            m = n_epi
            if g == 1 or m > 0:
                ph = m if g == 1 else m - 1
                yield ("wait", B[f"epi_turn{g}"], ph & 1)
            # order: tile pend_j's epilogue after tile pend_j - 1's
            assert (not epi_done and pend_j == 0) or (epi_done and epi_done[-1] == pend_j - 1), (epi_done[-3:], pend_j)
            assert O[g] == ("done", pend_j), ("epilogue before O complete", O[g], pend_j)
            O[g] = ("read", pend_j)
            epi_done.append(pend_j)
            B[f"epi_turn{g ^ 1}"].arrive()
            n_epi += 1
        while True:
            st, use = n & 1, n >> 1
            if widened_kind and st == g:
                yield ("wait", B[f"stg_full{st}"], use & 1)
                nt0, item0 = info[st]
                if nt0 > 0:
                    if kind == "fp8":
                        assert stage_raw[st] == item0, ("widening rows of another item", stage_raw[st], item0)
                    else:
                        assert staging[0] == item0, ("widening the wrong staged block", staging[0], item0)
                    assert item0 < 2 or stage_readers.get(item0 - 2, 0) == 4, ("stage not free for widening", item0)
                    stage_item[st] = item0
                    widened[item0] = True
                    if kind == "fp4":
                        B["stg_empty"].arrive()
                B[f"kv_full{st}"].arrive()
            yield ("wait", B[f"kv_full{st}"], use & 1)
            nt, item_n = info[st]
            if nt == 0:
                break
            stage_readers[item_n] = stage_readers.get(item_n, 0) + 1
            B[f"kv_empty{st}"].arrive()
            for t in range(nt):
                if (j & 1) == g:
                    # q of tile j into the group's buffer: the previous q k^T is complete
                    assert S[g] is None or S[g][1] == j - 2 or S[g][1] < j, S[g]
                    def qland(g=g, j=j):
                        q_buf[g] = j
                        B[f"q_full{g}"].arrive()
                    later(f"tma_q{g}", qland)
                    if pend_j >= 0:
                        yield ("wait", B[f"o_full{g}"], (pend_j >> 1) & 1)
                        yield from epilogue()
                    yield ("wait", B[f"s_full{g}"], (j >> 1) & 1)
                    assert S[g] == ("S", j)
                    S[g] = ("P", j)
                    B[f"p_full{g}"].arrive()
                    pend_j = j
                    yield None
                j += 1
            n += 1
        if pend_j >= 0:
            yield ("wait", B[f"o_full{g}"], (pend_j >> 1) & 1)
            yield from epilogue()

    agents = {"prod": producer(), "i0": issuer(0), "i1": issuer(1), "s0": softmax(0), "s1": softmax(1)}
    state = {k: None for k in agents}
    done = set()
    steps = 0
    while len(done) < len(agents) or any(pending.values()):
        steps += 1
        assert steps < 500000
        progressed = False
        srcs = [s for s in pending if pending[s]]
        if srcs and rnd.random() < 0.5:
            pending[rnd.choice(srcs)].pop(0)()
            progressed = True
        order = list(agents); rnd.shuffle(order)
        for k in order:
            if k in done:
                continue
            w = state[k]
            if w is not None:
                if not w[1].ready(w[2]):
                    continue
                state[k] = None
            try:
                state[k] = next(agents[k])
            except StopIteration:
                done.add(k)
            progressed = True
            break
        if not progressed and not any(pending.values()):
            raise AssertionError(f"deadlock: {[(k, state[k][1].name, state[k][2]) for k in agents if state[k]]}")
    total_tiles = sum(items)
    assert epi_done == list(range(total_tiles)), (epi_done, total_tiles)
    return steps


def run_dense(tiles, seed, fix=True):
    rnd = random.Random(seed)
    B = {}
    def bar(n, c=1): B[n] = Bar(n, c)
    for g in range(2):
        for nm in ("q_full", "q_empty", "s_full", "p_full", "p_empty", "o_full", "o_empty"):
            bar(f"{nm}{g}")
    for st in range(2):
        bar(f"kv_full{st}"); bar(f"kv_empty{st}", 2)
    bar("go1")
    pending = {}
    def later(src, cb): pending.setdefault(src, []).append(cb)
    O = {0: None, 1: None}
    def producer():
        blk = 0
        for n, nb in enumerate(tiles):
            for h in range(2):
                yield ("wait", B[f"q_empty{h}"], (n & 1) ^ 1)
                later(f"tq{h}", lambda h=h: B[f"q_full{h}"].arrive())
            for b in range(nb):
                st, us = blk & 1, blk >> 1
                yield ("wait", B[f"kv_empty{st}"], (us & 1) ^ 1)
                later(f"tkv{st}", lambda st=st: B[f"kv_full{st}"].arrive())
                blk += 1
    def issuer(g):
        blk, ng = 0, 0
        for n, nb in enumerate(tiles):
            yield ("wait", B[f"q_full{g}"], n & 1)
            if nb == 0:
                later(f"m{g}", lambda: B[f"q_empty{g}"].arrive())
                if fix and n > 0:
                    yield ("wait", B[f"o_empty{g}"], (n - 1) & 1)
            if g == 1 and nb > 0:
                yield ("wait", B["go1"], ng & 1); ng += 1
            for b in range(nb):
                st = blk & 1
                yield ("wait", B[f"kv_full{st}"], (blk >> 1) & 1)
                if blk > 0:
                    yield ("wait", B[f"p_empty{g}"], (blk - 1) & 1)
                if b == nb - 1:
                    later(f"m{g}", lambda: B[f"q_empty{g}"].arrive())
                later(f"m{g}", lambda: B[f"s_full{g}"].arrive())
                yield ("wait", B[f"p_full{g}"], blk & 1)
                if g == 0 and b == 0:
                    B["go1"].arrive()
                if b == 0 and n > 0:
                    yield ("wait", B[f"o_empty{g}"], (n - 1) & 1)
                assert b > 0 or n == 0 or O[g] == ("read", n - 1) or tiles[n - 1] == 0 and O[g][0] == "read"
                O[g] = ("pend", n)
                def pv(st=st, n=n):
                    O[g] = ("done", n)
                    B[f"p_empty{g}"].arrive(); B[f"kv_empty{st}"].arrive()
                later(f"m{g}", pv)
                blk += 1
            def of(n=n, nb=nb):
                if nb == 0: O[g] = ("done", n)
                B[f"o_full{g}"].arrive()
            later(f"m{g}", of)
    def softmax(g):
        blk = 0
        for n, nb in enumerate(tiles):
            for b in range(nb):
                yield ("wait", B[f"s_full{g}"], blk & 1)
                B[f"p_full{g}"].arrive()
                blk += 1
                yield None
            yield ("wait", B[f"o_full{g}"], n & 1)
            assert O[g] == ("done", n), ("epilogue reads the wrong O", O[g], n)
            O[g] = ("read", n)
            B[f"o_empty{g}"].arrive()
    agents = {"p": producer(), "i0": issuer(0), "i1": issuer(1), "s0": softmax(0), "s1": softmax(1)}
    state = {k: None for k in agents}; done = set(); steps = 0
    while len(done) < len(agents) or any(pending.values()):
        steps += 1; assert steps < 200000
        prog = False
        srcs = [s for s in pending if pending[s]]
        if srcs and rnd.random() < 0.5:
            pending[rnd.choice(srcs)].pop(0)(); prog = True
        order = list(agents); rnd.shuffle(order)
        for k in order:
            if k in done: continue
            w = state[k]
            if w is not None:
                if not w[1].ready(w[2]): continue
                state[k] = None
            try: state[k] = next(agents[k])
            except StopIteration: done.add(k)
            prog = True; break
        if not prog and not any(pending.values()):
            raise AssertionError(f"deadlock {[(k, state[k][1].name) for k in agents if state[k]]}")



def run_decode(items, seed, fp8=False):
    """items: key counts (>= 1) of the CTA's decode items, in order.  Three
    K/V stages; widened caches (FP8, NVFP4) land a block's narrow rows in
    its own stage, where the widening warps widen them in place."""
    NS = 3
    rnd = random.Random(seed)
    B = {}
    def bar(n, c=1): B[n] = Bar(n, c)
    for i in range(NS):
        bar(f"kv_full{i}"); bar(f"kv_empty{i}")
    for i in range(2):
        for nm in ("q_full", "q_empty", "s_full", "p_full", "p_empty", "o_full", "o_empty"):
            bar(f"{nm}{i}")
    for i in range(NS):
        bar(f"stg_full{i}")
    pending = {}
    def later(src, cb): pending.setdefault(src, []).append(cb)
    stage = {}     # st -> block (landed / widened)
    stage_raw = {}  # st -> block whose narrow rows landed there
    Sbuf = {}      # sb -> ('S'|'read', blk)
    Pbuf = {}      # sb -> ('P'|'used', blk)
    Obuf = {}      # ib -> ('acc'|'done'|'read', item)
    pv_done = [-1]
    nblk = sum(items)
    def producer():
        blk = 0
        for n_it, nk in enumerate(items):
            ib, ui = n_it & 1, n_it >> 1
            yield ("wait", B[f"q_empty{ib}"], (ui & 1) ^ 1)
            later(f"tq{ib}", lambda ib=ib: B[f"q_full{ib}"].arrive())
            for j in range(nk):
                st, us = blk % NS, blk // NS
                yield ("wait", B[f"kv_empty{st}"], (us & 1) ^ 1)
                assert blk < NS or pv_done[0] >= blk - NS, ("stage refilled before its p v", blk)
                if fp8:
                    assert blk < NS or stage.get(st) == blk - NS, ("narrow rows over an unwidened block", blk)
                    def sl(st=st, blk=blk):
                        stage_raw[st] = blk
                        B[f"stg_full{st}"].arrive()
                    later(f"tkv{st}", sl)
                else:
                    def land(st=st, blk=blk):
                        stage[st] = blk
                        B[f"kv_full{st}"].arrive()
                    later(f"tkv{st}", land)
                blk += 1
    def issuer_qk():
        # S^T of block b: its q (item start), its K, and the S buffer it
        # reuses read out (P of block b - 2 written)
        b = 0
        for n_it, nk in enumerate(items):
            ib = n_it & 1
            for j in range(nk):
                st, sb = b % NS, b & 1
                if j == 0:
                    yield ("wait", B[f"q_full{ib}"], (n_it >> 1) & 1)
                yield ("wait", B[f"kv_full{st}"], (b // NS) & 1)
                if b >= 2:
                    yield ("wait", B[f"p_full{sb}"], ((b - 2) >> 1) & 1)
                assert stage.get(st) == b, ("S from the wrong K", stage.get(st), b)
                assert Sbuf.get(sb) in (None, ("read", b - 2)), ("S overwritten before read", Sbuf.get(sb), b)
                def qk(sb=sb, b=b):
                    Sbuf[sb] = ("S", b)
                    B[f"s_full{sb}"].arrive()
                later("mma_qk", qk)
                if j == nk - 1:
                    later("mma_qk", lambda ib=ib: B[f"q_empty{ib}"].arrive())
                b += 1
                yield None
    def issuer_pv():
        # O^T += V^T P^T of block b: its P, and at an item start the O
        # buffer it reuses read out
        b = 0
        for n_it, nk in enumerate(items):
            ib = n_it & 1
            for j in range(nk):
                st, sb = b % NS, b & 1
                yield ("wait", B[f"p_full{sb}"], (b >> 1) & 1)
                if j == 0:
                    yield ("wait", B[f"o_empty{ib}"], ((n_it >> 1) & 1) ^ 1)
                assert Pbuf.get(sb) == ("P", b), (Pbuf.get(sb), b)
                assert stage.get(st) == b
                if j == 0:
                    assert Obuf.get(ib) in (None, ("read", n_it - 2)), ("O overwritten before read", Obuf.get(ib))
                    Obuf[ib] = ("acc", n_it)
                def pv(sb=sb, st=st, b=b):
                    Pbuf[sb] = ("used", b)
                    pv_done[0] = b
                    B[f"p_empty{sb}"].arrive(); B[f"kv_empty{st}"].arrive()
                later("mma_pv", pv)
                if j == nk - 1:
                    def of(ib=ib, it=n_it):
                        Obuf[ib] = ("done", it)
                        B[f"o_full{ib}"].arrive()
                    later("mma_pv", of)
                b += 1
                yield None
    def softmax():
        blk = 0
        for n_it, nk in enumerate(items):
            ib, ui = n_it & 1, n_it >> 1
            for j in range(nk):
                st, us, sb, ub = blk % NS, blk // NS, blk & 1, blk >> 1
                yield ("wait", B[f"kv_full{st}"], us & 1)
                assert stage.get(st) == blk, ("softmax on the wrong block", stage.get(st), blk)
                yield ("wait", B[f"s_full{sb}"], ub & 1)
                assert Sbuf.get(sb) == ("S", blk)
                Sbuf[sb] = ("read", blk)
                yield ("wait", B[f"p_empty{sb}"], (ub & 1) ^ 1)
                assert blk < 2 or pv_done[0] >= blk - 2
                if j > 0 and rnd.random() < 0.3:  # raise m: the previous p v must be done
                    pb = blk - 1
                    yield ("wait", B[f"p_empty{pb & 1}"], (pb >> 1) & 1)
                    assert pv_done[0] >= blk - 1 and Obuf.get(ib) == ("acc", n_it)
                Pbuf[sb] = ("P", blk)
                B[f"p_full{sb}"].arrive()
                blk += 1
                yield None
            # the previous item's epilogue at this item's end; the last
            # item's own epilogue follows at once
            last = n_it == len(items) - 1
            for q in range(max(0, n_it - 1), n_it + 1 if last else n_it):
                qb = q & 1
                yield ("wait", B[f"o_full{qb}"], (q >> 1) & 1)
                assert Obuf.get(qb) == ("done", q)
                Obuf[qb] = ("read", q)
                B[f"o_empty{qb}"].arrive()
    def widen():
        # widened caches: warps 6-9 widen each block's narrow rows in place
        for blk in range(nblk):
            st, us = blk % NS, blk // NS
            yield ("wait", B[f"stg_full{st}"], us & 1)
            assert stage_raw.get(st) == blk, ("widening rows of another block", stage_raw.get(st), blk)
            assert blk < NS or pv_done[0] >= blk - NS, ("widening into a busy stage", blk)
            stage[st] = blk
            B[f"kv_full{st}"].arrive()
            yield None
    agents = {"p": producer(), "mq": issuer_qk(), "mp": issuer_pv(), "s": softmax()}
    if fp8:
        agents["w"] = widen()
    state = {k: None for k in agents}; done = set(); steps = 0
    while len(done) < len(agents) or any(pending.values()):
        steps += 1; assert steps < 500000
        prog = False
        srcs = [s for s in pending if pending[s]]
        if srcs and rnd.random() < 0.5:
            pending[rnd.choice(srcs)].pop(0)(); prog = True
        order = list(agents); rnd.shuffle(order)
        for k in order:
            if k in done: continue
            w = state[k]
            if w is not None:
                if w[0] == "pred":
                    if not w[1](): continue
                elif not w[1].ready(w[2]): continue
                state[k] = None
            try: state[k] = next(agents[k])
            except StopIteration: done.add(k)
            prog = True; break
        if not prog and not any(pending.values()):
            raise AssertionError(f"deadlock {[(k, state[k][0], getattr(state[k][1], 'name', '')) for k in agents if state[k]]}")

@pytest.mark.parametrize("kind", ["16", "fp8", "fp4"])
def test_fwd_kv_stationary_protocol(kind):
    rnd = random.Random(11 + ["16", "fp8", "fp4"].index(kind))
    for trial in range(400):
        items = [rnd.randint(1, 4) for _ in range(rnd.randint(0, 7))]
        run_fwd_kv_stationary(items, trial, kind)


@pytest.mark.parametrize("fp8", [False, True])
def test_fwd_decode_protocol(fp8):
    rnd = random.Random(3 + fp8)
    for trial in range(400):
        items = [rnd.randint(1, 8) for _ in range(rnd.randint(1, 7))]
        run_decode(items, trial, fp8)


def test_dense_protocol():
    rnd = random.Random(5)
    for trial in range(400):
        tiles = [rnd.choice([0, 1, 2, 3]) for _ in range(rnd.randint(1, 6))]
        run_dense(tiles, trial)


def test_dense_model_finds_the_empty_tile_race():
    """Negative control: without the empty tile's o_empty wait some
    schedule fails, so the model does see this kind of race."""
    rnd = random.Random(5)
    failures = 0
    for trial in range(2000):
        tiles = [rnd.choice([0, 1, 2, 3]) for _ in range(rnd.randint(1, 6))]
        try:
            run_dense(tiles, trial, fix=False)
        except AssertionError:
            failures += 1
    assert failures > 0
