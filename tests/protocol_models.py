"""Random-interleaving models of the barrier protocols of the persistent
tensor-core kernels (test infrastructure).

Each model runs the roles of one CTA (TMA producer, MMA thread, softmax or
compute warps, dQ reducer) as generators that yield at every poll of a wait;
the copy engine lands loads in random order, the tensor pipe executes issued
products and commits in order, and the bulk-reduction engine reads its
buffers in order, each at random times, with per-run role speeds spanning two
orders of magnitude.  A run fails if an arrival exceeds a barrier's count, a
product or reduction reads a buffer holding other data, a load overwrites a
buffer a pending product still reads, an accumulate-0 product overwrites
accumulators not yet read out, a consumer sees another step's scores, or a
role waits for a phase that never comes.  `skip` names waits to leave out,
to show that the checks catch their absence.
"""
import random

class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arr, self.tx, self.done = name, count, 0, 0, 0
    def arrive(self, tx=0):
        assert self.arr < self.count, f"arrive overflow on {self.name} phase {self.done}"
        self.arr += 1; self.tx += tx; self._check()
    def complete_tx(self, tx):
        self.tx -= tx; assert self.tx >= 0, f"tx underflow {self.name}"; self._check()
    def _check(self):
        if self.arr == self.count and self.tx == 0:
            self.done += 1; self.arr = 0
    def try_wait(self, parity):
        return (self.done & 1) != parity

def pairs_for(rng, n):
    out = []
    for _ in range(n):
        nkv0 = rng.randint(1, 5)
        two = rng.random() < 0.8
        nkv1 = (nkv0 + rng.randint(0, 1)) if two else 0
        out.append((nkv0, nkv1))
    return out

def run_forward(pairs, seed, S=2, skip=()):
    rng = random.Random(seed)
    q = Bar("q", 1); qfree = Bar("qfree", 1)
    kv = [Bar(f"kv{s}", 1) for s in range(S)]
    kfree = [Bar(f"kfree{s}", 1) for s in range(S)]; vfree = [Bar(f"vfree{s}", 1) for s in range(S)]
    bs = [Bar(f"s{t}", 1) for t in range(2)]; bp = [Bar(f"p{t}", 1) for t in range(2)]; epi = [Bar(f"epi{t}", 1) for t in range(2)]
    nmaxs = [max(a, b) for a, b in pairs]
    G0 = [sum(nmaxs[:i]) for i in range(len(pairs))]
    # buffer contents: Q -> pair, K[s] -> global step, V[s] -> global step
    qbuf = None; kbuf = [None] * S; vbuf = [None] * S
    loads = []          # (kind, slot, value, bar)
    pipe = []           # ("s", t, pair, g) | ("pv", t, pair, g, acc) | ("commit", bar, tag)
    readers = {("q",): 0}
    reads = {}          # buffer key -> count of issued-not-executed MMAs reading it
    o_read = {}         # t -> pair whose O the softmax has read out (epilogue done)
    s_last = [None, None]  # last executed S per tile: (pair, j)
    def rd(key, d):
        reads[key] = reads.get(key, 0) + d
    def issue(op):
        pipe.append(op)
        if op[0] == "s": rd(("q",), 1); rd(("k", op[3] % S), 1)
        if op[0] == "pv": rd(("v", op[3] % S), 1)
    def execute(op):
        nonlocal qbuf
        if op[0] == "s":
            _, t, pr, g = op
            assert qbuf == pr, f"S of pair {pr} reads Q of pair {qbuf}"
            assert kbuf[g % S] == g, f"S step {g} reads K {kbuf[g % S]}"
            rd(("q",), -1); rd(("k", g % S), -1)
            s_last[t] = (pr, g - G0[pr])
        elif op[0] == "pv":
            _, t, pr, g, acc = op
            assert vbuf[g % S] == g, f"PV step {g} reads V {vbuf[g % S]}"
            if not acc:
                prev = [i for i in range(pr) if pairs[i][t] > 0]
                if prev: assert o_read.get(t) == prev[-1], f"PV acc=0 of pair {pr} tile {t} over unread O of pair {prev[-1]}"
            rd(("v", g % S), -1)
        else:
            op[1].arrive()
    def land(ld):
        nonlocal qbuf
        kind, slot, val, bar, tx = ld
        key = ("q",) if kind == "q" else (kind, slot)
        assert reads.get(key, 0) == 0, f"load {kind}{slot}={val} over a buffer an MMA still reads"
        if kind == "q": qbuf = val
        elif kind == "k": kbuf[slot] = val
        else: vbuf[slot] = val
        bar.complete_tx(tx)
    def producer():
        G = 0
        q.arrive(tx=2); loads.append(("q", 0, 0, q, 1)); loads.append(("k", 0, 0, q, 1))
        for ii, (n0, n1) in enumerate(pairs):
            nmax = max(n0, n1); has_next = ii + 1 < len(pairs)
            for j in range(nmax):
                g = G + j; s = g % S
                k_next = j + 1 < nmax or has_next
                if g >= S:
                    if "vfree" not in skip:
                        while not vfree[s].try_wait((g // S - 1) & 1): yield
                if k_next and g + 1 >= S:
                    if "kfree" not in skip:
                        while not kfree[(g + 1) % S].try_wait(((g + 1) // S - 1) & 1): yield
                kv[s].arrive(tx=2 if k_next else 1)
                loads.append(("v", s, g, kv[s], 1))
                if k_next: loads.append(("k", (g + 1) % S, g + 1, kv[s], 1))
                yield
            G += nmax
            if has_next:
                if "qfree" not in skip:
                    while not qfree.try_wait(ii & 1): yield
                q.arrive(tx=1); loads.append(("q", 0, ii + 1, q, 1))
            yield
    def mma():
        G = 0; cp = [0, 0]; used = [0, 0]
        for ii, nk in enumerate(pairs):
            nmax = max(nk)
            while not q.try_wait(ii & 1): yield
            for t in range(2):
                if nk[t] == 0: continue
                if used[t] > 0:
                    if "epi" not in skip:
                        while not epi[t].try_wait((used[t] - 1) & 1): yield
                used[t] += 1
                issue(("s", t, ii, G)); issue(("commit", bs[t], (ii, 0)))
                yield
            for j in range(nmax):
                g = G + j; s = g % S
                while not kv[s].try_wait((g // S) & 1): yield
                for t in range(2):
                    if j >= nk[t]: continue
                    while not bp[t].try_wait(cp[t] & 1): yield
                    cp[t] += 1
                    issue(("pv", t, ii, g, j > 0))
                    if j + 1 < nk[t]: issue(("s", t, ii, g + 1))
                    issue(("commit", bs[t], (ii, j + 1)))
                    yield
            G += nmax
    def softmax(t):
        cs = 0
        for ii, nk in enumerate(pairs):
            n = nk[t]
            if n == 0: continue
            nmax = max(nk); t_last = 1 if nk[1] > 0 else 0; G = G0[ii]
            for j in range(n):
                while not bs[t].try_wait(cs & 1): yield
                cs += 1
                assert s_last[t] == (ii, j), f"softmax {t} pair {ii} step {j} sees S {s_last[t]}"
                if t == t_last:
                    g = G + j
                    kfree[g % S].arrive()
                    if g > 0: vfree[(g - 1) % S].arrive()
                    if j == n - 1: qfree.arrive()
                yield
                bp[t].arrive()
                yield
            while not bs[t].try_wait(cs & 1): yield
            cs += 1
            epi[t].arrive()
            yield
            o_read[t] = ii
            yield
    roles = [producer(), mma(), softmax(0), softmax(1)]
    speed = [10 ** rng.uniform(-2, 0) for _ in range(4)]
    alive = [True] * 4
    idle = 0; steps = 0
    while any(alive) or pipe or loads:
        steps += 1
        assert steps < 3000000, "no progress: a role waits for a phase that never comes" 
        progressed = False
        choice = rng.random()
        if choice < 0.15 and loads:
            land(loads.pop(rng.randrange(len(loads)))); progressed = True
        elif choice < 0.35 and pipe:
            execute(pipe.pop(0)); progressed = True
        else:
            r = rng.choices(range(4), weights=speed)[0]
            if alive[r]:
                try:
                    next(roles[r])
                except StopIteration:
                    alive[r] = False
                progressed = True
        idle = 0 if progressed else idle + 1
        assert idle < 100000, "stuck"
    for i in range(4): assert not alive[i]
    return True



def run_backward(items, seed, skip=(), ring_slots=4, pieces=False):
    """items: list of step counts (one per key tile of this CTA).  Only the
    producer knows them: it hands each tile to the MMA thread and the compute
    warps through a ring of records in shared memory (bar_item per slot,
    bar_itemfree counting the three readers), then an end record.
    pieces: the head-width-128 scheme, in which the dS^T buffer is two query
    halves and half 0 of dQ goes to the copy engine as two pieces, each staged
    over one of them and each releasing its own half (bar_dsfree / bar_dsfree1);
    half 1 is staged after the second piece.  Otherwise (head width 64) half 0
    is one piece over the whole buffer."""
    rng = random.Random(seed)
    B = lambda n, c=1: Bar(n, c)
    kv = B("kv"); qf = [B("qf0", 2), B("qf1", 2)]; qe = [B("qe0"), B("qe1")]; of = B("of"); oe = B("oe")
    bs = B("s"); dp = B("dp"); bp = B("p", 2); ds = B("ds", 2); dq = B("dq"); dqfree = B("dqfree", 2)
    dsfree = B("dsfree"); staged = [B("staged0"), B("staged1")]; stfree = B("stfree")
    staged0b = B("staged0b"); dsfree1 = B("dsfree1")
    DS = ["dSa", "dSb"] if pieces else ["dS"]   # the dS^T buffer: two query halves, or one
    itemdone = B("itemdone"); accfree = B("accfree", 2)
    G0 = [sum(items[:i]) for i in range(len(items))]
    buf = {"K": None, "V": None, "Q0": None, "Q1": None, "dO": None, "dS": None, "dSa": None, "dSb": None,
           "stage": None}
    reads = {}
    loads = []
    pipe = []
    engine = []        # copy-engine reductions in order: (buffer, expected content, bar to arrive when read)
    tm = {"DP": None, "S": None, "acc": None}   # tensor-memory contents (what the last writer put there)
    drained = set()    # dQ steps read out of TMEM
    acc_read = set()   # items whose dK/dV the epilogue read out
    R = ring_slots
    ring = [None] * R          # (tile, step count) per slot; step count None = end
    bitem = [B(f"item{s}") for s in range(R)]
    bitemfree = [B(f"itemfree{s}", 3) for s in range(R)]   # MMA thread + two compute halves
    def read_record(ii):
        """generator: wait for tile ii's record, read it, free the slot; returns the step count"""
        slot = ii % R
        while not bitem[slot].try_wait((ii // R) & 1): yield
        tag, n = ring[slot]
        assert tag == ii, f"role reads the record of tile {tag} for tile {ii}"
        bitemfree[slot].arrive()
        return n
    def rd(k, d): reads[k] = reads.get(k, 0) + d
    def issue(op):
        pipe.append(op)
        for k in op[2]: rd(k, 1)
    def execute(op):
        kind, args, rks = op
        for k, want in zip(rks, args["want"]):
            assert buf[k] == want, f"{kind} reads {k}={buf[k]} expected {want}"
            rd(k, -1)
        if kind == "commit":
            args["bar"].arrive(); return
        g = args.get("g")
        if kind == "dP":
            assert tm["DP"] is None or tm["DP"][0] != "dQ" or tm["DP"][1] in drained, f"dP {g} over undrained {tm['DP']}"
            tm["DP"] = ("dP", g)
        elif kind == "dQ":
            tm["DP"] = ("dQ", g)
        elif kind == "S":
            tm["S"] = ("S", g)
        elif kind in ("dV", "dK") and args["acc0"] == 0:
            it = args["item"]
            assert it == 0 or (it - 1) in acc_read, f"{kind} acc=0 of item {it} over unread accumulators"
    def land(ld):
        k, val, bar, tx = ld
        assert reads.get(k, 0) == 0, f"load {k}={val} over a buffer an MMA still reads"
        buf[k] = val; bar.complete_tx(tx)
    def engine_step():
        k, want, bar = engine.pop(0)
        assert buf[k] == want, f"reduction reads {k}={buf[k]} expected {want}"
        bar.arrive()
    # ---- roles
    def producer():
        G = 0
        def load_kv(ii):
            kv.arrive(tx=2); loads.append(("K", ii, kv, 1)); loads.append(("V", ii, kv, 1))
        def publish(ii):
            slot = ii % R
            if ii >= R and "itemfree" not in skip:
                while not bitemfree[slot].try_wait((ii // R - 1) & 1): yield
            ring[slot] = (ii, items[ii] if ii < len(items) else None)
            bitem[slot].arrive()
        yield from publish(0)
        for ii, n in enumerate(items):
            if ii == 0: load_kv(0)
            for k in range(n):
                g = G + k; st = g & 1
                if g >= 2:
                    while not qe[st].try_wait(((g >> 1) - 1) & 1): yield
                qf[st].arrive(tx=1); loads.append((f"Q{st}", g, qf[st], 1))
                yield
                qf[st].arrive()  # L / D written
                if g >= 1:
                    while not oe.try_wait((g - 1) & 1): yield
                of.arrive(tx=1); loads.append(("dO", g, of, 1))
                if k == 0 and ii > 0:
                    if "itemdone" not in skip:
                        while not itemdone.try_wait((ii - 1) & 1): yield
                    load_kv(ii)
                yield
            G += n
            yield from publish(ii + 1)
    def mma():
        G = 0
        for ii in range(len(items) + 1):
            n = yield from read_record(ii)
            if n is None: return
            while not kv.try_wait(ii & 1): yield
            while not qf[G & 1].try_wait((G >> 1) & 1): yield
            issue(("S", {"g": G, "want": [ii, G]}, ["K", f"Q{G & 1}"])); issue(("commit", {"bar": bs, "want": []}, []))
            if G > 0:
                if "dqfree_first" not in skip:
                    while not dqfree.try_wait((G - 1) & 1): yield
            while not of.try_wait(G & 1): yield
            issue(("dP", {"g": G, "want": [ii, G]}, ["V", "dO"])); issue(("commit", {"bar": dp, "want": []}, []))
            yield
            for k in range(n):
                g = G + k; st = g & 1
                if k > 0:
                    while not dqfree.try_wait((g - 1) & 1): yield
                    while not of.try_wait(g & 1): yield
                    issue(("dP", {"g": g, "want": [ii, g]}, ["V", "dO"])); issue(("commit", {"bar": dp, "want": []}, []))
                while not bp.try_wait(g & 1): yield
                if k == 0 and ii > 0:
                    if "accfree" not in skip:
                        while not accfree.try_wait((ii - 1) & 1): yield
                issue(("dV", {"g": g, "acc0": k > 0, "item": ii, "want": [g]}, ["dO"])); issue(("commit", {"bar": oe, "want": []}, []))
                if k + 1 < n:
                    while not qf[st ^ 1].try_wait(((g + 1) >> 1) & 1): yield
                    issue(("S", {"g": g + 1, "want": [ii, g + 1]}, ["K", f"Q{st ^ 1}"])); issue(("commit", {"bar": bs, "want": []}, []))
                while not ds.try_wait(g & 1): yield
                issue(("dK", {"g": g, "acc0": k > 0, "item": ii, "want": [g]}, [f"Q{st}"])); issue(("commit", {"bar": qe[st], "want": []}, []))
                issue(("dQ", {"g": g, "want": [ii] + [("dS", g)] * len(DS)}, ["K"] + DS)); issue(("commit", {"bar": dq, "want": []}, []))
                yield
            issue(("commit", {"bar": itemdone, "want": []}, []))
            G += n
    def compute(ch):
        G = 0
        def drain(gg):
            while not dq.try_wait(gg & 1): yield
            drained.add(gg); dqfree.arrive()   # (each half arrives; count 2)
            yield
            if ch == 1:
                while not (staged0b if pieces else staged[0]).try_wait(gg & 1): yield
                if gg > 0:
                    if "stfree" not in skip:
                        while not stfree.try_wait((gg - 1) & 1): yield
            if ch == 0 and pieces:
                for half, bar_st, bar_free in (("dSa", staged[0], dsfree), ("dSb", staged0b, dsfree1)):
                    assert reads.get(half, 0) == 0, "staging over dS while dQ still reads it"
                    buf[half] = ("h0", gg); engine.append((half, ("h0", gg), bar_free))
                    bar_st.arrive()
                    yield
                return
            if ch == 0:
                assert reads.get("dS", 0) == 0, "staging over dS while dQ still reads it"
                buf["dS"] = ("h0", gg); engine.append(("dS", ("h0", gg), dsfree))
            else:
                buf["stage"] = ("h1", gg); engine.append(("stage", ("h1", gg), stfree))
            staged[ch].arrive()
            yield
        for ii in range(len(items) + 1):
            n = yield from read_record(ii)
            if n is None: return
            for k in range(n):
                g = G + k
                while not qf[g & 1].try_wait((g >> 1) & 1): yield
                while not bs.try_wait(g & 1): yield
                assert tm["S"] == ("S", g), f"compute {ch} step {g} sees {tm['S']}"
                bp.arrive()
                yield
                if k > 0: yield from drain(g - 1)
                while not dp.try_wait(g & 1): yield
                assert tm["DP"] == ("dP", g), f"compute {ch} step {g} sees {tm['DP']}"
                if g > 0:
                    if "dsfree" not in skip:
                        while not (dsfree1 if pieces and ch == 1 else dsfree).try_wait((g - 1) & 1): yield
                if pieces:
                    half = DS[ch]
                    assert reads.get(half, 0) == 0, "dS^T written while dQ still reads it"
                    buf[half] = ("dS", g)
                elif ch == 0:
                    buf["dS"] = ("dS", g)   # both halves write; model the buffer's content once
                ds.arrive()
                yield
            yield from drain(G + n - 1)
            while not itemdone.try_wait(ii & 1): yield
            acc_read_half[ch].add(ii)
            if ii in acc_read_half[1 - ch]: acc_read.add(ii)
            accfree.arrive()
            yield
            G += n
    acc_read_half = [set(), set()]
    roles = [producer(), mma(), compute(0), compute(1)]
    speed = [10 ** rng.uniform(-2, 0) for _ in range(4)]
    alive = [True] * 4
    steps = 0
    while any(alive) or pipe or loads or engine:
        steps += 1
        assert steps < 3000000, "no progress"
        c = rng.random()
        if c < 0.12 and loads:
            land(loads.pop(rng.randrange(len(loads))))
        elif c < 0.3 and pipe:
            execute(pipe.pop(0))
        elif c < 0.36 and engine:
            engine_step()
        else:
            r = rng.choices(range(4), weights=speed)[0]
            if alive[r]:
                try: next(roles[r])
                except StopIteration: alive[r] = False
    return True

