"""A discrete-event model of the attention kernel's barrier protocol (host-side, no GPU).

The kernel's roles are modelled as generators that block on mbarrier phases:

- the Q/K(/V) producer warp;
- the V producer warp (split rings only);
- the MMA warp;
- the two softmax warpgroups.

The tensor pipe executes issued MMAs and commits in order, at random times. TMA loads land after
random delays. The model checks, at every step:

- no deadlock;
- no phase aliasing: a parity wait is answered the way the hardware answers it, and an answer that
  differs from the intended one (the phase two ahead, or the phase before) is reported;
- no K/V slot or Q tile overwritten while an MMA still reads it;
- no score tile overwritten before its warpgroup copied it out;
- no P tile overwritten while its PV is pending;
- every PV reads the P and V tiles it should;
- no output accumulator overwritten by a unit's first PV before the previous unit's output was read
  out of it, and no output read out while a PV into it is pending or before its unit's last PV.

Each rule mirrors a statement of the kernel source (zyfa_fwd.cuh).  For example, K and V have
rings of their own exactly when the ring holds three slots or fewer.  The last PV of a query tile
is issued after the next unit's first score MMA.
"""
import random

ROWS = 128  # query rows per tile


class Barrier:
    def __init__(self, count=1):
        self.count, self.arrivals, self.done = count, 0, 0

    def arrive(self):
        self.arrivals += 1
        if self.arrivals == self.count:
            self.arrivals, self.done = 0, self.done + 1


def tiles_for(S, BN, r0, t):
    """K/V tiles of query tile t of a unit.  A unit is either an int r0 (rows [r0, r0 + 256) of one
    head: tile t starts at r0 + 128 t) or a pair (r0, r0) (the same 128 rows of two heads that share
    a KV head: both tiles start at r0)."""
    first = r0[t] if isinstance(r0, tuple) else r0 + t * ROWS
    if first >= S:
        return 0
    return (min(first + ROWS, S) + BN - 1) // BN


def simulate(S, BN, stages, units, seed, wrong_release=False, steady_without_q1_release=False,
             max_steps=2_000_000):
    """Run one random schedule; returns the list of protocol violations (empty when clean).

    wrong_release and steady_without_q1_release plant a mistake (in the K/V release rule, or a
    steady block that never releases query tile 1's Q buffer) that the checks must catch."""
    rnd = random.Random(seed)
    split = stages <= 3
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Barrier(count)
        return bars[name]

    for st in range(stages):
        for n in ("k_full", "k_empty", "v_full", "v_empty"):
            bar(f"{n}{st}")
    for t in range(2):
        for n in ("q_full", "q_empty", "s_full", "pv_done"):
            bar(f"{n}{t}")
        bar(f"p_full{t}", 4)
    bar("s_free", 4)

    errors = []
    k_refs, v_refs, q_refs = [0] * stages, [0] * stages, [0, 0]
    k_data, v_data, q_data = [None] * stages, [None] * stages, [None, None]
    score = {"owner": None, "read": True}
    p_tile, pv_pending = [None, None], [0, 0]
    o_state = [{"owner": None, "free": True, "pvs": 0}, {"owner": None, "free": True, "pvs": 0}]
    pipe, loads = [], []

    def wait(name, k):
        # answered as the hardware answers a parity wait: complete when the barrier's completed-phase
        # count has the other parity; any answer that differs from "phase k has completed" is aliasing
        b = bars[name]

        def ready():
            hw = (b.done % 2) != (k % 2)
            if hw != (b.done >= k + 1):
                errors.append(f"phase aliasing on {name}: {b.done} phases done, waiting for phase {k}")
                return True
            return hw
        return ready

    def producer():
        kv = 0
        q_cnt = [0, 0]
        for r0 in units:
            n = (tiles_for(S, BN, r0, 0), tiles_for(S, BN, r0, 1))
            for t in range(2):
                if n[t] == 0:
                    continue
                if q_cnt[t] > 0:
                    yield wait(f"q_empty{t}", q_cnt[t] - 1)
                if q_refs[t]:
                    errors.append(f"Q{t} overwritten while read")
                q_data[t] = r0
                loads.append([rnd.randint(1, 30), f"q_full{t}"])
                q_cnt[t] += 1
            for j in range(max(n)):
                st = kv % stages
                if kv >= stages:
                    yield wait(f"k_empty{st}", kv // stages - 1)
                if k_refs[st]:
                    errors.append(f"K slot {st} overwritten while read")
                k_data[st] = (r0, j)
                if not split:
                    if v_refs[st]:
                        errors.append(f"V slot {st} overwritten while read")
                    v_data[st] = (r0, j)
                loads.append([rnd.randint(1, 60), f"k_full{st}"])
                kv += 1

    def v_producer():
        if not split:
            return
        yield lambda: True
        kv = 0
        for r0 in units:
            for j in range(max(tiles_for(S, BN, r0, 0), tiles_for(S, BN, r0, 1))):
                st = kv % stages
                if kv >= stages:
                    yield wait(f"v_empty{st}", kv // stages - 1)
                if v_refs[st]:
                    errors.append(f"V slot {st} overwritten while read")
                v_data[st] = (r0, j)
                loads.append([rnd.randint(1, 60), f"v_full{st}"])
                kv += 1

    def mma():
        kv_cnt, s_seq = 0, 0
        q_cnt, p_cnt = [0, 0], [0, 0]
        read_pending, last = False, (0, 0)
        tail = None  # (n0, n1, kv base, r0) of the unit whose last PVs are pending

        def do_pv(t, j, kvb, n0, n1, r0):
            st = (kvb + j) % stages
            if split:
                yield wait(f"v_full{st}", (kvb + j) // stages)
            if p_tile[t] != (r0, j):
                errors.append(f"PV{t}({j}) of unit {r0} reads P of {p_tile[t]}")
            if v_data[st] != (r0, j):
                errors.append(f"PV{t}({j}) of unit {r0} reads V of {v_data[st]}")
            pv_pending[t] += 1
            v_refs[st] += 1
            pipe.append(("pv", t, st, r0, j))
            pipe.append(("commit", f"pv_done{t}"))
            pv0_last = n1 == 0 or (j == n0 - 1 and n1 > n0)
            if wrong_release and j == n0 - 1 and n1 > 0:
                pv0_last = not pv0_last
            if (t == 0) == pv0_last:
                pipe.append(("commit", f"v_empty{st}" if split else f"k_empty{st}"))

        def issue_s(t, j, st, r0, n, q1_release=True):
            # one score MMA and its commits, as the steady block issues it
            nonlocal s_seq
            if k_data[st] != (r0, j) or q_data[t] != r0:
                errors.append(f"S{t}({j}) of unit {r0} reads K of {k_data[st]}, Q of {q_data[t]}")
            k_refs[st] += 1
            q_refs[t] += 1
            pipe.append(("s", t, j, st, r0))
            pipe.append(("commit", f"s_full{t}"))
            if split and (t == 1 or j >= n[1]):
                pipe.append(("commit", f"k_empty{st}"))
            s_seq += 1
            if j == n[t] - 1 and (t == 0 or q1_release):
                pipe.append(("commit", f"q_empty{t}"))

        def issue_tail():
            n0, n1, kvb, r0 = tail
            for t, nt in ((0, n0), (1, n1)):
                if nt:
                    yield wait(f"p_full{t}", p_cnt[t])
                    p_cnt[t] += 1
                    yield from do_pv(t, nt - 1, kvb, n0, n1, r0)

        for r0 in units:
            n = (tiles_for(S, BN, r0, 0), tiles_for(S, BN, r0, 1))
            for t in range(2):
                if n[t]:
                    yield wait(f"q_full{t}", q_cnt[t])
                    q_cnt[t] += 1
            for j in range(max(n)):
                if j >= 1 and j < n[0] and n[1] > 0:
                    # steady state (both query tiles active), the kernel's branch-free block:
                    # S0(j), PV1(j-2), S1(j), PV0(j-1); each score MMA after the read of the previous one
                    st = (kv_cnt + j) % stages
                    yield wait(f"k_full{st}", (kv_cnt + j) // stages)
                    yield wait("s_free", s_seq - 1)
                    issue_s(0, j, st, r0, n)
                    if j >= 2:
                        yield from do_pv(1, j - 2, kv_cnt, n[0], n[1], r0)
                    yield wait("s_free", s_seq - 1)
                    issue_s(1, j, st, r0, n, q1_release=not steady_without_q1_release)
                    yield from do_pv(0, j - 1, kv_cnt, n[0], n[1], r0)
                    read_pending, last = True, (1, j)
                    continue
                for t in range(2):
                    if j >= n[t]:
                        continue
                    st = (kv_cnt + j) % stages
                    if t == 0 or j >= n[0]:  # first score tile of K tile j
                        yield wait(f"k_full{st}", (kv_cnt + j) // stages)
                    unlock = None
                    if read_pending:
                        yield wait("s_free", s_seq - 1)
                        read_pending = False
                        if last[1] >= 1:
                            unlock = (last[0], last[1] - 1)
                    pv_first = unlock is not None and unlock[0] == t
                    if pv_first:
                        yield from do_pv(*unlock, kv_cnt, n[0], n[1], r0)
                    if k_data[st] != (r0, j) or q_data[t] != r0:
                        errors.append(f"S{t}({j}) of unit {r0} reads K of {k_data[st]}, Q of {q_data[t]}")
                    k_refs[st] += 1
                    q_refs[t] += 1
                    pipe.append(("s", t, j, st, r0))
                    pipe.append(("commit", f"s_full{t}"))
                    if split and (t == 1 or j >= n[1]):
                        pipe.append(("commit", f"k_empty{st}"))
                    s_seq += 1
                    read_pending, last = True, (t, j)
                    if j == n[t] - 1:
                        pipe.append(("commit", f"q_empty{t}"))
                    if unlock is not None and not pv_first:
                        yield from do_pv(*unlock, kv_cnt, n[0], n[1], r0)
                    if t == 0 and j == 0 and tail is not None:
                        yield from issue_tail()
                        tail = None
            if read_pending:
                yield wait("s_free", s_seq - 1)
                read_pending = False
                if last[1] >= 1:
                    yield from do_pv(last[0], last[1] - 1, kv_cnt, n[0], n[1], r0)
            tail = (n[0], n[1], kv_cnt, r0)
            kv_cnt += max(n)
        if tail is not None:
            yield from issue_tail()

    def softmax(t):
        s_cnt = pv_ph = 0
        for r0 in units:
            nt = tiles_for(S, BN, r0, t)
            for j in range(nt):
                yield wait(f"s_full{t}", s_cnt)
                s_cnt += 1
                if score["owner"] != (t, r0, j):
                    errors.append(f"warpgroup {t} reads score tile {score['owner']}, expected {(t, r0, j)}")
                score["read"] = True
                for _ in range(4):
                    bars["s_free"].arrive()
                for _ in range(rnd.randint(0, 3)):
                    yield lambda: True  # the softmax arithmetic
                if j > 0:
                    yield wait(f"pv_done{t}", pv_ph)
                    pv_ph += 1
                if pv_pending[t]:
                    errors.append(f"warpgroup {t} overwrites P while its PV is pending")
                p_tile[t] = (r0, j)
                if j == nt - 1:
                    for _ in range(4):
                        bars[f"p_full{t}"].arrive()
            if nt:
                yield wait(f"pv_done{t}", pv_ph)  # epilogue: the tile's last PV
                pv_ph += 1
                if pv_pending[t]:
                    errors.append(f"epilogue of warpgroup {t} with a PV pending")
                if o_state[t] != {"owner": r0, "free": False, "pvs": nt}:
                    errors.append(f"warpgroup {t} reads out {o_state[t]} for unit {r0} ({nt} PVs)")
                o_state[t]["free"] = True

    roles = [producer(), v_producer(), mma(), softmax(0), softmax(1)]
    blocked = [None] * len(roles)
    finished = [False] * len(roles)
    for _ in range(max_steps):
        progressed = False
        if pipe and rnd.random() < 0.5:  # the tensor pipe retires its oldest operation
            op = pipe.pop(0)
            progressed = True
            if op[0] == "s":
                _, t, j, st, r0 = op
                if not score["read"]:
                    errors.append(f"score tile S{t}({j}) overwrites an unread one")
                score.update(owner=(t, r0, j), read=False)
                k_refs[st] -= 1
                q_refs[t] -= 1
            elif op[0] == "pv":
                _, t, st, r0, j = op
                if j == 0:
                    if not o_state[t]["free"]:
                        errors.append(f"first PV of tile {t} of unit {r0} overwrites the output of "
                                      f"{o_state[t]['owner']} before it was read out")
                    o_state[t] = {"owner": r0, "free": False, "pvs": 1}
                elif o_state[t]["owner"] != r0:
                    errors.append(f"PV of tile {t} of unit {r0} accumulates into the output of {o_state[t]['owner']}")
                else:
                    o_state[t]["pvs"] += 1
                pv_pending[t] -= 1
                v_refs[st] -= 1
            else:
                bars[op[1]].arrive()
        for ld in list(loads):
            ld[0] -= 1
            if ld[0] <= 0:
                loads.remove(ld)
                bars[ld[1]].arrive()
                progressed = True
        order = list(range(len(roles)))
        rnd.shuffle(order)
        for i in order:
            if finished[i] or (blocked[i] is not None and not blocked[i]()):
                continue
            try:
                blocked[i] = next(roles[i])
                progressed = True
            except StopIteration:
                finished[i], blocked[i] = True, None
        if errors:
            return errors
        if all(finished) and not pipe and not loads:
            return []
        if not progressed and not pipe and not loads:
            return [f"deadlock (roles finished: {finished})"]
    return ["no end within the step limit"]
