"""A model of the persistent decode matvec's barrier protocol (csrc/matvec_kq.cu), run under
random schedules on the CPU.  Agents: the copy warp (weight tiles of the CTA's chunk
sequence through an NS-stage ring, the first ring round ramped), the x warps of each chunk
parity that have batch rows (or, with an activation fragment plane, one bulk copier per
parity), and the sixteen compute warps in two teams by chunk parity.  A compute warp waits
for its chunk's weight stage, reads it, releases it, waits for the fragment slot, reads it
and releases it; at the end of each unit (row group) the team-1 warp hands its partial sums
to the team-0 warp of the same rows through a buffer per unit parity.  Bulk copies land in
any order.  Every run must finish and every read must see the chunk (or unit) it is meant
for.  The index arithmetic is the kernel's, restated.  Planted mistakes must be caught: an
odd ring depth and teams by the unit-local chunk parity (the two failures met while the
kernel was built) and a copy warp that does not wait for a stage to be released.  The
split-K kernel's simpler pipeline (csrc/matvec.cu) is modelled at the end."""
import pytest

from tests.protocol_model import Bar, Violation, run

KFS = 4       # fragment slots
KTEAM = 8     # compute warps per team


def run_cta(groups, grid, b, nchunk, xlive, plane, seed, ns=4, bug=None):
    units = list(range(b, groups, grid))  # this CTA's row groups
    seq = [(u, c) for u in range(len(units)) for c in range(nchunk)]  # its chunk sequence
    wfull, wempty = [Bar(1) for _ in range(ns)], [Bar(KTEAM) for _ in range(ns)]
    ffull = [Bar(1 if plane else xlive) for _ in range(KFS)]
    fempty = [Bar(KTEAM) for _ in range(KFS)]
    pfull = [[Bar(1) for _ in range(2)] for _ in range(KTEAM)]
    pempty = [[Bar(1) for _ in range(2)] for _ in range(KTEAM)]
    w_tag = [None] * ns
    f_tag = [[None] * max(xlive, 1) for _ in range(KFS)]
    xch = [[None] * KTEAM for _ in range(2)]
    events = []

    def copies():
        for i in range(len(seq)):
            s = i % ns
            if i >= ns:
                if bug != "copy_skips_empty":
                    yield wempty[s], ((i // ns) - 1) & 1
            elif i >= 2:  # ramp: after the tile two before has landed
                yield wfull[i - 2], 0
            wfull[s].expect_tx(1)

            def land(s=s, i=i):
                w_tag[s] = i
                wfull[s].complete_tx(1)
            events.append(land)

    def x_warp(xi, par):
        for i in range(par, len(seq), 2):
            fs = i % KFS
            if i >= KFS:
                yield fempty[fs], ((i // KFS) - 1) & 1
            f_tag[fs][xi] = i
            ffull[fs].arrive()

    def plane_copier(par):
        for i in range(par, len(seq), 2):
            fs = i % KFS
            if i >= KFS:
                yield fempty[fs], ((i // KFS) - 1) & 1
            ffull[fs].expect_tx(1)

            def land(fs=fs, i=i):
                for k in range(len(f_tag[fs])):
                    f_tag[fs][k] = i
                ffull[fs].complete_tx(1)
            events.append(land)

    def compute(team, wq):
        at, base = 0, 0
        wpos, wph, fpos, fph = 0, 0, 0, 0
        for u in range(len(units)):
            nch = nchunk
            j0 = team & 1 if bug == "unit_local_parity" else (team + base) & 1
            for j in range(j0, nch, 2):
                d = base + j - at
                wpos += d
                while wpos >= ns:
                    wpos -= ns
                    wph ^= 1
                fpos += d
                while fpos >= KFS:
                    fpos -= KFS
                    fph ^= 1
                at = base + j
                s, fs = wpos, fpos
                yield wfull[s], wph
                if w_tag[s] != at:
                    raise Violation(f"warp {team}/{wq} read weight chunk {w_tag[s]} for {at}")
                wempty[s].arrive()
                yield ffull[fs], fph
                if any(v != at for v in f_tag[fs]):
                    raise Violation(f"warp {team}/{wq} read fragments {f_tag[fs]} for {at}")
                fempty[fs].arrive()
            base += nch
            par = u & 1
            if team == 1:
                if u >= 2:
                    yield pempty[wq][par], ((u >> 1) - 1) & 1
                xch[par][wq] = u
                pfull[wq][par].arrive()
                continue
            yield pfull[wq][par], (u >> 1) & 1
            if xch[par][wq] != u:
                raise Violation(f"team-0 warp {wq} read partial sums of unit {xch[par][wq]} for {u}")
            pempty[wq][par].arrive()

    agents = [copies()]
    if plane:
        agents += [plane_copier(0), plane_copier(1)]
    else:
        agents += [x_warp(xi, par) for xi in range(xlive) for par in (0, 1)]
    agents += [compute(team, wq) for team in (0, 1) for wq in range(KTEAM)]
    return run(agents, events, [], seed)


# row groups, grid, chunks per group (K / 256): several groups per CTA, odd and even chunk
# counts, one chunk
SHAPES = [(1, 1, 14), (5, 2, 14), (7, 3, 3), (6, 2, 1), (4, 1, 5), (9, 4, 2)]


@pytest.mark.parametrize("xlive,plane", [(1, False), (2, False), (1, True)])
def test_random_schedules_finish_and_read_what_they_should(xlive, plane):
    for groups, grid, nchunk in SHAPES:
        for b in range(min(grid, groups)):
            for seed in range(25):
                run_cta(groups, grid, b, nchunk, xlive, plane, seed=977 * nchunk + 31 * b + seed)


@pytest.mark.parametrize("bug,ns,nchunk", [(None, 3, 7), ("unit_local_parity", 4, 3),
                                           ("copy_skips_empty", 4, 14)])
def test_planted_protocol_mistakes_are_caught(bug, ns, nchunk):
    caught = 0
    for seed in range(200):
        try:
            run_cta(4, 1, 0, nchunk, 1, False, seed=seed, ns=ns, bug=bug)
        except Violation:
            caught += 1
    assert caught > 0


# ---- the split-K matvec (csrc/matvec.cu): one CTA per (row group, K slice) -------------
# The copy warp fills a stage with the weight tile and the x chunk of every batch row (one
# transaction barrier; the first ring round's weights before the wait for the previous
# kernel, its x after); the x warps convert the staged x into a fragment slot and release the
# stage (before the conversion with x in registers, "early", or after it); the eight compute
# warps read their weights, release the stage, wait for the slot, read it and release it.

def run_split(nch, xwarps, early, seed, ns=2, fs_n=2, bug=None):
    ncomp = 8
    wfull, wempty = [Bar(1) for _ in range(ns)], [Bar(ncomp + xwarps) for _ in range(ns)]
    ffull, fempty = [Bar(xwarps) for _ in range(fs_n)], [Bar(ncomp) for _ in range(fs_n)]
    w_tag, x_tag = [None] * ns, [None] * ns
    f_tag = [[None] * xwarps for _ in range(fs_n)]
    events = []

    def fill(i, weights=True, x=True):
        s = i % ns
        if weights:
            wfull[s].expect_tx(2)
            events.append(lambda s=s, i=i: (w_tag.__setitem__(s, i), wfull[s].complete_tx(1)))
        if x:
            events.append(lambda s=s, i=i: (x_tag.__setitem__(s, i), wfull[s].complete_tx(1)))

    def copies():
        pre = min(nch, ns)
        for i in range(pre):
            fill(i, x=False)
        for i in range(pre):
            fill(i, weights=False)
        for i in range(pre, nch):
            if bug != "copy_skips_empty":
                yield wempty[i % ns], ((i // ns) - 1) & 1
            fill(i)

    def x_warp(xi):
        for i in range(nch):
            s, fs = i % ns, i % fs_n
            yield wfull[s], (i // ns) & 1
            if early:
                if x_tag[s] != i:
                    raise Violation(f"x warp {xi} read x of chunk {x_tag[s]} for {i}")
                wempty[s].arrive()
            if i >= fs_n:
                yield fempty[fs], ((i // fs_n) - 1) & 1
            if not early and x_tag[s] != i:
                raise Violation(f"x warp {xi} read x of chunk {x_tag[s]} for {i}")
            f_tag[fs][xi] = i
            ffull[fs].arrive()
            if not early:
                wempty[s].arrive()

    def compute(w):
        for i in range(nch):
            s, fs = i % ns, i % fs_n
            yield wfull[s], (i // ns) & 1
            if w_tag[s] != i:
                raise Violation(f"compute warp {w} read weights of chunk {w_tag[s]} for {i}")
            if bug == "release_slot_first":
                fempty[fs].arrive()
            wempty[s].arrive()
            yield ffull[fs], (i // fs_n) & 1
            if any(v != i for v in f_tag[fs]):
                raise Violation(f"compute warp {w} read fragments {f_tag[fs]} for {i}")
            if bug != "release_slot_first":
                fempty[fs].arrive()

    agents = [copies()] + [x_warp(k) for k in range(xwarps)] + [compute(w) for w in range(8)]
    return run(agents, events, [], seed)


@pytest.mark.parametrize("fs_n", [2, 3])  # fragment slots: 3 for Q4_K / Q5_K, else 2
@pytest.mark.parametrize("xwarps,early", [(1, False), (1, True), (2, False), (2, True)])
def test_split_k_random_schedules_finish_and_read_what_they_should(xwarps, early, fs_n):
    for nch in (1, 2, 3, 5, 8, 14):
        for seed in range(40):
            run_split(nch, xwarps, early, seed=101 * nch + seed, fs_n=fs_n)


@pytest.mark.parametrize("bug", ["copy_skips_empty", "release_slot_first"])
def test_split_k_planted_mistakes_are_caught(bug):
    caught = 0
    for seed in range(200):
        try:
            run_split(8, 2, True, seed=seed, bug=bug)
        except Violation:
            caught += 1
    assert caught > 0
