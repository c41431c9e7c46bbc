"""A model of the prefill MMQ's barrier protocol (csrc/mmq.cu), run under random schedules on
the CPU: the TMA producer, the two MMA issuers, the epilogue and, in the decode-plane form
(MQ_REG_MMQ_FROM_DECODE_PLANE), the four weight decoders are agents; TMA copies and MMA
completions are asynchronous events that land in any order (a CTA's MMAs complete in issue
order).  mbarriers follow the PTX phase rules (a wait on parity p returns once the phase of
parity p has completed, at once on a fresh barrier for p = 1).  Every run must finish (no
deadlock) and every read must see the data meant for it: the MMA the stage's activation and
weight tiles of its fill (at issue and at completion), the decoders the chunk of their fill,
the epilogue the accumulator of its use and the scales of its group.  The index arithmetic
of each role is the kernel's, restated.  Planted protocol mistakes must be caught."""
import pytest

from tests.protocol_model import Bar, Violation, run

K_RAMP = 3
PK_SLOTS = 3


def run_cta(ntiles, grid, b, ntm, nb, dots, pw, seed, bug=None):
    """One CTA (blockIdx b of `grid`) of a Q4_K MMQ over ntiles output tiles (ntm along M),
    nb 32-element blocks along K.  Returns the number of scheduling steps."""
    NST = 4 if pw else 6
    SR = NST // 2
    npairs, ngroups, nchk = (nb + 1) // 2, (nb + 7) >> 3, nb // 8
    nms = 0 if dots else (3 * nb + 63) // 64
    nmu = 2 if nms > 0 else 0
    nuse = npairs + nmu
    full = [Bar(5 if pw else 1) for _ in range(NST)]
    empty = [Bar(1) for _ in range(NST)]
    tfull, tempty = [Bar(1) for _ in range(2)], [Bar(1) for _ in range(2)]
    gfull, gempty = [Bar(1) for _ in range(2)], [Bar(1) for _ in range(2)]
    pfull, pempty = [Bar(1) for _ in range(PK_SLOTS)], [Bar(4) for _ in range(PK_SLOTS)]
    a_tag, b_tag = [None] * NST, [None] * NST
    bpart = [[None] * 4 for _ in range(NST)]  # decode-plane form: each decoder's rows
    pk_tag, gs_tag, acc_tag = [None] * PK_SLOTS, [None] * 2, [None] * 2
    events = []        # TMA copies: land in any order
    mma_q = [[], []]   # per issuer: MMA completions and commits, in order
    tiles = list(range(b, ntiles, grid))

    def fill_stage(tl, f, c_ctr):
        pr = f if f < npairs else -1
        i = (tl * nuse + (f if f < npairs else npairs + ((f - npairs) & 1))) & 1
        c = c_ctr[i]
        c_ctr[i] += 1
        return pr, i, i + 2 * (c % SR), c // SR

    def land(bar, n, fn):
        def ev():
            fn()
            bar.complete_tx(n)
        events.append(ev)

    def chunk_copy(cg):
        ps = (cg + (bug == "chunk_slot_off_by_one")) % PK_SLOTS
        pfull[ps].expect_tx(1)
        land(pfull[ps], 1, lambda: pk_tag.__setitem__(ps, cg))

    def producer():
        nchunks = len(tiles) * nchk if pw else 0
        pre = 0
        if pw:
            for cg in range(min(PK_SLOTS, nchunks)):
                chunk_copy(cg)
        elif tiles:
            pre = min(npairs, K_RAMP)
            for f in range(pre):
                full[f].expect_tx(2)
                land(full[f], 1, lambda f=f: b_tag.__setitem__(f, (0, f)))
        c_ctr = [0, 0]
        for tl, t in enumerate(tiles):
            for f in range(npairs + nms):
                pr, i, s, q = fill_stage(tl, f, c_ctr)
                if not dots and pr >= 0 and pr % 4 == 0:
                    g = pr >> 2
                    G = tl * ngroups + g
                    slot = G & 1
                    if G >= 2:
                        yield gempty[slot], ((G >> 1) - 1) & 1
                    gfull[slot].expect_tx(2)
                    land(gfull[slot], 2, lambda slot=slot, v=(tl, g): gs_tag.__setitem__(slot, v))
                if q >= 1:
                    yield empty[s], (q - 1) & 1
                elif tl == 0 and s >= K_RAMP:
                    yield full[s - K_RAMP], 0
                if pr < 0:
                    full[s].expect_tx(2)
                    v = ("min", tl, f)
                    land(full[s], 1, lambda s=s, v=v: a_tag.__setitem__(s, v))
                    land(full[s], 1, lambda s=s, v=v: b_tag.__setitem__(s, v))
                    continue
                if tl == 0 and f < pre:
                    land(full[s], 1, lambda s=s, v=(tl, pr): a_tag.__setitem__(s, v))
                    continue
                full[s].expect_tx(1 if pw else 2)
                land(full[s], 1, lambda s=s, v=(tl, pr): a_tag.__setitem__(s, v))
                if pw:
                    cg = tl * nchk + (pr >> 2)
                    cn = cg + PK_SLOTS - 1
                    if pr % 4 == 0 and cg >= 1 and cn < nchunks:
                        if bug != "producer_skips_pempty":
                            yield pempty[cn % PK_SLOTS], (cn // PK_SLOTS - 1) & 1
                        chunk_copy(cn)
                else:
                    land(full[s], 1, lambda s=s, v=(tl, pr): b_tag.__setitem__(s, v))

    def decoder(dw):
        c_ctr = [0, 0]
        for tl, t in enumerate(tiles):
            for f in range(npairs + nms):
                pr, i, s, q = fill_stage(tl, f, c_ctr)
                if q >= 1 and bug != "decoder_skips_empty":
                    yield empty[s], (q - 1) & 1
                cg = tl * nchk + (pr >> 2)
                ps = cg % PK_SLOTS
                if pr >= 0:
                    if pr % 4 == 0:
                        yield pfull[ps], (cg // PK_SLOTS) & 1
                    if pk_tag[ps] != cg:
                        raise Violation(f"decoder {dw} read chunk {pk_tag[ps]} for {cg}")
                    bpart[s][dw] = (tl, pr)
                full[s].arrive()
                if pr >= 0 and pr % 4 == 3:
                    pempty[ps].arrive()

    def weight_ok(s, want):
        if pw and not (isinstance(want, tuple) and want[0] == "min"):
            return all(v == want for v in bpart[s])
        return b_tag[s] == want

    def issuer(i):
        c = 0
        for tl, t in enumerate(tiles):
            u = (i - tl * nuse) & 1
            while u < nuse:
                use = (tl * nuse + u) >> 1
                if use >= 1 and bug != "issuer_skips_tempty":
                    yield tempty[i], (use - 1) & 1
                if u >= npairs:
                    j = u - npairs
                    ks = (nms - j + 1) >> 1
                    for k in range(ks):
                        s = i + 2 * (c % SR)
                        want = ("min", tl, npairs + j + 2 * k)
                        yield full[s], (c // SR) & 1
                        c += 1
                        issue_mma(i, s, want)
                    commit_acc(i, ("min", tl, npairs + j))
                    u += 2
                    continue
                s = i + 2 * (c % SR)
                yield full[s], (c // SR) & 1
                c += 1
                issue_mma(i, s, (tl, u))
                commit_acc(i, (tl, u))
                u += 2

    def issue_mma(i, s, want):
        if a_tag[s] != want or not weight_ok(s, want):
            raise Violation(f"MMA on stage {s} found {a_tag[s]}/{b_tag[s]}/{bpart[s]} for {want}")

        def done():
            if a_tag[s] != want or not weight_ok(s, want):
                raise Violation(f"stage {s} overwritten before its MMA for {want} completed")
            empty[s].arrive()
        mma_q[i].append(done)

    def commit_acc(i, v):
        def done():
            acc_tag[i] = v
            tfull[i].arrive()
        mma_q[i].append(done)

    def epilogue():
        for tl, t in enumerate(tiles):
            ub = (tl * nuse) >> 1
            for g in range(ngroups):
                G = tl * ngroups + g
                slot = G & 1
                if not dots:
                    yield gfull[slot], (G >> 1) & 1
                    if gs_tag[slot] != (tl, g):
                        raise Violation(f"epilogue read scales {gs_tag[slot]} for {(tl, g)}")
                for pp in range(4):
                    pr = 4 * g + pp
                    i = pp & 1
                    yield tfull[i], (ub + (pp >> 1)) & 1
                    if acc_tag[i] != (tl, pr):
                        raise Violation(f"epilogue read accumulator {acc_tag[i]} for {(tl, pr)}")
                    tempty[i].arrive()
                if not dots:
                    gempty[slot].arrive()
            for j in range(nmu):
                U = tl * nuse + npairs + j
                i = U & 1
                yield tfull[i], (U >> 1) & 1
                if nms - j > 0 and acc_tag[i] != ("min", tl, npairs + j):
                    raise Violation(f"epilogue read min term {acc_tag[i]}")
                tempty[i].arrive()

    agents = [producer(), issuer(0), issuer(1), epilogue()]
    if pw:
        agents += [decoder(d) for d in range(4)]
    return run(agents, events, mma_q, seed)


SHAPES = [  # ntiles, grid, ntm, nb: one tile, several per CTA, one chunk per tile, many
    (1, 1, 1, 8), (3, 1, 1, 16), (5, 2, 2, 8), (6, 2, 3, 24), (4, 1, 2, 32), (7, 3, 1, 16),
]


@pytest.mark.parametrize("pw", [False, True])
@pytest.mark.parametrize("dots", [False, True])
def test_random_schedules_finish_and_read_what_they_should(pw, dots):
    runs = 0
    for ntiles, grid, ntm, nb in SHAPES:
        for b in range(min(grid, ntiles)):
            for seed in range(40):
                run_cta(ntiles, grid, b, ntm, nb, dots, pw, seed=1000 * nb + 10 * b + seed)
                runs += 1
    assert runs > 0


@pytest.mark.parametrize("bug,pw", [("decoder_skips_empty", True), ("producer_skips_pempty", True),
                                    ("chunk_slot_off_by_one", True), ("issuer_skips_tempty", True),
                                    ("issuer_skips_tempty", False)])
def test_planted_protocol_mistakes_are_caught(bug, pw):
    """A decoder that writes a stage before the MMA has released it, a producer that reuses a
    chunk slot before the decoders are done with it or copies a chunk into the wrong slot, and
    an issuer that overwrites an accumulator the epilogue has not read must each fail some
    schedule."""
    caught = 0
    for seed in range(300):
        try:
            run_cta(4, 1, 0, 2, 32, False, pw, seed=seed, bug=bug)
        except Violation:
            caught += 1
    assert caught > 0
