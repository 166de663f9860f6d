"""Model checks of the exchange flow control of the D = 512 CTA pairs (the
forward's in smqa_fwd.cu, the backward's in smqa_bwd.cu), run on the CPU.

Two CTAs, each with three score tiles, a four-stage kv ring and X exchange
buffers per receiver.  Per block i each CTA:
  gather(i)   needs kv stage i % 4 free (P.V of block i - 4 done);
  scores(i)   needs gather(i) and score tile i % 3 free (softmax read i - 3);
  send(i)     needs scores(i) and, for i >= X, the peer's block i - X + 3 to
              have arrived here; it writes block i into the peer's buffer
              i % X, and the block arrives there some time later;
  combine(i)  needs the peer's block i in buffer i % X (then consumes it)
              and this CTA's send(i) (the rounded own partial);
  softmax(i)  needs combine(i); frees score tile i % 3;
  pv(i)       needs softmax(i); frees kv stage i % 4.
Each role runs its blocks in order.  A random scheduler picks among the
enabled steps (message deliveries included) until both CTAs finish.

Checked: a send never overwrites a buffer block the peer has not consumed;
every wait on a receive barrier (phase i // X of barrier i % X, tested by
parity as mbarriers are) is never two or more phases behind the barrier,
where a parity test would misread it; and the run never deadlocks.  X = 3
must deadlock (each sender would wait for the peer's same block), which
shows that the model can fail."""
import random

import pytest

ROLES = ("gather", "scores", "send", "combine", "softmax", "pv")


def run_model(X: int, nblk: int, seed: int, tiles: int = 3, stages: int = 4):
    rng = random.Random(seed)
    nxt = [{r: 0 for r in ROLES} for _ in range(2)]  # next block of each role
    arrived = [set(), set()]        # blocks that have arrived in CTA c's buffers
    in_flight = []                  # (dest CTA, block) messages not yet delivered
    consumed = [set(), set()]       # blocks CTA c's combiner has consumed
    phases = [[0] * X for _ in range(2)]  # completed phases of CTA c's receive barriers

    def done(c, role, i):
        return i < nxt[c][role]

    def check_wait(c, blk):
        # waiting for phase blk // X of barrier blk % X: the barrier must not
        # have completed phase blk // X + 1 already
        assert phases[c][blk % X] <= blk // X + 1, ("phase aliasing", c, blk)

    def enabled(c):
        out = []
        i = nxt[c]["gather"]
        if i < nblk and (i < stages or done(c, "pv", i - stages)):
            out.append("gather")
        i = nxt[c]["scores"]
        if i < nblk and done(c, "gather", i) and (i < tiles or done(c, "softmax", i - tiles)):
            out.append("scores")
        i = nxt[c]["send"]
        if i < nblk and done(c, "scores", i):
            if i >= X:
                j = i - X + tiles
                check_wait(c, j)
                if j in arrived[c]:
                    out.append("send")
            else:
                out.append("send")
        i = nxt[c]["combine"]
        if i < nblk and done(c, "send", i):
            check_wait(c, i)
            if i in arrived[c]:
                out.append("combine")
        i = nxt[c]["softmax"]
        if i < nblk and done(c, "combine", i):
            out.append("softmax")
        i = nxt[c]["pv"]
        if i < nblk and done(c, "softmax", i):
            out.append("pv")
        return out

    while any(nxt[c][r] < nblk for c in range(2) for r in ROLES):
        choices = [(c, r) for c in range(2) for r in enabled(c)]
        choices += [("deliver", k) for k in range(len(in_flight))]
        if not choices:
            return "deadlock"
        c, r = rng.choice(choices)
        if c == "deliver":
            dest, blk = in_flight.pop(r)
            arrived[dest].add(blk)
            phases[dest][blk % X] += 1
            continue
        i = nxt[c][r]
        if r == "send":
            peer = 1 - c
            if i >= X:  # the buffer's previous block must have been consumed
                assert (i - X) in consumed[peer], ("overwrite", c, i)
            in_flight.append((peer, i))
        elif r == "combine":
            consumed[c].add(i)
        nxt[c][r] += 1
    return "ok"


@pytest.mark.parametrize("X", [4, 5, 6])
@pytest.mark.parametrize("seed", range(40))
@pytest.mark.parametrize("stages", [4, 5])
def test_exchange_protocol_is_safe_and_live(X, seed, stages):
    assert run_model(X, nblk=24, seed=seed, stages=stages) == "ok"


def test_three_buffers_deadlock():
    assert all(run_model(3, nblk=12, seed=s) == "deadlock" for s in range(5))


# ---------------------------------------------------------------------------
# The backward pair (smqa_bwd.cu): one S/dP tile, a two-stage kv ring, one
# P/dS shared-memory buffer and NB exchange buffers with an explicit
# consumed-signal (SendOk).  The P/dS threads both send this CTA's partials
# and consume the peer's; with G groups, group g handles blocks i = g mod G
# in order (G = 2: the two groups alternate blocks and overlap).  Per block:
#   gather(i)    needs kv stage i % 2 free (the kernel frees it after the dQ
#                MMAs of block i - 2; the model waits for all of grad(i - 2),
#                which is stricter);
#   sdp(i)       needs gather(i) and the S/dP tile read by read(i - 1);
#   read(i)      needs sdp(i) and pds(i - G) (the same threads, in order);
#   send(i)      needs read(i) and, for i >= NB, the peer's SendOk for block
#                i - NB; writes buffer i % NB of the peer (in flight);
#   pds(i)       needs send(i), grad(i - 1) (the single P/dS buffer) and the
#                peer's block i; consumes it and, if i + NB < nblk, sends
#                SendOk for buffer i % NB to the peer (in flight);
#   grad(i)      needs pds(i) and drain(i - 1) (single dKV tile);
#   drain(i)     needs grad(i).
# A barrier that a group waits on is only ever completed for that group's
# blocks (per-parity barriers), so the parity tests below check phases per
# group.
BWD_ROLES = ("gather", "sdp", "read", "send", "pds", "grad", "drain")


def run_bwd_model(NB: int, nblk: int, seed: int, G: int = 1):
    rng = random.Random(seed)
    nxt = [{r: 0 for r in BWD_ROLES} for _ in range(2)]
    done_set = [{r: set() for r in BWD_ROLES} for _ in range(2)]
    arrived = [set(), set()]
    sendok = [set(), set()]        # consumed-signals received by CTA c (block numbers)
    consumed = [set(), set()]
    recv_ph = [[0] * NB for _ in range(2)]
    ok_ph = [[0] * NB for _ in range(2)]
    in_flight = []                 # (kind, dest, block)
    # The per-group roles (read, send, pds) keep one cursor per group.
    gnxt = [[{r: g for r in ("read", "send", "pds")} for g in range(G)] for _ in range(2)]

    def done(c, role, i):
        return i in done_set[c][role]

    def enabled(c):
        out = []
        n = nxt[c]
        i = n["gather"]
        if i < nblk and (i < 2 or done(c, "grad", i - 2)):
            out.append(("gather", i))
        i = n["sdp"]
        if i < nblk and done(c, "gather", i) and (i == 0 or done(c, "read", i - 1)):
            out.append(("sdp", i))
        for g in range(G):
            cur = gnxt[c][g]
            i = cur["read"]
            if i < nblk and done(c, "sdp", i) and (i < G or done(c, "pds", i - G)):
                out.append(("read", i))
            i = cur["send"]
            if i < nblk and done(c, "read", i):
                if i >= NB:
                    assert ok_ph[c][i % NB] <= (i // NB - 1) + 1, ("sendok aliasing", c, i)
                    if (i - NB) in sendok[c]:
                        out.append(("send", i))
                else:
                    out.append(("send", i))
            i = cur["pds"]
            if i < nblk and done(c, "send", i) and (i == 0 or done(c, "grad", i - 1)):
                assert recv_ph[c][i % NB] <= i // NB + 1, ("recv aliasing", c, i)
                if i in arrived[c]:
                    out.append(("pds", i))
        i = n["grad"]
        if i < nblk and done(c, "pds", i) and (i == 0 or done(c, "drain", i - 1)):
            out.append(("grad", i))
        i = n["drain"]
        if i < nblk and done(c, "grad", i):
            out.append(("drain", i))
        return out

    def finished():
        return all(len(done_set[c]["drain"]) == nblk for c in range(2))

    while not finished():
        choices = [(c, e) for c in range(2) for e in enabled(c)]
        choices += [("deliver", k) for k in range(len(in_flight))]
        if not choices:
            return "deadlock"
        c, e = rng.choice(choices)
        if c == "deliver":
            kind, dest, blk = in_flight.pop(e)
            if kind == "data":
                arrived[dest].add(blk)
                recv_ph[dest][blk % NB] += 1
            else:
                sendok[dest].add(blk)
                ok_ph[dest][blk % NB] += 1
            continue
        r, i = e
        peer = 1 - c
        if r == "send":
            if i >= NB:
                assert (i - NB) in consumed[peer], ("overwrite", c, i)
            in_flight.append(("data", peer, i))
        elif r == "pds":
            consumed[c].add(i)
            if i + NB < nblk:
                in_flight.append(("ok", peer, i))
        done_set[c][r].add(i)
        if r in ("read", "send", "pds"):
            gnxt[c][i % G][r] += G
        else:
            nxt[c][r] += 1
    return "ok"


@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("NB", [2, 3, 4])
@pytest.mark.parametrize("seed", range(30))
def test_backward_exchange_protocol_is_safe_and_live(NB, seed, G):
    assert run_bwd_model(NB, nblk=24, seed=seed, G=G) == "ok"


# ---------------------------------------------------------------------------
# The persistent kernels' token layer (smqa_fwd.cu, smqa_bwd.cu): one CTA
# works through a sequence of tokens, each of nblk[k] blocks (zero allowed),
# as one sequence of blocks G.  A four-entry ring publishes each token; every
# reader releases an entry once done with it, and the producer (the gather
# warps) publishes token k only once all readers have released token k - 4.
# Per token the CTA has one Q buffer (forward; Q and dO in the backward),
# reloaded once the previous loaded token's MMAs that read it have completed,
# and one accumulator (O / dQ in TMEM) that the next token with blocks may
# overwrite only after the current one's read-out.  The forward sets up token
# k + 1 after `pre` blocks of token k are gathered (pre = min(nblk, 2)), the
# backward after all of them.
#
# Forward roles: gather(G) needs kv stage G % 5 free (pv(G - 5)); scores(G)
# needs gather(G), score tile G % 3 free (softmax(G - 3)) and its token's Q;
# softmax(G) needs scores(G) (the pair's exchange, modelled above, sits in
# between), the P buffer G % 2 free (pv(G - 2)) and, for any but a token's
# first block, pv(G - 1) (the rescale; always taken here, which only adds
# waits); pv(G) needs softmax(G) and, for a token's first block, the previous
# token's read-out; the read-out of token k needs pv of its last block.  The
# Q of token k may load once every scores MMA of the previous loaded token is
# done.  Readers of the ring: the MMA thread (releases a token once its P.V
# cursor is past it) and the softmax (at the token's start); the combiner and
# sender release at the token's start like the softmax and add nothing here.
#
# Backward roles: gather(G) needs kv stage G % 2 free (grad(G - 2)); sdp(G)
# needs gather(G), the S/dP tile read (pds(G - 1)) and its token's Q / dO;
# pds(G) needs sdp(G) and the P/dS buffer (grad(G - 1)); grad(G) needs pds(G),
# the dKV^T tile drained (drain(G - 1)) and, for a token's first block, the
# previous token's dQ read-out; drain(G) needs grad(G); the read-out of token
# k (by the drain warps) needs drain and grad of its last block.  Q / dO of
# token k load once every MMA of the previous loaded token is done.  Readers:
# the MMA thread (releases after its gradient cursor), the P/dS warps and the
# drain (at the token's start).
RING = 4


def run_persistent_model(kind: str, nblks, seed: int, mutant: str = ""):
    rng = random.Random(seed)
    ntok = len(nblks)
    first = []                       # G of each token's first block
    g = 0
    for n in nblks:
        first.append(g)
        g += n
    total = g
    tok_of = []
    for k, n in enumerate(nblks):
        tok_of += [k] * n
    fwd = kind == "fwd"
    blk_roles = ("gather", "s", "soft", "pv") if fwd else ("gather", "s", "pds", "grad", "drain")
    done = {r: set() for r in blk_roles}
    readout = set()                  # tokens whose accumulator has been read out
    published = []                   # tokens published so far (in order)
    released = {}                    # token -> readers that released it
    readers = ("mma", "soft") if fwd else ("mma", "pds", "drain")
    tok_ph = [0] * RING              # completed phases of each ring entry's full barrier
    loaded = []                      # tokens whose Q (Q / dO) load was issued, in order
    role_tok = {r: 0 for r in readers if r != "mma"}  # next token each reader starts
    mma_rel = 0                      # next token the MMA thread releases
    gcur = [0, 0]                    # producer: next token to gather, next block in it
    pending_setup = [0]              # next token to set up (publish)

    def non_empty_before(k):
        return [j for j in range(k) if nblks[j] > 0]

    def q_of_ok(G):
        return tok_of[G] in loaded

    def entry_free(k):
        if k < RING:
            return True
        return released.get(k - RING, set()) == set(readers)

    def entry_gate(k):  # what the producer waits for (a mutant drops the MMA's release)
        if k < RING:
            return True
        need = set(readers) - ({"mma"} if mutant == "ring_ignores_mma" else set())
        return need <= released.get(k - RING, set())

    def reader_wait(k):
        # a reader waiting for token k: the entry must not be two phases ahead
        assert tok_ph[k % RING] <= k // RING + 1, ("ring aliasing", k)
        return k < len(published)

    def last_block_done(role, k):
        n = nblks[k]
        return n == 0 or (first[k] + n - 1) in done[role]

    def enabled():
        out = []
        # producer: setup, or the next gather
        ks, (kg, ig) = pending_setup[0], gcur
        setup_due = ks < ntok + 1 and ks <= kg + 1 and (
            ks == 0 or (ks == kg + 1 and (ig >= min(nblks[kg], 2 if fwd else nblks[kg]))))
        if setup_due and ks <= ntok and entry_gate(ks):
            out.append(("setup", ks))
        elif kg < ntok and kg < len(published) and ig < nblks[kg]:
            G = first[kg] + ig
            stages = 5 if fwd else 2
            free = G < stages or ((G - stages) in done["pv" if fwd else "grad"])
            if free:
                out.append(("gather", G))
        # Q load of the next token with blocks
        nxt_load = [k for k in range(ntok) if nblks[k] > 0 and k not in loaded]
        if nxt_load:
            k = nxt_load[0]
            if k < len(published):
                prev = [j for j in loaded]
                if not prev or mutant == "q_no_wait" or all(
                        (first[prev[-1]] + b) in done["s" if fwd else "grad"] for b in range(nblks[prev[-1]])):
                    out.append(("load", k))
        for G in range(total):
            k = tok_of[G]
            ib = G - first[k]
            if fwd:
                if G not in done["s"] and (G == 0 or (G - 1) in done["s"]) and G in done["gather"] \
                        and (G < 3 or (G - 3) in done["soft"]) and q_of_ok(G):
                    out.append(("s", G))
                if G not in done["soft"] and (G == 0 or (G - 1) in done["soft"]) and G in done["s"] \
                        and (G < 2 or (G - 2) in done["pv"]) and (ib == 0 or (G - 1) in done["pv"]) \
                        and role_tok["soft"] > k:
                    out.append(("soft", G))
                prev = non_empty_before(k)
                if G not in done["pv"] and (G == 0 or (G - 1) in done["pv"]) and G in done["soft"] \
                        and (ib > 0 or not prev or prev[-1] in readout or mutant == "acc_no_wait"):
                    out.append(("pv", G))
            else:
                if G not in done["s"] and (G == 0 or (G - 1) in done["s"]) and G in done["gather"] \
                        and (G == 0 or (G - 1) in done["pds"]) and q_of_ok(G):
                    out.append(("s", G))
                if G not in done["pds"] and (G == 0 or (G - 1) in done["pds"]) and G in done["s"] \
                        and (G == 0 or (G - 1) in done["grad"]) and role_tok["pds"] > k:
                    out.append(("pds", G))
                prev = non_empty_before(k)
                if G not in done["grad"] and (G == 0 or (G - 1) in done["grad"]) and G in done["pds"] \
                        and (G == 0 or (G - 1) in done["drain"]) \
                        and (ib > 0 or not prev or prev[-1] in readout or mutant == "acc_no_wait"):
                    out.append(("grad", G))
                if G not in done["drain"] and (G == 0 or (G - 1) in done["drain"]) \
                        and G in done["grad"] and role_tok["drain"] > k:
                    out.append(("drain", G))
        # readers starting a token (waiting for its publication)
        for r in role_tok:
            k = role_tok[r]
            if k < ntok and reader_wait(k):
                # the reader finishes its previous token first
                if k == 0 or (r == "soft" and last_block_done("soft", k - 1) and (k - 1) in readout) \
                        or (r == "pds" and last_block_done("pds", k - 1)) \
                        or (r == "drain" and last_block_done("drain", k - 1) and (k - 1) in readout):
                    out.append(("start_" + r, k))
        # read-out of the accumulator (forward: the softmax; backward: the drain)
        owner = "soft" if fwd else "drain"
        for k in range(ntok):
            if k not in readout and role_tok[owner] > k and last_block_done(owner, k) \
                    and last_block_done("pv" if fwd else "grad", k) \
                    and all(j in readout for j in range(k)):
                out.append(("readout", k))
        # the MMA thread releases a token once its last P.V / gradient is issued
        k = mma_rel
        if k < ntok and k < len(published) and last_block_done("pv" if fwd else "grad", k):
            out.append(("mma_release", k))
        return out

    steps = 0
    while True:
        all_done = len(readout) == ntok and all(len(done[r]) == total for r in blk_roles)
        if all_done:
            return "ok"
        choices = enabled()
        if not choices:
            return "deadlock"
        ev, x = rng.choice(choices)
        steps += 1
        assert steps < 200000
        if ev == "setup":
            k = x
            if k < ntok:
                assert k < RING or mma_rel > k - RING, ("ring entry overwritten while the MMA reads it", k)
                assert entry_free(k), ("overwrite of a live ring entry", k)
                published.append(k)
                tok_ph[k % RING] += 1
            pending_setup[0] = k + 1
            if k == 0:
                gcur[0], gcur[1] = 0, 0
        elif ev == "gather":
            done["gather"].add(x)
            gcur[1] += 1
            while gcur[0] < ntok and gcur[1] >= nblks[gcur[0]] and pending_setup[0] > gcur[0] + 1:
                gcur[0] += 1
                gcur[1] = 0
        elif ev == "load":
            if loaded:
                last = loaded[-1]
                assert all((first[last] + b) in done["s" if fwd else "grad"] for b in range(nblks[last])), \
                    ("Q reloaded under pending MMAs", x)
            loaded.append(x)
        elif ev.startswith("start_"):
            r = ev[6:]
            released.setdefault(x, set()).add(r)
            role_tok[r] = x + 1
        elif ev == "readout":
            readout.add(x)
        elif ev == "mma_release":
            released.setdefault(x, set()).add("mma")
            mma_rel = x + 1
        else:
            if ev in ("pv", "grad"):
                k = tok_of[x]
                if x == first[k]:
                    prev = non_empty_before(k)
                    assert not prev or prev[-1] in readout, ("accumulator overwritten", k)
            done[ev].add(x)
        # the producer moves to the next token once its blocks are gathered and
        # the next one is set up
        while gcur[0] < ntok and gcur[1] >= nblks[gcur[0]] and pending_setup[0] > gcur[0] + 1:
            gcur[0] += 1
            gcur[1] = 0


def _token_mix(rng, ntok):
    out = []
    for _ in range(ntok):
        r = rng.random()
        out.append(0 if r < 0.25 else 1 if r < 0.4 else 2 if r < 0.5 else rng.randint(3, 9))
    return out


@pytest.mark.parametrize("kind", ["fwd", "bwd"])
@pytest.mark.parametrize("seed", range(40))
def test_persistent_token_layer_is_safe_and_live(kind, seed):
    rng = random.Random(1000 + seed)
    nblks = _token_mix(rng, 14)
    if seed % 5 == 0:
        nblks[3:8] = [0] * 5      # a run of empty tokens
    if seed % 7 == 0:
        nblks = [0] * 6           # no token has a block
    assert run_persistent_model(kind, nblks, seed) == "ok"


@pytest.mark.parametrize("kind,mutant", [("fwd", "ring_ignores_mma"), ("fwd", "q_no_wait"),
                                          ("bwd", "ring_ignores_mma"), ("bwd", "q_no_wait"),
                                          ("bwd", "acc_no_wait")])
def test_persistent_model_catches_planted_mistakes(kind, mutant):
    """Each planted mistake -- the producer not waiting for the MMA thread's
    release of a ring entry, Q (Q / dO) reloaded without waiting for the
    MMAs that read it, the backward's first gradient of a token not waiting
    for the previous token's dQ read-out -- trips a safety check on some
    schedule.  (In the forward the O read-out is done by the softmax threads
    before they write the next token's first P, which that token's first P.V
    needs anyway: the kernel's wait for it is implied, and dropping it here
    is no mistake.)"""
    caught = 0
    for seed in range(60):
        rng = random.Random(2000 + seed)
        nblks = _token_mix(rng, 14)
        try:
            run_persistent_model(kind, nblks, seed, mutant=mutant)
        except AssertionError:
            caught += 1
    assert caught > 0
