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
