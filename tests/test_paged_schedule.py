"""CPU model of the paged kernel's balanced schedule and of its merge pass.

Worker w of W takes global 16-token steps [w T / W, (w+1) T / W) of the
requests laid end to end (request b holds ceil(len_b / 16) steps starting at
P_b), walks them as segments of consecutive requests, writes a request whole
when one segment covers it and otherwise leaves a partial in slot 0 (its first
segment) or slot 1 (its last); the merge pass recomputes which workers hold a
request from P_b alone.  The model applies the same formulas and checks, on
random length mixes and worker counts, that every step is walked exactly once,
that every request (empty ones included) is written exactly once, and that the
merge pass finds exactly the partials the workers left, in the slots they left
them in.  (The GPU tests check the kernel itself against the oracle.)"""
import random

STEP = 16


def _walk(lens, W):
    steps = [(n + STEP - 1) // STEP for n in lens]
    T, B = sum(steps), len(lens)
    P = [0] * (B + 1)
    for b in range(B):
        P[b + 1] = P[b] + steps[b]
    covered, final, partials = {}, {}, {}
    for w in range(W):
        start, end = w * T // W, (w + 1) * T // W
        # the worker's first request: the first b with P_b + max(steps_b, 1) > start
        seg_b, seg_p = B, T
        for b in range(B):
            if P[b] + max(steps[b], 1) > start:
                seg_b, seg_p = b, P[b]
                break
        seg_t = start
        last = w == W - 1
        while seg_b < B and (seg_t < end or (last and seg_t == end)):
            b = seg_b
            seg_next = min(end, seg_p + steps[b])
            n_tok = min((seg_next - seg_p) * STEP, lens[b]) - (seg_t - seg_p) * STEP
            assert n_tok >= 0
            for st in range(seg_t, seg_next):
                assert (b, st) not in covered, ("step walked twice", b, st)
                covered[(b, st)] = w
            if seg_t == seg_p and seg_next == seg_p + steps[b]:
                assert b not in final, ("request written twice", b)
                final[b] = w
            else:
                assert (b, w) not in partials
                partials[(b, w)] = 0 if seg_t == start else 1
            if seg_next == seg_p + steps[b]:
                seg_p = seg_next
                seg_b += 1
            seg_t = seg_next
    return steps, T, P, covered, final, partials


def _check(lens, W):
    steps, T, P, covered, final, partials = _walk(lens, W)
    B = len(lens)
    for b in range(B):
        for st in range(P[b], P[b + 1]):
            assert (b, st) in covered, ("step not walked", b, st)
    for b in range(B):
        if steps[b] == 0:
            assert b in final, ("empty request not written", b)
            continue
        w_first = ((P[b] + 1) * W - 1) // T
        w_last = ((P[b] + steps[b]) * W - 1) // T
        if w_first == w_last:
            assert final.get(b) == w_first, ("whole request written by another worker", b)
            continue
        assert b not in final
        found = set()
        for w in range(w_first, w_last + 1):
            ws, wn = w * T // W, (w + 1) * T // W
            if ws == wn:
                continue  # a worker with no steps holds nothing
            slot = 1 if (w == w_first and ws < P[b]) else 0
            assert partials.get((b, w)) == slot, ("merge looks in the wrong slot", b, w)
            found.add((b, w))
        assert {k for k in partials if k[0] == b} == found, ("partial the merge does not read", b)


def test_schedule_edges():
    for lens, W in [([0], 1), ([0, 0, 0], 5), ([1], 7), ([16, 17, 0, 1], 3), ([3000], 304),
                    ([512] * 256, 304), ([512] * 256, 256), ([0, 5000, 0, 1], 40), ([31, 32, 33], 100)]:
        _check(lens, W)


def test_schedule_random_mixes():
    rng = random.Random(1)
    for _ in range(4000):
        B = rng.randint(1, 12)
        lens = [rng.choice([0, 0, 1, 5, 16, 17, 31, 32, 100, 1000, rng.randint(0, 3000)]) for _ in range(B)]
        _check(lens, rng.randint(1, 40))
