"""A host model of the one-launch kernel's grid barrier (its per-CTA arrival
tags and generation word), explored over random interleavings: no CTA may
leave a barrier before every CTA of the launch has arrived at it, whatever
the words held when the launch started (another tensor's data, a byte fill,
tags equal to the next generation), across launches that run back to back
on the same words, and after a CTA gives up (its timeout adds 2 to the
generation).  The model takes the kernel's steps as atomic actions of a
random scheduler:
  every CTA       reads the generation g
  CTA b > 0       writes its tag (g + 1) ^ salt, then waits until the
                  generation differs from g; it passes iff it reads g + 1
  CTA 0           waits until every tag reads (g + 1) ^ salt, then writes
                  g + 1
  a waiting CTA   may give up: it adds 2 to the generation and fails.
Two mutants must be caught: without the salt, by a planted tag; without the
generation's advance on a timeout, by the tags a failed launch left behind.
"""
import random

import pytest

MASK = (1 << 64) - 1


class Launch:
    def __init__(self, words, G, salt, rng, give_up_rate, poison=True):
        self.w, self.G, self.salt, self.rng, self.p_give_up = words, G, salt, rng, give_up_rate
        self.poison = 2 if poison else 0  # what a CTA that gives up adds to the generation
        self.g = [None] * G        # generation each CTA read
        self.arrived = [False] * G
        self.state = ["read"] * G  # read -> (tag) -> wait -> pass / fail
        self.passed_early = False

    def runnable(self):
        return [b for b in range(self.G) if self.state[b] not in ("pass", "fail")]

    def step(self, b):
        w, salt = self.w, self.salt
        st = self.state[b]
        if st == "read":
            self.g[b] = w[0]
            if b == 0:
                self.arrived[0] = True
                self.state[b] = "wait"
            else:
                self.state[b] = "tag"
        elif st == "tag":
            w[b] = ((self.g[b] + 1) & MASK) ^ salt
            self.arrived[b] = True
            self.state[b] = "wait"
        elif st == "wait":
            if self.rng.random() < self.p_give_up:
                w[0] = (w[0] + self.poison) & MASK
                self.state[b] = "fail"
                return
            g = self.g[b]
            if b == 0:
                want = ((g + 1) & MASK) ^ salt
                if all(w[c] == want for c in range(1, self.G)):
                    if not all(self.arrived):
                        self.passed_early = True
                    w[0] = (g + 1) & MASK
                    self.state[b] = "pass"
            else:
                v = w[0]
                if v != g:
                    if v == (g + 1) & MASK:
                        if not all(self.arrived):
                            self.passed_early = True
                        self.state[b] = "pass"
                    else:
                        self.state[b] = "fail"

    def run(self, max_steps=100000):
        for _ in range(max_steps):
            r = self.runnable()
            if not r:
                return
            # a CTA that waits for a barrier nobody can complete any more
            # (its generation moved on, or CTA 0 failed) stops on its timeout
            self.step(self.rng.choice(r))
        for b in self.runnable():  # every remaining wait runs out
            self.state[b] = "fail"
            self.w[0] = (self.w[0] + self.poison) & MASK


def initial_words(kind, G, rng):
    if kind == "random":
        return [rng.getrandbits(64) for _ in range(G)]
    if kind == "zeros":
        return [0] * G
    if kind == "ones":
        return [MASK] * G
    if kind == "next_generation":  # every tag equal to the unsalted next generation
        g = rng.getrandbits(64)
        return [g] + [(g + 1) & MASK] * (G - 1)
    if kind == "arange":           # int64 data of another tensor
        base = rng.randrange(1 << 20)
        return [base + i for i in range(G)]
    raise KeyError(kind)


KINDS = ["random", "zeros", "ones", "next_generation", "arange"]


@pytest.mark.parametrize("kind", KINDS)
def test_no_cta_passes_before_all_arrive(kind):
    rng = random.Random(1000 + KINDS.index(kind))
    for trial in range(60):
        G = rng.choice([1, 2, 3, 5, 8])
        words = initial_words(kind, G, rng)
        salt = rng.getrandbits(64) | 1
        give_up = rng.choice([0.0, 0.0, 0.002, 0.02])
        for launch in range(4):  # back to back on the same words
            L = Launch(words, G, salt, rng, give_up)
            L.run()
            assert not L.passed_early, (kind, trial, launch, G)
            if give_up == 0.0:
                # with every CTA resident and no timeout, every CTA passes
                assert all(s == "pass" for s in L.state), (kind, trial, launch, L.state)


def test_unsalted_mutant_is_caught():
    """Without the salt, tags left equal to the next generation release CTA 0
    before the others arrive: the model must see it."""
    rng = random.Random(7)
    caught = False
    for trial in range(200):
        G = 4
        words = initial_words("next_generation", G, rng)
        L = Launch(words, G, 0, rng, 0.0)
        L.run()
        caught = caught or L.passed_early
    assert caught


def test_mutant_without_timeout_advance_is_caught():
    """If a CTA that gives up left the generation alone, a launch after a
    failed one would read the same generation, and the tags the failed launch
    wrote would release CTA 0 early: the model must see it."""
    rng = random.Random(8)
    caught = False
    for trial in range(300):
        G = 5
        words = initial_words("random", G, rng)
        salt = rng.getrandbits(64) | 1
        for launch in range(4):
            L = Launch(words, G, salt, rng, 0.05, poison=False)
            L.run()
            caught = caught or L.passed_early
    assert caught
