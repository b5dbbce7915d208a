"""Counting identities the CUDA path relies on, checked by brute force on CPU.

The backoff kernel counts the corpus ends of exactly m matching tokens
(m = 2, 3) without measuring them: an end e matches at least m tokens of the
tail exactly when the last m-gram of the tail ends at e, so with Q_m = the
number of valid occurrences of the last m-gram (valid: a continuation follows
that is neither the sentinel nor past the end of the text),

    #{valid e : L(e) >= m} = Q_m   and   #{valid e : L(e) == m} = Q_m - Q_(m+1),

where L(e) is capped at min(D, n) and at e + 1 (SuffixGPU (PyPI), How it
works, step 1: every match length of every end).  This is what lets the
kernel take the ends of length 2 and 3 from the gram draft blocks' counts
and walk only the interval of the next longer gram.  Here both sides are
computed from their definitions on random tiny texts, with sentinels and
repeats, and random tails.
"""
import random

import pytest

from bruteforce import ends_of


def _L(X, t, e, D):
    n = len(t)
    lim = min(D, n, e + 1)
    l = 0
    while l < lim and X[e - l] == t[n - 1 - l]:
        l += 1
    return l


def _valid(X, Z, e):
    return e + 1 < len(X) and X[e + 1] != Z


@pytest.mark.parametrize("seed", range(6))
def test_exact_length_counts_from_gram_counts(seed):
    rng = random.Random(seed)
    for _ in range(200):
        V = rng.choice([2, 3, 5])
        Z = V
        X = []
        for _d in range(rng.randint(1, 6)):  # docs, each followed by the sentinel
            X += [rng.randrange(V) for _ in range(rng.randint(0, 30))] + [Z]
        n = rng.randint(1, 12)
        t = [rng.randrange(V) for _ in range(n)]
        D = rng.randint(1, 8)
        dl = min(D, n)
        valid_ends = [e for e in range(len(X)) if X[e] != Z and _valid(X, Z, e)]
        lengths = {e: _L(X, t, e, D) for e in valid_ends}
        for m in (2, 3):
            if dl < m:
                continue
            q_m = sum(1 for e in ends_of(X, t[n - m:]) if _valid(X, Z, e))
            assert sum(1 for e in valid_ends if lengths[e] >= m) == q_m
            if dl >= m + 1:
                q_m1 = sum(1 for e in ends_of(X, t[n - m - 1:]) if _valid(X, Z, e))
                assert sum(1 for e in valid_ends if lengths[e] == m) == q_m - q_m1
            else:  # the cap: every end of the m-gram matches exactly m
                assert sum(1 for e in valid_ends if lengths[e] == m) == q_m
