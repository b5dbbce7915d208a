"""Brute-force drafter for tiny inputs, formulated differently from the oracle.

The oracle computes per-position backward match lengths and runs the vote on
an explicit occurrence set.  Here everything is re-derived by naive substring
search instead:

* the match length M is the largest l for which the last l tokens occur
  somewhere else followed by a continuation (for the corpus: by a token other
  than the sentinel);
* with an unbounded occurrence budget, the survivors after emitting
  tau_0..tau_{d-1} are exactly the occurrences of the string
  tail[-M:] + tau_0..tau_{d-1}, so the depth-d vote counts occurrences of
  that string extended by each candidate token;
* with a budget R, the occurrence list is the R largest end positions of
  tail[-M:], found by the same substring search, and each later depth looks
  the continuation up directly.

Pure Python, quadratic or worse: only for n, N up to a few dozen tokens.
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Optional, Sequence, Tuple


def ends_of(text: Sequence[int], pat: Sequence[int]) -> List[int]:
    """All e with text[e-len(pat)+1 .. e] == pat."""
    m = len(pat)
    out = []
    for s in range(0, len(text) - m + 1):
        if list(text[s:s + m]) == list(pat):
            out.append(s + m - 1)
    return out


def count_occ(text: Sequence[int], pat: Sequence[int]) -> int:
    return len(ends_of(text, pat))


class Result:
    def __init__(self):
        self.drafts: List[int] = []
        self.probs: List[Fraction] = []
        self.M = 0
        self.source = 0
        self.c0 = 0

    @property
    def score(self) -> Fraction:
        return sum(self.probs, Fraction(0))


def _self_M(t: List[int], D: int) -> int:
    n = len(t)
    for l in range(min(D, n - 1), 0, -1):
        # an occurrence of the last l tokens that ends at or before n-2
        if any(e <= n - 2 for e in ends_of(t, t[n - l:])):
            return l
    return 0


def _corpus_M(X: List[int], Z: int, t: List[int], D: int) -> int:
    n = len(t)
    if D < 2 or n < 2:
        return 0
    for l in range(min(D, n), 1, -1):
        pat = t[n - l:]
        for e in ends_of(X, pat):
            if e + 1 < len(X) and X[e + 1] != Z:
                return l
    return 0


def brute_propose(t: Sequence[int], n: int, k: int, D: int, R: Optional[int], S: int,
                  factor: Tuple[int, int], offset: int, min_prob: Tuple[int, int],
                  X: Optional[Sequence[int]] = None, Z: int = -1,
                  depth_sum_cap: bool = False) -> Result:
    """R=None means an unbounded occurrence budget."""
    t = list(t[:n])
    res = Result()
    if n == 0:
        return res
    Ms = _self_M(t, D) if n >= 2 else 0
    Mc = _corpus_M(list(X), Z, t, D) if X is not None and len(X) > 0 else 0
    if Mc > Ms:
        src, M, text = 2, Mc, list(X)
    else:
        src, M, text = (1 if Ms > 0 else 0), Ms, t
    res.M, res.source = M, src
    if M == 0:
        return res

    tail = t[n - M:]

    def has_cont(e):
        if src == 1:
            return e <= n - 2
        return e + 1 < len(text) and text[e + 1] != Z

    occ = sorted((e for e in ends_of(text, tail) if has_cont(e)), reverse=True)
    if R is not None:
        occ = occ[:R]
    c0 = len(occ)
    res.c0 = c0
    cap = min(k, (factor[0] * M) // factor[1] + offset, max(0, S - n - 1))
    if depth_sum_cap:
        cap = min(cap, D - M)

    def cont(e, d):
        q = e + 1 + d
        if src == 1:
            return t[q] if q <= n - 1 else None
        return text[q] if q < len(text) and text[q] != Z else None

    if R is None:
        # survivors are occurrences of tail + emitted; count by substring search
        W = list(tail)
        alphabet = sorted(set(x for x in text if not (src == 2 and x == Z)))
        for d in range(max(cap, 0)):
            counts = {x: count_occ(text, W + [x]) for x in alphabet}
            best = max(counts.values()) if counts else 0
            if best == 0:
                break
            tau = min(x for x, c in counts.items() if c == best)
            if best * min_prob[1] < min_prob[0] * c0:
                break
            res.drafts.append(tau)
            res.probs.append(Fraction(best, c0))
            W.append(tau)
        return res

    alive = list(occ)
    for d in range(max(cap, 0)):
        vals = [(e, cont(e, d)) for e in alive]
        vals = [(e, v) for e, v in vals if v is not None]
        if not vals:
            break
        counts = {}
        for _, v in vals:
            counts[v] = counts.get(v, 0) + 1
        best = max(counts.values())
        tau = min(v for v, c in counts.items() if c == best)
        if best * min_prob[1] < min_prob[0] * c0:
            break
        res.drafts.append(tau)
        res.probs.append(Fraction(best, c0))
        alive = [e for e, v in vals if v == tau]
    return res


def brute_backoff(t: Sequence[int], n: int, k: int, D: int, R: int, S: int,
                  factor: Tuple[int, int], offset: int, min_prob: Tuple[int, int],
                  nb: int, X: Optional[Sequence[int]] = None, Z: int = -1) -> Result:
    """Multi-length backoff read literally: for support threshold t the
    candidate length is the largest l whose last-l-token string occurs (with a
    continuation) at least t times, found by counting substring occurrences
    for every l; each candidate votes with the R most recent occurrences of
    its string; the best score wins, then the longer length, then the row."""
    t = list(t[:n])
    best: Optional[Result] = None
    if n == 0:
        return Result()
    paths = [(1, t, 1, min(D, n - 1))]
    if X is not None and len(X) > 0 and D >= 2 and n >= 2:
        paths.append((2, list(X), 2, min(D, n)))
    for src, text, lmin, lmax in paths:
        def valid(e):
            if src == 1:
                return e <= n - 2
            return e + 1 < len(text) and text[e + 1] != Z

        occ_of = {l: sorted((e for e in ends_of(text, t[n - l:]) if valid(e)), reverse=True)
                  for l in range(lmin, lmax + 1)}
        lengths = []
        for th in range(1, nb + 1):
            ok = [l for l in occ_of if len(occ_of[l]) >= th]
            if ok and max(ok) not in lengths:
                lengths.append(max(ok))
        for l in lengths:
            occ = occ_of[l][:R]
            res = Result()
            res.M, res.source, res.c0 = l, src, len(occ)
            cap = min(k, (factor[0] * l) // factor[1] + offset, max(0, S - n - 1))
            alive = list(occ)
            for d in range(max(cap, 0)):
                vals = []
                for e in alive:
                    q = e + 1 + d
                    if src == 1:
                        v = t[q] if q <= n - 1 else None
                    else:
                        v = text[q] if q < len(text) and text[q] != Z else None
                    if v is not None:
                        vals.append((e, v))
                if not vals:
                    break
                counts = {}
                for _, v in vals:
                    counts[v] = counts.get(v, 0) + 1
                top = max(counts.values())
                tau = min(v for v, c in counts.items() if c == top)
                if top * min_prob[1] < min_prob[0] * res.c0:
                    break
                res.drafts.append(tau)
                res.probs.append(Fraction(top, res.c0))
                alive = [e for e, v in vals if v == tau]
            if best is None or res.score > best.score or (res.score == best.score and l > best.M):
                best = res
    return best if best is not None else Result()


def brute_suffix_array(X: Sequence[int]) -> List[int]:
    """Python's list order is lexicographic with a proper prefix first."""
    X = list(X)
    return sorted(range(len(X)), key=lambda i: X[i:])
