"""Saving and restoring the cross-request corpus (sgd_save / sgd_load).

A context restored from a file drafts exactly as the one that saved it --
same ring, same snapshot, same delta -- and keeps working (ingest, rebuild,
swap) the same way afterwards.  Files that are not such a save, or do not fit
the context, are refused before anything changes.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _mods():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from model_free_suffix_gb300 import build
    build.build()
    from model_free_suffix_gb300 import SuffixDrafter, _lib as L
    from oracle import oracle as O
    import harness as H
    return SuffixDrafter, L, O, H


def _docs(rng, base, m, S, lo=20, hi=300):
    buf = np.zeros((m, S), dtype=np.int32)
    lens = rng.integers(lo, hi, size=m).astype(np.int32)
    for i in range(m):
        off = int(rng.integers(0, base.shape[0] - lens[i]))
        buf[i, :lens[i]] = base[off:off + lens[i]]
    return buf, lens


def _ingest(dr, ring, buf, lens):
    m = buf.shape[0]
    rows = torch.arange(m, dtype=torch.int32, device="cuda")
    dr.ingest(torch.from_numpy(buf).cuda(), rows, torch.zeros_like(rows), torch.from_numpy(lens).cuda())
    ring.ingest(buf, np.arange(m), np.zeros(m), lens)


@pytest.mark.parametrize("delta", [0, 4096], ids=["no-delta", "delta"])
def test_save_load_round_trip(tmp_path, delta):
    SuffixDrafter, L, O, H = _mods()
    V, S, B, C = 37, 512, 32, 4096
    rng = np.random.default_rng(12)
    base = rng.integers(0, V, size=2000).astype(np.int32)
    kw = dict(max_batch=B, seq_capacity=S, vocab_size=V, k=8, max_tree_depth=16, max_occurrences=16,
              corpus_capacity=C, max_docs=256, delta_capacity=delta)
    A = SuffixDrafter(**kw)
    ring = O.Ring(C, 256, V)
    p = O.Params(S=S, V=V, k=8, D=16, R=16)
    side = torch.cuda.Stream()
    # enough docs to wrap the ring, a snapshot, then more docs after it
    for _ in range(4):
        _ingest(A, ring, *_docs(rng, base, 6, S))
    A.build_sa(side)
    assert A.poll(wait=True)[0] == 1
    X, since = ring.snapshot(), ring.pushed
    _ingest(A, ring, *_docs(rng, base, 5, S))
    path = os.path.join(str(tmp_path), "corpus.sgd")
    A.save(path)
    assert os.path.getsize(path) == 88 + 4 * C + 12 * 256 + 4 * X.shape[0]
    Bd = SuffixDrafter(**kw)
    Bd.load(path)
    assert Bd.corpus_stats() == A.corpus_stats() == (ring.live, ring.ndocs)
    ta, sa_a, _ = A.export_snapshot()
    tb, sa_b, _ = Bd.export_snapshot()
    assert torch.equal(ta, tb) and torch.equal(sa_a, sa_b)
    tok = np.zeros((B, S), dtype=np.int32)
    n = rng.integers(10, 300, size=B).astype(np.int32)
    for b in range(B):
        off = int(rng.integers(0, base.shape[0] - n[b]))
        tok[b, :n[b]] = base[off:off + n[b]]
    g_tok, g_n = torch.from_numpy(tok).cuda(), torch.from_numpy(n).cuda()
    Xc = O.corpus_text(X, ring.delta(since, delta)) if delta else X
    want = O.propose(p, tok, n, X=Xc)
    for dr in (A, Bd):
        H.compare(dr.propose(g_tok, g_n), want, ctx="restored" if dr is Bd else "saved")
    # both keep working alike: more docs, a rebuild, a swap
    buf, lens = _docs(rng, base, 4, S)
    for dr in (A, Bd):
        m = buf.shape[0]
        rows = torch.arange(m, dtype=torch.int32, device="cuda")
        dr.ingest(torch.from_numpy(buf).cuda(), rows, torch.zeros_like(rows),
                  torch.from_numpy(lens).cuda())
        dr.build_sa(side)
        assert dr.poll(wait=True)[0] == 1
    ring.ingest(buf, np.arange(buf.shape[0]), np.zeros(buf.shape[0]), lens)
    want = O.propose(p, tok, n, X=ring.snapshot())
    for dr in (A, Bd):
        H.compare(dr.propose(g_tok, g_n), want, ctx="after a rebuild")
        assert dr.get_error() == 0
    A.close()
    Bd.close()


def test_load_refuses_foreign_or_damaged_files(tmp_path):
    SuffixDrafter, L, O, H = _mods()
    V, S, C = 37, 256, 2048
    rng = np.random.default_rng(5)
    base = rng.integers(0, V, size=800).astype(np.int32)
    kw = dict(max_batch=4, seq_capacity=S, vocab_size=V, k=4, corpus_capacity=C, max_docs=64)
    A = SuffixDrafter(**kw)
    ring = O.Ring(C, 64, V)
    _ingest(A, ring, *_docs(rng, base, 5, S))
    A.build_sa(torch.cuda.Stream())
    assert A.poll(wait=True)[0] == 1
    good = os.path.join(str(tmp_path), "good.sgd")
    A.save(good)
    raw = bytearray(open(good, "rb").read())
    Bd = SuffixDrafter(**kw)
    before = Bd.corpus_stats()

    def refused(data, status, other=None):
        path = os.path.join(str(tmp_path), "bad.sgd")
        open(path, "wb").write(bytes(data))
        with pytest.raises(L.SgdError) as ei:
            (other or Bd).load(path)
        assert ei.value.status == status
        assert (other or Bd).corpus_stats() == before

    bad = bytearray(raw); bad[0:8] = b"NOTACORP"
    refused(bad, L.SGD_EINVAL)                       # not a save
    refused(raw[:100], L.SGD_EIO)                    # cut short
    bad = bytearray(raw); bad[88] = 0xff; bad[89] = 0xff; bad[90] = 0xff; bad[91] = 0x7f
    refused(bad, L.SGD_EINVAL)                       # a ring id out of range
    bad = bytearray(raw); bad[56:60] = (7).to_bytes(4, "little")
    refused(bad, L.SGD_EINVAL)                       # head no longer the oldest doc
    bad = bytearray(raw); bad[40:48] = (123).to_bytes(8, "little")
    refused(bad, L.SGD_EINVAL)                       # live tokens that the docs do not add up to
    other = SuffixDrafter(**dict(kw, corpus_capacity=4096))
    before = other.corpus_stats()
    refused(raw, L.SGD_EINVAL, other)                # another ring size
    with pytest.raises(L.SgdError) as ei:
        Bd.load(os.path.join(str(tmp_path), "missing.sgd"))
    assert ei.value.status == L.SGD_EIO
    Bd.load(good)                                    # and the good file still loads
    assert Bd.corpus_stats() == A.corpus_stats()
    for dr in (A, Bd, other):
        dr.close()
