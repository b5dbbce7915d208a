"""The seeded generators are deterministic and have the stated shapes."""
import numpy as np

from model_free_suffix_gb300 import workload as W


def test_trace_deterministic_and_shaped():
    cfg = W.CONFIGS["c2"]
    a = W.ServingTrace(cfg, seed=3, steps=4, B=8)
    b = W.ServingTrace(cfg, seed=3, steps=4, B=8)
    ta, na = a.initial()
    tb, nb = b.initial()
    assert (ta == tb).all() and (na == nb).all()
    assert ta.shape == (8, cfg.S)
    assert ((na >= cfg.n_lo) & (na <= cfg.n_hi)).all()
    for b_ in range(8):
        assert (ta[b_, na[b_]:] == -1).all()
        assert (ta[b_, :na[b_]] >= 0).all() and (ta[b_, :na[b_]] < cfg.V).all()
    for _ in range(4):
        sa, sb = a.next_step(), b.next_step()
        assert (sa.sampled == sb.sampled).all()
        acc = (sa.sampled >= 0).sum(1)
        assert ((acc >= 1) & (acc <= cfg.T)).all()
        for r in range(8):  # leading prefix, then -1
            assert (sa.sampled[r, acc[r]:] == -1).all()


def test_finishing_rows_and_reset():
    cfg = W.CONFIGS["c3"]
    tr = W.ServingTrace(cfg, seed=0, steps=3, B=40)
    st = tr.next_step()
    assert st.finished.shape[0] == 2 and len(set(st.finished.tolist())) == 2
    assert st.reset_tokens.shape == (2, cfg.S)
    assert (st.ingest_lengths >= 1).all()


def test_corpus_docs_fit():
    cfg = W.CONFIGS["c3"]
    docs, lens = W.corpus_docs(cfg, capacity=1 << 14)
    assert int(lens.sum() + lens.shape[0]) <= 1 << 14
    assert ((lens >= cfg.doc_lo) & (lens <= cfg.doc_hi)).all()


def test_sa_corpus_exact_length():
    X = W.sa_corpus(1 << 14, seed=1, V=151936)
    assert X.shape == (1 << 14,) and X[-1] == 151936
    assert ((X >= 0) & (X <= 151936)).all()
    docs, lens = W.docs_from_text(X, 151936)
    assert int(lens.sum() + lens.shape[0]) == 1 << 14
