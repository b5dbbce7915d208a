#!/usr/bin/env python
"""Benchmark of the GPU-resident suffix-decoding drafter.

Metric: propose steps/s and us/step at B=256, S=4096 (one step = the whole
drafting path on one batch: update + self match + corpus probe + expansion,
the ingest of the rows that finish in that step, the background suffix-array
rebuild policy and the swap poll), plus suffix-array build Mtok/s and the HBM
GB/s of the dominant kernel against the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica of the workload on its
own GPU (rows shard across GPUs; there is no data-path collective); rank 0
prints one JSON line.  `--impl reference` times the CPU oracle instead.

Secondary lines in the same JSON object (each its own workload, named in it):
  warm / latency_floor  the headline step without the L2 flush, and one graph
                        of one minimal kernel between the same events;
  delta, backoff        the headline loop with the delta scan / multi-length
                        backoff drafting;
  long_context          the long-context serving loop (B=1024, S=32768, 4M
                        corpus, 64 steps, 5% of rows finishing per step);
  sa_build              standalone suffix-array builds (1M, 16M tokens);
  sa_concurrent         drafting steps with and without a suffix-array build
                        running on a side stream, the build's wall time and
                        the swap cost;
  cpu_baseline          the CPU oracle on the host's cores and on one core,
                        and the naive comparison-sort suffix array.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "propose steps/s & µs/step at B=256,S=4096; SA build Mtok/s; HBM GB/s"
WORKLOADS = {
    "c1": ("self-match loop: B=4 rows, S=2048 int32, vocab 32000 (uniform fresh tokens, p=0.7 "
           "repeats from 64 spans of 8-64), num_tokens U[512,2048], k=8, max_tree_depth=24, "
           "T=9 sampled ids, no corpus"),
    "c2": ("self-match loop: B=64 rows, S=8192 int32, vocab 151936 (Zipf 1.1 fresh tokens, "
           "p=0.5 repeats from 256 spans of 16-128), num_tokens U[1024,8192], k=16, "
           "max_tree_depth=24, T=17 sampled ids, no corpus"),
    "c3": ("serving loop: B=256 rows, S=4096 int32, vocab 151936 (Zipf 1.1 fresh tokens, "
           "p=0.5 repeats from 256 spans of 16-128), num_tokens U[1024,4096], k=16, "
           "max_tree_depth=24, max_occurrences=64, T=17 sampled ids (U[1,17] accepted), "
           "1M-token corpus ring prefilled with 64-512-token responses; per step 5% of rows "
           "finish and are ingested, a side-stream rebuild starts once 2^16 tokens arrived"),
    "c5": ("long-context serving loop: B=1024 rows, S=32768 int32, vocab 151936 (Zipf 1.1 "
           "fresh tokens, p=0.8 repeats from 1024 spans of 32-512), num_tokens U[8192,32768], "
           "k=32, max_tree_depth=32, max_occurrences=64, T=33 sampled ids, 4M-token corpus "
           "ring prefilled; per step 5% of rows (51) finish and are ingested, a side-stream "
           "rebuild starts once 2^16 tokens arrived and none is in flight"),
}
TIMING_NOTE = {
    "l2": "flushed before every timed step (a write of twice the L2 size, outside the events)",
    "launch": "each step replays one CUDA graph (the fused sgd_step launch: update + propose + "
              "ingest, or the separate calls where the step cannot fuse) on a highest-priority "
              "stream; rebuilds run on a lowest-priority side stream",
}


def kernel_traffic(kernel, items=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel's current sources (else None).  A per-item record is scaled by
    the items one launch processes."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kernel]
        h = hashlib.sha256()
        for f in rec["sources"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != rec["sha256"]:
            return None
        if "bytes_per_launch" in rec:
            return int(rec["bytes_per_launch"])
        if items is None:
            return None
        return int(float(rec["bytes_per_item"]) * items)
    except Exception:
        return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi samples of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _us(ms_list):
    return {"mean": round(1e3 * float(np.mean(ms_list)), 2),
            "median": round(1e3 * float(np.median(ms_list)), 2),
            "p90": round(1e3 * float(np.percentile(ms_list, 90)), 2)}


# ---------------------------------------------------------------------------
def make_steps(cfg, seed, n_steps):
    from model_free_suffix_gb300 import workload as W
    tr = W.ServingTrace(cfg, seed=seed, steps=n_steps)
    tok, n = tr.initial()
    steps = [tr.next_step() for _ in range(n_steps)]
    return tr, tok, n, steps


def algorithmic_bytes_propose(sum_n, B, T, k, N, ingest_tokens=0):
    """Bytes one step launch must touch, the data-independent lower bound:
    every valid token of every row once, the sampled ids, the outputs, the
    sectors of two suffix-array binary searches per row, and the ingested
    docs (read once, written once into the ring)."""
    probe = 0 if N <= 0 else B * 2 * int(np.ceil(np.log2(N + 1))) * 2 * 32
    return 4 * sum_n + 4 * B * T + B * (8 * k + 16) + probe + 8 * ingest_tokens


class RowStats:
    """Per-row statistics the drafting kernel writes (sgd_set_row_stats),
    summed over the timed steps: the suffix-array hits each row's probe
    scanned and the continuation gathers of rows drafted from the corpus.
    Each scanned hit costs an SA entry and a text sector (4 + 32 bytes); each
    corpus occurrence that votes reads ceil(4 cap / 32) sectors."""

    def __init__(self, dr, B, dev):
        import torch
        self.buf = torch.zeros(dr.cfg.max_batch * 4, dtype=torch.int32, device=dev)
        self.acc = torch.zeros(5, dtype=torch.int64, device=dev)
        self.steps = 0
        self.B = B
        dr.set_row_stats(self.buf)

    def add(self):
        import torch
        st = self.buf[:4 * self.B].view(self.B, 4).to(torch.int64)
        src, how = st[:, 3] & 255, (st[:, 3] >> 8) & 15
        corpus = (src == 2).to(torch.int64)
        gather = st[:, 1] * ((4 * st[:, 2] + 31) // 32 * 32) * corpus
        # (a corpus draft read from a gram draft gathers nothing)
        gather = gather * (1 - ((st[:, 3] >> 12) & 1))
        self.acc += torch.stack([st[:, 0].sum(), gather.sum(), corpus.sum(), (how == 0).sum(),
                                 ((st[:, 3] >> 12) & 1).sum()])
        self.steps += 1

    def per_step(self):
        a = self.acc.cpu().numpy().astype(np.float64) / max(1, self.steps)
        return {"hits_scanned": round(float(a[0]), 1), "gather_bytes": round(float(a[1]), 1),
                "corpus_rows": round(float(a[2]), 2), "rows_scanned": round(float(a[3]), 2),
                "gram_draft_rows": round(float(a[4]), 2)}


def workload_config(cfg, world):
    """The workload both arms run, by what it is and its sizes."""
    return {"workload": WORKLOADS[cfg.name], "B": cfg.B, "S": cfg.S, "k": cfg.k, "D": cfg.D,
            "R": cfg.R, "T": cfg.T, "corpus_tokens": cfg.corpus_tokens,
            "rebuild_tokens": cfg.rebuild_tokens,
            "parallelism": "replicas" if world > 1 else "single"}


def _prefill(dr, cfg, tr, dev, side, rank, chunk=2048):
    """Corpus prefill (setup, untimed): docs until the ring is full, then the
    first snapshot, built and swapped in."""
    import torch
    from model_free_suffix_gb300 import workload as W
    docs, lens = W.corpus_docs(cfg, seed=rank, capacity=cfg.corpus_tokens, pool=tr.pool)
    for s0 in range(0, docs.shape[0], chunk):
        d = docs[s0:s0 + chunk]
        m = d.shape[0]
        buf = torch.full((m, cfg.S), -1, dtype=torch.int32, device=dev)
        buf[:, :d.shape[1]] = torch.from_numpy(d).to(dev)
        dr.ingest(buf, torch.arange(m, dtype=torch.int32, device=dev),
                  torch.zeros(m, dtype=torch.int32, device=dev),
                  torch.from_numpy(np.ascontiguousarray(lens[s0:s0 + chunk])).to(dev))
        del buf
    dr.build_sa(side)
    assert dr.poll(wait=True)[0] == 1


def serve_loop(args, rank, world, cfg_name="c3", delta=0, backoff=1, K=None, Wm=None,
               headline=False, row_index=0):
    """The serving loop of `cfg_name`: per step the update, propose and ingest
    of the rows that finish (one captured graph), then the host's rebuild
    policy and swap poll.  delta > 0: the docs ingested since the current
    snapshot are matched too; backoff > 1: multi-length backoff drafting;
    row_index: each row's own match from its bigram position index (the rows
    a step restarts are reset outside the timed region, like their contents).
    headline: also the warm and latency-floor timings, the end-to-end leg
    through host buffers and the standalone suffix-array builds."""
    import torch
    from model_free_suffix_gb300 import SuffixDrafter
    from model_free_suffix_gb300 import workload as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[cfg_name]
    K = args.steps if K is None else K
    Wm = args.warmup if Wm is None else Wm
    K_warm = min(K, args.warm_steps) if headline else 0
    K_e2e = min(K, args.e2e_steps) if headline else 0
    tr, tok, n, steps = make_steps(cfg, seed=rank, n_steps=Wm + K + K_warm + K_e2e)
    dr = SuffixDrafter(max_batch=cfg.B, seq_capacity=cfg.S, vocab_size=cfg.V, k=cfg.k,
                       max_tree_depth=cfg.D, max_occurrences=cfg.R, max_sampled=cfg.T,
                       max_spec_factor=cfg.factor, max_spec_offset=cfg.offset,
                       min_token_prob=cfg.min_prob, corpus_capacity=cfg.corpus_tokens,
                       delta_capacity=delta, num_backoff=backoff, row_index=row_index,
                       device=dev.index)
    # drafting at the device's highest stream priority, snapshot builds at the lowest
    least, greatest = torch.cuda.Stream.priority_range()
    stream = torch.cuda.Stream(device=dev, priority=greatest)
    side = torch.cuda.Stream(device=dev, priority=least)
    torch.cuda.set_stream(stream)
    if cfg.corpus_tokens:
        _prefill(dr, cfg, tr, dev, side, rank, chunk=2048 if cfg.S <= 8192 else 256)

    g_tok = torch.from_numpy(tok).to(dev)
    g_n = torch.from_numpy(n).to(dev)
    if row_index:
        dr.reset_rows(g_tok, g_n, torch.arange(cfg.B, dtype=torch.int32, device=dev))
    out = dr.new_outputs(cfg.B)
    stats = RowStats(dr, cfg.B, dev) if backoff == 1 else None
    m_fin = int(np.floor(cfg.finish_frac * cfg.B))
    # fixed device inputs of one step; each step's values are staged into them
    d_samp = torch.full((cfg.B, cfg.T), -1, dtype=torch.int32, device=dev)
    d_rows = torch.zeros(max(1, m_fin), dtype=torch.int32, device=dev)
    d_st = torch.zeros(max(1, m_fin), dtype=torch.int32, device=dev)
    d_ln = torch.zeros(max(1, m_fin), dtype=torch.int32, device=dev)
    n_dev_steps = Wm + K + K_warm
    samp = [torch.from_numpy(s.sampled).to(dev) for s in steps[:n_dev_steps]]
    fin = [(torch.from_numpy(s.finished).to(dev), torch.from_numpy(s.ingest_starts).to(dev),
            torch.from_numpy(s.ingest_lengths).to(dev), int(s.ingest_lengths.sum()),
            torch.from_numpy(s.finished.astype(np.int64)).to(dev),
            None if s.reset_tokens is None else torch.from_numpy(s.reset_tokens).to(dev),
            torch.from_numpy(s.reset_n).to(dev)) for s in steps[:n_dev_steps]]
    # the step, captured once: update + propose + ingest of the finished rows
    ingest = bool(m_fin and cfg.corpus_tokens)
    g_step = torch.cuda.CUDAGraph()
    dr.propose_with_update(g_tok, g_n, d_samp, out=out)  # warm the launch path
    torch.cuda.synchronize()
    l_cap = dr.launch_count()
    with torch.cuda.graph(g_step, stream=stream):
        if ingest:
            dr.step(g_tok, g_n, d_samp, d_rows, d_st, d_ln, out=out, stream=stream)
        else:
            dr.propose_with_update(g_tok, g_n, d_samp, out=out, stream=stream)
    graph_kernels = dr.launch_count() - l_cap   # library kernels one replay runs
    g_tok.copy_(torch.from_numpy(tok))   # undo the warm-up update
    g_n.copy_(torch.from_numpy(n))
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or (126 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    # ring tokens each step's docs take (a sentinel after each)
    ring_tok = [int(s.ingest_lengths.sum()) + int((s.ingest_lengths > 0).sum()) for s in steps]
    state = {"pending": False, "ingested": 0, "swaps": 0, "builds": 0, "build_stats": [],
             # ring tokens placed since the current / the pending snapshot was linearised
             "since_front": 0, "since_pending": 0, "delta_tok": []}

    def stage(i, cold=True):
        """Outside the timed region: the previous step's finished rows restart
        (workload bookkeeping), this step's inputs land in the fixed buffers,
        and (cold) L2 is flushed."""
        if i > 0:
            rows0, _, _, _, idx, rt, rn = fin[i - 1]
            if idx.numel():
                g_tok[idx] = rt
                g_n[idx] = rn
                if row_index:
                    dr.reset_rows(g_tok, g_n, rows0)
        d_samp.copy_(samp[i])
        rows, st_, ln, _, _, _, _ = fin[i]
        if rows.numel():
            d_rows.copy_(rows)
            d_st.copy_(st_)
            d_ln.copy_(ln)
        if cold:
            flush.fill_(i)

    def account(i):
        """The trace's bookkeeping for step i (host only, before its events):
        the docs it ingests count toward the rebuild policy."""
        state["delta_tok"].append(min(delta, state["since_front"]))  # what this step's rows scanned
        state["ingested"] += fin[i][3]
        state["since_front"] += ring_tok[i]
        state["since_pending"] += ring_tok[i]

    def policy(i):
        """The step's library calls after its launch: the rebuild policy and the
        swap poll (a swap launches on the step's stream, inside its events)."""
        if cfg.corpus_tokens:
            if not state["pending"] and state["ingested"] >= cfg.rebuild_tokens:
                dr.build_sa(side, stream=stream)
                state["pending"] = True
                state["ingested"] = 0
                state["since_pending"] = 0
                state["builds"] += 1
            if state["pending"]:  # (nothing to poll for otherwise)
                st, _ = dr.poll(wait=False, stream=stream)
                if st == 1:
                    state["pending"] = False
                    state["swaps"] += 1
                    state["since_front"] = state["since_pending"]
                    state["build_stats"].append(dr.build_stats())

    def one_step(i, ev=None, cold=True, collect=False):
        stage(i, cold)
        account(i)
        if ev:
            ev[0].record(stream)
        g_step.replay()
        if ev:
            ev[1].record(stream)
        policy(i)
        if ev:
            ev[2].record(stream)
        if collect and stats is not None:
            stats.add()   # (after the events: device work of the statistics is not timed)

    for i in range(Wm):
        one_step(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    l0 = dr.launch_count()
    nb0 = len(state["build_stats"])
    clk = Clocks(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clk.start()
    time.sleep(0.05)
    b0 = state["builds"]
    t_wall = time.perf_counter()
    for j in range(K):
        one_step(Wm + j, evs[j], collect=True)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks = clk.stop()
    barrier(world)
    torch.cuda.synchronize()
    launches = dr.launch_count() - l0 + graph_kernels * K
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    prop_ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = float(np.sum(step_ms))
    total_ms_max = allreduce_max(total_ms, world)
    builds_in_region = state["builds"] - b0
    region_builds = state["build_stats"][nb0:]
    n_sum = int(g_n.sum().item())
    peak, peak_kind = peaks()
    ing_tok = float(np.mean([fin[Wm + j][3] for j in range(K)])) if ingest else 0.0
    lower = algorithmic_bytes_propose(n_sum, cfg.B, cfg.T, cfg.k, cfg.corpus_tokens, ing_tok)
    prop_avg_s = float(np.mean(prop_ms)) / 1e3
    row = stats.per_step() if stats is not None else None
    full = None if row is None else int(lower + 36 * row["hits_scanned"] + row["gather_bytes"])
    dev_bytes, pinned_bytes = dr.memory()
    caller_bytes = (g_tok.numel() + g_n.numel() + d_samp.numel() + 3 * d_rows.numel()) * 4 + sum(
        t.numel() * t.element_size() for t in (out.drafts, out.num_valid, out.score, out.probs,
                                               out.match_info))
    memory = {"context_device_bytes": int(dev_bytes), "context_pinned_bytes": int(pinned_bytes),
              "caller_device_bytes": int(caller_bytes)}

    def roofline(kernel, byts, traffic_key):
        ach = byts / prop_avg_s / 1e9
        return {"bound": "hbm", "kernel": kernel, "achieved": round(ach, 2), "peak": peak,
                "unit": "GB/s", "frac": round(ach / peak, 4), "bytes_per_launch": int(byts),
                "traffic": kernel_traffic(traffic_key), "avg_launch_us": round(prop_avg_s * 1e6, 2),
                "peak_kind": peak_kind}

    res = {"steps": K, "us_per_step": round(1e3 * total_ms_max / K, 2),
           "steps_per_s": round(world * K / (total_ms_max / 1e3), 2),
           "graph_us": _us(prop_ms), "kernels_per_step": int(graph_kernels),
           "builds_in_timed_region": builds_in_region, "swaps_in_timed_region": len(region_builds),
           "memory": memory, "clocks": clocks}
    if row is not None:
        res["row_stats"] = row
        res["bytes_per_step"] = {"lower_bound": int(lower), "with_scans_and_gathers": full}
    if backoff > 1:
        res["roofline"] = roofline("backoff_kernel (the update included; with the ingest launch of "
                                   "the step)", lower, "backoff_kernel")
    elif delta:
        dv = float(np.mean(state["delta_tok"][Wm:Wm + K]))
        res["mean_delta_tokens"] = round(dv, 1)
        # the delta is read from HBM once per step (every row then finds it in L2)
        res["roofline"] = roofline("propose_kernel", full + 4 * dv, "propose_kernel_delta")
    else:
        res["roofline"] = roofline("propose_kernel", full,
                                   "propose_kernel" if cfg_name == "c3" else "propose_kernel_c5")
        res["roofline"]["bytes_lower_bound"] = int(lower)
    if not headline:
        if state["pending"]:
            dr.poll(wait=True, stream=stream)
        dr.close()
        return res

    # warm: the same step back to back, no flush between steps
    evw = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K_warm)]
    for j in range(K_warm):
        one_step(Wm + K + j, evw[j], cold=False)
    torch.cuda.synchronize()
    warm_ms = [e[0].elapsed_time(e[2]) for e in evw]
    res["warm"] = {"steps": K_warm, "us_per_step": round(1e3 * float(np.mean(warm_ms)), 2),
                   "graph_us": _us([e[0].elapsed_time(e[1]) for e in evw]),
                   "l2": "not flushed: steps back to back"}
    # latency floor: one graph holding one minimal kernel, between the same events
    tiny = torch.zeros(1, dtype=torch.int32, device=dev)
    g_tiny = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_tiny, stream=stream):
        tiny.fill_(1)
    floor = {}
    for mode in ("cold", "warm"):
        ms = []
        for j in range(64):
            if mode == "cold":
                flush.fill_(j)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_tiny.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        floor[mode] = _us(ms)
    res["latency_floor_us"] = {"what": "one CUDA graph of one minimal kernel replayed between "
                                       "the step's CUDA events", **floor}
    # e2e: host buffers through the public API, copies inside the timed region
    if state["pending"]:
        dr.poll(wait=True, stream=stream)
        state["pending"] = False
    res["e2e"] = e2e_leg(dr, cfg, steps, Wm + K + K_warm, K_e2e, g_tok, g_n, flush, side, state,
                         dev, stream, row_index)
    pass_ms = float(sum(b["pass_ms"] for b in region_builds))
    pass_elems = int(sum(b["pass_elems"] for b in region_builds))
    n_passes = int(sum(b["passes"] for b in region_builds))
    res["kernels"] = {"propose_kernel": {"launches": K, "total_ms": round(float(np.sum(prop_ms)), 3)},
                      "k_onesweep (side stream)": {"launches": n_passes, "total_ms": round(pass_ms, 3)}}
    res["gpu_launches"] = int(launches)
    res["wall_s_timed_region"] = round(t_wall, 4)
    res["roofline_propose"] = res["roofline"]
    if pass_ms > float(np.sum(prop_ms)) and n_passes:
        ach_p = 24.0 * pass_elems / (pass_ms / 1e3) / 1e9
        res["roofline"] = {"bound": "hbm", "kernel": "k_onesweep", "achieved": round(ach_p, 2),
                           "peak": peak, "unit": "GB/s", "frac": round(ach_p / peak, 4),
                           "traffic": kernel_traffic("k_onesweep", pass_elems / n_passes),
                           "bytes_per_launch": int(24 * pass_elems / n_passes),
                           "avg_launch_us": round(1e3 * pass_ms / n_passes, 2),
                           "peak_kind": peak_kind}
    dr.close()
    return res


def e2e_leg(dr, cfg, steps, first, K, g_tok, g_n, flush, side, state, dev, stream, row_index=0):
    """Same steps through the public API with pinned host buffers
    (SuffixDrafter.step_host): each step copies its sampled ids and ingest
    arguments host->device and reads the drafts and valid counts back, all
    inside the timed region."""
    import torch
    n_avail = len(steps) - first
    K = min(K, n_avail)
    # the step's inputs arrive in one fixed pinned block [sampled | rows | starts |
    # lengths] and the outputs leave through one [drafts | num_valid]: the library
    # moves each in one copy, and the call is bound to the buffers once
    BT = cfg.B * cfg.T
    m = max(s.finished.shape[0] for s in steps[first:first + K]) if cfg.corpus_tokens else 0
    assert all(s.finished.shape[0] == m for s in steps[first:first + K]) or not cfg.corpus_tokens
    blocks = [np.concatenate([s.sampled.ravel(), s.finished[:m], s.ingest_starts[:m],
                              s.ingest_lengths[:m]]).astype(np.int32) for s in steps[first:first + K]]
    ingested = [int(s.ingest_lengths[:m].sum()) for s in steps[first:first + K]]
    h_in = torch.empty(BT + 3 * m, dtype=torch.int32).pin_memory()
    h_in_np = h_in.numpy()
    h_out = torch.empty(cfg.B * cfg.k + cfg.B, dtype=torch.int32).pin_memory()
    h_drafts, h_nv = h_out[:cfg.B * cfg.k].view(cfg.B, cfg.k), h_out[cfg.B * cfg.k:]
    step_host = dr.bind_step_host(g_tok, g_n, h_in[:BT].view(cfg.B, cfg.T), h_in[BT:BT + m],
                                  h_in[BT + m:BT + 2 * m], h_in[BT + 2 * m:], h_drafts, h_nv,
                                  stream=stream)
    times = []
    bi = bo = 0
    for j in range(K):
        if first + j > 0:
            p = steps[first + j - 1]
            if p.finished.shape[0]:
                idx = torch.from_numpy(p.finished.astype(np.int64)).to(dev)
                g_tok[idx] = torch.from_numpy(p.reset_tokens).to(dev)
                g_n[idx] = torch.from_numpy(p.reset_n).to(dev)
                if row_index:
                    dr.reset_rows(g_tok, g_n, idx.to(torch.int32))
        flush.fill_(j)
        h_in_np[:] = blocks[j]       # this step's inputs land in pinned host memory
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        # one library call: host->device copy of the step's inputs, the fused
        # launch, device->host copy of the drafts and valid counts
        step_host()
        state["ingested"] += ingested[j]
        if cfg.corpus_tokens:
            if not state["pending"] and state["ingested"] >= cfg.rebuild_tokens:
                dr.build_sa(side)
                state["pending"] = True
                state["ingested"] = 0
            if state["pending"]:  # (nothing to swap in otherwise)
                st, _ = dr.poll(wait=False)
                if st == 1:
                    state["pending"] = False
        stream.synchronize()
        times.append(time.perf_counter() - t0)
        bi = (BT + 3 * m) * 4
        bo = h_drafts.numel() * 4 + h_nv.numel() * 4
    if state["pending"]:
        dr.poll(wait=True)
        state["pending"] = False
    tot = float(np.sum(times))
    return {"value": round(K / tot, 2), "unit": "steps/s", "h2d_bytes_per_step": int(bi),
            "d2h_bytes_per_step": int(bo), "us_per_step": round(1e6 * tot / K, 2), "steps": K}


def sa_build_leg(args, dev, sizes=None):
    """Standalone suffix-array builds of the suffix-array workload (1M and 16M)."""
    import torch
    from model_free_suffix_gb300 import SuffixDrafter
    from model_free_suffix_gb300 import workload as W
    peak, peak_kind = peaks()
    out = {}
    if sizes is None:
        sizes = [1 << 20] + ([] if args.no_sa16m else [1 << 24])
    for N in sizes:
        X = torch.from_numpy(W.sa_corpus(N, seed=0)).to(dev)
        dr = SuffixDrafter(max_batch=1, seq_capacity=8, vocab_size=151936, corpus_capacity=N,
                           device=dev.index)
        sa = torch.empty(N, dtype=torch.int32, device=dev)
        runs = []
        flush = torch.empty(256 << 20 >> 2, dtype=torch.int32, device=dev)
        for r in range(3 if N <= 1 << 20 else 2):
            flush.fill_(r)  # L2 flushed before every timed build
            dr.suffix_array(X, out=sa)
            runs.append(dr.build_stats())
        del flush
        best = min(runs, key=lambda s: s["ms"])
        pass_bytes = 24 * best["pass_elems"]
        r_pass = pass_bytes / (best["pass_ms"] / 1e3) / 1e9 if best["pass_ms"] > 0 else None
        r_all = best["model_bytes"] / (best["ms"] / 1e3) / 1e9
        out["%dM" % (N >> 20)] = {
            "workload": "suffix-array workload: %d int32 tokens, docs of 64-512 Zipf(1.1) tokens "
                        "over 151936 each followed by the sentinel, 30%% repeats of 512 spans "
                        "of 32-256" % N,
            "n": N, "ms": round(best["ms"], 3), "mtok_s": round(N / best["ms"] / 1e3, 1),
            "rounds": best["rounds"], "passes": best["passes"],
            "sorted_elems": best["sorted_elems"],
            "model_bytes": int(best["model_bytes"]),
            "model_gbs": round(r_all, 1), "model_frac": round(r_all / peak, 4),
            "radix_pass": {"bound": "hbm", "achieved": None if r_pass is None else round(r_pass, 1),
                           "peak": peak, "unit": "GB/s",
                           "traffic": kernel_traffic("k_onesweep",
                                                     best["pass_elems"] / max(1, best["passes"])),
                           "frac": None if r_pass is None else round(r_pass / peak, 4),
                           "avg_launch_us": round(1e3 * best["pass_ms"] / max(1, best["passes"]), 2),
                           "peak_kind": peak_kind},
        }
        dr.close()
        del X, sa
        torch.cuda.empty_cache()
    return out


def sa_concurrent_leg(args, dev, N):
    """Drafting steps while a suffix-array build runs on a side stream.

    A context over the N-token suffix-array workload (its docs ingested, the
    first snapshot built) drafts the serving rows (B=256, S=4096, k=16) with
    one captured graph per step.  Timed per step (L2 flushed before each):
    steps with no build in flight; then a build started on a lowest-priority
    side stream and steps back to back, each followed by a non-blocking poll,
    until the poll swaps the new snapshot in.  Reported: step us without and
    with the build, the build's wall time from the call to the swap, its own
    GPU time, and the swap (the poll that swaps: host us and the GPU time of
    its descriptor write on the drafting stream).  The graph was captured
    before the swap and keeps running after it (the descriptor's address does
    not change)."""
    import torch
    from model_free_suffix_gb300 import SuffixDrafter
    from model_free_suffix_gb300 import workload as W
    cfg = W.CONFIGS["c3"]
    X = W.sa_corpus(N, seed=0)
    docs, lens = W.docs_from_text(X, cfg.V)
    dr = SuffixDrafter(max_batch=cfg.B, seq_capacity=cfg.S, vocab_size=cfg.V, k=cfg.k,
                       max_tree_depth=cfg.D, max_occurrences=cfg.R, max_sampled=cfg.T,
                       corpus_capacity=N, device=dev.index)
    least, greatest = torch.cuda.Stream.priority_range()
    stream = torch.cuda.Stream(device=dev, priority=greatest)
    side = torch.cuda.Stream(device=dev, priority=least)
    torch.cuda.set_stream(stream)
    chunk = 2048
    for s0 in range(0, docs.shape[0], chunk):
        d = docs[s0:s0 + chunk]
        m = d.shape[0]
        buf = torch.full((m, cfg.S), -1, dtype=torch.int32, device=dev)
        buf[:, :d.shape[1]] = torch.from_numpy(d).to(dev)
        dr.ingest(buf, torch.arange(m, dtype=torch.int32, device=dev),
                  torch.zeros(m, dtype=torch.int32, device=dev),
                  torch.from_numpy(np.ascontiguousarray(lens[s0:s0 + chunk])).to(dev))
        del buf
    dr.build_sa(side, stream=stream)
    assert dr.poll(wait=True, stream=stream)[0] == 1
    # the rows are not updated: every step drafts the same batch, so the steps
    # before, during and after the build do identical work
    tr = W.ServingTrace(cfg, seed=0, steps=1)
    tok, n = tr.initial()
    g_tok, g_n = torch.from_numpy(tok).to(dev), torch.from_numpy(n).to(dev)
    out = dr.new_outputs(cfg.B)
    dr.propose(g_tok, g_n, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        dr.propose(g_tok, g_n, out=out, stream=stream)
    flush = torch.empty(256 << 20 >> 2, dtype=torch.int32, device=dev)
    counter = [0]

    def step():
        counter[0] += 1
        flush.fill_(counter[0])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        return e0, e1

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    idle = [step() for _ in range(args.concurrent_steps)]
    torch.cuda.synchronize()
    idle_ms = [a.elapsed_time(b) for a, b in idle]
    gen0 = dr.poll(wait=False, stream=stream)[1]
    # the build, and steps until its swap
    busy, swap = [], None
    t0 = time.perf_counter()
    dr.build_sa(side, stream=stream)
    for _ in range(args.concurrent_max_steps):
        busy.append(step())
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        h0 = time.perf_counter()
        st, gen = dr.poll(wait=False, stream=stream)
        h1 = time.perf_counter()
        eb.record(stream)
        if st == 1:
            swap = (h1 - t0, h1 - h0, ea, eb, gen)
            break
    torch.cuda.synchronize()
    busy_ms = [a.elapsed_time(b) for a, b in busy]
    after = [step() for _ in range(32)]
    torch.cuda.synchronize()
    after_ms = [a.elapsed_time(b) for a, b in after]
    bs = dr.build_stats()
    if swap is None:
        dr.poll(wait=True, stream=stream)
    res = {"workload": "serving rows (B=256, S=4096, k=16, D=24, R=64) drafting over the "
                       "suffix-array workload's %d-token corpus; one captured propose graph "
                       "per step (the same rows every step), L2 flushed before each" % N,
           "n": N, "step_us_no_build": _us(idle_ms),
           "step_us_during_build": _us(busy_ms) if busy_ms else None,
           "steps_during_build": len(busy_ms),
           "step_us_after_swap": _us(after_ms) if after_ms else None,
           "build_gpu_ms": round(bs["ms"], 3)}
    if swap is not None:
        res["build_wall_ms"] = round(1e3 * swap[0], 3)
        res["swap"] = {"poll_host_us": round(1e6 * swap[1], 2),
                       "poll_gpu_us": round(1e3 * swap[2].elapsed_time(swap[3]), 2),
                       "generation": [int(gen0), int(swap[4])]}
    dr.close()
    del flush
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
def cpu_oracle_leg(cfg, seconds, rank=0, threads=None):
    """The CPU oracle as it stands, on the same workload, rows spread over
    `threads` host threads (all cores by default); a bounded sample of steps."""
    from oracle import oracle as O
    from model_free_suffix_gb300 import workload as W
    O.build()
    threads = threads or os.cpu_count() or 1
    tr, tok, n, steps = make_steps(cfg, seed=rank, n_steps=400)
    ring, X = None, None
    if cfg.corpus_tokens:
        docs, lens = W.corpus_docs(cfg, seed=rank, capacity=cfg.corpus_tokens, pool=tr.pool)
        ring = O.Ring(cfg.corpus_tokens, 65536, cfg.V)
        buf = np.full((docs.shape[0], cfg.S), -1, dtype=np.int32)
        buf[:, :docs.shape[1]] = docs
        ring.ingest(buf, np.arange(docs.shape[0]), np.zeros(docs.shape[0]), lens)
        X = ring.snapshot()
    p = O.Params(S=cfg.S, V=cfg.V, k=cfg.k, D=cfg.D, R=cfg.R, factor=cfg.factor,
                 offset=cfg.offset, min_prob=cfg.min_prob)
    done = 0
    t0 = time.perf_counter()
    while done < len(steps):
        s = steps[done]
        O.update_state(tok, n, s.sampled, cfg.V)
        O.propose(p, tok, n, X=X, threads=threads)
        if s.finished.shape[0]:
            if ring is not None:
                ring.ingest(tok, s.finished, s.ingest_starts, s.ingest_lengths, num_tokens=n)
            for i, b in enumerate(s.finished):
                tok[b] = s.reset_tokens[i]
                n[b] = s.reset_n[i]
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return {"value": round(done / el, 3), "unit": "steps/s", "cores": threads, "kind": "oracle",
            "us_per_step": round(1e6 * el / done, 1),
            "sample": "%d steps of the same workload (update + propose of all %d rows + ingest; "
                      "no suffix-array rebuild in the sample), %.1f s" % (done, cfg.B, el)}


def cpu_sa_leg(sizes):
    """The oracle's naive suffix array (a comparison sort of every suffix, one
    thread) on the suffix-array workload."""
    from oracle import oracle as O
    from model_free_suffix_gb300 import workload as W
    O.build()
    out = {}
    for N in sizes:
        X = W.sa_corpus(N, seed=0)
        t0 = time.perf_counter()
        O.suffix_array(X)
        el = time.perf_counter() - t0
        out["%dM" % (N >> 20)] = {"n": N, "s": round(el, 3), "mtok_s": round(N / el / 1e6, 3),
                                  "cores": 1, "kind": "oracle naive comparison sort"}
    return out


# ---------------------------------------------------------------------------
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--e2e-steps", type=int, default=256)
    ap.add_argument("--warm-steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c3")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-single-seconds", type=float, default=6.0)
    ap.add_argument("--no-sa16m", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--long-context-steps", type=int, default=64,
                    help="steps of the long-context serving loop, a secondary line (0: skip)")
    ap.add_argument("--sa-only", type=int, default=0,
                    help="only time suffix-array builds of this many tokens and print them")
    ap.add_argument("--backoff-steps", type=int, default=64,
                    help="steps of the serving loop with num_backoff=8, a secondary line (0: skip)")
    ap.add_argument("--delta-steps", type=int, default=256,
                    help="steps of the serving loop with the delta scan on, a secondary line (0: skip)")
    ap.add_argument("--concurrent-steps", type=int, default=64,
                    help="steps timed with no build in flight in the concurrent-build line (0: skip)")
    ap.add_argument("--concurrent-max-steps", type=int, default=4096)
    ap.add_argument("--row-index-steps", type=int, default=256,
                    help="steps of the serving loop with row_index=1, a secondary line (0: skip)")
    ap.add_argument("--long-only", action="store_true",
                    help="only time the long-context serving loop and print its line")
    ap.add_argument("--long-row-index", type=int, default=0,
                    help="with --long-only: row_index of the long-context loop")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    from model_free_suffix_gb300 import workload as W
    cfg = W.CONFIGS[args.config]
    if args.impl == "reference":
        if rank == 0:
            cb = cpu_oracle_leg(cfg, args.cpu_seconds)
            res = {"metric": METRIC, "value": cb["value"], "unit": "steps/s", "n_gpus": world,
                   "steps": args.steps, "warmup": args.warmup,
                   "ms_per_step": round(1e3 / cb["value"], 3), "higher_is_better": True,
                   "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
                   "config": workload_config(cfg, world),
                   "impl": "reference", "cpu_baseline": cb,
                   "e2e": {"value": cb["value"], "unit": "steps/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}}
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    from __graft_entry__ import build
    build()
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if args.sa_only:
        if rank == 0:
            print(json.dumps(sa_build_leg(args, dev, sizes=[args.sa_only])), flush=True)
        return
    if args.long_only:
        r = serve_loop(args, rank, world, "c5", K=args.long_context_steps, Wm=3,
                       row_index=args.long_row_index)
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    h = serve_loop(args, rank, world, args.config, headline=True)
    K = args.steps
    res = {
        "metric": METRIC, "value": h["steps_per_s"], "unit": "steps/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(h["us_per_step"] / 1e3, 5),
        "us_per_step": h["us_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic", "config": workload_config(cfg, world), "timing": TIMING_NOTE,
    }
    res.update({k: v for k, v in h.items() if k not in ("steps", "us_per_step", "steps_per_s")})
    if args.config == "c3":
        if args.delta_steps > 0:
            res["delta"] = dict(workload="the serving loop above with delta_capacity=%d: the docs "
                                         "ingested since the current snapshot was linearised are "
                                         "matched too" % cfg.rebuild_tokens,
                                **serve_loop(args, rank, world, "c3", delta=cfg.rebuild_tokens,
                                             K=args.delta_steps))
        if args.backoff_steps > 0:
            res["backoff"] = dict(workload="the serving loop above with num_backoff=8: for support "
                                           "thresholds 1..8 the t-th largest match length of each "
                                           "path is a candidate, every candidate voted, the best "
                                           "score wins",
                                  **serve_loop(args, rank, world, "c3", backoff=8,
                                               K=args.backoff_steps))
        if args.row_index_steps > 0:
            res["row_index"] = dict(workload="the serving loop above with row_index=1: each row's "
                                             "own match from its bigram position index",
                                    **serve_loop(args, rank, world, "c3", K=args.row_index_steps,
                                                 row_index=1))
        if args.long_context_steps > 0:
            res["long_context"] = dict(workload=WORKLOADS["c5"],
                                       **serve_loop(args, rank, world, "c5",
                                                    K=args.long_context_steps, Wm=3))
            res["long_context_row_index"] = dict(
                workload=WORKLOADS["c5"] + "; row_index=1: each row's own match from its bigram "
                                           "position index",
                **serve_loop(args, rank, world, "c5", K=args.long_context_steps, Wm=3, row_index=1))
    res["sa_build"] = sa_build_leg(args, dev)
    if args.concurrent_steps > 0:
        res["sa_concurrent"] = {("%dM" % (N >> 20)): sa_concurrent_leg(args, dev, N)
                                for N in ([1 << 20] + ([] if args.no_sa16m else [1 << 24]))}
    if rank == 0:
        if not args.no_cpu_baseline:
            cb = cpu_oracle_leg(cfg, args.cpu_seconds)
            cb["single_thread"] = cpu_oracle_leg(cfg, args.cpu_single_seconds, threads=1)
            cb["naive_suffix_array"] = cpu_sa_leg([1 << 20] + ([] if args.no_sa16m else [1 << 24]))
            res["cpu_baseline"] = cb
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
