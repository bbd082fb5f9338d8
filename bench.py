#!/usr/bin/env python
"""Tiered decode attention benchmark (QEvict three-tier KV cache, decode path).

Workload: the Llama-3.1-8B-shaped cache of 32 layers, 32 query / 8 KV heads,
head_dim 128, batch 1, 32768-token context in 64-token windows, a 20 % byte
budget (tiers from routing on seeded Zipf(1.1) scores), synthetic bf16 K/V
N(0, 1) with 1 % Student-t(3) outlier channels. Inputs are seeded and resident
in HBM before timing; the 32 layers hold about 860 MB of tiered cache, far
more than the 129 MB L2, so no layer is served from L2 when it comes round.

One step = one decode token through all 32 layers: per layer one fused call
that appends the token's K/V and runs tiered decode attention with the
per-window mass added to the cumulative scores; every 64th step ends with a
routing event on every layer (rank, evict, demote with the write-once ledger,
promote; the layers' routes run side by side on 8 streams, since no layer's
routing depends on another's). Steps are replayed as CUDA graphs captured
from the C ABI calls.

Prints one JSON line. ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama8b_b1_32k_20pct"
METRIC = "tiered decode attention µs/layer-step and effective HBM GB/s (% of GB300 peak)"
ROUTE_EVERY = 64
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- helpers

def all_workloads():
    """Every benchmark workload by name: the fixed ones, then the Mistral-7B-shaped
    sweep points (batch 4), named by context, window and budget."""
    from tiered_kv_cache_decode_gb300 import synth
    out = {k: dict(v) for k, v in synth.WORKLOADS.items() if k != "tiny"}
    for p in synth.mistral_sweep():
        out[f"mistral7b_b4_{p['L'] // 1024}k_w{p['w']}_{round(p['beta'] * 100)}pct"] = dict(p)
    return out


def workload(name=None):
    return dict(all_workloads()[name or WORKLOAD])


def costs(wl):
    d = 128
    c_fp = wl["w"] * wl["Hkv"] * d * 4
    c_q = wl["w"] * wl["Hkv"] * 2 * (d // 4 + 4 * (d // 32))
    return c_fp, c_q


def route_counts(wl, n_cand, L):
    """(n_fp, n_q) a routing event yields at length L (same rule as the kernels)."""
    c_fp, c_q = costs(wl)
    Bt = math.floor(wl["beta"] * (L * wl["Hkv"] * 128 * 4))
    n_fp = min(n_cand, max(1, math.floor((wl["rho"] * Bt) / c_fp)))
    n_q = min(n_cand - n_fp, (Bt - n_fp * c_fp) // c_q)
    return n_fp, n_q


class TierTracker:
    """Host-side bookkeeping of how many windows each tier holds (per layer;
    every layer and sequence has the same counts), to count algorithmic bytes."""

    def __init__(self, wl, L):
        self.wl, self.L = wl, L
        W = -(-L // wl["w"])
        self.n_fp, self.n_q = route_counts(wl, W, L)

    def append(self):
        if self.L % self.wl["w"] == 0:
            self.n_fp += 1
        self.L += 1

    def route(self):
        self.n_fp, self.n_q = route_counts(self.wl, self.n_fp + self.n_q, self.L)

    def decode_bytes(self):
        """Algorithmic bytes of one decode launch (one layer, all sequences):
        resident tiered cache (the open window at its token count), the query,
        the fp32 output and the read + write of one cumulative score per window."""
        wl = self.wl
        c_fp, c_q = costs(wl)
        W = -(-self.L // wl["w"])
        ntok = self.L - (W - 1) * wl["w"]
        resident = (self.n_fp - 1) * c_fp + ntok * wl["Hkv"] * 128 * 4 + self.n_q * c_q
        aux = wl["Hq"] * 128 * 2 + wl["Hq"] * 128 * 4 + W * 8
        return wl["B"] * (resident + aux)

    def append_bytes(self):
        return self.wl["B"] * self.wl["Hkv"] * 128 * 4 * 2     # read the token, write it to its slot


def sample_clocks():
    q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    try:
        return subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100"],
                                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
    except OSError:
        return None


def finish_clocks(proc, gpu_index):
    if proc is None:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    proc.terminate()
    try:
        out, _ = proc.communicate(timeout=5)
    except subprocess.TimeoutExpired:
        proc.kill()
        out, _ = proc.communicate()
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in out.splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9 or f[0] != str(gpu_index):
            continue
        try:
            sm.append(float(f[1]))
            mx.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(sm)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in p:
                v = p[key]
                if isinstance(v, dict):
                    v = v.get("value") or v.get("gbs")
                return float(v), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def run_config(wl, NL, world, route_events=None):
    """The workload description both arms print."""
    per_layer = TierTracker(wl, wl["L"]).decode_bytes()
    c = {"workload": WORKLOAD if NL == wl["layers"] else f"{WORKLOAD} ({NL} of {wl['layers']} layers)",
         "batch": wl["B"], "layers": NL, "q_heads": wl["Hq"], "kv_heads": wl["Hkv"],
         "head_dim": 128, "context": wl["L"], "window": wl["w"], "budget_frac": wl["beta"],
         "fp_share": wl["rho"], "route_every": ROUTE_EVERY, "parallelism": f"replicas x{world}",
         "l2": f"inputs larger than L2 ({NL} layers x {per_layer / 1e6:.1f} MB of tiered cache)"}
    if route_events is not None:
        c["route_events_in_timed_steps"] = route_events
    return c


def combine_ranks(ms, e2e_s, nbytes, e2e_bytes, world, device):
    """Whole-job figures over the ranks (each runs its own replica): the
    slowest rank's times and the bytes of all ranks."""
    if world == 1:
        return ms, e2e_s, float(nbytes), float(e2e_bytes)
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, e2e_s], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([float(nbytes), float(e2e_bytes)], dtype=torch.float64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t[0]), float(t[1]), float(n[0]), float(n[1])


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source (else None)."""
    src = os.path.join(ROOT, "tiered_kv_cache_decode_gb300", "csrc", "qevict_decode.cu")
    summ = os.path.join(ROOT, "profiles", f"decode_{WORKLOAD}.md")
    if not os.path.exists(summ):
        return None
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        fields = {}
        for line in open(summ):
            item = line.strip().lstrip("-* ").strip()
            if ":" in item and item.startswith(("kernel_sha", "dram_bytes_per_launch")):
                k, v = item.split(":", 1)
                fields[k.strip(" -*`")] = v.strip(" `\n")
        if fields.get("kernel_sha") == sha:
            return int(float(fields["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        pass
    return None


# --------------------------------------------------------------------------- CPU oracle leg

def _oracle_worker(args):
    """One layer of the workload on the CPU oracle: prefill, then timed decode
    steps (append + attention + score accumulation) for about `budget_s` s."""
    layer, budget_s, max_steps, name = args
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    import torch
    torch.set_num_threads(1)
    import oracle as O
    from tiered_kv_cache_decode_gb300 import synth
    wl = workload(name)
    B, Hq, Hkv, w, L = wl["B"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"]
    k, v = synth.kv_tokens(0, layer, B, 0, L, Hkv, 128, wl["outliers"])
    c = O.OracleCache(B, Hq, Hkv, 128, w, beta=wl["beta"], rho=wl["rho"])
    c.prefill(k.float().numpy(), v.float().numpy(), scores=synth.zipf_scores(0, layer, B, L // w).numpy())
    del k, v
    tr = TierTracker(wl, L)
    done, nbytes, spent = 0, 0, 0.0
    while done < max_steps and (spent < budget_s or done == 0):
        kn, vn = synth.kv_tokens(0, layer, B, c.L, 1, Hkv, 128, wl["outliers"])
        q = synth.queries(0, layer, done, B, Hq, 128).float().numpy()
        kn, vn = kn.float().numpy(), vn.float().numpy()
        t0 = time.perf_counter()
        c.append(kn, vn)
        c.decode(q, accumulate=True)
        spent += time.perf_counter() - t0
        tr.append()
        nbytes += tr.decode_bytes() + tr.append_bytes()
        done += 1
    return nbytes, spent, done


def oracle_throughput(n_workers, budget_s, max_steps):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(n_workers) as pool:
        res = pool.map(_oracle_worker, [(l, budget_s, max_steps, WORKLOAD) for l in range(n_workers)])
    wall = time.perf_counter() - t0
    nbytes = sum(r[0] for r in res)
    spent = max(r[1] for r in res)
    steps = sum(r[2] for r in res)
    return nbytes / spent / 1e9, spent, steps, wall


# --------------------------------------------------------------------------- native arm

def measure_diagnostics(cache, wl, NL, pool, nq, nkv, stream, reps, dev):
    """Routing diagnostics after the timed steps: the last routing event's tier
    moves on every layer (selection churn, reactivation) and the future missed
    mass of a fresh query over the full keys, timed over four layers in turn
    (256 MiB of keys, more than L2 holds)."""
    import torch
    from tiered_kv_cache_decode_gb300 import synth
    B, Hq, Hkv, w, L0, d, seed = wl["B"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"], 128, 0
    cnt = torch.stack([cache.tier_move_counts(l) for l in range(NL)]).double()   # [NL][B][8]
    churn = (1 - cnt[..., 4] / cnt[..., 2].clamp(min=1)).mean().item()
    react = (cnt[..., 5] / cnt[..., 1].clamp(min=1)).mean().item()
    nd = min(NL, 4)
    Lc = cache.length(0)
    n_app = Lc - L0
    kfull, qd = [], []
    for l in range(nd):
        k0, _ = synth.kv_tokens(seed, l, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
        ka = pool[:n_app, l, nq:nq + nkv].reshape(n_app, B, Hkv, d).permute(1, 0, 2, 3)
        kfull.append(torch.cat([k0, ka], dim=1).contiguous())
        qd.append(synth.queries(seed + 1, l, 0, B, Hq, d, device=dev))
        del k0
    fmm = torch.empty(nd, B, Hq, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for l in range(nd):   # eager first: the launch shape is set up outside the capture
            cache.future_missed_mass(l, qd[l], kfull[l], out=fmm[l], stream=stream)
        with torch.cuda.graph(g, stream=stream):
            for l in range(nd):
                cache.future_missed_mass(l, qd[l], kfull[l], out=fmm[l], stream=stream)
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for r in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    assert cache.status() == 0, cache.last_error()
    us = e0.elapsed_time(e1) * 1e3 / (reps * nd)
    # keys and queries read, one tier byte per window read, one float written per query head
    nbytes = B * Lc * Hkv * d * 2 + B * Hq * d * 2 + B * (-(-Lc // w)) + B * Hq * 4
    return {
        "tier_move": {"layers": NL, "churn": round(churn, 4), "reactivation": round(react, 4),
                      "counts_layer0_seq0": [int(x) for x in cnt[0, 0].tolist()]},
        "future_missed_mass": {"mean": round(fmm.mean().item(), 5), "max": round(fmm.max().item(), 5),
                               "us_per_launch": round(us, 3), "bytes_per_launch": int(nbytes),
                               "gbs": round(nbytes / (us * 1e-6) / 1e9, 2), "context": Lc},
    }


def measure_management(cache, wl, NL, g_route, stream, dev):
    """Routing events and the tier moves they make, on the headline workload.
    One 32-layer routing event of the main cache after the timed steps (its
    CUDA graph, 8 streams). Then the quantise (K4) and dequantise (K5) paths,
    timed through routing events on a fresh 4-layer cache whose windows start
    in full precision: a first event on seeded scores quantises every window
    it demotes for the first time; a second event on re-drawn scores promotes
    INT2 windows back and quantises the full-precision windows it demotes.
    Each call (plan + quantise + promote kernels) is timed with CUDA events;
    bytes are the window rows moved, counted from the statistics counters: a
    first quantisation reads 512 B and writes 96 B per token and KV head, a
    promotion reads 96 B and writes 512 B (evictions and ledger reuses move
    no data)."""
    import torch
    from tiered_kv_cache_decode_gb300 import binding, synth
    B, Hq, Hkv, w, L0, d, seed = wl["B"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"], 128, 0
    W0 = L0 // w
    # a routing event on every layer, once to warm up, then the median of five (the
    # tiers have settled, so these time the ranking and the few moves it makes)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    with torch.cuda.stream(stream):
        g_route.replay()
        for _ in range(5):
            e0.record(stream)
            g_route.replay()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
    torch.cuda.synchronize()
    route_us = statistics.median(times)
    st = cache.status()
    assert st == 0, f"device status {st}: {cache.last_error()}"
    nl = 4
    mc = binding.TieredCache(B, nl, Hq, Hkv, w, L0, budget_frac=wl["beta"], fp_share=wl["rho"],
                             fp_capacity=W0, ledger_capacity=W0)
    for l in range(nl):
        k, v = synth.kv_tokens(seed, l, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
        mc.prefill(l, k, v, tiers=torch.zeros(B, W0, dtype=torch.uint8, device=dev))
        del k, v
    row = Hkv * w * (512 + 96)
    out = {"route_event_us_32_layers": round(route_us, 2)}
    for name, sd in (("route_first_quantisations", seed + 400), ("route_promotions", seed + 401)):
        ov = [synth.zipf_scores(sd, l, B, W0, device=dev) for l in range(nl)]
        s0 = mc.stats()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for l in range(nl):
                mc.route(l, scores_override=ov[l], stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3
        s1 = mc.stats()
        nq = s1["ledger_writes"] - s0["ledger_writes"]
        npr = s1["promotions"] - s0["promotions"]
        nbytes = (nq + npr) * row
        out[name] = {"quantised_per_layer": nq / nl, "promoted_per_layer": npr / nl,
                     "us_per_layer_event": round(us / nl, 2), "bytes_per_layer_event": int(nbytes // nl),
                     "gbs": round(nbytes / (us * 1e-6) / 1e9, 2)}
    st = mc.status()
    assert st == 0, f"device status {st}: {mc.last_error()}"
    mc.close()
    return out


def measure_variants(wl, NL, reps, dev, peak):
    """The workload with per-KV-head tiers: every (sequence, KV head) routed on
    its own seeded scores. Times the decode kernel over all layers (CUDA graph,
    the same algorithmic bytes as the shared mode plus one score per window per
    extra KV head), then routing events on fresh seeded scores: one event under
    one budget across all layers and KV heads (qevict_route_global) against one
    routing per layer, both captured as CUDA graphs on one stream."""
    import torch
    from tiered_kv_cache_decode_gb300 import binding, synth
    B, Hq, Hkv, w, L0, d, seed = wl["B"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"], 128, 0
    W0 = L0 // w
    units = B * Hkv
    # pools for every window: a global event may give one layer more than its own share
    ph = binding.TieredCache(B, NL, Hq, Hkv, w, L0, budget_frac=wl["beta"], fp_share=wl["rho"], per_head=True,
                             fp_capacity=W0, ledger_capacity=W0)
    ph.set_launch_overlap(True)
    ph.set_cooperative_launch(False)   # the decodes run alone on the GPU
    for l in range(NL):
        k, v = synth.kv_tokens(seed, l, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
        ph.prefill(l, k, v, scores=synth.zipf_scores(seed, l, units, W0, device=dev))
        del k, v
    q = [synth.queries(seed, l, 0, B, Hq, d, device=dev) for l in range(NL)]
    xo = torch.empty(NL, B, Hq, d, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ovs = [torch.empty(units, W0, dtype=torch.float32, device=dev) for _ in range(NL)]
    g_dec, g_glob, g_layer, g_ls, g_rd = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                          torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph())
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_dec, stream=stream):
            for l in range(NL):
                ph.decode(l, q[l], out=xo[l], want_mass=False, accumulate=True, stream=stream)
        with torch.cuda.graph(g_glob, stream=stream):
            ph.route_global(ovs, stream=stream)
        with torch.cuda.graph(g_layer, stream=stream):
            for l in range(NL):
                ph.route(l, scores_override=ovs[l], stream=stream)
        with torch.cuda.graph(g_ls, stream=stream):
            for l in range(NL):
                ph.route_logsparse(l, recent=2, stream=stream)
        with torch.cuda.graph(g_rd, stream=stream):
            for l in range(NL):
                ph.route_rd(l, scores_override=ovs[l], stream=stream)
        for _ in range(3):
            g_dec.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g_dec.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us_dec = e0.elapsed_time(e1) * 1e3 / (reps * NL)
    nbytes = TierTracker(wl, L0).decode_bytes() + B * (Hkv - 1) * W0 * 8
    route_us = {}
    for name, g in (("global", g_glob), ("per_layer", g_layer), ("rd", g_rd)):
        tot = 0.0
        for r in range(8):
            for l in range(NL):
                ovs[l].copy_(synth.zipf_scores(seed + 100 + r, l, units, W0, device=dev) * (1.0 + 0.02 * l))
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1) * 1e3
        route_us[name] = round(tot / 8, 2)
        if name == "global":   # windows each layer keeps after a global event
            kept = [int((ph.tables(l)[0] != 2).sum()) for l in range(NL)]
    # log-sparse events: positions do not move between replays, so each timed
    # event follows an untimed global event on fresh scores that scrambles the tiers
    tot = 0.0
    for r in range(8):
        for l in range(NL):
            ovs[l].copy_(synth.zipf_scores(seed + 200 + r, l, units, W0, device=dev))
        with torch.cuda.stream(stream):
            g_glob.replay()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            g_ls.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1) * 1e3
    route_us["logsparse"] = round(tot / 8, 2)
    # decode on the tiers of a rate-distortion event (its counts differ from the fp_share split)
    for l in range(NL):
        ovs[l].copy_(synth.zipf_scores(seed + 300, l, units, W0, device=dev))
    with torch.cuda.stream(stream):
        g_rd.replay()
        for _ in range(3):
            g_dec.replay()
        e0.record(stream)
        for _ in range(reps):
            g_dec.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us_dec_rd = e0.elapsed_time(e1) * 1e3 / (reps * NL)
    c_fp_u, c_q_u = w * d * 4, w * 2 * (d // 4 + 4 * (d // 32))
    tiers_rd = torch.stack([ph.tables(l)[0] for l in range(NL)])   # [NL][units][W]
    n_fp_rd = (tiers_rd == 0).sum(dim=2).double()
    n_q_rd = (tiers_rd == 1).sum(dim=2).double()
    bytes_rd = ((n_fp_rd * c_fp_u + n_q_rd * c_q_u).sum(dim=1).mean().item()
                + B * (Hq * d * 2 + Hq * d * 4 + Hkv * W0 * 8))
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g_dec.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us_dec_ls = e0.elapsed_time(e1) * 1e3 / (reps * NL)
    st = ph.status()
    assert st == 0, f"device status {st}: {ph.last_error()}"
    return {
        "per_kv_head_decode": {"us_per_launch": round(us_dec, 3), "bytes_per_launch": int(nbytes),
                               "gbs": round(nbytes / (us_dec * 1e-6) / 1e9, 2),
                               "frac_of_peak": round(nbytes / (us_dec * 1e-6) / 1e9 / peak, 4),
                               "us_per_launch_after_logsparse_route": round(us_dec_ls, 3)},
        "rate_distortion": {"route_us_per_event_32_layers": route_us["rd"],
                            "fp_int2_evicted_per_unit_mean": [round(n_fp_rd.mean().item(), 2),
                                                              round(n_q_rd.mean().item(), 2),
                                                              round(W0 - n_fp_rd.mean().item() - n_q_rd.mean().item(),
                                                                    2)],
                            "decode_us_per_launch": round(us_dec_rd, 3), "decode_bytes_per_launch": int(bytes_rd),
                            "decode_gbs": round(bytes_rd / (us_dec_rd * 1e-6) / 1e9, 2),
                            "decode_frac_of_peak": round(bytes_rd / (us_dec_rd * 1e-6) / 1e9 / peak, 4)},
        "routing_event_us": {"global_all_layers_and_heads": route_us["global"],
                             "one_per_layer": route_us["per_layer"],
                             "logsparse_one_per_layer": route_us["logsparse"], "layers": NL,
                             "keys_per_sequence": NL * Hkv * W0,
                             "windows_kept_per_layer_after_global_min_max": [min(kept), max(kept)]},
    }


def measure_mixed_widths(wl, NL, reps, dev, peak):
    """The workload with INT4 and INT8 allowed, routed by the rate-distortion
    allocation over widths {0, 2, 4, 8, 16} (qevict_route_rd_mixed) on seeded
    scores: one event per layer captured as a CUDA graph on one stream, timed
    over 8 fresh score sets, then the decode kernel over all layers on the
    tiers the last event left (CUDA graph; algorithmic bytes: every kept
    window at its width, plus the query, output and scores)."""
    import torch
    from tiered_kv_cache_decode_gb300 import binding, synth
    B, Hq, Hkv, w, L0, d, seed = wl["B"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"], 128, 0
    W0 = L0 // w
    mc = binding.TieredCache(B, NL, Hq, Hkv, w, L0, budget_frac=wl["beta"], fp_share=wl["rho"], max_ledger_bits=8,
                             fp_capacity=W0, ledger_capacity=W0)
    mc.set_launch_overlap(True)
    mc.set_cooperative_launch(False)   # the decodes run alone on the GPU
    zeros = torch.zeros(B, W0, dtype=torch.uint8, device=dev)
    for l in range(NL):
        k, v = synth.kv_tokens(seed, l, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
        mc.prefill(l, k, v, tiers=zeros)
        del k, v
    q = [synth.queries(seed, l, 0, B, Hq, d, device=dev) for l in range(NL)]
    xo = torch.empty(NL, B, Hq, d, dtype=torch.float32, device=dev)
    ovs = [torch.empty(B, W0, dtype=torch.float32, device=dev) for _ in range(NL)]
    stream = torch.cuda.Stream(device=dev)
    g_route, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_route, stream=stream):
            for l in range(NL):
                mc.route_rd_mixed(l, scores_override=ovs[l], stream=stream)
        with torch.cuda.graph(g_dec, stream=stream):
            for l in range(NL):
                mc.decode(l, q[l], out=xo[l], want_mass=False, accumulate=True, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    for r in range(8):
        for l in range(NL):
            ovs[l].copy_(synth.zipf_scores(seed + 400 + r, l, B, W0, device=dev))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            g_route.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1) * 1e3
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_dec.replay()
        e0.record(stream)
        for _ in range(reps):
            g_dec.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us_dec = e0.elapsed_time(e1) * 1e3 / (reps * NL)
    cost = {0: w * Hkv * d * 4, 1: w * Hkv * 2 * (d // 4 + 16), 3: w * Hkv * 2 * (d // 2 + 16),
            4: w * Hkv * 2 * (d + 16), 2: 0}
    tiers = torch.stack([mc.tables(l)[0] for l in range(NL)])   # [NL][B][W]
    per_tier = {t: (tiers == t).sum().item() / (NL * B) for t in (0, 4, 3, 1, 2)}
    nbytes = sum(cost[t] * n for t, n in per_tier.items()) * B + B * (Hq * d * 2 + Hq * d * 4 + Hkv * W0 * 8)
    st = mc.status()
    assert st == 0, f"device status {st}: {mc.last_error()}"
    return {"route_us_per_event_all_layers": round(tot / 8, 2), "layers": NL,
            "windows_bf16_int8_int4_int2_evicted_per_sequence_mean": [round(per_tier[t], 2) for t in (0, 4, 3, 1, 2)],
            "decode_us_per_launch": round(us_dec, 3), "decode_bytes_per_launch": int(nbytes),
            "decode_gbs": round(nbytes / (us_dec * 1e-6) / 1e9, 2),
            "decode_frac_of_peak": round(nbytes / (us_dec * 1e-6) / 1e9 / peak, 4)}


def measure_k_channels(wl, NL, reps, dev, peak):
    """RDKV's K-channel half on the workload: per layer the channel weights
    from 64 seeded query vectors and the prefill keys, then one K-channel
    routing event (window widths {0, 2, 4, 8, 16}, K group widths {0, 2, 4, 8}
    within the quantised windows' K bytes) on seeded scores, then the decode
    kernel over all layers on those tiers (CUDA graph; algorithmic bytes: the
    full-precision windows, the quantised windows' K groups at their widths
    with the K meta and their V at the window width, plus the query, output
    and scores)."""
    import torch
    from tiered_kv_cache_decode_gb300 import binding, synth
    B, Hq, Hkv, w, L0, d, seed = wl["B"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"], 128, 0
    W0 = L0 // w
    kc = binding.TieredCache(B, NL, Hq, Hkv, w, L0, budget_frac=wl["beta"], fp_share=wl["rho"], max_ledger_bits=8,
                             fp_capacity=W0, ledger_capacity=W0)
    kc.set_launch_overlap(True)
    kc.set_cooperative_launch(False)   # the decodes run alone on the GPU
    zeros = torch.zeros(B, W0, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_w = t_r = 0.0
    for l in range(NL):
        k, v = synth.kv_tokens(seed, l, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
        kc.prefill(l, k, v, tiers=zeros)
        q_obs = torch.stack([synth.queries(seed, l, 1000 + i, B, Hq, d, device=dev) for i in range(64)], dim=1)
        sc = synth.zipf_scores(seed + 500, l, B, W0, device=dev)
        wts = kc.k_channel_weights(l, q_obs, k)
        if l == 0:
            # the weights kernel alone: a CUDA graph of repeated calls (the call only
            # reads the cache), timed after a warm-up replay
            s_w, g_w = torch.cuda.Stream(device=dev), torch.cuda.CUDAGraph()
            torch.cuda.synchronize()
            with torch.cuda.stream(s_w):
                with torch.cuda.graph(g_w, stream=s_w):
                    for _ in range(8):
                        kc.k_channel_weights(l, q_obs, k, stream=s_w)
                g_w.replay()
                e0.record(s_w)
                for _ in range(4):
                    g_w.replay()
                e1.record(s_w)
            torch.cuda.synchronize()
            t_w = e0.elapsed_time(e1) * 1e3 / 32
            del g_w
        torch.cuda.synchronize()
        e0.record()
        kc.route_rd_kv(l, wts, scores_override=sc)
        e1.record()
        torch.cuda.synchronize()
        t_r += e0.elapsed_time(e1) * 1e3
        del k, v, q_obs
    q = [synth.queries(seed, l, 0, B, Hq, d, device=dev) for l in range(NL)]
    xo = torch.empty(NL, B, Hq, d, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    g_dec = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_dec, stream=stream):
            for l in range(NL):
                kc.decode(l, q[l], out=xo[l], want_mass=False, accumulate=True, stream=stream)
        for _ in range(3):
            g_dec.replay()
        e0.record(stream)
        for _ in range(reps):
            g_dec.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us_dec = e0.elapsed_time(e1) * 1e3 / (reps * NL)
    nbytes, hist = 0, {b: 0 for b in (0, 2, 4, 8)}
    n_fp = n_q = 0
    for l in range(NL):
        tiers = kc.tables(l)[0]
        kgw = kc.k_group_bits(l)
        for b in range(B):
            kbytes = sum(4 * int(x) + 4 for x in kgw[b].reshape(-1))   # per token, all KV heads
            for x in kgw[b].reshape(-1):
                hist[int(x)] += 1
            for t in tiers[b].tolist():
                if t == 0:
                    nbytes += w * Hkv * d * 4
                    n_fp += 1
                elif t in (1, 3, 4):
                    vb = {1: 2, 3: 4, 4: 8}[t]
                    nbytes += w * (kbytes + Hkv * (d * vb // 8 + 16))
                    n_q += 1
    nbytes = nbytes / NL + B * (Hq * d * 2 + Hq * d * 4 + Hkv * W0 * 8)
    st = kc.status()
    assert st == 0, f"device status {st}: {kc.last_error()}"
    kbytes_w = B * L0 * Hkv * d * 2 + B * 64 * Hq * d * 2   # keys and observed queries read
    return {"layers": NL, "weights_us_per_layer": round(t_w, 2), "weights_gbs": round(kbytes_w / (t_w * 1e-6) / 1e9, 1),
            "route_us_per_layer": round(t_r / NL, 2),
            "k_group_widths_0_2_4_8": [hist[b] for b in (0, 2, 4, 8)],
            "windows_fp_quantised_per_sequence_mean": [round(n_fp / (NL * B), 2), round(n_q / (NL * B), 2)],
            "decode_us_per_launch": round(us_dec, 3), "decode_bytes_per_launch": int(nbytes),
            "decode_gbs": round(nbytes / (us_dec * 1e-6) / 1e9, 2),
            "decode_frac_of_peak": round(nbytes / (us_dec * 1e-6) / 1e9 / peak, 4)}


def measure_per_config(reps, dev, peak, which="all"):
    """The decode kernel on every other workload: the Llama-3.1-8B-shaped batch
    8 at 32K and 5 %, the Qwen2.5-7B-shaped batch 16 at 16K and 10 %, and the 27
    Mistral-7B-shaped sweep points (batch 4; 8K / 32K / 128K tokens, windows of
    32 / 64 / 128, budgets of 5 / 10 / 20 %). Each runs as many layers as make
    its tiered cache at least three times the 129 MB L2 (at most its model's
    layer count), routed on seeded Zipf scores; one CUDA graph decodes every
    layer once, timed over `reps` replays. Then, at each sweep context (64-token
    windows, 10 %), routing events on a fresh two-layer cache starting in full
    precision time the quantise path (first quantisations) and the promote
    path (promotions), with the bytes of the window rows they move."""
    import torch
    from tiered_kv_cache_decode_gb300 import binding, synth
    names = [n for n in all_workloads() if n != WORKLOAD]
    if which != "all":
        names = [n for n in names if n in which.split(",")]
    out = {}
    d, seed = 128, 0
    for name in names:
        wl = workload(name)
        B, Hq, Hkv, w, L0 = wl["B"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"]
        W0 = -(-L0 // w)
        per_layer = TierTracker(wl, L0).decode_bytes()
        NL = int(min(wl["layers"], max(2, math.ceil(3 * 129e6 / per_layer))))
        cache = binding.TieredCache(B, NL, Hq, Hkv, w, L0, budget_frac=wl["beta"], fp_share=wl["rho"])
        cache.set_launch_overlap(True)
        cache.set_cooperative_launch(False)   # the decodes run alone on the GPU
        for l in range(NL):
            k, v = synth.kv_tokens(seed, l, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
            cache.prefill(l, k, v, scores=synth.zipf_scores(seed, l, B, W0, device=dev))
            del k, v
        q = [synth.queries(seed, l, 0, B, Hq, d, device=dev) for l in range(NL)]
        xo = torch.empty(NL, B, Hq, d, dtype=torch.float32, device=dev)
        stream = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for l in range(NL):
                    cache.decode(l, q[l], out=xo[l], want_mass=False, accumulate=True, stream=stream)
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        st = cache.status()
        assert st == 0, f"{name}: device status {st}: {cache.last_error()}"
        us = e0.elapsed_time(e1) * 1e3 / (reps * NL)
        tr = TierTracker(wl, L0)
        gbs = per_layer / (us * 1e-6) / 1e9
        out[name] = {"layers_timed": NL, "windows_fp_int2_evicted": [tr.n_fp, tr.n_q, W0 - tr.n_fp - tr.n_q],
                     "us_per_launch": round(us, 3), "bytes_per_launch": int(per_layer),
                     "gbs": round(gbs, 2), "frac_of_peak": round(gbs / peak, 4)}
        del cache, q, xo, g
        torch.cuda.empty_cache()
    # quantise / promote throughput against context (64-token windows, 10 %)
    moves = {}
    for L0 in (8192, 32768, 131072):
        name = f"mistral7b_b4_{L0 // 1024}k_w64_10pct"
        if which != "all" and name not in which.split(","):
            continue
        wl = workload(name)
        B, Hq, Hkv, w = wl["B"], wl["Hq"], wl["Hkv"], wl["w"]
        W0 = L0 // w
        nl = 2
        mc = binding.TieredCache(B, nl, Hq, Hkv, w, L0, budget_frac=wl["beta"], fp_share=wl["rho"],
                                 fp_capacity=W0, ledger_capacity=W0)
        for l in range(nl):
            k, v = synth.kv_tokens(seed, l, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
            mc.prefill(l, k, v, tiers=torch.zeros(B, W0, dtype=torch.uint8, device=dev))
            del k, v
        row = Hkv * w * (512 + 96)
        stream = torch.cuda.Stream(device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        res = {}
        for kind, sd in (("quantise", seed + 500), ("promote", seed + 501)):
            ov = [synth.zipf_scores(sd, l, B, W0, device=dev) for l in range(nl)]
            s0 = mc.stats()
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                e0.record(stream)
                for l in range(nl):
                    mc.route(l, scores_override=ov[l], stream=stream)
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3
            s1 = mc.stats()
            nq = s1["ledger_writes"] - s0["ledger_writes"]
            npr = s1["promotions"] - s0["promotions"]
            res[kind] = {"quantised_per_layer": nq / nl, "promoted_per_layer": npr / nl,
                         "us_per_layer_event": round(us / nl, 2),
                         "gbs": round((nq + npr) * row / (us * 1e-6) / 1e9, 2)}
        st = mc.status()
        assert st == 0, f"{name}: device status {st}: {mc.last_error()}"
        mc.close()
        del mc
        torch.cuda.empty_cache()
        moves[f"{L0 // 1024}k"] = res
    out["mistral7b_b4_w64_10pct_route_moves"] = moves
    return out


def run_native(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import __graft_entry__
    from tiered_kv_cache_decode_gb300 import binding, synth

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = workload()
    B, NL, Hq, Hkv, w, L0 = wl["B"], wl["layers"], wl["Hq"], wl["Hkv"], wl["w"], wl["L"]
    if args.layers:
        NL = args.layers
    d = 128
    K, Wm = args.steps, args.warmup
    total_steps = Wm + 2 * K + 8
    maxc = L0 + total_steps + 64
    seed = 0

    # Start the CPU oracle pool first (spawned workers never touch the GPU).
    cpu = None
    pool_async = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import multiprocessing as mp
        nw = max(1, min(8, (os.cpu_count() or 2) // 2))
        ctx = mp.get_context("spawn")
        cpu_pool = ctx.Pool(nw)
        pool_async = (cpu_pool, nw, cpu_pool.map_async(_oracle_worker, [(l, args.cpu_seconds, 200, WORKLOAD)
                                                                         for l in range(nw)]),
                      time.perf_counter())

    cache = binding.TieredCache(B, NL, Hq, Hkv, w, maxc, budget_frac=wl["beta"], fp_share=wl["rho"])
    # inside the step graph every decode follows the previous layer's decode kernel
    cache.set_launch_overlap(True)
    cache.set_cooperative_launch(False)   # the decodes run alone on the GPU
    W0 = L0 // w
    for layer in range(NL):
        k, v = synth.kv_tokens(seed, layer, B, 0, L0, Hkv, d, wl["outliers"], device=dev)
        sc = synth.zipf_scores(seed, layer, B, W0, device=dev)
        cache.prefill(layer, k, v, scores=sc)
        del k, v
    torch.cuda.synchronize()
    assert cache.status() == 0, cache.last_error()

    # per-step inputs, resident in HBM: [step][layer][q | k | v] bf16
    nq, nkv = B * Hq * d, B * Hkv * d
    per_layer = nq + 2 * nkv
    pool = torch.empty(total_steps, NL, per_layer, dtype=torch.bfloat16, device=dev)
    for layer in range(NL):
        kn, vn = synth.kv_tokens(seed, layer, B, L0, total_steps, Hkv, d, wl["outliers"], device=dev)
        for s in range(total_steps):
            pool[s, layer, :nq] = synth.queries(seed, layer, s, B, Hq, d, device=dev).reshape(-1)
            pool[s, layer, nq:nq + nkv] = kn[:, s].reshape(-1)
            pool[s, layer, nq + nkv:] = vn[:, s].reshape(-1)
    xin = torch.empty(NL, per_layer, dtype=torch.bfloat16, device=dev)
    xout = torch.empty(NL, B, Hq, d, dtype=torch.float32, device=dev)
    qv = [xin[l, :nq].view(B, Hq, d) for l in range(NL)]
    kv_ = [xin[l, nq:nq + nkv].view(B, Hkv, d) for l in range(NL)]
    vv = [xin[l, nq + nkv:].view(B, Hkv, d) for l in range(NL)]

    stream = torch.cuda.Stream(device=dev)
    route_streams = [torch.cuda.Stream(device=dev) for _ in range(8)]
    g_step, g_route, g_decode = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_step, stream=stream):
            for l in range(NL):
                cache.decode_step(l, qv[l], kv_[l], vv[l], out=xout[l], want_mass=False, accumulate=True,
                                  stream=stream)
        # a routing event: the layers are independent, so their routes run
        # side by side on a few streams, forked from and joined back to the step's
        with torch.cuda.graph(g_route, stream=stream):
            fork = torch.cuda.Event()
            fork.record(stream)
            for rs in route_streams:
                rs.wait_event(fork)
            for l in range(NL):
                cache.route(l, stream=route_streams[l % len(route_streams)])
            for rs in route_streams:
                join = torch.cuda.Event()
                join.record(rs)
                stream.wait_event(join)
        with torch.cuda.graph(g_decode, stream=stream):
            for l in range(NL):
                cache.decode(l, qv[l], out=xout[l], want_mass=False, accumulate=True, stream=stream)
    torch.cuda.synchronize()

    tracker = TierTracker(wl, L0)
    gstep = [0]

    def one_step(s_idx, host_in=None, host_out=None):
        if host_in is not None:
            xin.copy_(host_in, non_blocking=True)
        else:
            xin.copy_(pool[s_idx], non_blocking=True)
        g_step.replay()
        tracker.append()
        nbytes = NL * (tracker.decode_bytes() + tracker.append_bytes())
        launches = NL
        gstep[0] += 1
        routed = gstep[0] % ROUTE_EVERY == 0
        if routed:
            g_route.replay()
            tracker.route()
            launches += 3 * NL
        if host_out is not None:
            host_out.copy_(xout, non_blocking=True)
        return nbytes, launches, int(routed)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for s in range(Wm):
            one_step(s)
        barrier()
        clk = sample_clocks()
        # The timed steps last tens of ms, less than one sampling period, so the
        # GPU is kept at the same work while the sampler starts: the decode-only
        # graph (no appends, the context stays put) for about 0.6 s, then the
        # timed steps. Every sample falls under the decode kernel's load.
        t_soak = time.perf_counter() + 0.6
        while time.perf_counter() < t_soak:
            for _ in range(8):
                g_decode.replay()
            stream.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        ev0.record(stream)
        nbytes, launches, route_events = 0, 0, 0
        for s in range(K):
            b_, l_, r_ = one_step(Wm + s)
            nbytes += b_
            launches += l_
            route_events += r_
        ev1.record(stream)
        barrier()
        clocks = finish_clocks(clk, local_rank)
        ms = ev0.elapsed_time(ev1)

        # the dominant kernel alone: decode over all 32 layers, no appends
        dec_bytes = tracker.decode_bytes()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(K):
            g_decode.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        dec_ms = e0.elapsed_time(e1) / (K * NL)

        # end to end: inputs from pinned host memory, outputs back to the host every step
        if args.no_e2e:
            host_pool = None
        else:
            host_pool = pool[Wm + K:Wm + 2 * K].cpu().pin_memory()
        host_out = torch.empty(NL, B, Hq, d, dtype=torch.float32).pin_memory()
        barrier()
        t0 = time.perf_counter()
        e2e_bytes = 0
        for s in range(0 if args.no_e2e else K):
            b_, _, _ = one_step(Wm + K + s, host_in=host_pool[s], host_out=host_out)
            e2e_bytes += b_
            stream.synchronize()
        e2e_s = max(time.perf_counter() - t0, 1e-9)
    torch.cuda.synchronize()
    st = cache.status()
    assert st == 0, f"device status {st}: {cache.last_error()}"
    cache.refresh_lengths()
    diagnostics = None if args.no_diag else measure_diagnostics(cache, wl, NL, pool, nq, nkv, stream, K, dev)
    management = None if args.no_diag else measure_management(cache, wl, NL, g_route, stream, dev)

    ms, e2e_s, tot_bytes, tot_e2e_bytes = combine_ranks(ms, e2e_s, nbytes, e2e_bytes, world, dev)

    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    value = tot_bytes / (ms / 1e3) / 1e9
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": round(ms / K, 5),
        "us_per_layer_step": round(ms / K / NL * 1e3, 4),
        "pct_of_hbm_peak": round(100 * (value / world) / peak, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": dict(run_config(wl, NL, world, route_events),
                       launch="CUDA graphs of decode launches with programmatic dependent launch; "
                              "non-cooperative grids (nothing else runs on the GPU)"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                     "kernel": "decode_kernel (tiered split-K decode + combine + score + append)",
                     "peak_source": peak_kind, "us_per_launch": round(dec_ms * 1e3, 3),
                     "bytes_per_launch": dec_bytes},
        "e2e": None if args.no_e2e else {"value": round(tot_e2e_bytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(NL * per_layer * 2), "d2h_bytes_per_step": int(xout.numel() * 4),
                "ms_per_step": round(e2e_s / K * 1e3, 4)},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if diagnostics is not None:
        diagnostics["future_missed_mass"]["frac_of_peak"] = round(diagnostics["future_missed_mass"]["gbs"] / peak, 4)
        line["diagnostics"] = diagnostics
    if management is not None:
        line["management"] = management
    if not args.no_variants:
        del cache, pool
        torch.cuda.empty_cache()
        legs = set(args.variants.split(","))
        line["variants"] = measure_variants(wl, NL, K, dev, peak) if "all" in legs or "per_head" in legs else {}
        if "all" in legs or "mixed_widths" in legs:
            line["variants"]["mixed_widths"] = measure_mixed_widths(wl, NL, K, dev, peak)
        if "all" in legs or "k_channels" in legs:
            line["variants"]["k_channels"] = measure_k_channels(wl, NL, K, dev, peak)
    if not args.no_per_config:
        line["per_config"] = measure_per_config(K, dev, peak, args.per_config)
    if pool_async is not None:
        cpu_pool, nw, res, t_start = pool_async
        out = res.get()
        cpu_pool.close()
        nb = sum(r[0] for r in out)
        spent = max(r[1] for r in out)
        line["cpu_baseline"] = {"value": round(nb / spent / 1e9, 4), "unit": "GB/s", "cores": nw,
                                "host_cores": os.cpu_count(), "kind": "oracle",
                                # each worker is one single-threaded process: its rate is the one-core figure
                                "one_core_value": round(sum(r[0] / r[1] for r in out if r[1] > 0) / len(out) / 1e9, 4),
                                "sample": f"{nw} layers of the workload, one per single-threaded process, "
                                          f"{sum(r[2] for r in out)} decode steps in total (append + fp64 attention "
                                          f"+ score accumulation) after a 32K-token prefill"}
    return line


# --------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return None
    nw = max(1, min(8, (os.cpu_count() or 2) // 2))
    per_step = max(1, args.steps + args.warmup)
    gbs, spent, steps, wall = oracle_throughput(nw, budget_s=1e9, max_steps=per_step)
    wl = workload()
    sample = (f"{nw} of the {wl['layers']} layers, one per single-threaded process; {per_step} decode steps "
              f"each (append + fp64 attention + score accumulation) after a 32K-token prefill")
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(spent / max(1, per_step) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": run_config(wl, wl["layers"], world),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": nw, "host_cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="run fewer layers of the same per-layer workload (profiling captures)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) leg")
    ap.add_argument("--no-diag", action="store_true", help="skip the routing diagnostics leg")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the per-KV-head and global-routing leg")
    ap.add_argument("--variants", default="all",
                    help="comma-separated variant legs: per_head (with the routers), mixed_widths, k_channels "
                         "(default: all)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the decode measurement on the other workloads")
    ap.add_argument("--per-config", default="all",
                    help="comma-separated workload names for the per-config leg (default: all)")
    ap.add_argument("--workload", default=WORKLOAD, help="headline workload (see --list-workloads)")
    ap.add_argument("--list-workloads", action="store_true")
    args = ap.parse_args()
    if args.list_workloads:
        print("\n".join(all_workloads()))
        return
    if args.workload not in all_workloads():
        ap.error(f"unknown workload {args.workload}")
    globals()["WORKLOAD"] = args.workload
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        line = run_native(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
