"""Benchmark of the collective datapath on one GB300 (emulated ranks).

Default workload (one "step"): the tensor-parallel decode all-reduce — R=8 emulated ranks,
4096 bf16 (8 KiB) per rank, N(0,1) values from seed 2, a pool of 7 input sets, 10,000
back-to-back epochs in one persistent launch with the speculative protocol (dual
buffers, fence-free content-tagged validation of the reduced flag, 200 ns speculation
delay). Metric: microseconds per epoch.

Also measured in the same run and reported as extra keys: the other protocols and checks,
a staggered-start stress run, per-epoch latency percentiles, and every large-payload
configuration (eight collectives at 16, 64 and 256 MiB per rank, the prefill all-reduce
one-shot and two-shot, MoE dispatch and combine) as achieved HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|sweep|prefill|moe|moe_combine|fig15|fused|single]
                    [--max-bytes B] [--collective C --mib M --datapath D] [--protocols P]

Under torchrun each rank runs an independent replica on its own GPU (the emulated
collective needs no inter-GPU exchange); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

R_DECODE, N_DECODE, POOL, EPOCHS = 8, 4096, 7, 10000
FLUSH_BYTES = 256 << 20  # > 129 MB L2


ENGINE_SOURCES = ["engine.cu", "atom.cuh", "engine.cuh", "coll_internal.h", "tma.cuh"]
BULK_SOURCES = ["bulk.cu", "atom.cuh", "engine.cuh", "coll_internal.h", "tma.cuh"]


def sources_sha256(names):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "collective_datapath_copy_gb300", "csrc")
    for n in names:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(kernel, names):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json), only if
    it was taken on the current sources of that kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("sources_sha256") != sources_sha256(names):
        return None
    return d.get("dram_bytes_per_launch")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid):
        self.rows = []
        self.proc = None
        self.uuid = device_uuid

    def __enter__(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.25)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.rows)}


# ------------------------------------------------------------------ our arm

def _decode_inputs(torch, dev):
    rng = synth.seeded_rng(2)
    pool_np = [[synth.normal_bf16(rng, N_DECODE) for _ in range(R_DECODE)] for _ in range(POOL)]
    host = [np.ascontiguousarray(np.stack([pool_np[p][r] for p in range(POOL)])).view(np.int16)
            for r in range(R_DECODE)]
    ins = [torch.from_numpy(h).to(dev) for h in host]
    return pool_np, host, ins


def max_over_ranks(value, dist, device):
    """The slowest replica's time (every rank must call this; dist None = one process)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_flush(torch, dev):
    """L2 flush between timed steps: write a 256 MiB buffer (> L2), then read another
    256 MiB buffer so the dirty lines of the write are written back before the timed step
    starts rather than during it."""
    wbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush():
        wbuf.fill_(1)
        rbuf.max()
    return flush


def _time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before every step."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e))
    return times


def _stats_us(times_ms, per=1):
    """median / min / max of per-step times (ms), divided by `per`, in microseconds."""
    t = sorted(x * 1000.0 / per for x in times_ms)
    return {"us_median": round(t[len(t) // 2], 3), "us_min": round(t[0], 3),
            "us_max": round(t[-1], 3), "steps": len(t)}


def _time_stream(torch, fns, steps, warmup, flush, stream):
    """Per-step CUDA-event times (ms) of the launches `fns` issued back to back (L2 flushed
    before each step, not between the launches of a step)."""
    def run_all():
        for f in fns:
            f()
    return _time_steps(torch, run_all, steps, warmup, flush, stream)


def measure_zero_copy(torch, cdc, nm, in_sets, out_sets, steps, warmup, flush, stream, peak,
                      **cfg):
    """One zero-copy plan, timed two ways, each the median (with min and max) of `steps`
    steps:
    - single: one launch right after an L2 flush (CUDA events around the launch; the time
      includes the launch and the event pair, about 5 us that a one-element kernel timed the
      same way also takes);
    - stream: launches back to back (six, or four when the sets are large), cycling over
      input/output sets that together exceed L2, so every launch reads inputs no recent
      launch left in L2; per-launch time = the step's time / launches (launch overheads
      overlap the previous launch).
    GB/s and the fraction of `peak` are over the plan's minimal bytes (each input byte a
    named output depends on read once, each named output byte written once)."""
    pl = cdc.Plan(nm, zero_copy=1, **cfg)
    runs = [pl.bind(i, o) for i, o in zip(in_sets, out_sets)]
    b = int(pl.info.min_bytes)
    one = _time_steps(torch, runs[0], steps, warmup, flush, stream)
    seq = runs * max(2, 6 // len(runs))
    many = _time_stream(torch, seq, steps, 1, flush, stream)
    st = pl.status()
    if st["code"] != 0:
        raise RuntimeError(f"run failed: {st}")
    kern = "bulk_kernel" if pl.info.bulk_tile_bytes else "zc_kernel"
    pl.free()
    res = {"min_bytes": b, "kernel": kern}
    for key, tt, per in (("single", one, 1), ("stream", many, len(seq))):
        r = _stats_us(tt, per)
        r["gbs"] = round(b / (r["us_median"] * 1e-6) / 1e9, 1)
        r["frac"] = round(r["gbs"] / peak, 4)
        res[key] = r
    res["stream"]["launches_per_step"] = len(seq)
    return res


def _cold_sets(set_bytes):
    """Input/output sets to cycle through in the back-to-back measurement so that no launch
    finds its data in L2: three below L2's size, two up to four times it, one beyond (a
    launch then evicts everything the previous one touched)."""
    return 3 if set_bytes < L2_BYTES else (2 if set_bytes < 4 * L2_BYTES else 1)


LARGE_KINDS = ("allreduce", "reduce_scatter", "allgather", "broadcast", "alltoall",
               "reduce_to_root", "gather", "scatter")
L2_BYTES = 129e6


def large_collectives(torch, cdc, dev, flush, stream, peak, steps, warmup,
                      sizes_mib=(16, 64, 256)):
    """Every collective at every large size per rank: zero-copy datapath, R=8 emulated ranks,
    bf16 uniform[-1,1] (synth.device_uniform_bf16), timed by measure_zero_copy."""
    R = 8
    rows = []
    for mib in sizes_mib:
        n = (mib << 20) // 2
        for kind in LARGE_KINDS:
            nm = getattr(cdc, kind)(R, n, "bf16")
            nsets = _cold_sets(2 * (sum(nm.in_len) + sum(nm.out_len)))
            in_sets = [[synth.device_uniform_bf16(torch, 3000 + 100 * k + r, n, dev)
                        for r in range(R)] for k in range(nsets)]
            out_sets = [[torch.empty(L, dtype=torch.int16, device=dev) for L in nm.out_len]
                        for _ in range(nsets)]
            cfg = {"datapath": "twoshot"} if kind == "allreduce" else {}
            r = measure_zero_copy(torch, cdc, nm, in_sets, out_sets, steps, warmup, flush,
                                  stream, peak, **cfg)
            r.update({"collective": kind + ("-twoshot" if kind == "allreduce" else ""),
                      "mib_per_rank": mib, "sets": nsets})
            rows.append(r)
            del in_sets, out_sets
        torch.cuda.empty_cache()
    return rows


def prefill_allreduce(torch, cdc, dev, flush, stream, peak, steps, warmup):
    """The prefill all-reduce, 8 x 8192 x 4096 bf16 (64 MiB per rank), N(0,1): two-shot
    (reduce once, push to every rank) and one-shot (every rank reduces all eight)."""
    R, n = 8, 8192 * 4096
    nm = cdc.allreduce(R, n, "bf16")
    ns = _cold_sets(2 * 2 * R * n)
    in_sets = [[synth.device_normal_bf16(torch, 4000 + 100 * k + r, n, dev) for r in range(R)]
               for k in range(ns)]
    out_sets = [[torch.empty(n, dtype=torch.int16, device=dev) for _ in range(R)]
                for _ in range(ns)]
    res = {dp: measure_zero_copy(torch, cdc, nm, in_sets, out_sets, steps, warmup, flush,
                                 stream, peak, datapath=dp)
           for dp in ("twoshot", "oneshot")}
    del in_sets, out_sets
    torch.cuda.empty_cache()
    return res


def moe_collectives(torch, cdc, dev, flush, stream, peak, steps, warmup,
                    which=("dispatch", "combine")):
    """MoE dispatch (each token row to every rank hosting one of its top-8 of 256 experts,
    Zipf(1.1) popularity; 8 x 4096 tokens x 7168 bf16) and its reverse, the combine (a sum
    over the destination ranks)."""
    R, T, H, E, k = 8, 4096, 7168, 256, 8
    routing = synth.zipf_topk_routing(5, R, T, E, k, 1.1)
    res = {}
    for name in which:
        nm = (cdc.moe_dispatch if name == "dispatch" else cdc.moe_combine)(routing, E // R, H)
        ns = _cold_sets(2 * (sum(nm.in_len) + sum(nm.out_len)))
        in_sets = [[synth.device_normal_bf16(torch, 5000 + 100 * s_ + r, L, dev)
                    for r, L in enumerate(nm.in_len)] for s_ in range(ns)]
        out_sets = [[torch.empty(L, dtype=torch.int16, device=dev) for L in nm.out_len]
                    for _ in range(ns)]
        res[name] = measure_zero_copy(torch, cdc, nm, in_sets, out_sets, steps, warmup, flush,
                                      stream, peak)
        res[name]["rows_per_rank"] = [int(c) for c in nm.meta["counts"]]
        del in_sets, out_sets
        torch.cuda.empty_cache()
    return res


def large_payloads(torch, cdc, dev, flush, stream, peak, steps, warmup):
    """Every large-payload configuration: the collectives at 16, 64 and 256 MiB per rank,
    the prefill all-reduce and MoE dispatch / combine."""
    a = (torch, cdc, dev, flush, stream, peak, steps, warmup)
    return {"method": "zero-copy datapath, R=8 emulated ranks, bf16; 'single' = one launch "
                      "right after an L2 flush, 'stream' = launches back to back over input "
                      "sets that together exceed L2; median (min, max) of the steps; GB/s "
                      "over the minimal bytes",
            "collectives": large_collectives(*a), "prefill_allreduce_64MiB": prefill_allreduce(*a),
            "moe": moe_collectives(*a)}


def large_rooflines(large, peak, peak_kind):
    """Roofline records of the two zero-copy kernels at full size: the bulk (TMA) ring on the
    prefill two-shot all-reduce and the warp kernel on MoE combine (uneven producer counts).
    achieved = minimal bytes per launch / the per-launch time of the back-to-back ('stream')
    measurement; traffic = DRAM bytes per launch from the committed ncu summary, if it was
    taken on the kernel's current sources."""
    out = {}
    for what, r in (("prefill all-reduce two-shot, 8 x 64 MiB",
                     large["prefill_allreduce_64MiB"]["twoshot"]),
                    ("MoE combine, 8 x 4096 x 7168", large["moe"]["combine"])):
        st = r["stream"]
        kern = r["kernel"]
        srcs = BULK_SOURCES if kern == "bulk_kernel" else ENGINE_SOURCES
        out[f"{kern}: {what}"] = {
            "bound": "hbm", "achieved": st["gbs"], "peak": peak, "unit": "GB/s",
            "frac": round(st["gbs"] / peak, 4), "peak_kind": f"of {peak_kind}",
            "traffic": recorded_traffic(f"{kern}/{what.split(',')[0]}", srcs),
            "algorithmic_bytes": r["min_bytes"], "us_per_launch": st["us_median"]}
    return out


def run_ours(args, rank, world, dist):
    import torch
    import collective_datapath_copy_gb300 as cdc
    from collective_datapath_copy_gb300.build import build

    build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = make_flush(torch, dev)
    peak, peak_kind = peaks()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None

    nm = cdc.allreduce(R_DECODE, N_DECODE, "bf16")
    pool_np, host_in, ins = _decode_inputs(torch, dev)
    outs = [torch.empty(EPOCHS, N_DECODE, dtype=torch.int16, device=dev) for _ in range(R_DECODE)]
    kw = dict(n_epochs=EPOCHS, in_epoch_stride=2 * N_DECODE, in_pool=POOL,
              out_epoch_stride=2 * N_DECODE)
    plans = {name: cdc.Plan(nm, **cfg) for name, cfg in [
        ("spec", dict(protocol="spec")),
        ("dual", dict(protocol="dual")),
        ("barrier", dict(protocol="barrier")),
        ("spec_stagger", dict(protocol="spec", inject="stagger", inject_seed=2,
                              inject_prob_ppm=100000, inject_max_ns=20000, inject_start_ns=5000)),
        ("spec_fenced", dict(protocol="spec", spec_check="tagged")),
        ("spec_no_delay", dict(protocol="spec", spec_delay_ns=0)),
        ("spec_literal", dict(protocol="spec", spec_check="literal")),
        ("spec_twoshot", dict(protocol="spec", datapath="twoshot")),
        ("spec_twoshot_pull", dict(protocol="spec", datapath="twoshot_pull")),
        ("ll", dict(protocol="ll")),
        ("ll_chain", dict(protocol="ll", chain=1)),
        ("spec_chain", dict(protocol="spec", chain=1)),
        ("dual_chain", dict(protocol="dual", chain=1)),
        ("barrier_chain", dict(protocol="barrier", chain=1)),
    ]}

    def step(name):
        return lambda: plans[name].run(ins, outs, **kw)

    # headline: speculative protocol, timed K steps, clocks sampled during the region
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(uuid) as clk:
        t_wall0 = time.perf_counter()
        times = _time_steps(torch, step("spec"), args.steps, args.warmup, flush, stream)
        t_wall = time.perf_counter() - t_wall0
    torch.cuda.synchronize()
    st = plans["spec"].status()
    if st["code"] != 0:
        raise RuntimeError(f"spec run failed: {st}")
    ms = max_over_ranks(sum(times) / len(times), dist, dev)
    us_epoch = ms * 1000.0 / EPOCHS

    # other protocols (same K/W)
    proto = {}
    for name in ("dual", "barrier", "spec_stagger", "spec_fenced", "spec_no_delay", "spec_literal",
                 "spec_twoshot", "spec_twoshot_pull", "ll", "ll_chain", "spec_chain", "dual_chain",
                 "barrier_chain"):
        tt = _time_steps(torch, step(name), max(3, args.steps // 2), 1, flush, stream)
        s2 = plans[name].status()
        if s2["code"] != 0:
            raise RuntimeError(f"{name} failed: {s2}")
        proto[name] = _stats_us(tt, EPOCHS)
        proto[name]["us_per_epoch"] = proto[name]["us_median"]
        if name.startswith("spec"):
            proto[name]["retries_per_check"] = (s2["spec_retries"] / s2["spec_checks"]
                                                if s2["spec_checks"] else 0.0)
    proto["spec"] = dict(_stats_us(times, EPOCHS), us_per_epoch=round(us_epoch, 4),
                         retries_per_check=(st["spec_retries"] / st["spec_checks"]
                                            if st["spec_checks"] else 0.0))

    # per-epoch latency percentiles from %globaltimer stamps (spec)
    sp = cdc.Plan(nm, protocol="spec", record_stamps=1, stamp_capacity=EPOCHS)
    sp.run(ins, outs, **kw)
    sp.run(ins, outs, **kw)
    stamps = sp.stamps(EPOCHS).astype(np.int64)
    d = np.diff(stamps) / 1000.0
    lat = {"p50_us": round(float(np.percentile(d, 50)), 3),
           "p99_us": round(float(np.percentile(d, 99)), 3),
           "p999_us": round(float(np.percentile(d, 99.9)), 3),
           "engine": "the specialised variant of the timed run, with one %globaltimer stamp "
                     "per epoch (first warp)"} if d.size else {}
    sp.free()
    # where an epoch's time goes (first warp): stage+notify, wait/validate, store+rest
    # (four stamps per epoch run the general engine)
    phases = {}
    for name, cfg in [("spec", dict(protocol="spec")), ("dual", dict(protocol="dual")),
                      ("spec_fenced", dict(protocol="spec", spec_check="tagged")),
                      ("ll", dict(protocol="ll"))]:
        pp = cdc.Plan(nm, record_stamps=2, stamp_capacity=EPOCHS, **cfg)
        pp.run(ins, outs, **kw)
        pp.run(ins, outs, **kw)
        st4 = pp.stamps(EPOCHS).astype(np.int64)[1:].reshape(-1, 4)
        pp.free()
        med = lambda x: round(float(np.median(x)) / 1000.0, 3)
        phases[name] = {"stage_notify_us": med(st4[:, 1] - st4[:, 0]),
                        "wait_validate_us": med(st4[:, 2] - st4[:, 1]),
                        "store_rest_us": med(st4[:, 3] - st4[:, 2]),
                        "epoch_us": med(np.diff(st4[:, 0]))}
    # the latency floor: one flag round trip between two blocks (near: blocks 0 and 1;
    # far: block 0 and the last block of an SM-count grid)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    rtt = {}
    for tag, peer in (("near", 1), ("far", nsm - 1)):
        ns, sa, sb = cdc.probe_flag_rtt(peer, 20000)
        rtt[tag] = {"rtt_ns": round(ns, 1), "sm": [sa, sb]}

    # end to end through the C ABI with host buffers: H2D of the step's inputs (pinned),
    # the run, D2H of every epoch's outputs. The epochs run in chunks whose first epoch is a
    # multiple of the pool size (so every epoch reads the same pool entry as in one run);
    # each chunk's outputs go to the host on a second stream while the next chunk runs, and
    # the step ends when the last copy has landed.
    host_pinned_in = [torch.from_numpy(h).pin_memory() for h in host_in]
    host_pinned_out = [torch.empty(EPOCHS, N_DECODE, dtype=torch.int16).pin_memory()
                       for _ in range(R_DECODE)]
    h2d = sum(h.numel() * 2 for h in host_pinned_in)
    d2h = sum(h.numel() * 2 for h in host_pinned_out)
    chunk = POOL * 200
    chunks = [(e0, min(chunk, EPOCHS - e0)) for e0 in range(0, EPOCHS, chunk)]
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_step():
        for r in range(R_DECODE):
            ins[r].copy_(host_pinned_in[r], non_blocking=True)
        for e0, n in chunks:
            plans["spec"].run(ins, [o[e0:e0 + n] for o in outs], n_epochs=n,
                              in_epoch_stride=2 * N_DECODE, in_pool=POOL,
                              out_epoch_stride=2 * N_DECODE, stream=stream)
            ready = torch.cuda.Event()
            ready.record(stream)
            copy_stream.wait_event(ready)
            with torch.cuda.stream(copy_stream):
                for r in range(R_DECODE):
                    host_pinned_out[r][e0:e0 + n].copy_(outs[r][e0:e0 + n], non_blocking=True)
        stream.wait_stream(copy_stream)

    te = _time_steps(torch, e2e_step, max(3, args.steps // 2), 2, flush, stream)
    e2e_us = sum(te) / len(te) * 1000 / EPOCHS
    # the copies landed: check the last step's outputs on the host against the device
    torch.cuda.synchronize()
    e2e_exact = all(torch.equal(host_pinned_out[r], outs[r].cpu()) for r in range(R_DECODE))
    # the host link's rate for these copies alone (one rank's outputs, device to pinned host)
    copy_ms = _time_steps(torch, lambda: host_pinned_out[0].copy_(outs[0], non_blocking=True),
                          3, 1, flush, stream)
    d2h_gbs = outs[0].numel() * 2 / (sorted(copy_ms)[1] * 1e-3) / 1e9

    # the smallest configuration: all-reduce of 2 x 1024 fp32, barrier protocol, one epoch per
    # launch; median of 1000 launches, each timed with CUDA events
    s_rng = synth.seeded_rng(1)
    s_in = [torch.from_numpy(synth.uniform_f32(s_rng, 1024)).to(dev) for _ in range(2)]
    s_out = [torch.empty(1024, device=dev) for _ in range(2)]
    s_plan = cdc.Plan(cdc.allreduce(2, 1024, "f32"), protocol="barrier")
    for _ in range(20):
        s_plan.run(s_in, s_out)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(1000)]
    for a_, b_ in ev:
        a_.record(stream)
        s_plan.run(s_in, s_out, stream=stream)
        b_.record(stream)
    torch.cuda.synchronize()
    assert s_plan.status()["code"] == 0
    small_us = sorted(a_.elapsed_time(b_) for a_, b_ in ev)[500] * 1000
    s_plan.free()

    # large payloads: every collective at 16 / 64 / 256 MiB per rank, the prefill
    # all-reduce and MoE dispatch / combine (zero-copy datapath)
    large = None
    if not args.skip_large:
        for p in plans.values():
            p.free()
        plans.clear()
        del outs
        torch.cuda.empty_cache()
        large = large_payloads(torch, cdc, dev, flush, stream, peak, max(10, args.steps // 2),
                               args.warmup)

    algo_bytes = 2 * R_DECODE * N_DECODE * 2 * EPOCHS
    achieved = algo_bytes / (ms / 1000) / 1e9
    for p in plans.values():
        p.free()
    clocks = clk.summary()
    res = {
        "metric": "us per small All-Reduce epoch (TP decode, 8 emulated ranks x 8 KiB bf16)",
        "value": round(us_epoch, 4),
        "unit": "us/epoch",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, pool of 7 input sets)",
        "config": {"workload": "TP decode all-reduce: R=8 emulated ranks x 4096 bf16 per rank, "
                               "10000 epochs per step in one persistent launch, speculative "
                               "protocol (dual buffers, fence-free content-tagged validation, "
                               "adaptive speculation window from 200 ns), oneshot",
                   "ranks": R_DECODE, "elems_per_rank": N_DECODE, "epochs_per_step": EPOCHS,
                   "input_pool": POOL, "protocol": "spec", "l2": "flushed before every timed "
                   "step (256 MiB written, then another 256 MiB read)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 5),
                     "traffic": recorded_traffic("engine_kernel", ENGINE_SOURCES),
                     "peak_kind": f"of {peak_kind}",
                     "note": "latency-bound: 128 KiB of algorithmic bytes per epoch"},
        "value_stats": dict(_stats_us(times, EPOCHS), note="per-step spread of the timed steps "
                            "(value = their total / (steps x epochs))"),
        "latency": lat,
        "phases": phases,
        "flag_round_trip": rtt,
        "protocols": proto,
        "large_payloads": large,
        "rooflines_large": large_rooflines(large, peak, peak_kind) if large else None,
        "small_allreduce_2x1024_f32": {"median_us": round(small_us, 3), "launches": 1000,
                                       "protocol": "barrier", "epochs_per_launch": 1},
        "e2e": {"value": round(e2e_us, 4), "unit": "us/epoch", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "runs_per_step": len(chunks),
                "overlap": "each run's outputs copied to pinned host memory on a second "
                           "stream while the next run computes",
                "host_copy_matches_device": bool(e2e_exact),
                "step_stats": _stats_us(te, EPOCHS),
                "d2h_copy_gbs": round(d2h_gbs, 1)},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(pool_np, seconds=args.cpu_seconds)
        res["cpu_baseline_all_cores_throughput"] = cpu_baseline_all_cores(
            seconds=args.cpu_seconds / 2)
    return res


# ------------------------------------------------------------------ oracle timing

def cpu_baseline(pool_np, seconds=10.0):
    """The oracle, as it stands, on the host: fixed-order all-reduce epochs of the decode
    workload until about `seconds` have passed (a bounded sample of the 10,000 epochs)."""
    from oracle import collectives
    t0 = time.perf_counter()
    n = 0
    while True:
        for r_out in collectives.allreduce(pool_np[n % POOL], "bf16"):
            pass
        n += 1
        if n % 50 == 0 and time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(dt / n * 1e6, 3), "unit": "us/epoch", "cores": 1, "kind": "oracle",
            "sample": f"{n} epochs of the 8 x 4096 bf16 all-reduce (numpy, one thread)"}


def _oracle_worker(seconds):
    """One host process of the all-cores oracle timing: the same oracle loop as above."""
    from oracle import collectives
    rng = synth.seeded_rng(2)
    pool_np = [[synth.normal_bf16(rng, N_DECODE) for _ in range(R_DECODE)] for _ in range(POOL)]
    collectives.allreduce(pool_np[0], "bf16")  # warm
    t0 = time.perf_counter()
    n = 0
    while True:
        collectives.allreduce(pool_np[n % POOL], "bf16")
        n += 1
        if n % 20 == 0 and time.perf_counter() - t0 > seconds:
            break
    return n, time.perf_counter() - t0


def cpu_baseline_all_cores(seconds=5.0):
    """The same oracle run as independent epochs in one spawned process per allowed host
    core (the oracle is single-threaded numpy): the host's aggregate rate of independent
    epochs, not the latency of one epoch (that stays the single-thread figure)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    env_keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
    os.environ["OMP_NUM_THREADS"] = os.environ["OPENBLAS_NUM_THREADS"] = "1"
    try:
        with mp.get_context("spawn").Pool(cores) as p:
            res = p.map(_oracle_worker, [seconds] * cores)
    finally:
        for k, v in env_keep.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    total = sum(n for n, _ in res)
    window = max(dt for _, dt in res)
    return {"value": round(window / total * 1e6, 3), "unit": "us/epoch", "cores": cores,
            "kind": "oracle",
            "sample": f"{total} independent epochs of the 8 x 4096 bf16 all-reduce in {cores} "
                      f"processes (numpy, one thread each), {window:.1f} s: aggregate "
                      f"throughput, not one epoch's latency"}


def cpu_oracle_collectives(m_bytes=4 << 20, seconds=0.5, R=8):
    """The oracle timed on the host for the sweep's collectives: each collective of M bytes
    of bf16 per rank (a bounded sample of the sweep's sizes) repeated for about `seconds`,
    reported in GB/s over the same minimal bytes as the GPU rows (one thread, numpy)."""
    import collective_datapath_copy_gb300 as cdc
    from oracle import collectives
    n = m_bytes // 2
    rng = synth.seeded_rng(3)
    xs = [synth.uniform_bf16(rng, n) for _ in range(R)]
    calls = {"allreduce": lambda: collectives.allreduce(xs, "bf16"),
             "reduce_scatter": lambda: collectives.reduce_scatter(xs, "bf16"),
             "allgather": lambda: collectives.allgather(xs),
             "broadcast": lambda: collectives.broadcast(xs, 0),
             "alltoall": lambda: collectives.alltoall(xs),
             "reduce_to_root": lambda: collectives.reduce_to_root(xs, "bf16", 0),
             "gather": lambda: collectives.gather(xs, 0),
             "scatter": lambda: collectives.scatter(xs, 0)}
    rows = []
    for kind, fn in calls.items():
        min_bytes = int(cdc.validate(getattr(cdc, kind)(R, n, "bf16"), zero_copy=1).min_bytes)
        fn()
        t0 = time.perf_counter()
        reps = 0
        while True:
            fn()
            reps += 1
            if time.perf_counter() - t0 > seconds:
                break
        dt = (time.perf_counter() - t0) / reps
        rows.append({"collective": kind, "bytes_per_rank": m_bytes,
                     "gbs": round(min_bytes / dt / 1e9, 3), "ms": round(dt * 1e3, 3)})
    return {"kind": "oracle", "cores": 1, "rows": rows,
            "sample": f"each collective at {m_bytes >> 20} MiB per rank, repeated for about "
                      f"{seconds} s (numpy, one thread)"}


def run_reference(args):
    rng = synth.seeded_rng(2)
    pool_np = [[synth.normal_bf16(rng, N_DECODE) for _ in range(R_DECODE)] for _ in range(POOL)]
    from oracle import collectives
    per_step = max(20, int(args.ref_epochs))
    for _ in range(args.warmup):
        for e in range(per_step):
            collectives.allreduce(pool_np[e % POOL], "bf16")
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for e in range(per_step):
            collectives.allreduce(pool_np[e % POOL], "bf16")
        times.append(time.perf_counter() - t0)
    us = sum(times) / len(times) / per_step * 1e6
    cb = {"value": round(us, 3), "unit": "us/epoch", "cores": 1, "kind": "oracle",
          "sample": f"{per_step} epochs per step of the 8 x 4096 bf16 all-reduce"}
    return {
        "impl": "reference",
        "metric": "us per small All-Reduce epoch (TP decode, 8 emulated ranks x 8 KiB bf16)",
        "value": round(us, 3), "unit": "us/epoch", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sum(times) / len(times) * 1000, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, pool of 7 input sets)",
        "config": {"workload": "TP decode all-reduce: R=8 emulated ranks x 4096 bf16 per rank "
                               "(CPU oracle, bounded sample of the 10000 epochs)",
                   "ranks": R_DECODE, "elems_per_rank": N_DECODE, "input_pool": POOL},
        "cpu_baseline": cb,
        "e2e": {"value": round(us, 3), "unit": "us/epoch", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ other workloads

def _zc_measure(torch, cdc, nm, ins, outs, steps, warmup, flush, stream, graph_reps=50, **cfg):
    """A small zero-copy collective: the per-collective time of `graph_reps` launches
    replayed back to back from a CUDA graph (no host work; the inputs stay in L2), median of
    the steps, in microseconds; and, for context, one launch right after an L2 flush, whose
    CUDA-event time is mostly the launch and the event pair at these sizes."""
    pl = cdc.Plan(nm, zero_copy=1, **cfg)
    tt = _time_steps(torch, lambda: pl.run(ins, outs), steps, warmup, flush, stream)
    st = pl.status()
    if st["code"] != 0:
        raise RuntimeError(f"run failed: {st}")
    r = {"min_bytes": int(pl.info.min_bytes), "tiles": int(pl.info.n_tiles),
         "single_launch": _stats_us(tt)}
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pl.run(ins, outs)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for _ in range(graph_reps):
            pl.run(ins, outs)
    g.replay()
    torch.cuda.synchronize()
    tg = _time_steps(torch, g.replay, max(3, steps // 2), 1, lambda: None, stream)
    r["graph"] = _stats_us(tg, graph_reps)
    r["graph"]["launches_per_replay"] = graph_reps
    del g
    pl.free()
    return r


def run_workload(args):
    """Non-default workloads: the layout-named sweep, the prefill all-reduce, MoE dispatch.
    Each prints its own JSON line (median of K steps, L2 flushed before each)."""
    import torch
    import collective_datapath_copy_gb300 as cdc
    from collective_datapath_copy_gb300.build import build
    build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = make_flush(torch, dev)
    peak, peak_kind = peaks()
    R = 8
    res = {"workload": args.workload, "peak_gbs": peak, "peak_kind": peak_kind}
    # context for the single-launch times: a one-element kernel timed the same way (L2
    # flush, then CUDA events around one launch)
    one = torch.zeros(1, device=dev)
    tfl = _time_steps(torch, lambda: one.add_(1), max(5, args.steps), args.warmup, flush, stream)
    res["one_element_kernel_us"] = _stats_us(tfl)
    if args.workload == "sweep":
        # small sizes (1 KiB .. 4 MiB per rank): a single launch is dominated by its launch,
        # so the per-collective time comes from 50 launches replayed from a CUDA graph;
        # large sizes (16 MiB and up): measure_zero_copy
        sizes = [1 << k for k in range(10, 29, 2)]
        if args.max_bytes:
            sizes = [m for m in sizes if m <= args.max_bytes]
        rows = []
        for m in [m for m in sizes if m <= (4 << 20)]:
            n = m // 2
            ins = [synth.device_uniform_bf16(torch, 3000 + r, n, dev) for r in range(R)]
            for kind in LARGE_KINDS:
                nm = getattr(cdc, kind)(R, n, "bf16")
                outs = [torch.empty(L, dtype=torch.int16, device=dev) for L in nm.out_len]
                cfgs = {"twoshot": dict(datapath="twoshot"), "oneshot": dict(datapath="oneshot")} \
                    if kind == "allreduce" else {"": {}}
                for tag, cfg in cfgs.items():
                    r = _zc_measure(torch, cdc, nm, ins, outs, args.steps, args.warmup, flush,
                                    stream, graph_reps=50, **cfg)
                    r.update({"collective": kind + (f"-{tag}" if tag else ""), "bytes_per_rank": m})
                    rows.append(r)
                del outs
            del ins
            torch.cuda.empty_cache()
        res["small"] = rows
        big = [m >> 20 for m in sizes if m >= (16 << 20)]
        if big:
            res["large"] = large_collectives(torch, cdc, dev, flush, stream, peak, args.steps,
                                             args.warmup, sizes_mib=big)
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_oracle_collectives()
    elif args.workload == "prefill":
        res.update(prefill_allreduce(torch, cdc, dev, flush, stream, peak, args.steps,
                                     args.warmup))
    elif args.workload == "single":
        # one collective at one size (zero-copy datapath, R=8, bf16 uniform[-1,1]): `steps`
        # launches, each right after an L2 flush (a short run to profile one kernel)
        n = (args.mib << 20) // 2
        nm = getattr(cdc, args.collective)(R, n, "bf16")
        ins = [synth.device_uniform_bf16(torch, 3000 + r, n, dev) for r in range(R)]
        outs = [torch.empty(L, dtype=torch.int16, device=dev) for L in nm.out_len]
        cfg = {"datapath": args.datapath} if args.datapath else {}
        if args.warp_kernel:
            cfg["tma_min_bytes"] = (1 << 64) - 1
        if args.tile_bytes:
            cfg["tile_bytes"] = args.tile_bytes
        pl = cdc.Plan(nm, zero_copy=1, **cfg)
        tt = _time_steps(torch, pl.bind(ins, outs), args.steps, args.warmup, flush, stream)
        if pl.status()["code"] != 0:
            raise RuntimeError(f"run failed: {pl.status()}")
        r = _stats_us(tt)
        r["gbs"] = round(pl.info.min_bytes / (r["us_median"] * 1e-6) / 1e9, 1)
        r["frac"] = round(r["gbs"] / peak, 4)
        res.update({"collective": args.collective, "mib_per_rank": args.mib,
                    "datapath": args.datapath or "default", "min_bytes": int(pl.info.min_bytes),
                    "kernel": "bulk_kernel" if pl.info.bulk_tile_bytes else "zc_kernel",
                    "single": r})
        pl.free()
    elif args.workload == "fig15":
        # SiFAR Fig. 15 grid: R = 2/4/8 ranks x 8/16/32 KB payloads, every protocol and
        # datapath, 2000 epochs per launch; microseconds per epoch (median of K launches)
        rows = []
        E = 2000
        for Rr in (2, 4, 8):
            for kb in (8, 16, 32):
                n = kb * 1024 // 2
                ins = [synth.device_normal_bf16(torch, 1500 + 10 * Rr + r, (7, n), dev)
                       for r in range(Rr)]
                outs = [torch.empty(E, n, dtype=torch.int16, device=dev) for _ in range(Rr)]
                nm = cdc.allreduce(Rr, n, "bf16")
                for proto in ("barrier", "dual", "spec", "ll"):
                    for dp in ("oneshot", "twoshot", "twoshot_pull"):
                        if proto == "ll" and dp == "twoshot_pull":
                            continue  # tagged data has no flags to pull on
                        pl = cdc.Plan(nm, protocol=proto, datapath=dp)
                        tt = _time_steps(torch, lambda: pl.run(ins, outs, n_epochs=E,
                                                               in_epoch_stride=2 * n, in_pool=7,
                                                               out_epoch_stride=2 * n),
                                         args.steps, args.warmup, flush, stream)
                        st = pl.status()
                        if st["code"] != 0:
                            raise RuntimeError(f"fig15 {Rr} {kb} {proto} {dp}: {st}")
                        t = sorted(tt)[len(tt) // 2]
                        rows.append({"R": Rr, "kb": kb, "protocol": proto, "datapath": dp,
                                     "us_per_epoch": round(t * 1000 / E, 4),
                                     "retries_per_check": (st["spec_retries"] / st["spec_checks"]
                                                           if st["spec_checks"] else 0.0)})
                        pl.free()
        res["rows"] = rows
    elif args.workload == "fused":
        # producer fusion: each rank's payload is a row-parallel GEMV shard y_r = W_r x_r
        # (8 ranks, 4096 outputs, k = 512 per rank) computed in the stage step, then
        # all-reduced; compared with the all-reduce alone on the same payload size
        Rr, n, k, E, pool = 8, 4096, 512, 2000, 7
        wts = [synth.device_normal_bf16(torch, 900 + r, (k, n), dev) for r in range(Rr)]
        xs = [synth.device_normal_bf16(torch, 910 + r, (pool, k), dev) for r in range(Rr)]
        ys = [synth.device_normal_bf16(torch, 920 + r, (pool, n), dev) for r in range(Rr)]
        outs = [torch.empty(E, n, dtype=torch.int16, device=dev) for _ in range(Rr)]
        nm = cdc.allreduce(Rr, n, "bf16")
        # units: the default 512 bytes (16 pieces per rank, 128 CTAs), and the smallest that
        # spreads the pieces over every SM (8 ranks x 19 units of 432 bytes on 152 SMs)
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        per_rank = max(1, nsm // Rr)
        fill = -(-(2 * n) // per_rank)
        fill = max(64, -(-fill // 16) * 16)
        units = [512] + ([fill] if fill < 512 else [])
        rows = []
        for proto, unit, chain in [(p_, u_, c_) for p_ in args.protocols.split(",")
                                   for u_ in units for c_ in (0, 1)]:
            pl = cdc.Plan(nm, protocol=proto, chain=chain, unit_bytes=unit)
            tf = _time_steps(torch, lambda: pl.run_gemv(wts, xs, k, outs, n_epochs=E,
                                                        x_epoch_stride=2 * k, x_pool=pool,
                                                        out_epoch_stride=2 * n),
                             args.steps, args.warmup, flush, stream)
            ta = _time_steps(torch, lambda: pl.run(ys, outs, n_epochs=E, in_epoch_stride=2 * n,
                                                   in_pool=pool, out_epoch_stride=2 * n),
                             args.steps, args.warmup, flush, stream)
            if pl.status()["code"] != 0:
                raise RuntimeError(f"fused {proto}: {pl.status()}")
            med = lambda t: round(sorted(t)[len(t) // 2] * 1000 / E, 4)
            rows.append({"protocol": proto, "chain": chain, "unit_bytes": unit,
                         "ctas": int(pl.info.n_warps), "fused_us_per_epoch": med(tf),
                         "allreduce_only_us_per_epoch": med(ta)})
            pl.free()
        res["rows"] = rows
        res["gemv"] = {"ranks": Rr, "outputs": n, "k_per_rank": k,
                       "weight_bytes_per_epoch": Rr * n * k * 2}
    elif args.workload in ("moe", "moe_combine"):
        which = ("dispatch",) if args.workload == "moe" else ("combine",)
        res.update(moe_collectives(torch, cdc, dev, flush, stream, peak, args.steps, args.warmup,
                                   which=which))
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-epochs", type=int, default=2000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-large", action="store_true",
                    help="leave out the large-payload collectives of the default run")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "sweep", "prefill", "moe", "moe_combine", "fig15",
                             "fused", "single"])
    ap.add_argument("--max-bytes", type=int, default=0, help="sweep: largest bytes per rank")
    ap.add_argument("--collective", default="allreduce", choices=list(LARGE_KINDS),
                    help="single: the collective")
    ap.add_argument("--mib", type=int, default=16, help="single: MiB per rank")
    ap.add_argument("--datapath", default="", help="single: oneshot or twoshot (sums)")
    ap.add_argument("--warp-kernel", action="store_true",
                    help="single: the warp kernel instead of the bulk (TMA) ring")
    ap.add_argument("--tile-bytes", type=int, default=0,
                    help="single: warp kernel bytes per tile (0: the plan's choice)")
    ap.add_argument("--protocols", default="barrier,dual,spec",
                    help="fused: protocols to run, comma-separated")
    ap.add_argument("--print-sources-sha", action="store_true",
                    help="print the sha256 of the engine kernel's sources and exit")
    args = ap.parse_args()
    if args.print_sources_sha:
        print(sources_sha256(ENGINE_SOURCES))
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if args.workload != "decode":
        if rank == 0:
            print(json.dumps(run_workload(args)), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    res = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
