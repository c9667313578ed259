"""Benchmark of the DSpark per-round hot path on one GB300.

A step is one whole round -- Markov draft of gamma positions, confidence head,
prefix scheduler, rejection-sampling verification -- over one batch of the
synthetic workload (default: batch-128 engine point, B=128, gamma=16,
V=151936).  The metric is verified draft tokens per second: the sum over
requests of the scheduled verify lengths l_r, per round, divided by the round
time.  T is an input of the round, so in the headline round the draft takes
the softmax statistics of the target rows the accept chains reach while it
runs, testing each position as its inputs come out and skipping the rows past
a known rejection (DSPARK_CHAIN_TARGET_STATS), and verification decides on
them.  The same round verifying along each request's accept chain after the
draft (dspark_round's default), with the draft taking every row j < gamma
(DSPARK_EARLY_TARGET_STATS) and with verification taking every row j < l_r
first (DSPARK_ALL_ROW_STATS) are reported beside it, with the other
workloads, a truncating schedule and a CUDA-graph replay of the round.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                        [--impl gb300|reference] [--no-cpu-baseline] [--no-e2e]
                        [--no-workloads] [--form chain|early|all|lazy]
        python bench.py --profile-draft [--workload NAME] [--form lazy] [--plain-draft]   (the first stage alone)
        python bench.py --profile-label [--workload NAME]   (the acceptance labels alone)
        python bench.py --profile-round [--workload NAME] [--form F]   (whole rounds, for launch lists)

Prints one JSON line.  With N > 1 (torchrun) each rank runs an independent
replica of the workload (the path shards over requests with no exchange), the
timing is the max over ranks and `value` counts all ranks' tokens.
"""
import argparse
import hashlib
import json
import os
import subprocess
import tempfile
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/s (B=128,γ=16,V=151936) on 1 GB300; % HBM roofline"
UNIT = "tokens/s"

# Forms of a round, by where verification gets the softmax statistics of the
# target rows its accept tests use:
#   chain  verification reads only the rows the accept tests reach (row j of a
#          request once its positions 1..j were accepted): dspark_round's default
#   early  the draft takes the rows j < gamma while it runs (T given at draft
#          time; DSPARK_EARLY_TARGET_STATS)
#   all    verification takes every row j < l_r first (DSPARK_ALL_ROW_STATS)
#   lazy   the draft takes only the rows the accept chains reach, running the
#          accept tests itself as their inputs come out (T given at draft
#          time; DSPARK_CHAIN_TARGET_STATS)
FORMS = {"chain": "verification along the accept chains",
         "early": "target-row statistics taken by the draft",
         "all": "verification's pass over every row j < l_r",
         "lazy": "target-row statistics of the rows the accept chains reach, taken by the draft"}
DRAFT_T_FORMS = ("early", "lazy")   # forms whose draft takes T along


def form_flags(form):
    """Keyword arguments of ds.round for a form."""
    return dict(early_stats=form == "early", all_row_stats=form == "all", chain_stats=form == "lazy")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="batch128")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the records of the other workloads")
    ap.add_argument("--soak", type=float, default=0.5,
                    help="seconds of untimed rounds just before the timed ones (clock samples under load)")
    ap.add_argument("--profile-draft", action="store_true",
                    help="run only the Markov draft of the workload a few times (small ncu captures)")
    ap.add_argument("--plain-draft", action="store_true",
                    help="with --profile-draft: the draft without the target-row statistics")
    ap.add_argument("--profile-label", action="store_true",
                    help="the acceptance labels alone, 4 calls on a draft's statistics (for ncu)")
    ap.add_argument("--profile-round", action="store_true",
                    help="run a few whole rounds of the workload (ncu launch lists and kernel captures)")
    ap.add_argument("--form", default="lazy", choices=list(FORMS),
                    help="the headline round's form (and --profile-round's): where the target rows' "
                         "statistics come from")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes of one round (each input byte counted once)
# ---------------------------------------------------------------------------
def t_rows(form, B, G, ell_sum, n_acc, n_full):
    """Target rows one round reads once (a rejecting request's row k* - 1 is
    counted here; the residual's second read of it is in round_bytes):
    chain, lazy -- rows 0..n_r of every request, n_r + 1 each (the row of the
    rejected position, or the bonus row after a whole accept); early -- every
    row j < gamma, and the bonus rows; all -- every row j < l_r, and the bonus
    rows."""
    if form in ("chain", "lazy"):
        return n_acc + B
    if form == "early":
        return B * G + n_full
    return ell_sum + n_full


def round_bytes(w, rows, n_reject):
    """Algorithmic bytes of one round that reads `rows` target rows once and
    has n_reject rejecting requests (each re-reads its U and T rows at k*)."""
    sw = 2 if w.wdtype == torch.bfloat16 else 4
    B, G, V, r, H = w.B, w.gamma, w.V, w.r, w.H
    return (4 * B * G * V                 # U
            + 4 * V * rows                # target rows read once
            + sw * r * V                  # W2 once
            + sw * B * G * r              # W1 gathers
            + sw * B * G * H              # h
            + 4 * (H + r)                 # w
            + 8 * V * n_reject            # residual U and T rows
            + 16 * B * G + 8 * B)         # outputs


def draft_bytes_per_launch(w):
    """Algorithmic bytes of one draft call (all gamma positions): U once, W2
    once, the gamma W1 row gathers, x/p/lse out."""
    sw = 2 if w.wdtype == torch.bfloat16 else 4
    return 4 * w.B * w.gamma * w.V + sw * w.r * w.V + sw * w.B * w.gamma * w.r + 12 * w.B * w.gamma


def fused_draft_bytes_per_launch(w):
    """The draft call that also takes the statistics of the target rows
    j < gamma along (T_early): the draft's bytes plus those rows once."""
    return draft_bytes_per_launch(w) + 4 * w.B * w.gamma * w.V


def stage_bytes_per_launch(w, early=True, rows=None):
    """The first stage of a round (dspark_draft_schedule: draft, confidences,
    schedule): the draft's bytes, the target rows it takes along once (every
    row j < gamma when early; `rows` of them when given, the rows j < gamma
    the accept chains reach), the hidden states h and the head's w once, and
    c and ell out."""
    sw = 2 if w.wdtype == torch.bfloat16 else 4
    b = draft_bytes_per_launch(w) + sw * w.B * w.gamma * w.H + 4 * (w.H + w.r) + 4 * w.B * w.gamma + 4 * w.B
    if rows is not None:
        return b + 4 * w.V * rows
    return b + (4 * w.B * w.gamma * w.V if early else 0)


def stage_bytes_of(w, r, form):
    """The first stage's algorithmic bytes in a RoundTimer result's form
    (lazy: the rows j < gamma of the chains, n_r + 1 per rejecting request
    and gamma per whole accept)."""
    if form == "lazy":
        return stage_bytes_per_launch(w, rows=(r["n_acc"] + r["n_rej"]) / r["steps"])
    return stage_bytes_per_launch(w, form == "early")


def kernels_per_round(w, form="chain"):
    """Launches of this library's kernels in one round (cudaMemsetAsync not
    counted).  First stage: on the tensor-core path (bf16, r = 256,
    V >= 192) one persistent kernel, which also finishes x, p, lse and the
    confidences after a last grid barrier and runs the schedule in its last
    CTA; else a CUDA-core step and finalize per position (with early
    statistics a prep and a row-statistics kernel follow), the confidence
    and the schedule kernels.  Verify: the accept tests (verify_chain; or
    verify_decide, after prep and row statistics for the full row pass),
    bonus race, residual (the draft kernel in residual mode, whose last CTA
    and the bonus race's write the tokens; or its CUDA-core form and then the
    residual finalize)."""
    tc = w.wdtype == torch.bfloat16 and w.r == 256 and w.V >= 192
    stage = 1 if tc else 2 * w.gamma + (2 if form in DRAFT_T_FORMS else 0) + 2
    verify = (3 if tc else 4) + (2 if form == "all" else 0)
    return stage + verify


# Source files of a profiled kernel: a committed ncu figure counts only while
# they are unchanged since the capture.  The figure itself is a small JSON
# record beside the prose summary in profiles/.
DRAFT_SOURCES = ["draft_tc.cu", "tc_common.cuh", "common.cuh", "conf.cuh", "sched.cuh"]
DRAFT_PROFILE = os.path.join(ROOT, "profiles", "draft_step_tc_batch128.json")
LABEL_SOURCES = ["label_tc.cu", "tc_common.cuh", "common.cuh"]
LABEL_PROFILE = os.path.join(ROOT, "profiles", "label_tc_batch128.json")


def source_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "speculative_decoding_02_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def draft_source_hash():
    return source_hash(DRAFT_SOURCES)


def profile_records(path):
    """The committed ncu records of a file (one record or a list of them)."""
    with open(path) as f:
        recs = json.load(f)
    return recs if isinstance(recs, list) else [recs]


def profile_traffic(path, sources, w, **match):
    """DRAM bytes (read + write) of one launch from a committed ncu record, or
    None if it is missing, for another workload or mode, or stale."""
    try:
        for rec in profile_records(path):
            if rec.get("workload") != w.name or rec.get("source_sha256_16") != source_hash(sources):
                continue
            if any(rec.get(k) != v for k, v in match.items()):
                continue
            return int(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def draft_traffic(w, form="early"):
    """DRAM bytes of one first-stage launch of a form from the committed ncu
    record (None if missing, for another workload or mode, or stale): the
    draft alone (chain, all), with every row j < gamma (early), with the rows
    the accept chains reach (lazy)."""
    return profile_traffic(DRAFT_PROFILE, DRAFT_SOURCES, w, early_target_stats=form in DRAFT_T_FORMS,
                           chain_target_stats=True if form == "lazy" else None)


def label_traffic(w):
    """DRAM bytes of one acceptance-label launch from the committed ncu record."""
    return profile_traffic(LABEL_PROFILE, LABEL_SOURCES, w)


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during timing."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"dspark_clocks_{os.getpid()}.csv")

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def oracle_round_sample(w, inp_host, nreq, rnd=0):
    """One oracle round over the first `nreq` requests as a batch of their own.
    Returns (verified draft tokens, seconds, threads)."""
    import oracle
    h = inp_host
    sub = {k: (v[:nreq] if k in ("U", "T", "h", "anchor") else v) for k, v in h.items()}
    t0 = time.perf_counter()
    d = oracle.draft(sub["U"], sub["W1"], sub["W2"], sub["anchor"], w.seed, rnd)
    c = oracle.confidence(sub["h"], sub["W1"], sub["w"], sub["anchor"], d["x"])
    if w.mode == 0:
        ell = np.full(nreq, w.gamma, np.int32)
    else:
        b = np.arange(nreq * (w.gamma + 1) + 1, dtype=np.float64)
        sps = (b / (1.0 + b / w.sps_b0)).astype(np.float32)
        ell = oracle.schedule(c, sps, oracle.MODE_GREEDY)["ell"]
    oracle.verify(sub["T"], sub["U"], sub["W1"], sub["W2"], sub["anchor"], d["x"], ell, w.seed, rnd)
    dt = time.perf_counter() - t0
    return int(ell.sum()), dt, oracle.num_threads()


def host_sample(w, nreq, device):
    from speculative_decoding_02_gb300 import workloads as wl
    wsmall = w
    weights = wl.make_weights(w, device)
    rin = wl.make_round_inputs(w, 0, device)
    d = {k: wl.to_numpy(v) for k, v in weights.items()}
    for k in ("U", "T", "h"):
        d[k] = wl.to_numpy(rin[k][:nreq])
    d["anchor"] = d["anchor"][:nreq]
    del rin
    return wsmall, d


def single_thread_sample(w, hs):
    """The oracle on one core: one round of the first request alone."""
    import oracle
    thr = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        tok, dt, _ = oracle_round_sample(w, hs, 1)
    finally:
        oracle.set_num_threads(thr)
    return {"value": tok / dt, "unit": UNIT, "cores": 1,
            "sample": f"one oracle round over 1 of {w.B} requests (full gamma, V), {dt:.1f} s wall"}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine
    type); never raises."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


def cpu_sample_size(w):
    import oracle
    return max(1, min(w.B, oracle.num_threads()))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from speculative_decoding_02_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    nreq = cpu_sample_size(w)
    _, hs = host_sample(w, nreq, "cpu")
    for i in range(args.warmup):
        oracle_round_sample(w, hs, nreq, rnd=i)
    tot_tok, tot_t, thr = 0, 0.0, 1
    for i in range(args.steps):
        tok, dt, thr = oracle_round_sample(w, hs, nreq, rnd=args.warmup + i)
        tot_tok += tok
        tot_t += dt
    value = tot_tok / tot_t
    sample = f"{nreq} of {w.B} requests per step (full gamma={w.gamma}, V={w.V}), scheduled as their own batch"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, "B": w.B, "gamma": w.gamma, "V": w.V},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Across ranks (one process per GPU; each rank runs its own replica)
# ---------------------------------------------------------------------------
def slowest_rank_ms(ms, device):
    """The timed region's length on the slowest rank (the job's time)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_units(units, device):
    """The units (verified draft tokens) that all ranks processed together."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return int(units)
    t = torch.tensor([int(units)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class RoundTimer:
    """Rounds of one workload through the public entry points that
    dspark_round runs (draft_schedule: draft, confidences and schedule; then
    verify), on the current stream; events around the first stage give its
    duration inside the same timed rounds."""

    def __init__(self, ds, w, inp, dev, form, sps=None, khist=None, ws=None):
        assert form in FORMS, form
        self.ds, self.w, self.inp, self.dev, self.form = ds, w, inp, dev, form
        self.early = form in DRAFT_T_FORMS
        self.sps = inp["sps"] if sps is None else sps
        self.khist = khist
        self.ws = ds.workspace(w.B, w.gamma, w.V, dev) if ws is None else ws
        self.out = ds.RoundOutputs(w.B, w.gamma, dev)
        self.stream = torch.cuda.current_stream(dev)

    def step(self, i, d0=None, d1=None, out=None):
        ds, w, inp = self.ds, self.w, self.inp
        if d0 is not None:
            d0.record(self.stream)
        o = ds.draft_schedule(inp["U"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], w.seed, i,
                              sps=self.sps, mode=w.mode, khist=self.khist, out=self.out if out is None else out,
                              ws=self.ws,
                              T_early=inp["T"] if self.early else None, chain_stats=self.form == "lazy")
        if d1 is not None:
            d1.record(self.stream)
        n, _ = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], o.x, o.p, o.lse, o.ell, w.seed, i,
                         self.ws, early_stats=self.early, scratch_from_draft=True, all_row_stats=self.form == "all")
        return o.ell, n

    def run(self, steps, warmup, rnd0=0, barrier=None, soak_s=0.0):
        """Warm-up rounds, an optional untimed soak, then `steps` timed rounds.
        Returns dict(ms (total), draft_ms (mean per call), ell_sum, n_acc, n_rej,
        n_full (requests that accepted every verified position))."""
        for i in range(warmup):
            self.step(rnd0 + i)
        torch.cuda.synchronize()
        st = self.ds.read_status(self.ws)
        if st != self.ds.OK:
            raise RuntimeError(f"{self.w.name}: device status {st} after warm-up")
        if soak_s > 0:
            # keeps the GPU under the same load for a few clock-sampling periods
            t0 = time.perf_counter()
            j = 0
            while time.perf_counter() - t0 < soak_s:
                self.step(rnd0 + warmup + (j % 64))
                j += 1
                if j % 32 == 0:
                    torch.cuda.synchronize()
        # each timed round writes outputs of its own (no copies in the timed region)
        bufs = [self.ds.RoundOutputs(self.w.B, self.w.gamma, self.dev) for _ in range(steps)]
        dstart = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        dend = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        (barrier or torch.cuda.synchronize)()
        e0.record(self.stream)
        outs = [self.step(rnd0 + warmup + i, dstart[i], dend[i], bufs[i]) for i in range(steps)]
        e1.record(self.stream)
        (barrier or torch.cuda.synchronize)()
        st = self.ds.read_status(self.ws)
        if st != self.ds.OK:
            raise RuntimeError(f"{self.w.name}: device status {st} in the timed rounds")
        return dict(ms=e0.elapsed_time(e1),
                    draft_ms=float(np.mean([dstart[i].elapsed_time(dend[i]) for i in range(steps)])),
                    ell_sum=sum(int(e.sum()) for e, _ in outs), n_acc=sum(int(n.sum()) for _, n in outs),
                    n_rej=sum(int((n < e).sum()) for e, n in outs), n_full=sum(int((n == e).sum()) for e, n in outs),
                    steps=steps)


def round_rows(w, r, form):
    """Target rows per round that a RoundTimer result's form reads once."""
    steps = r["steps"]
    return t_rows(form, w.B, w.gamma, r["ell_sum"] / steps, r["n_acc"] / steps, r["n_full"] / steps)


def round_record(w, r, hbm, form):
    """Per-round figures of a RoundTimer result."""
    steps = r["steps"]
    ms = r["ms"] / steps
    per_round = r["ell_sum"] / steps
    rows = round_rows(w, r, form)
    rb = round_bytes(w, rows, r["n_rej"] / steps)
    db = stage_bytes_of(w, r, form)
    return {"form": FORMS[form], "ms": ms, "verified_per_round": per_round,
            "accepted_per_round": r["n_acc"] / steps,
            "verified_tokens_per_s": r["ell_sum"] / (r["ms"] / 1e3),
            "accepted_tokens_per_s": r["n_acc"] / (r["ms"] / 1e3),
            "target_rows_per_round": rows,
            "round_GB": rb / 1e9, "round_hbm_frac": rb / (ms / 1e3) / 1e9 / hbm,
            "draft_ms": r["draft_ms"], "draft_GB": db / 1e9,
            "draft_hbm_frac": db / (r["draft_ms"] / 1e3) / 1e9 / hbm, "early_target_stats": form in DRAFT_T_FORMS}


def gated_round_ms(ds, w, inp, dev, steps):
    """Rounds with the gated recurrent head instead of the Markov head: its
    draft, the confidences, the schedule and verification of the gated draft
    (along the accept chains), K rounds timed with CUDA events."""
    from speculative_decoding_02_gb300 import workloads as wl
    gates = wl.make_gates(w, dev)
    khist = torch.zeros(2, dtype=torch.int32, device=dev) if w.mode == 2 else None
    ws = ds.workspace(w.B, w.gamma, w.V, dev)
    stream = torch.cuda.current_stream(dev)

    def step(i, d0=None, d1=None):
        if d0 is not None:
            d0.record(stream)
        x, p, lse = ds.gated_markov_draft(inp["U"], inp["W1"], inp["W2"], gates["gate_g"], gates["gate_c"],
                                          inp["anchor"], w.seed, i, ws=ws)
        if d1 is not None:
            d1.record(stream)
        c = ds.confidence(inp["h"], inp["W1"], inp["w"], inp["anchor"], x)
        ell, _, _ = ds.schedule(c, inp["sps"], w.mode, i, khist, ws)
        n, _ = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, i, ws,
                         gated=True)
        return ell, n

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    if ds.read_status(ws) != ds.OK:
        raise RuntimeError("device status after the gated-head rounds")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    outs = [step(3 + i, *ev[i]) for i in range(steps)]
    e1.record(stream)
    torch.cuda.synchronize()
    if ds.read_status(ws) != ds.OK:
        raise RuntimeError("device status in the gated-head rounds")
    ms = e0.elapsed_time(e1) / steps
    ell_sum = sum(int(e.sum()) for e, _ in outs)
    return {"ms": ms, "draft_ms": float(np.mean([a.elapsed_time(b) for a, b in ev])),
            "verified_tokens_per_s": ell_sum / (ms * steps / 1e3),
            "accepted_per_round": sum(int(n.sum()) for _, n in outs) / steps,
            "note": "gated recurrent head (gates N(0, 1)); draft, confidence, schedule and verify as separate calls"}


def graph_round_ms(ds, w, inp, dev, steps, form):
    """One round of the given form captured into a CUDA graph with the round
    index in device memory (advanced by the round's last kernel), replayed
    `steps` times."""
    khist = torch.zeros(2, dtype=torch.int32, device=dev) if w.mode == 2 else None
    out = ds.RoundOutputs(w.B, w.gamma, dev)
    n = ds.workspace_size(w.B, w.gamma, w.V)
    buf = torch.zeros(n + 256, dtype=torch.uint8, device=dev)
    ws = buf[(-buf.data_ptr()) % 256:][:n]
    round_dev = torch.zeros(1, dtype=torch.int64, device=dev)

    def call():
        ds.round(inp["U"], inp["T"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], seed=w.seed, rnd=0,
                 sps=inp["sps"], mode=w.mode, khist=khist, out=out, ws=ws, round_dev=round_dev,
                 advance_round=True, **form_flags(form))

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    if ds.read_status(ws) != ds.OK:
        raise RuntimeError("device status after the graph replays")
    ms = e0.elapsed_time(e1) / steps
    ell = int(out.ell.sum())
    del g, buf
    return {"ms": ms, "verified_per_round": ell, "verified_tokens_per_s": ell / (ms / 1e3),
            "rounds_replayed": steps + 4, "round_index_after": int(round_dev[0])}


def other_workload(ds, wl, name, dev, steps, warmup, hbm):
    """Rounds of every form of another workload (serving512: 100 consecutive
    rounds with the top-K schedule taking K from two rounds earlier); the
    inputs are freed afterwards."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, 0, dev)
    rec = {"B": w.B, "gamma": w.gamma, "V": w.V}
    for form in FORMS:
        khist = torch.zeros(2, dtype=torch.int32, device=dev) if w.mode == wl.MODE_TOPK else None
        rt = RoundTimer(ds, w, inp, dev, form, khist=khist)
        k = 100 if name == "serving512" else steps
        r = rt.run(k, warmup)
        rec[form] = round_record(w, r, hbm, form)
    if name == "serving512":
        rec["note"] = "100 consecutive timed rounds; top-K with K from two rounds earlier; inputs fixed, the " \
                      "round index advancing"
    del inp
    torch.cuda.empty_cache()
    return rec


def run_gpu(args):
    import speculative_decoding_02_gb300 as ds
    from speculative_decoding_02_gb300 import build as lib_build
    from speculative_decoding_02_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        lib_build.build()
    if world > 1:
        dist.barrier()
    ds.library()
    hbm, bf16, peak_kind = peaks()

    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w, 0, dev)
    khist = torch.zeros(2, dtype=torch.int32, device=dev) if w.mode == wl.MODE_TOPK else None
    tc = w.wdtype == torch.bfloat16 and w.r == 256 and w.V >= 192
    form = args.form
    early = form in DRAFT_T_FORMS

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # the headline: rounds of the chosen form (default: verification along
    # the accept chains)
    timer = RoundTimer(ds, w, inp, dev, form, khist=khist)
    with Clocks(local) as clk:
        r = timer.run(args.steps, args.warmup, barrier=barrier, soak_s=args.soak)
    ms = slowest_rank_ms(r["ms"], dev)
    ell_sum, n_acc, n_rej = r["ell_sum"], r["n_acc"], r["n_rej"]
    per_round = ell_sum / args.steps
    rows = round_rows(w, r, form)
    value = job_units(ell_sum, dev) / (ms / 1e3)

    # dominant kernel: the round's first stage (one persistent launch: the
    # Markov draft, with the target-row statistics in the early form, the
    # confidences and the schedule), timed inside the timed region
    draft_ms = r["draft_ms"]
    dbytes = stage_bytes_of(w, r, form)
    achieved = dbytes / (draft_ms / 1e3) / 1e9

    extra = {}
    if rank == 0:
        # the same workload in the other forms (same round indices)
        extra["other_forms"] = {f: round_record(w, RoundTimer(ds, w, inp, dev, f, khist=khist).run(
            args.steps, 3), hbm, f) for f in FORMS if f != form and (tc or f not in DRAFT_T_FORMS)}
        # a falling steps-per-second curve, so that the greedy truncates (the
        # scheduler's sorting path; only the verified rows are read)
        if w.mode == wl.MODE_GREEDY:
            b = torch.arange(inp["sps"].numel(), dtype=torch.float64, device=dev)
            sps_fall = (1.0 / (1.0 + b / 256.0)).float()
            rt = RoundTimer(ds, w, inp, dev, form, sps=sps_fall)
            rec = round_record(w, rt.run(args.steps, 3, rnd0=2000), hbm, form)
            rec["sps"] = "1 / (1 + B / 256)"
            extra["truncating_schedule"] = rec
        if tc:
            extra["graph_replay"] = graph_round_ms(ds, w, inp, dev, args.steps, form)
            extra["gated_head"] = gated_round_ms(ds, w, inp, dev, args.steps)

    # the acceptance labels of one round's verified positions (a widening of
    # the path: sum_v min(p_d, p_t) per position), timed on their own; the
    # target rows' statistics are the ones the round's draft took along
    label = None
    ws = timer.ws
    if rank == 0 and tc:
        x, p, lse = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 7, ws=ws,
                                    T_early=inp["T"])
        c = ds.confidence(inp["h"], inp["W1"], inp["w"], inp["anchor"], x)
        ell, _, _ = ds.schedule(c, inp["sps"], w.mode, 7, khist, ws)

        def lab():
            return ds.acceptance_label(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, lse, ell, ws=ws,
                                       stats="early")

        for _ in range(3):
            lab()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream(dev)
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_lab = 5
        l0.record(stream)
        for _ in range(n_lab):
            lab()
        l1.record(stream)
        torch.cuda.synchronize()
        if ds.read_status(ws) != ds.OK:
            raise RuntimeError("device status after the acceptance labels")
        lms = l0.elapsed_time(l1) / n_lab
        npos = int(ell.sum())
        # every position's U and T rows (the kernel streams each once) and W2
        lbytes = 8 * w.V * w.B * w.gamma + (2 if w.wdtype == torch.bfloat16 else 4) * w.r * w.V
        label = {"ms": lms, "positions": npos, "algorithmic_GB": lbytes / 1e9,
                 "achieved_GBs": lbytes / (lms / 1e3) / 1e9, "frac": lbytes / (lms / 1e3) / 1e9 / hbm,
                 "launches_per_call": 2, "target_stats": "taken by the round's draft",
                 "traffic": label_traffic(w)}

    # sequential temperature scaling over held-out samples of this batch size
    # (1024 rounds of the workload's requests), timed on its own
    sts_fit = None
    if rank == 0:
        g = torch.Generator(device=dev)
        g.manual_seed(11)
        N = 1024 * w.B
        zs = torch.randn((N, w.gamma), generator=g, device=dev) * 1.8 + 1.2
        ells = torch.randint(0, w.gamma + 1, (N,), generator=g, device=dev, dtype=torch.int32)
        accs = torch.minimum(torch.randint(0, w.gamma + 1, (N,), generator=g, device=dev, dtype=torch.int32), ells)
        grid = torch.exp(torch.linspace(np.log(0.25), np.log(4.0), 49, device=dev)).float()
        ds.sts_fit(zs, ells, accs, grid)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(3):
            ds.sts_fit(zs, ells, accs, grid)
        s1.record()
        torch.cuda.synchronize()
        sms = s0.elapsed_time(s1) / 3
        # every observed (sample, position) evaluates one sigmoid per grid value
        # plus its prefix product (fp64)
        obs = int(sum(int((ells >= k).sum()) for k in range(1, w.gamma + 1)))
        sts_fit = {"ms": sms, "samples": N, "grid": 49, "observed_positions": obs,
                   "fp64_sigmoids_per_s": obs * (49 + (w.gamma - 1) / 2) / (sms / 1e3)}
        del zs, ells, accs

    # end to end through host buffers: per-round inputs copied in, results out
    e2e = None
    if rank == 0 and not args.no_e2e:
        e2e = run_e2e(w, inp, ds, dev, args, khist, form)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nreq = cpu_sample_size(w)
        _, hs = host_sample(w, nreq, dev)
        tok, dt, thr = oracle_round_sample(w, hs, nreq)
        cpu = {"value": tok / dt, "unit": UNIT, "cores": thr, "kind": "oracle", "cpu_model": cpu_model(),
               "sample": f"one oracle round over {nreq} of {w.B} requests (full gamma, V), "
                         f"{dt:.1f} s wall",
               "single_thread": single_thread_sample(w, hs)}

    # the other workloads (after the headline's inputs are freed)
    if rank == 0 and args.workload == "batch128" and not args.no_workloads:
        del inp
        torch.cuda.empty_cache()
        extra["workloads"] = {n: other_workload(ds, wl, n, dev, args.steps, 3, hbm)
                              for n in ("qwen3_4b", "large_vocab", "serving512")}

    if rank == 0:
        rbytes = round_bytes(w, rows, n_rej / args.steps)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "gamma": w.gamma, "V": w.V, "r": w.r, "H": w.H,
                       "weights": "bf16" if w.wdtype == torch.bfloat16 else "f32",
                       "l2": "inputs larger than L2 (U+T %.2f GB)" % ((4 * w.B * (2 * w.gamma + 1) * w.V) / 1e9),
                       "form": FORMS[form], "early_target_stats": early,
                       "verified_per_round": per_round, "accepted_per_round": n_acc / args.steps,
                       "target_rows_per_round": rows,
                       "round_GB": rbytes / 1e9,
                       "round_hbm_frac": rbytes / (ms / args.steps / 1e3) / 1e9 / hbm,
                       "parallelism": f"replicas x{world}"},
            "roofline": {"kernel": "the round's first stage, one persistent launch (dspark_draft_schedule: "
                                   "draft_step_tc drafting, taking the statistics of the target rows the accept "
                                   "chains reach along, then its fused finalize with the confidences and the "
                                   "schedule)"
                         if form == "lazy" else
                         "the round's first stage, one persistent launch (dspark_draft_schedule: "
                                   "draft_step_tc drafting, taking the target rows' statistics along, then its "
                                   "fused finalize with the confidences and the schedule)"
                         if early else "the round's first stage, one persistent launch (dspark_draft_schedule: "
                                       "draft_step_tc drafting, then its fused finalize with the confidences and "
                                       "the schedule)",
                         "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": draft_traffic(w, form),
                         "peak_kind": peak_kind,
                         "algorithmic_bytes_per_launch": dbytes, "ms_per_launch": draft_ms},
            "clocks": clk.summary(),
            "acceptance_label": label,
            "sts_fit": sts_fit,
            "e2e": e2e,
            "gpu_launches": args.steps * kernels_per_round(w, form),
            "cpu_baseline": cpu,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(w, inp, ds, dev, args, khist, form):
    """Rounds through the public API with the per-round inputs in pinned host
    memory: H2D of U, T, h, anchor and D2H of tokens, counts and lengths are
    inside the timed region.  The inputs are double-buffered on the device and
    the next round's upload runs on a copy stream while the current round
    computes."""
    names = ["U", "T", "h", "anchor"]
    hostb = {k: inp[k].cpu().pin_memory() for k in names}
    devb = [{k: torch.empty_like(inp[k]) for k in names} for _ in range(2)]
    outs = ["x", "ell", "n", "tok"]
    out = ds.RoundOutputs(w.B, w.gamma, dev)
    hosto = {k: torch.empty(getattr(out, k).shape, dtype=getattr(out, k).dtype).pin_memory() for k in outs}
    ws = ds.workspace(w.B, w.gamma, w.V, dev)
    bi = sum(t.numel() * t.element_size() for t in hostb.values())
    bo = sum(t.numel() * t.element_size() for t in hosto.values())
    stream = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    steps = max(3, min(args.steps, 10))
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def upload(slot):
        copy.wait_event(consumed[slot])
        with torch.cuda.stream(copy):
            for k in names:
                devb[slot][k].copy_(hostb[k], non_blocking=True)
            uploaded[slot].record(copy)

    def compute(i, slot):
        stream.wait_event(uploaded[slot])
        b = devb[slot]
        ds.round(b["U"], b["T"], inp["W1"], inp["W2"], b["h"], inp["w"], b["anchor"], seed=w.seed, rnd=i,
                 sps=inp["sps"], mode=w.mode, khist=khist, out=out, ws=ws, **form_flags(form))
        consumed[slot].record(stream)
        for k in outs:
            hosto[k].copy_(getattr(out, k), non_blocking=True)

    for slot in range(2):
        consumed[slot].record(stream)
    upload(0)
    compute(0, 0)
    torch.cuda.synchronize()
    # steady state: each timed step uploads the next round's inputs while it
    # computes this round's (round 0's inputs are uploaded before timing; the
    # last step's upload is for a round outside the timed region)
    upload(1)
    torch.cuda.synchronize()
    ell_sum = 0
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        slot = (i + 1) % 2
        upload((i + 2) % 2)   # the next round's inputs while this one computes
        compute(i + 1, slot)
        stream.synchronize()
        ell_sum += int(hosto["ell"].sum())
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    del hostb, devb
    return {"value": ell_sum / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": steps, "wall_s": time.perf_counter() - t0, "uploads": "double-buffered on a copy stream"}


def run_profile_draft(args):
    """The round's first stage of the workload alone (dspark_draft_schedule:
    draft, confidences, schedule), 4 calls, taking the target rows'
    statistics along unless --plain-draft (for ncu: U, T, h, the weights and
    the anchors are all it holds on the device)."""
    import speculative_decoding_02_gb300 as ds
    from speculative_decoding_02_gb300 import build as lib_build
    from speculative_decoding_02_gb300 import workloads as wl
    dev = torch.device("cuda", 0)
    lib_build.build()
    w = wl.WORKLOADS[args.workload]
    weights = wl.make_weights(w, dev)
    rin = wl.make_round_inputs(w, 0, dev)
    sps = wl.sps_table(w)
    sps = None if sps is None else sps.to(dev)
    khist = torch.zeros(2, dtype=torch.int32, device=dev)
    T = None if args.plain_draft else rin["T"]
    chain = T is not None and args.form == "lazy"
    ws = ds.workspace(w.B, w.gamma, w.V, dev)
    for i in range(4):
        ds.draft_schedule(rin["U"], weights["W1"], weights["W2"], rin["h"], weights["w"], weights["anchor"], w.seed,
                          i, sps=sps, mode=w.mode, khist=khist, ws=ws, T_early=T, chain_stats=chain)
    torch.cuda.synchronize()
    st = ds.read_status(ws)
    rec = {"profile_draft": w.name, "early_target_stats": T is not None, "chain_target_stats": chain, "status": st,
           "source_sha256_16": draft_source_hash()}
    if chain and st == ds.OK:
        # the rows j < gamma the accept chains of the third call (the one a
        # capture with -s 2 -c 1 takes) reach: n_r + 1 per rejecting request,
        # n_r per whole accept (the same round again, then its verification)
        o = ds.draft_schedule(rin["U"], weights["W1"], weights["W2"], rin["h"], weights["w"], weights["anchor"],
                              w.seed, 2, sps=sps, mode=w.mode, khist=torch.zeros(2, dtype=torch.int32, device=dev),
                              ws=ws, T_early=T, chain_stats=True)
        n, _ = ds.verify(rin["T"], rin["U"], weights["W1"], weights["W2"], weights["anchor"], o.x, o.p, o.lse, o.ell,
                         w.seed, 2, ws, early_stats=True, scratch_from_draft=True)
        n, ell = n.cpu(), o.ell.cpu()
        rec["chain_rows"] = int(n.sum()) + int((n < ell).sum())
        rec["algorithmic_bytes_per_launch"] = stage_bytes_per_launch(w, rows=rec["chain_rows"])
        st = ds.read_status(ws)
        rec["status"] = st
    print(json.dumps(rec))
    if st != ds.OK:
        sys.exit(1)


def run_profile_label(args):
    """The acceptance labels of the workload, 4 calls, reading the target
    rows' statistics a draft took along (for ncu: U, T, W1, W2, the anchors
    and the draft's outputs are all it holds on the device)."""
    import speculative_decoding_02_gb300 as ds
    from speculative_decoding_02_gb300 import build as lib_build
    from speculative_decoding_02_gb300 import workloads as wl
    dev = torch.device("cuda", 0)
    lib_build.build()
    w = wl.WORKLOADS[args.workload]
    weights = wl.make_weights(w, dev)
    rin = wl.make_round_inputs(w, 0, dev)
    del rin["h"]
    ws = ds.workspace(w.B, w.gamma, w.V, dev)
    x, _, lse = ds.markov_draft(rin["U"], weights["W1"], weights["W2"], weights["anchor"], w.seed, 0, ws=ws,
                                T_early=rin["T"])
    ell = torch.full((w.B,), w.gamma, dtype=torch.int32, device=dev)
    for _ in range(4):
        ds.acceptance_label(rin["T"], rin["U"], weights["W1"], weights["W2"], weights["anchor"], x, lse, ell, ws=ws,
                            stats="early")
    torch.cuda.synchronize()
    st = ds.read_status(ws)
    print(json.dumps({"profile_label": w.name, "status": st, "source_sha256_16": source_hash(LABEL_SOURCES)}))
    if st != ds.OK:
        sys.exit(1)


def run_profile_round(args):
    """A few whole rounds of the workload through the entry points (the form
    of --form): two warm-up rounds, then args.steps rounds, for ncu launch
    lists and captures of round kernels."""
    import speculative_decoding_02_gb300 as ds
    from speculative_decoding_02_gb300 import build as lib_build
    from speculative_decoding_02_gb300 import workloads as wl
    dev = torch.device("cuda", 0)
    lib_build.build()
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w, 0, dev)
    khist = torch.zeros(2, dtype=torch.int32, device=dev) if w.mode == wl.MODE_TOPK else None
    r = RoundTimer(ds, w, inp, dev, args.form, khist=khist).run(args.steps, 2)
    print(json.dumps({"profile_round": w.name, "form": args.form, "steps": args.steps,
                      "ms_per_round": r["ms"] / args.steps, "kernels_per_round": kernels_per_round(w, args.form)}))


def main():
    args = parse()
    if args.profile_draft:
        run_profile_draft(args)
    elif args.profile_round:
        run_profile_round(args)
    elif args.profile_label:
        run_profile_label(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
